"""Planted mistakes in the CPU oracle must trip at least one pin (CPU only).

Each mutant is the oracle source with one plausible slip (a swapped nibble, a
wrong shift, an inclusive prefix where an exclusive one belongs, a reversed
tie-break, a skipped overwrite ...).  It is compiled into a temporary shared
object and run through the same pin battery as the real oracle; a mutant that
passes every pin would mean the pins cannot tell that mistake apart.
"""
import os

import pytest

from oracle import oracle as O
from tests.oracle_pins import CHECKS

MUTANTS = [
    ("nibble order swapped on encode",
     "out[n + i / 2] |= (uint8_t)(code << (4 * (i % 2)));",
     "out[n + i / 2] |= (uint8_t)(code << (4 * (1 - i % 2)));"),
    ("sign stored at bit 6 of the sm byte",
     "out[i] = (uint8_t)((sign << 7) | mant);",
     "out[i] = (uint8_t)((sign << 6) | mant);"),
    ("escape position not chunk-relative",
     "put_u16(rec + 3 * j, (unsigned)(i % ORC_CHUNK));",
     "put_u16(rec + 3 * j, (unsigned)(i % 65535u));"),
    ("escaped element gets code 15",
     "            code = 0;\n",
     "            code = 15;\n"),
    ("tie-break toward the larger exponent",
     "if (best < 0 || hist[e] > hist[best]) best = e;",
     "if (best < 0 || hist[e] >= hist[best]) best = e;"),
    ("codebook listed in descending order",
     "    for (int e = 0; e < bins; e++)\n        if (taken[e]) cb[k++] = (uint8_t)e;",
     "    for (int e = bins - 1; e >= 0; e--)\n        if (taken[e]) cb[k++] = (uint8_t)e;"),
    ("inclusive header offset",
     "put_u32(hdr + 8 * c, offset);",
     "put_u32(hdr + 8 * c, offset + count);"),
    ("chunk count off by one on exact multiples",
     "uint64_t orc_num_chunks(uint64_t n) { return ceil_div(n, ORC_CHUNK); }",
     "uint64_t orc_num_chunks(uint64_t n) { return n / ORC_CHUNK + 1; }"),
    ("E5M2 field with code on top",
     "unsigned field = code | (((sign << 2) | mant) << 4); /* R1, R8 */",
     "unsigned field = (code << 3) | ((sign << 2) | mant); /* R1, R8 */"),
    ("E5M2 exponent read from the wrong bits",
     "return ((unsigned)x[i] >> 2) & 0x1Fu;",
     "return ((unsigned)x[i] >> 3) & 0x1Fu;"),
    ("BF16 decode puts the sign at bit 14",
     "unsigned v = ((sm >> 7) << 15) | ((unsigned)cb[code] << 7) | (sm & 0x7Fu);",
     "unsigned v = ((sm >> 7) << 14) | ((unsigned)cb[code] << 7) | (sm & 0x7Fu);"),
    ("decode skips the escape overwrite (BF16)",
     "v = (v & 0x807Fu) | (e << 7);",
     "v = v | (e & 0u);"),
    ("decode reads the high nibble first",
     "unsigned code = (in[n + i / 2] >> (4 * (i % 2))) & 0xFu;",
     "unsigned code = (in[n + i / 2] >> (4 * (1 - i % 2))) & 0xFu;"),
    ("validate accepts unsorted positions",
     "if (k > 0 && pos <= get_u16(rec + 3 * (offset + k - 1))) return ORC_CORRUPT;",
     "if (k > 0 && pos == 0xFFFFFu) return ORC_CORRUPT;"),
    ("validate accepts a repeated codebook exponent",
     "if (cb[a] == cb[b]) return 0;",
     "if (cb[a] == cb[b] && a < 0) return 0;"),
    ("histogram drops the last element",
     "for (uint64_t i = 0; i < n; i++) hist[exponent_at(dt, x, i)]++;",
     "for (uint64_t i = 0; i + 1 < n; i++) hist[exponent_at(dt, x, i)]++;"),
    ("E5M2 decode drops the mantissa",
     "y[i] = (uint8_t)(((sm3 >> 2) << 7) | ((unsigned)cb[code] << 2) | (sm3 & 0x3u));",
     "y[i] = (uint8_t)(((sm3 >> 2) << 7) | ((unsigned)cb[code] << 2));"),
    ("Top-8 ablation codes packed 4 bits apart",
     "unsigned bit = 3 * (unsigned)(i % 8);",
     "unsigned bit = 4 * (unsigned)(i % 8);"),
    ("sentinel ablation marks escapes with code 14",
     "                code = 15;",
     "                code = 14;"),
]


@pytest.fixture(scope="module")
def source():
    with open(O.SOURCE) as f:
        return f.read()


@pytest.mark.parametrize("name,old,new", MUTANTS, ids=[m[0] for m in MUTANTS])
def test_mutant_is_caught(tmp_path, source, name, old, new):
    assert source.count(old) == 1, f"mutation site for '{name}' not found exactly once"
    lib = O.compile_source(source.replace(old, new), os.path.join(tmp_path, "mutant.so"))
    mutant = O.Oracle(lib)
    tripped = []
    for check in CHECKS:
        try:
            check(mutant)
        except (AssertionError, RuntimeError, ValueError, IndexError):
            tripped.append(check.__name__)
    assert tripped, f"no pin catches the planted mistake: {name}"
