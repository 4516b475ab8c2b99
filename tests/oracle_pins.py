"""Pins for the CPU oracle: facts fixed by the pages and by arithmetic.

Each ``check_*`` takes an oracle wrapper and raises AssertionError when the
oracle disagrees with a fact that does not come from the oracle itself:

* hand-worked byte streams (tests/golden/*.txt, each with its derivation and
  the section of the SplitZip pages it follows);
* brute force over every BF16 bit pattern and every E5M2 byte, where the
  escape count and stream size have closed forms (each exponent value owns
  exactly 256 BF16 patterns / 8 E5M2 patterns);
* the closed-form stream size N + ceil(N/2) + 3E + 16 + 8C (BF16) and
  7 ceil(N/8) + 3E + 16 + 8C (E5M2);
* escape-count and header invariants counted independently with numpy;
* bitwise round trip (the method is lossless: SplitZip abstract, arXiv
  2605.01708v2);
* rejection of corrupted streams.

``test_oracle_pins.py`` runs every check on the oracle; ``test_oracle_mutants.py``
runs them on oracle builds with a planted mistake and requires that each
mistake trips at least one check.
"""
import numpy as np

from oracle import oracle as O
from tests import _golden as G

CB_MID = np.arange(120, 136, dtype=np.uint8)        # contiguous BF16 codebook
CB_EDGES = np.array(list(range(0, 8)) + list(range(248, 256)), dtype=np.uint8)
CB_E5_MID = np.arange(14, 30, dtype=np.uint8)
CB_E5_EDGES = np.array(list(range(0, 8)) + list(range(24, 32)), dtype=np.uint8)


def _bf16_exponents(x):
    return (x.astype(np.uint32) >> 7) & 0xFF


def _e5_exponents(x):
    return (x.astype(np.uint32) >> 2) & 0x1F


def _roundtrip(orc, dt, cb, x):
    s = orc.encode(dt, cb, x)
    st, y = orc.decode(dt, s, O.Oracle.element_count(dt, x))
    assert st == O.OK, f"decode status {st}"
    assert y.tobytes() == np.ascontiguousarray(x).tobytes(), "round trip is not bitwise"
    return s


def _records(orc, dt, s, n):
    """Split a stream into (cb, [(offset, count)], [(pos, exp)])."""
    dense = orc.dense_bytes(dt, n)
    C = orc.num_chunks(n)
    cb = s[dense:dense + 16]
    h = s[dense + 16:dense + 16 + 8 * C].view(np.uint32).reshape(C, 2) if C else np.zeros((0, 2), np.uint32)
    r = s[dense + 16 + 8 * C:]
    assert r.size % 3 == 0
    r = r.reshape(-1, 3)
    pos = r[:, 0].astype(np.uint32) | (r[:, 1].astype(np.uint32) << 8)
    return cb, h, pos, r[:, 2]


# ---- hand-worked streams ---------------------------------------------------

def check_hand_bf16(orc):
    g = G.load("bf16_hand.txt")
    x = np.array(G.hexwords(g["input"]), dtype=np.uint16)
    cb = np.array(G.ints(g["codebook"]), dtype=np.uint8)
    s = _roundtrip(orc, O.BF16, cb, x)
    want = G.hexbytes(g["sm"]) + G.hexbytes(g["nibbles"]) + bytes(cb) + G.hexbytes(g["headers"]) + G.hexbytes(g["escapes"])
    assert s.tobytes() == want
    assert len(want) == int(g["size"]) == orc.encoded_size(O.BF16, 5, 1)


def check_hand_e5m2(orc):
    g = G.load("e5m2_hand.txt")
    x = np.array(G.hexwords(g["input"]), dtype=np.uint8)
    cb = np.array(G.ints(g["codebook"]), dtype=np.uint8)
    s = _roundtrip(orc, O.E5M2, cb, x)
    want = G.hexbytes(g["packed"]) + bytes(cb) + G.hexbytes(g["headers"]) + G.hexbytes(g["escapes"])
    assert s.tobytes() == want
    assert len(want) == int(g["size"]) == orc.encoded_size(O.E5M2, 5, 1)


def check_two_chunks_bf16(orc):
    g = G.load("bf16_two_chunks.txt")
    n = int(g["n"])
    x = np.full(n, int(g["fill"], 16), dtype=np.uint16)
    for i, v in G.assignments(g["set"]).items():
        x[i] = v
    cb = np.array(G.ints(g["codebook"]), dtype=np.uint8)
    s = _roundtrip(orc, O.BF16, cb, x)
    assert s.size == int(g["size"])
    sm = np.full(n, int(g["sm_fill"], 16), dtype=np.uint8)
    for i, v in G.assignments(g["sm_set"]).items():
        sm[i] = v
    nib = np.full((n + 1) // 2, int(g["nibble_fill"], 16), dtype=np.uint8)
    for i, v in G.assignments(g["nibble_set"]).items():
        nib[i] = v
    want = sm.tobytes() + nib.tobytes() + bytes(cb) + G.hexbytes(g["headers"]) + G.hexbytes(g["escapes"])
    assert s.tobytes() == want


def _sample_with_counts(dt, counts, rng):
    """Elements whose exponent fields have the given counts (random sign/mantissa)."""
    vals = []
    for e, c in counts.items():
        for _ in range(c):
            if dt == O.BF16:
                vals.append((int(rng.integers(0, 2)) << 15) | (e << 7) | int(rng.integers(0, 128)))
            else:
                vals.append((int(rng.integers(0, 2)) << 7) | (e << 2) | int(rng.integers(0, 4)))
    rng.shuffle(vals)
    return np.array(vals, dtype=np.uint16 if dt == O.BF16 else np.uint8)


def check_calibration_hand(orc):
    rng = np.random.default_rng(7)
    for g in G.load("calibration_hand.txt"):
        dt = O.BF16 if g["dtype"] == "bf16" else O.E5M2
        counts = G.assignments(g["counts"], value_base=10)
        want = np.array(G.ints(g["codebook"]), dtype=np.uint8)
        hist = np.zeros(256 if dt == O.BF16 else 32, dtype=np.uint64)
        for e, c in counts.items():
            hist[e] = c
        assert np.array_equal(orc.codebook_from_histogram(dt, hist), want), g["case"]
        x = _sample_with_counts(dt, counts, rng)
        assert np.array_equal(orc.histogram(dt, x), hist), g["case"]
        assert np.array_equal(orc.calibrate(dt, x), want), g["case"]


# ---- brute force -----------------------------------------------------------

def check_bruteforce_bf16(orc):
    x = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    for cb in (CB_MID, CB_EDGES):
        s = _roundtrip(orc, O.BF16, cb, x)
        # 240 exponents lie outside the codebook, 256 patterns each.
        assert orc.count_escapes(O.BF16, cb, x) == 61440
        assert s.size == 282648 == orc.encoded_size(O.BF16, 65536, 61440)
        sm = s[:65536]
        assert np.all(np.bincount(sm, minlength=256) == 256)  # (sign, mantissa) x 256 exponents
        nib = s[65536:65536 + 32768]
        codes = np.stack([nib & 0xF, nib >> 4], axis=1).reshape(-1)
        hist = np.bincount(codes, minlength=16)
        assert hist[0] == 256 + 61440 and np.all(hist[1:] == 256)
        _, h, pos, exp = _records(orc, O.BF16, s, 65536)
        assert h.tolist() == [[0, 61440]]
        assert np.array_equal(pos, np.flatnonzero(~np.isin(_bf16_exponents(x), cb)))
        assert np.array_equal(exp, _bf16_exponents(x)[pos].astype(np.uint8))
        # Codes follow ascending exponent order: code k <-> k-th smallest exponent.
        for k, e in enumerate(np.sort(cb)):
            assert np.all(codes[_bf16_exponents(x) == e] == k)


def check_bruteforce_e5m2(orc):
    x = np.arange(256, dtype=np.uint32).astype(np.uint8)
    for cb in (CB_E5_MID, CB_E5_EDGES):
        s = _roundtrip(orc, O.E5M2, cb, x)
        assert orc.count_escapes(O.E5M2, cb, x) == 128   # 16 exponents x 8 patterns
        assert s.size == 632 == orc.encoded_size(O.E5M2, 256, 128)
        _, h, pos, exp = _records(orc, O.E5M2, s, 256)
        assert h.tolist() == [[0, 128]]
        assert np.array_equal(pos, np.flatnonzero(~np.isin(_e5_exponents(x), cb)))
        assert np.array_equal(exp, _e5_exponents(x)[pos].astype(np.uint8))


# ---- invariants on random data ---------------------------------------------

def _gaussian_bf16(rng, n, scale=1.0):
    v = (rng.standard_normal(n) * scale).astype(np.float32)
    return (v.view(np.uint32) >> 16).astype(np.uint16)   # truncation: any pattern will do


def check_invariants_bf16(orc):
    rng = np.random.default_rng(11)
    n = 3 * 65536 + 4099
    x = _gaussian_bf16(rng, n, scale=np.exp(rng.standard_normal(n)))
    cb = orc.calibrate(O.BF16, x[: n // 3])
    s = _roundtrip(orc, O.BF16, cb, x)
    ex = _bf16_exponents(x)
    esc = ~np.isin(ex, cb)
    E = int(esc.sum())
    assert E > 0 and s.size == n + (n + 1) // 2 + 3 * E + 16 + 8 * 4
    cbs, h, pos, exp = _records(orc, O.BF16, s, n)
    assert np.array_equal(cbs, cb)
    counts = [int(esc[c * 65536:(c + 1) * 65536].sum()) for c in range(4)]
    assert h[:, 1].tolist() == counts
    assert h[:, 0].tolist() == [0, counts[0], counts[0] + counts[1], sum(counts[:3])]
    gidx = np.concatenate([c * 65536 + pos[h[c, 0]:h[c, 0] + h[c, 1]] for c in range(4)])
    assert np.array_equal(gidx, np.flatnonzero(esc))
    assert np.array_equal(exp, ex[gidx].astype(np.uint8))


def check_invariants_e5m2(orc):
    rng = np.random.default_rng(12)
    for n in list(range(1, 18)) + [65535, 65536, 65537, 65543, 2 * 65536 + 5]:
        x = rng.integers(0, 256, n, dtype=np.uint8)
        cb = CB_E5_MID
        s = _roundtrip(orc, O.E5M2, cb, x)
        E = int((~np.isin(_e5_exponents(x), cb)).sum())
        C = -(-n // 65536)
        assert s.size == 7 * (-(-n // 8)) + 3 * E + 16 + 8 * C
        if n % 8:
            # Unused fields of the last group are zero: its top (8 - n%8)*7 bits.
            last = int.from_bytes(s[7 * (n // 8):7 * (n // 8) + 7].tobytes(), "little")
            assert last >> (7 * (n % 8)) == 0


def check_edge_sizes(orc):
    rng = np.random.default_rng(13)
    # n = 0: the stream is the codebook alone.
    s = orc.encode(O.BF16, CB_MID, np.zeros(0, dtype=np.uint16))
    assert s.tobytes() == bytes(CB_MID)
    assert orc.decode(O.BF16, s, 0)[0] == O.OK
    s = orc.encode(O.E5M2, CB_E5_MID, np.zeros(0, dtype=np.uint8))
    assert s.tobytes() == bytes(CB_E5_MID)
    for n in (1, 2, 3, 65535, 65536, 65537, 131073):
        x = _gaussian_bf16(rng, n, scale=1e3)
        s = _roundtrip(orc, O.BF16, CB_MID, x)
        E = orc.count_escapes(O.BF16, CB_MID, x)
        assert s.size == n + (n + 1) // 2 + 3 * E + 16 + 8 * (-(-n // 65536))
        if n % 2:
            assert s[n + n // 2] >> 4 == 0   # unused high nibble of the last byte


def check_all_and_zero_escape(orc):
    rng = np.random.default_rng(14)
    n = 65536 + 1000
    x = _gaussian_bf16(rng, n)
    # Move every exponent outside CB_MID (to 10..109, sign/mantissa kept).
    x_all = ((x & 0x807F) | (rng.integers(10, 110, n).astype(np.uint16) << 7)).astype(np.uint16)
    s = _roundtrip(orc, O.BF16, CB_MID, x_all)
    assert s.size == (9 * n) // 2 + 16 + 8 * 2
    x_none = ((x & 0x807F) | (rng.integers(120, 136, n).astype(np.uint16) << 7)).astype(np.uint16)
    s = _roundtrip(orc, O.BF16, CB_MID, x_none)
    assert s.size == n + n // 2 + 16 + 8 * 2
    _, h, pos, _ = _records(orc, O.BF16, s, n)
    assert pos.size == 0 and h.tolist() == [[0, 0], [0, 0]]


def check_special_values(orc):
    specials = np.array([0x0000, 0x8000, 0x0001, 0x807F, 0x7F80, 0xFF80, 0x7FC0, 0x7F81,
                         0xFFFF, 0x7FFF, 0x0080, 0x3F80], dtype=np.uint16)
    for cb in (CB_MID, CB_EDGES):
        _roundtrip(orc, O.BF16, cb, specials)
    e5 = np.array([0x00, 0x80, 0x01, 0x03, 0x7C, 0xFC, 0x7D, 0x7F, 0xFF, 0x3C], dtype=np.uint8)
    for cb in (CB_E5_MID, CB_E5_EDGES):
        _roundtrip(orc, O.E5M2, cb, e5)


def check_dense_pass_then_overwrite(orc):
    """With the escapes stripped, decode must give code 0's exponent at each
    escaped element: escapes carry code 0 in the dense stream, and the dense
    pass runs before the overwrite."""
    g = G.load("bf16_hand.txt")
    x = np.array(G.hexwords(g["input"]), dtype=np.uint16)
    cb = np.array(G.ints(g["codebook"]), dtype=np.uint8)
    s = orc.encode(O.BF16, cb, x).copy()
    stripped = s[:-3].copy()
    stripped[5 + 3 + 16 + 4] = 0   # header count 1 -> 0
    st, y = orc.decode(O.BF16, stripped, 5)
    assert st == O.OK
    y = y.view(np.uint16)
    assert y[2] == (int(cb[0]) << 7) and np.array_equal(np.delete(y, 2), np.delete(x, 2))


def check_corrupt_rejected(orc):
    rng = np.random.default_rng(15)
    n = 65536 + 300
    x = _gaussian_bf16(rng, n, scale=np.exp(2 * rng.standard_normal(n)))
    s = orc.encode(O.BF16, CB_MID, x)
    dense = n + (n + 1) // 2
    hdr = dense + 16
    rec = hdr + 16
    cnt0 = int(s[hdr + 4:hdr + 8].view(np.uint32)[0])
    assert cnt0 >= 3
    assert orc.validate(O.BF16, s, n)[0] == O.OK

    def bad(mut):
        t = s.copy()
        t = mut(t)
        assert orc.validate(O.BF16, t, n)[0] == O.CORRUPT
        assert orc.decode(O.BF16, t, n)[0] == O.CORRUPT

    bad(lambda t: t[:-1])                                   # size not on a record boundary
    bad(lambda t: t[:-3])                                   # one record missing
    bad(lambda t: np.concatenate([t, t[-3:]]))              # one record too many
    bad(lambda t: (t.__setitem__(dense + 1, t[dense]), t)[1])           # duplicate codebook entry

    def hdr_offset(t):
        t[hdr + 8] ^= 1                                     # chunk 1 offset off by one
        return t
    bad(hdr_offset)

    def pos_order(t):
        a, b = rec, rec + 3                                 # swap the first two records
        ra, rb = t[a:a + 3].copy(), t[b:b + 3].copy()
        t[a:a + 3], t[b:b + 3] = rb, ra
        return t
    bad(pos_order)

    def pos_range(t):
        last = rec + 3 * (int(s[hdr + 8:hdr + 12].view(np.uint32)[0]) + int(s[hdr + 12:hdr + 16].view(np.uint32)[0]) - 1)
        t[last:last + 2] = np.array([0xFF, 0xFF], dtype=np.uint8)   # position 65535 >= 300 in chunk 1
        return t
    bad(pos_range)

    def count_too_big(t):
        t[hdr + 12:hdr + 16] = np.array([0xFF, 0xFF, 0, 0], dtype=np.uint8)
        return t
    bad(count_too_big)

    # E5M2: a codebook or escape exponent that does not fit 5 bits.
    x8 = rng.integers(0, 256, 1000, dtype=np.uint8)
    s8 = orc.encode(O.E5M2, CB_E5_MID, x8)
    d8 = 7 * 125
    t = s8.copy()
    t[d8 + 15] = 32
    assert orc.validate(O.E5M2, t, 1000)[0] == O.CORRUPT
    t = s8.copy()
    t[d8 + 16 + 8 + 2] = 40
    assert orc.validate(O.E5M2, t, 1000)[0] == O.CORRUPT


def check_invalid_codebook_refused(orc):
    x = np.zeros(4, dtype=np.uint16)
    bad = CB_MID.copy()
    bad[3] = bad[4]
    assert not orc.codebook_valid(O.BF16, bad)
    assert orc.codebook_valid(O.BF16, CB_MID)
    assert not orc.codebook_valid(O.E5M2, CB_MID)        # 120..135 do not fit 5 bits
    try:
        orc.encode(O.BF16, bad, x)
    except ValueError:
        return
    raise AssertionError("encode accepted a codebook with a repeated exponent")


def check_ablation_hand(orc):
    """Stream sizes under Top-16 / Top-8 / Top-15 + sentinel (golden)."""
    for g in G.load("ablation_hand.txt"):
        dt = O.BF16 if g["dtype"] == "bf16" else O.E5M2
        n = int(g["n"])
        if g["case"] == "bf16_all":
            x = np.arange(65536, dtype=np.uint32).astype(np.uint16)
        elif g["case"] == "e5m2_all":
            x = np.arange(256, dtype=np.uint32).astype(np.uint8)
        else:  # exponents ramp_from.. seen 20, 19, ..., 1 times
            e0 = int(g["ramp_from"])
            exps = np.concatenate([np.full(20 - k, e0 + k) for k in range(20)]).astype(np.uint32)
            x = (exps << 7).astype(np.uint16) if dt == O.BF16 else (exps << 2).astype(np.uint8)
        assert O.Oracle.element_count(dt, x) == n
        want = tuple(int(v) for v in g["sizes"].split())
        assert orc.ablation_sizes(dt, orc.histogram(dt, x), n) == want, g["case"]


def check_ablation_top16_is_the_stream(orc):
    """The Top-16 size of the ablation is the size of this format's stream."""
    rng = np.random.default_rng(12)
    for dt, x in ((O.BF16, (rng.standard_normal(70_001) * 40).astype(np.float32).view(np.uint32) >> 16),
                  (O.E5M2, rng.integers(0, 256, 9_999))):
        x = x.astype(np.uint16 if dt == O.BF16 else np.uint8)
        cb = orc.calibrate(dt, x)
        n = O.Oracle.element_count(dt, x)
        assert orc.ablation_sizes(dt, orc.histogram(dt, x), n)[0] == orc.encode(dt, cb, x).size


def check_ablation_codecs_hand(orc):
    """The Top-8 and sentinel streams of the five-element tensor (golden)."""
    for g in G.load("ablation_codecs_hand.txt"):
        variant = O.ABL_TOP8 if g["case"] == "top8" else O.ABL_SENTINEL
        x = np.array([int(v, 16) for v in g["x"].split()], dtype=np.uint16)
        cb = np.array([int(v) for v in g["codebook"].split()], dtype=np.uint8)
        want = np.array([int(v, 16) for v in g["stream"].split()], dtype=np.uint8)
        s = orc.abl_encode(variant, cb, x)
        assert np.array_equal(s, want), g["case"]
        st, y = orc.abl_decode(variant, s, 5)
        assert st == O.OK and y.tobytes() == x.tobytes()


def check_ablation_codecs_bruteforce(orc):
    """Every BF16 pattern: round trip, and the sizes arithmetic fixes (each
    exponent owns 256 patterns: E8 = 63,488, E15 = 61,696)."""
    x = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    rng = np.random.default_rng(21)
    for variant, k, size in ((O.ABL_TOP8, 8, 280592), (O.ABL_SENTINEL, 15, 160023)):
        for cb in (np.arange(120, 120 + k), np.sort(rng.choice(256, k, replace=False)),
                   np.array(list(range(k - 1)) + [255])):
            s = orc.abl_encode(variant, cb.astype(np.uint8), x)
            assert s.size == size
            st, y = orc.abl_decode(variant, s, 65536)
            assert st == O.OK and y.tobytes() == x.tobytes()
        # A shuffled tensor over three chunks: the order of escapes matters here.
        xs = x[rng.permutation(65536)][: 3 * 65536 // 2]
        xs = np.concatenate([xs, x[rng.permutation(65536)]])
        cb = orc.abl_codebook(variant, orc.histogram(O.BF16, xs))
        s = orc.abl_encode(variant, cb, xs)
        st, y = orc.abl_decode(variant, s, xs.size)
        assert st == O.OK and y.tobytes() == xs.tobytes()
        assert s.size == orc.ablation_sizes(O.BF16, orc.histogram(O.BF16, xs), xs.size)[1 if k == 8 else 2]


def check_ablation_codecs_reject_corruption(orc):
    x = (np.random.default_rng(5).standard_normal(70_000) * 50).astype(np.float32).view(np.uint32) >> 16
    x = x.astype(np.uint16)
    for variant in (O.ABL_TOP8, O.ABL_SENTINEL):
        cb = orc.abl_codebook(variant, orc.histogram(O.BF16, x))
        s = orc.abl_encode(variant, cb, x)
        assert orc.abl_decode(variant, s[:-1], x.size)[0] == O.CORRUPT       # size off
        k = 8 if variant == O.ABL_TOP8 else 15
        hdr = x.size + (3 * ((x.size + 7) // 8) if variant == O.ABL_TOP8 else (x.size + 1) // 2) + k
        bad = s.copy()
        bad[hdr + 4] ^= 1                                                     # chunk 0 count
        assert orc.abl_decode(variant, bad, x.size)[0] == O.CORRUPT


def _join_streams(dt, parts, ns):
    """The stream of the concatenated tensor assembled from shard streams by
    the layout alone (R9, R7): dense parts in order, the codebook once, each
    shard's headers with offsets shifted by the escapes before it, records
    in order.  Every shard but the last holds whole chunks."""
    dense_parts, nibs, hdrs, recs, e_before, cb = [], [], [], [], 0, None
    for s, n in zip(parts, ns):
        dense = n + (n + 1) // 2 if dt == O.BF16 else 7 * (-(-n // 8))
        C = -(-n // 65536)
        if dt == O.BF16:
            dense_parts.append(s[:n])
            nibs.append(s[n:dense])
        else:
            dense_parts.append(s[:dense])
        cb = s[dense:dense + 16] if cb is None else cb
        h = s[dense + 16:dense + 16 + 8 * C].copy().view(np.uint32).reshape(C, 2).copy()
        h[:, 0] += e_before
        hdrs.append(h.reshape(-1).view(np.uint8))
        rec = s[dense + 16 + 8 * C:]
        recs.append(rec)
        e_before += rec.size // 3
    return np.concatenate(dense_parts + nibs + [cb] + hdrs + recs)


def check_shard_join(orc):
    # Chunks are independent apart from the header offsets: shards of whole
    # chunks, encoded on their own and joined by the layout alone, give the
    # whole tensor's stream (positions are chunk-relative, offsets running sums).
    rng = np.random.default_rng(14)
    C = 65536
    for dt, cb in ((O.BF16, CB_MID), (O.E5M2, CB_E5_MID)):
        for ns in ([C, 2 * C + 77], [0, C, 0, C + 1], [3 * C], [C, C, 5]):
            n = sum(ns)
            if dt == O.BF16:
                x = _gaussian_bf16(rng, n, scale=np.exp(2 * rng.standard_normal(n))).view(np.uint8)
            else:
                x = rng.integers(0, 256, n, dtype=np.uint8)
            esize = 2 if dt == O.BF16 else 1
            parts, at = [], 0
            for m in ns:
                parts.append(orc.encode(dt, cb, x[at * esize:(at + m) * esize]))
                at += m
            whole = orc.encode(dt, cb, x)
            assert np.array_equal(_join_streams(dt, parts, ns), whole)


CHECKS = [
    check_hand_bf16,
    check_hand_e5m2,
    check_two_chunks_bf16,
    check_calibration_hand,
    check_bruteforce_bf16,
    check_bruteforce_e5m2,
    check_invariants_bf16,
    check_invariants_e5m2,
    check_edge_sizes,
    check_all_and_zero_escape,
    check_special_values,
    check_dense_pass_then_overwrite,
    check_corrupt_rejected,
    check_invalid_codebook_refused,
    check_ablation_hand,
    check_ablation_top16_is_the_stream,
    check_ablation_codecs_hand,
    check_ablation_codecs_bruteforce,
    check_ablation_codecs_reject_corruption,
    check_shard_join,
]
