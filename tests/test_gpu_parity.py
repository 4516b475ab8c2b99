"""CUDA codec vs the CPU oracle, element by element (GPU).

Encoded streams must be byte-identical to the oracle's and decoding must give
the input back bit for bit: the codec is integer bit manipulation, so the
tolerance is zero (SplitZip abstract, arXiv 2605.01708v2: the KV tensors are
preserved bitwise).
"""
import numpy as np
import pytest
import torch

from oracle import oracle as O
from tests import gpu_codec as G
from tests.oracle_pins import CB_EDGES, CB_E5_EDGES, CB_E5_MID, CB_MID

pytestmark = pytest.mark.gpu

ODT = {"bf16": O.BF16, "e5m2": O.E5M2}


def roundtrip_vs_oracle(orc, kind, cb, x: torch.Tensor, **kw):
    """Encode on the GPU, compare with the oracle byte for byte, decode on the
    GPU, compare with the input bit for bit."""
    dt, odt = G.DT[kind], ODT[kind]
    xh = G.as_bytes(x)
    n = G.elements(dt, x)
    want = orc.encode(odt, cb, xh)
    got, status, size = G.encode(dt, cb, x, out_offset=kw.get("out_offset", 0))
    assert status == 0, f"encode status {status}"
    assert size == want.size
    if not np.array_equal(got, want):
        bad = np.flatnonzero(got != want)
        pytest.fail(f"stream differs from the oracle at {bad.size} bytes, first at {bad[:8]} (size {size})")
    st, y, guard_ok = G.decode(dt, got, n, out_offset=kw.get("dec_out_offset", 0), in_offset=kw.get("dec_in_offset", 0))
    assert st == 0 and guard_ok
    assert np.array_equal(y, xh), "decode is not bit-exact"
    return got


def _gauss(n, scale_sigma=2.0, seed=0, device="cuda"):
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    s = torch.exp(scale_sigma * torch.randn(n, generator=g, device=device))
    return (torch.randn(n, generator=g, device=device) * s).to(torch.bfloat16)


def _bytes(n, seed=0):
    g = torch.Generator(device="cuda")
    g.manual_seed(seed)
    return torch.randint(0, 256, (n,), generator=g, device="cuda", dtype=torch.uint8)


EDGE_N = [0, 1, 2, 3, 7, 8, 9, 31, 32, 33, 255, 256, 257, 1023, 1024, 1025, 4095, 4097, 8191, 8192, 8193,
          16383, 16384, 16385, 65535, 65536, 65537, 131073, 200003, 3 * 65536 + 12345]


@pytest.mark.parametrize("n", EDGE_N)
def test_bf16_edge_sizes(orc, n):
    roundtrip_vs_oracle(orc, "bf16", CB_MID, _gauss(n, seed=n))


@pytest.mark.parametrize("n", EDGE_N)
def test_e5m2_edge_sizes(orc, n):
    roundtrip_vs_oracle(orc, "e5m2", CB_E5_MID, _bytes(n, seed=n))


def test_bf16_bruteforce_all_patterns(orc):
    x = torch.arange(65536, dtype=torch.int32, device="cuda").to(torch.int16).view(torch.bfloat16)
    # Contiguous codebooks (byte-parallel coding path) including both ends of
    # the exponent range, and a non-contiguous one (table path).
    cbs = (CB_MID, np.arange(0, 16, dtype=np.uint8), np.arange(240, 256, dtype=np.uint8), CB_EDGES)
    for cb in cbs:
        s = roundtrip_vs_oracle(orc, "bf16", cb, x)
        assert s.size == 282648
    # Every pattern in a shuffled order across several tiles and chunks.
    g = torch.Generator(device="cuda")
    g.manual_seed(5)
    perm = torch.cat([torch.randperm(65536, generator=g, device="cuda") for _ in range(5)])
    for cb in (CB_MID, CB_EDGES):
        roundtrip_vs_oracle(orc, "bf16", cb, x[perm].contiguous())


def test_e5m2_bruteforce_all_patterns(orc):
    x = torch.arange(256, dtype=torch.int32, device="cuda").to(torch.uint8)
    cbs = (CB_E5_MID, np.arange(0, 16, dtype=np.uint8), np.arange(16, 32, dtype=np.uint8), CB_E5_EDGES)
    for cb in cbs:
        s = roundtrip_vs_oracle(orc, "e5m2", cb, x)
        assert s.size == 632
    # Shuffled across several scan tiles and chunks (whole-warp load path).
    g = torch.Generator(device="cuda")
    g.manual_seed(6)
    perm = torch.randint(0, 256, (5 * 65536 + 77,), generator=g, device="cuda")
    for cb in cbs:
        roundtrip_vs_oracle(orc, "e5m2", cb, x[perm].contiguous())


def test_unaligned_buffers(orc):
    base = _gauss(3 * 65536 + 40, seed=11)
    roundtrip_vs_oracle(orc, "bf16", CB_MID, base[1:], out_offset=1, dec_out_offset=2, dec_in_offset=3)
    b8 = _bytes(2 * 65536 + 41, seed=12)
    roundtrip_vs_oracle(orc, "e5m2", CB_E5_MID, b8[3:], out_offset=5, dec_out_offset=1, dec_in_offset=7)


def test_all_escape_and_no_escape(orc):
    n = 3 * 65536 + 999
    x = _gauss(n, seed=13).view(torch.int16).to(torch.int32) & 0xFFFF
    g = torch.Generator(device="cuda")
    g.manual_seed(14)
    outside = torch.randint(10, 110, (n,), generator=g, device="cuda", dtype=torch.int32)
    inside = torch.randint(120, 136, (n,), generator=g, device="cuda", dtype=torch.int32)
    x_all = ((x & 0x807F) | (outside << 7)).to(torch.int16).view(torch.bfloat16)
    x_none = ((x & 0x807F) | (inside << 7)).to(torch.int16).view(torch.bfloat16)
    s = roundtrip_vs_oracle(orc, "bf16", CB_MID, x_all)
    assert s.size == n + (n + 1) // 2 + 3 * n + 16 + 8 * 4
    s = roundtrip_vs_oracle(orc, "bf16", CB_MID, x_none)
    assert s.size == n + (n + 1) // 2 + 16 + 8 * 4
    b = _bytes(n, seed=15).to(torch.int32)
    e_out = torch.randint(0, 14, (n,), generator=g, device="cuda", dtype=torch.int32)
    b_all = ((b & 0x83) | (e_out << 2)).to(torch.uint8)
    s = roundtrip_vs_oracle(orc, "e5m2", CB_E5_MID, b_all)
    assert s.size == 7 * ((n + 7) // 8) + 3 * n + 16 + 8 * 4


@pytest.mark.parametrize("escapes", ["fortieth_minus_one", "fortieth", "quarter", "sixty_percent"])
def test_escape_dense_streams(orc, escapes):
    """Streams with escapes in 1/40 of the elements and more, at exact counts
    spread uniformly over four and a fraction chunks.  From 1/40 on the
    decoder runs its escape-dense variant (exponents by byte adds for a
    contiguous codebook); one escape fewer keeps the other.  On both sides
    the stream is the oracle's byte for byte, and decoding gives the input
    back bit for bit, also into an output that is only 2-byte aligned (no
    vector stores) from an input at an odd address."""
    n = 4 * 65536 + 416                      # a multiple of 40: 1/40 is exact
    k = {"fortieth_minus_one": n // 40 - 1, "fortieth": n // 40, "quarter": n // 4,
         "sixty_percent": (3 * n) // 5}[escapes]
    g = torch.Generator(device="cuda")
    g.manual_seed(41)
    x = _gauss(n, scale_sigma=0.1, seed=42).view(torch.int16).to(torch.int32) & 0xFFFF
    inside = torch.randint(120, 136, (n,), generator=g, device="cuda", dtype=torch.int32)
    x = (x & 0x807F) | (inside << 7)
    idx = torch.randperm(n, generator=g, device="cuda")[:k]
    outside = torch.randint(10, 110, (k,), generator=g, device="cuda", dtype=torch.int32)
    x[idx] = (x[idx] & 0x807F) | (outside << 7)
    x = x.to(torch.int16).view(torch.bfloat16)
    s = roundtrip_vs_oracle(orc, "bf16", CB_MID, x)
    assert s.size == n + n // 2 + 16 + 8 * 5 + 3 * k
    roundtrip_vs_oracle(orc, "bf16", CB_MID, x, dec_out_offset=2, dec_in_offset=1)


def test_calibration_matches_oracle(orc):
    from lossless_kv_cache_bf16_gb300 import workloads as W

    for kind, sample in (("bf16", W.kv_tiny("cuda", 1)), ("e5m2", W.fp8_e5m2_kv("cuda", 1, layers=1, tokens=256)),
                         ("bf16", _gauss(100003, seed=3))):
        cb, hist = G.calibrate(G.DT[kind], sample)
        xh = G.as_bytes(sample)
        assert np.array_equal(hist, orc.histogram(ODT[kind], xh))
        assert np.array_equal(cb, orc.calibrate(ODT[kind], xh))


def test_tiny_config(orc):
    from lossless_kv_cache_bf16_gb300 import workloads as W

    x = W.kv_tiny("cuda", 0)
    cb, _ = G.calibrate(G.DT["bf16"], W.kv_tiny("cuda", 1))
    roundtrip_vs_oracle(orc, "bf16", cb, x)


def test_encode_on_side_stream(orc):
    x = _gauss(5 * 65536 + 3, seed=21)
    s = torch.cuda.Stream()
    want = orc.encode(O.BF16, CB_MID, G.as_bytes(x))
    with torch.cuda.stream(s):
        got, st, size = G.encode(G.DT["bf16"], CB_MID, x, stream=s)
    assert st == 0 and np.array_equal(got, want)


def test_capacity_overflow_reported(orc):
    from lossless_kv_cache_bf16_gb300 import splitzip as S

    x = _gauss(2 * 65536 + 5, seed=22)
    n = x.numel()
    want = orc.encode(O.BF16, CB_MID, G.as_bytes(x))
    cap = S.sz_encoded_size(S.SZ_BF16, n, 0) + 30  # room for 10 escapes only
    got, st, size = G.encode(S.SZ_BF16, CB_MID, x, capacity=cap)
    assert st == S.SZ_ERR_CAPACITY and size == want.size
    assert np.array_equal(got[:cap], want[:cap])  # everything that fits is right


def _unit_density_tensor(kind, n, seed, densities):
    """A tensor whose 1,024-element units each have their own escape density
    (drawn per unit from `densities`), so that scan tiles hold anywhere from
    no escapes to all escapes, with the staged-record limit falling inside
    units at varying places.  Escaped elements get an exponent outside CB_MID
    (BF16) or CB_E5_MID (E5M2), the others one inside it."""
    g = torch.Generator(device="cuda")
    g.manual_seed(seed)
    units = (n + 1023) // 1024
    d = torch.tensor(densities, dtype=torch.float32, device="cuda")
    per_unit = d[torch.randint(0, len(densities), (units,), generator=g, device="cuda")]
    p = per_unit.repeat_interleave(1024)[:n]
    esc = torch.rand(n, generator=g, device="cuda") < p
    r = torch.randint(0, 1 << 16, (n,), generator=g, device="cuda", dtype=torch.int32)
    if kind == "bf16":
        inside = torch.randint(120, 136, (n,), generator=g, device="cuda", dtype=torch.int32)
        outside = torch.randint(0, 120, (n,), generator=g, device="cuda", dtype=torch.int32)
        outside = torch.where(outside >= 110, outside + 26, outside)  # 0..109 and 136..145
        e = torch.where(esc, outside, inside)
        return ((r & 0x807F) | (e << 7)).to(torch.int16).view(torch.bfloat16)
    inside = torch.randint(14, 30, (n,), generator=g, device="cuda", dtype=torch.int32)
    outside = torch.randint(0, 16, (n,), generator=g, device="cuda", dtype=torch.int32)
    outside = torch.where(outside >= 14, outside + 16, outside)  # 0..13, 30, 31
    e = torch.where(esc, outside, inside)
    return ((r & 0x83) | (e << 2)).to(torch.uint8)


@pytest.mark.parametrize("kind", ["bf16", "e5m2"])
@pytest.mark.parametrize("seed,densities", [
    (31, (0.0, 0.002, 0.05, 0.3, 0.9, 1.0)),
    (32, (0.0, 1.0)),
    (33, (0.025, 0.035, 0.055, 0.065)),  # tiles around the staging limits (1,024 and 2,048 records)
    (34, (0.5,)),
])
def test_scan_tiles_beyond_staging(orc, kind, seed, densities):
    """Scan tiles with more escapes than the encoder stages have their
    remaining records re-derived unit by unit; the stream must still be the
    oracle's byte for byte, for tiles of every density mix and a ragged end."""
    n = 7 * 32768 + 1234
    cb = CB_MID if kind == "bf16" else CB_E5_MID
    x = _unit_density_tensor(kind, n, seed, densities)
    roundtrip_vs_oracle(orc, kind, cb, x)


@pytest.mark.parametrize("kind", ["bf16", "e5m2"])
def test_encode_status_needs_no_reset(orc, kind):
    """The encode writes its status word once, at its end, from what every
    block of the encode reported: whatever the word held before (another
    call's error, garbage) does not matter, and an error of one call does not
    stay for the next call on the same word and workspace."""
    from lossless_kv_cache_bf16_gb300 import splitzip as S

    dt = G.DT[kind]
    cb = CB_MID if kind == "bf16" else CB_E5_MID
    x = _unit_density_tensor(kind, 3 * 65536 + 777, 41, (0.0, 0.01, 0.5))
    n = G.elements(dt, x)
    want = orc.encode(ODT[kind], cb, G.as_bytes(x))
    ws = torch.empty(S.sz_workspace_size(dt, n), dtype=torch.uint8, device="cuda")
    ob = torch.zeros(1, dtype=torch.int64, device="cuda")
    st = torch.empty(1, dtype=torch.int32, device="cuda")
    full = torch.empty(S.sz_encoded_size(dt, n, n), dtype=torch.uint8, device="cuda")
    short = torch.empty(S.sz_encoded_size(dt, n, 0) + 30, dtype=torch.uint8, device="cuda")
    for before, out, expect in ((-1, full, S.SZ_OK), (99, short, S.SZ_ERR_CAPACITY), (S.SZ_ERR_CAPACITY, full, S.SZ_OK),
                                (S.SZ_ERR_TIMEOUT, short, S.SZ_ERR_CAPACITY), (0, full, S.SZ_OK)):
        st.fill_(before)
        S.sz_encode(dt, cb, x, out, ob, st, ws)
        torch.cuda.synchronize()
        assert int(st.item()) == expect, (before, expect)
        assert int(ob.item()) == want.size
        if expect == S.SZ_OK:
            assert np.array_equal(out[: want.size].cpu().numpy(), want)
