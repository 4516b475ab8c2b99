"""Online (per-tensor) calibration on the device, against the oracle.

The pages calibrate the codebook offline; their calibration ablation weighs
doing it per tensor instead.  These tests pin the device path to the oracle:
the device top-16 must equal the oracle's selection on the same counts, the
sampled device histogram must give the oracle's codebook for the gathered
sample, and an encode that reads the codebook from device memory must give
the oracle's stream byte for byte.  The whole chain also runs inside a
captured CUDA graph, which proves it needs no host synchronisation.
"""
import numpy as np
import pytest
import torch

from oracle import oracle as O
from tests import gpu_codec as G
from tests.oracle_pins import CB_E5_EDGES, CB_E5_MID, CB_EDGES, CB_MID

pytestmark = pytest.mark.gpu

S = None


@pytest.fixture(autouse=True)
def _lib():
    global S
    from lossless_kv_cache_bf16_gb300 import splitzip

    S = splitzip


ODT = {"bf16": O.BF16, "e5m2": O.E5M2}


def _dt(kind):
    return S.SZ_BF16 if kind == "bf16" else S.SZ_FP8_E5M2


def _device_cb(cb):
    return torch.tensor([int(v) for v in cb], dtype=torch.uint8, device="cuda")


def _histograms(bins, rng):
    """Counts that exercise the selection rule: ties, zeros, huge values."""
    yield np.zeros(bins, dtype=np.int64)                                   # all ties at 0
    yield np.arange(bins, dtype=np.int64)                                  # distinct
    yield np.full(bins, 7, dtype=np.int64)                                 # all tied
    h = np.zeros(bins, dtype=np.int64)
    h[[3, 9, bins - 1]] = 5                                                # fewer than 16 seen
    yield h
    for _ in range(40):
        h = rng.integers(0, 4, size=bins).astype(np.int64)                 # many ties
        yield h
        h = rng.integers(0, 1 << 40, size=bins).astype(np.int64)
        h[rng.integers(0, bins, size=8)] = h.max()                         # ties at the top
        yield h


@pytest.mark.parametrize("kind", ["bf16", "e5m2"])
def test_device_top16_matches_oracle(orc, kind):
    dt = _dt(kind)
    bins = S.sz_histogram_bins(dt)
    rng = np.random.default_rng(31)
    cb = torch.empty(16, dtype=torch.uint8, device="cuda")
    for h in _histograms(bins, rng):
        hist = torch.tensor(h, dtype=torch.int64, device="cuda")
        S.sz_codebook_from_histogram_device(dt, hist, cb)
        want = [int(v) for v in orc.codebook_from_histogram(ODT[kind], h.astype(np.uint64))]
        assert cb.cpu().tolist() == want, h


def _lowbias32(x):
    """C. Wellons' 32-bit integer hash, on uint64 arrays of 32-bit values."""
    m = np.uint64(0xFFFFFFFF)
    x = x.astype(np.uint64)
    x ^= x >> np.uint64(16)
    x = (x * np.uint64(0x7FEB352D)) & m
    x ^= x >> np.uint64(15)
    x = (x * np.uint64(0x846CA68B)) & m
    x ^= x >> np.uint64(16)
    return x


def _sampled(xb, esize, n, stride):
    """The sample, gathered on the host: 128-byte lines; run w of `stride`
    lines (the last may be shorter, L lines) contributes line
    w * stride + floor(lowbias32(w) * L / 2^32)."""
    per = 128 // esize
    lines = -(-n // per)
    w = np.arange(-(-lines // stride), dtype=np.uint64)
    first = w * np.uint64(stride)
    length = np.minimum(np.uint64(lines) - first, np.uint64(stride))
    sel = first + ((_lowbias32(w) * length) >> np.uint64(32))
    keep = np.zeros(lines, dtype=bool)
    keep[sel.astype(np.int64)] = True
    return xb.reshape(n, esize)[keep[np.arange(n) // per]].reshape(-1)


@pytest.mark.parametrize("kind", ["bf16", "e5m2"])
@pytest.mark.parametrize("stride", [1, 3, 16, 997])
def test_calibrate_device_matches_oracle_on_the_sample(orc, kind, stride):
    from lossless_kv_cache_bf16_gb300 import workloads as W

    dt = _dt(kind)
    if kind == "bf16":
        x = W.kv_tiny("cuda", 2).reshape(-1)[: 300_001]
    else:
        x = W.fp8_e5m2_kv("cuda", 2, layers=1, tokens=64).reshape(-1)[: 300_001]
    # aligned, misaligned (byte loads), then short tensors (one partial line)
    for xx in (x, x[1:], x[:65], x[:1]):
        n = xx.numel()
        hist = torch.empty(S.sz_histogram_bins(dt), dtype=torch.int64, device="cuda")
        cb = torch.empty(16, dtype=torch.uint8, device="cuda")
        S.sz_calibrate_device(dt, xx, hist, cb, sample_stride=stride)
        xb = G.as_bytes(xx)
        sample = _sampled(xb, 2 if kind == "bf16" else 1, n, stride)
        assert hist.cpu().numpy().astype(np.uint64).tolist() == orc.histogram(ODT[kind], sample).tolist()
        want = [int(v) for v in orc.calibrate(ODT[kind], sample)]
        assert cb.cpu().tolist() == want


@pytest.mark.parametrize("kind,cbv", [("bf16", CB_MID), ("bf16", CB_EDGES), ("e5m2", CB_E5_MID),
                                      ("e5m2", CB_E5_EDGES)])
@pytest.mark.parametrize("n", [0, 1, 7, 65_537, 3 * 32_768 + 5, 400_000])
def test_encode_dcb_matches_oracle(orc, kind, cbv, n):
    dt = _dt(kind)
    g = torch.Generator(device="cuda")
    g.manual_seed(n + 11)
    if kind == "bf16":
        x = (torch.randn(n, generator=g, device="cuda") * 30).to(torch.bfloat16)
    else:
        x = torch.randint(0, 256, (n,), generator=g, device="cuda", dtype=torch.uint8)
    cap = S.sz_encoded_size(dt, n, n)
    out = torch.empty(cap, dtype=torch.uint8, device="cuda")
    ws = torch.empty(S.sz_workspace_size(dt, n), dtype=torch.uint8, device="cuda")
    ob = torch.zeros(1, dtype=torch.int64, device="cuda")
    st = torch.full((1,), -1, dtype=torch.int32, device="cuda")
    S.sz_encode_dcb(dt, _device_cb(cbv), x, out, ob, st, ws)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    got = out[: int(ob.item())].cpu().numpy()
    want = orc.encode(ODT[kind], np.array(cbv, dtype=np.uint8), G.as_bytes(x))
    assert np.array_equal(got, want)


@pytest.mark.parametrize("kind,bad", [("bf16", list(range(15)) + [14]),          # repeated
                                      ("bf16", list(range(16, 0, -1))),          # descending
                                      ("e5m2", list(range(20, 36))),             # beyond 5 bits
                                      ("e5m2", [0] * 16)])
def test_encode_dcb_rejects_a_bad_codebook(kind, bad):
    dt = _dt(kind)
    n = 70_000
    x = torch.zeros(n * (2 if kind == "bf16" else 1), dtype=torch.uint8, device="cuda")
    out = torch.empty(S.sz_encoded_size(dt, n, n), dtype=torch.uint8, device="cuda")
    ws = torch.empty(S.sz_workspace_size(dt, n), dtype=torch.uint8, device="cuda")
    ob = torch.zeros(1, dtype=torch.int64, device="cuda")
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    S.sz_encode_dcb(dt, _device_cb(bad), x, out, ob, st, ws, n=n)
    torch.cuda.synchronize()
    assert int(st.item()) == S.SZ_ERR_INVALID_ARG


@pytest.mark.parametrize("kind", ["bf16", "e5m2"])
def test_online_chain_in_a_cuda_graph(orc, kind):
    """calibrate -> encode captured once in a CUDA graph (so neither call
    synchronises with the host), replayed on new data; decode follows eagerly
    with the stream size read back from the device."""
    from lossless_kv_cache_bf16_gb300 import workloads as W

    dt = _dt(kind)

    def data(seed):
        if kind == "bf16":
            return W.kv_tiny("cuda", seed).reshape(-1)
        return W.fp8_e5m2_kv("cuda", seed, layers=1, tokens=256).reshape(-1)

    x = data(3).clone()
    n = x.numel()
    hist = torch.empty(S.sz_histogram_bins(dt), dtype=torch.int64, device="cuda")
    cb = torch.empty(16, dtype=torch.uint8, device="cuda")
    out = torch.empty(S.sz_encoded_size(dt, n, n), dtype=torch.uint8, device="cuda")
    ws = torch.empty(S.sz_workspace_size(dt, n), dtype=torch.uint8, device="cuda")
    ob = torch.zeros(1, dtype=torch.int64, device="cuda")
    est = torch.zeros(1, dtype=torch.int32, device="cuda")
    dst = torch.zeros(1, dtype=torch.int32, device="cuda")
    y = torch.empty_like(x)

    def chain():
        S.sz_calibrate_device(dt, x, hist, cb, sample_stride=4)
        S.sz_encode_dcb(dt, cb, x, out, ob, est, ws)

    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        chain()  # warm-up outside the capture
    torch.cuda.current_stream().wait_stream(side)
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        chain()
    for seed in (5, 7):
        new = data(seed)
        xb = G.as_bytes(new)
        want_cb = orc.calibrate(ODT[kind], _sampled(xb, 2 if kind == "bf16" else 1, n, 4))
        want = orc.encode(ODT[kind], want_cb, xb)
        x.copy_(new)
        graph.replay()
        torch.cuda.synchronize()
        assert int(est.item()) == 0
        assert cb.cpu().tolist() == [int(v) for v in want_cb]
        size = int(ob.item())
        assert np.array_equal(out[:size].cpu().numpy(), want)
        S.sz_decode(dt, out, size, n, y, dst)
        torch.cuda.synchronize()
        assert int(dst.item()) == 0
        assert torch.equal(y.view(torch.uint8), x.view(torch.uint8))


@pytest.mark.parametrize("kind", ["bf16", "e5m2"])
def test_ablation_sizes_from_the_device_histogram(orc, kind):
    """Device histogram + the library's ablation arithmetic = the oracle's
    ablation sizes of the same tensor; the Top-16 size is the real stream's."""
    from lossless_kv_cache_bf16_gb300 import workloads as W

    dt = _dt(kind)
    x = (W.kv_tiny("cuda", 4) if kind == "bf16" else W.fp8_e5m2_kv("cuda", 4, layers=1, tokens=128)).reshape(-1)
    n = x.numel()
    hist = torch.empty(S.sz_histogram_bins(dt), dtype=torch.int64, device="cuda")
    S.sz_histogram(dt, x, hist)
    got = S.sz_ablation_sizes(dt, hist.cpu().tolist(), n)
    xb = G.as_bytes(x)
    assert got == orc.ablation_sizes(ODT[kind], orc.histogram(ODT[kind], xb), n)
    assert got[0] == orc.encode(ODT[kind], orc.calibrate(ODT[kind], xb), xb).size
