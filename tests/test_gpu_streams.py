"""Ordering and concurrency of the codec's launches (GPU).

The kernels that read what an earlier kernel wrote (finish after encode,
decode after its producer, top-16 selection after the histogram) are launched
as programmatic dependents and wait for that kernel before their first read.
These tests enqueue chains with no host synchronisation between the steps, so
that a read issued too early would see the previous iteration's bytes, and
compare every result with the oracle.  They also run several streams and
several host threads at once on separate buffers: the library keeps no state
between calls other than a cache of launch shapes.
"""
import threading

import numpy as np
import pytest
import torch

from oracle import oracle as O
from tests import gpu_codec as G
from tests.oracle_pins import CB_E5_MID, CB_MID

pytestmark = pytest.mark.gpu

ODT = {"bf16": O.BF16, "e5m2": O.E5M2}
CB = {"bf16": CB_MID, "e5m2": CB_E5_MID}


def _tensor(kind, n, seed, scale=30.0):
    g = torch.Generator(device="cuda")
    g.manual_seed(seed)
    if kind == "bf16":
        return (torch.randn(n, generator=g, device="cuda") * scale).to(torch.bfloat16)
    return (torch.randn(n, generator=g, device="cuda") * scale).to(torch.float8_e5m2).view(torch.uint8)


class Job:
    """One encode + decode of one tensor on one stream, with its own buffers."""

    def __init__(self, orc, kind, n, seed):
        from lossless_kv_cache_bf16_gb300 import splitzip as S

        self.kind, self.dt, self.n = kind, G.DT[kind], n
        self.x = _tensor(kind, n, seed)
        self.want = orc.encode(ODT[kind], CB[kind], G.as_bytes(self.x))
        self.out = torch.empty(S.sz_encoded_size(self.dt, n, n), dtype=torch.uint8, device="cuda")
        self.ws = torch.empty(S.sz_workspace_size(self.dt, n), dtype=torch.uint8, device="cuda")
        self.ob = torch.zeros(1, dtype=torch.int64, device="cuda")
        self.est = torch.full((1,), -1, dtype=torch.int32, device="cuda")
        self.dst = torch.full((1,), -1, dtype=torch.int32, device="cuda")
        self.y = torch.empty_like(self.x)
        self.stream = torch.cuda.Stream()

    def enqueue(self):
        from lossless_kv_cache_bf16_gb300 import splitzip as S

        # The stream's size is fixed by the input, so the decode can follow the
        # encode at once, with no host round trip for the size.
        S.sz_encode(self.dt, CB[self.kind], self.x, self.out, self.ob, self.est, self.ws, stream=self.stream)
        S.sz_decode(self.dt, self.out, self.want.size, self.n, self.y, self.dst, stream=self.stream)

    def check(self):
        assert int(self.est.item()) == 0 and int(self.dst.item()) == 0
        assert int(self.ob.item()) == self.want.size
        assert np.array_equal(self.out[: self.want.size].cpu().numpy(), self.want)
        assert torch.equal(self.y.view(torch.uint8), self.x.view(torch.uint8))


def test_streams_run_concurrently(orc):
    jobs = [Job(orc, kind, n, seed) for seed, (kind, n) in enumerate(
        [("bf16", 9 * 32_768 + 17), ("e5m2", 5 * 65_536 + 3), ("bf16", 200_000), ("e5m2", 1_000_001)])]
    torch.cuda.synchronize()
    for _ in range(3):  # interleaved on four streams, several calls deep
        for j in jobs:
            j.enqueue()
    torch.cuda.synchronize()
    for j in jobs:
        j.check()


@pytest.mark.parametrize("kind", ["bf16", "e5m2"])
def test_decode_waits_for_the_kernel_that_wrote_its_stream(orc, kind):
    from lossless_kv_cache_bf16_gb300 import splitzip as S

    dt, n = G.DT[kind], 600_000
    xs = [_tensor(kind, n, 100 + k, scale=s) for k, s in enumerate((30.0, 0.01))]
    streams = [torch.from_numpy(orc.encode(ODT[kind], CB[kind], G.as_bytes(x))).cuda() for x in xs]
    cap = max(s.numel() for s in streams)
    buf = torch.empty(cap, dtype=torch.uint8, device="cuda")
    ys = [torch.empty_like(xs[0]) for _ in range(8)]
    sts = torch.full((8,), -1, dtype=torch.int32, device="cuda")
    torch.cuda.synchronize()
    for i in range(8):
        src = streams[i % 2]
        # An elementwise kernel (not a copy-engine copy) writes the stream the
        # decode reads next; the two alternate, so an early read decodes the
        # other tensor or fails validation.
        torch.add(src, 0, out=buf[: src.numel()])
        S.sz_decode(dt, buf, src.numel(), n, ys[i], sts[i:i + 1])
    torch.cuda.synchronize()
    assert sts.cpu().tolist() == [0] * 8
    for i in range(8):
        assert torch.equal(ys[i].view(torch.uint8), xs[i % 2].view(torch.uint8)), f"decode {i}"


@pytest.mark.parametrize("kind", ["bf16", "e5m2"])
def test_selection_waits_for_the_histogram(orc, kind):
    from lossless_kv_cache_bf16_gb300 import splitzip as S

    dt, n = G.DT[kind], 300_000
    # Scales 2^10 apart: the exponent ranges, and so the codebooks, differ.
    xs = [_tensor(kind, n, 200 + k, scale=s) for k, s in enumerate((1.0, 1024.0))]
    want = [[int(v) for v in orc.calibrate(ODT[kind], G.as_bytes(x))] for x in xs]
    assert want[0] != want[1]
    hist = torch.empty(S.sz_histogram_bins(dt), dtype=torch.int64, device="cuda")
    cbs = torch.empty((8, 16), dtype=torch.uint8, device="cuda")
    torch.cuda.synchronize()
    for i in range(8):  # one histogram buffer for all: each selection must see its own counts
        S.sz_calibrate_device(dt, xs[i % 2], hist, cbs[i], sample_stride=1)
    torch.cuda.synchronize()
    for i in range(8):
        assert cbs[i].cpu().tolist() == want[i % 2], f"calibration {i}"


def test_host_threads_share_the_library(orc):
    jobs = [Job(orc, kind, n, 300 + k) for k, (kind, n) in enumerate(
        [("bf16", 131_073), ("e5m2", 262_151), ("bf16", 65_536 * 3), ("e5m2", 99_999)])]
    torch.cuda.synchronize()
    errors = []

    def worker(j):
        try:
            for _ in range(10):
                j.enqueue()
            j.stream.synchronize()
            j.check()
        except Exception as e:  # reported on the main thread
            errors.append(e)

    threads = [threading.Thread(target=worker, args=(j,)) for j in jobs]
    for t in threads:
        t.start()
    for t in threads:
        t.join()
    assert not errors, errors
