"""Pipelined offload to host memory and reload (transfer.Pipeline), against
the oracle: every segment's stream in host memory equals the oracle's stream
of that segment byte for byte, and the reloaded tensor is bit-exact."""
import numpy as np
import pytest
import torch

from oracle import oracle as O
from tests import gpu_codec as G
from tests.oracle_pins import CB_E5_EDGES, CB_E5_MID, CB_EDGES, CB_MID

pytestmark = pytest.mark.gpu

ODT = {"bf16": O.BF16, "e5m2": O.E5M2}


def _tensor(kind, n, seed):
    g = torch.Generator(device="cuda")
    g.manual_seed(seed)
    if kind == "bf16":
        return (torch.randn(n, generator=g, device="cuda") * 30).to(torch.bfloat16)
    return torch.randint(0, 256, (n,), generator=g, device="cuda", dtype=torch.uint8)


@pytest.mark.parametrize("kind,cb", [("bf16", CB_MID), ("bf16", CB_EDGES), ("e5m2", CB_E5_MID), ("e5m2", CB_E5_EDGES)])
@pytest.mark.parametrize("n,parts", [(0, 4), (1, 4), (65_537, 8), (5 * 65_536 + 123, 3), (1_000_000, 8),
                                     (1_000_000, 1)])
def test_offload_reload_matches_oracle(orc, kind, cb, n, parts):
    from lossless_kv_cache_bf16_gb300 import transfer as T

    dt = G.DT[kind]
    x = _tensor(kind, n, seed=n + parts)
    pipe = T.Pipeline(dt, cb, n, "cuda", parts=parts)
    hs = pipe.offload(x)
    assert hs.segs == T.segments(n, parts)
    xb = G.as_bytes(x)
    esize = 2 if kind == "bf16" else 1
    for (a0, a1), o, size in zip(hs.segs, hs.offsets, hs.sizes):
        want = orc.encode(ODT[kind], np.array(cb, dtype=np.uint8), xb[a0 * esize:a1 * esize])
        assert size == want.size
        assert np.array_equal(hs.host[o:o + size].numpy(), want)
    y = torch.full_like(x.view(torch.uint8), 0x5A).view(x.dtype)
    pipe.reload(hs, y)
    pipe.reload_status()
    torch.cuda.synchronize()
    assert torch.equal(y.view(torch.uint8), x.view(torch.uint8))


def test_pipeline_is_reusable_and_checks_sizes():
    from lossless_kv_cache_bf16_gb300 import transfer as T

    n = 3 * 65_536 + 7
    pipe = T.Pipeline(G.DT["bf16"], CB_MID, n, "cuda", parts=2)
    for seed in (1, 2):
        x = _tensor("bf16", n, seed)
        hs = pipe.offload(x)
        y = torch.empty_like(x)
        pipe.reload(hs, y)
        torch.cuda.synchronize()
        assert torch.equal(y.view(torch.uint8), x.view(torch.uint8))
    with pytest.raises(ValueError):
        pipe.offload(_tensor("bf16", n + 1, 3))
    with pytest.raises(ValueError):
        pipe.offload(_tensor("bf16", 2 * n, 3)[::2])


def test_encode_writes_its_size_to_pinned_host_memory():
    from lossless_kv_cache_bf16_gb300 import splitzip as S

    x = _tensor("bf16", 200_003, 5)
    n = x.numel()
    out = torch.empty(S.sz_encoded_size(S.SZ_BF16, n, n), dtype=torch.uint8, device="cuda")
    ws = torch.empty(S.sz_workspace_size(S.SZ_BF16, n), dtype=torch.uint8, device="cuda")
    dev_size = torch.zeros(1, dtype=torch.int64, device="cuda")
    host_size = torch.zeros(1, dtype=torch.int64, pin_memory=True)
    S.sz_encode(S.SZ_BF16, CB_MID, x, out, dev_size, None, ws)
    S.sz_encode(S.SZ_BF16, CB_MID, x, out, host_size, None, ws)
    torch.cuda.synchronize()
    assert int(host_size[0]) == int(dev_size.item()) > 0
    with pytest.raises(ValueError):
        S.sz_encode(S.SZ_BF16, CB_MID, x, out, torch.zeros(1, dtype=torch.int64), None, ws)


def test_packed_host_buffer_and_capacity():
    from lossless_kv_cache_bf16_gb300 import splitzip as S
    from lossless_kv_cache_bf16_gb300 import transfer as T

    n = 5 * 65_536 + 3
    x = _tensor("bf16", n, 8)
    need = T.Pipeline(G.DT["bf16"], CB_MID, n, "cuda", parts=3).offload(x).nbytes
    pipe = T.Pipeline(G.DT["bf16"], CB_MID, n, "cuda", parts=3, host_bytes=need)
    hs = pipe.offload(x)
    assert hs.nbytes == need and hs.offsets == [sum(hs.sizes[:i]) for i in range(len(hs.sizes))]
    y = torch.empty_like(x)
    pipe.reload(hs, y)
    pipe.reload_status()
    assert torch.equal(y.view(torch.uint8), x.view(torch.uint8))
    small = T.Pipeline(G.DT["bf16"], CB_MID, n, "cuda", parts=3, host_bytes=need - 1)
    with pytest.raises(S.SplitZipError) as e:
        small.offload(x)
    assert e.value.status == S.SZ_ERR_CAPACITY
