"""Shard streams joined into the stream of the whole tensor (GPU).

A tensor cut into shards of whole 65,536-element chunks is encoded shard by
shard; sz_concat must then give, byte for byte, the oracle's stream of the
whole tensor, and that stream must decode bit-exactly.  The oracle's own shard
streams are joined too, so the join is checked apart from the GPU encoder.
"""
import numpy as np
import pytest
import torch

from oracle import oracle as O
from tests import gpu_codec as G
from tests.oracle_pins import CB_E5_MID, CB_MID

pytestmark = pytest.mark.gpu

ODT = {"bf16": O.BF16, "e5m2": O.E5M2}
CB = {"bf16": CB_MID, "e5m2": CB_E5_MID}
C = 65536


def _tensor(kind, n, seed):
    g = torch.Generator(device="cuda")
    g.manual_seed(seed)
    x = torch.randn(n, generator=g, device="cuda") * 30
    if kind == "bf16":
        return x.to(torch.bfloat16)
    return x.to(torch.float8_e5m2).view(torch.uint8)


def _join(kind, streams, sizes, ns, n_total):
    from lossless_kv_cache_bf16_gb300 import splitzip as S

    dt = G.DT[kind]
    out = torch.full((S.sz_encoded_size(dt, n_total, n_total),), 0xA5, dtype=torch.uint8, device="cuda")
    st = torch.full((1,), -1, dtype=torch.int32, device="cuda")
    total = S.sz_concat(dt, streams, sizes, ns, out, st)
    torch.cuda.synchronize()
    return out, total, int(st.item())


SPLITS = [
    [C, 2 * C, 2 * C + 123],         # ragged last shard
    [0, 3 * C + 5],                  # an empty shard first
    [4 * C + 1],                     # one shard: a copy
    [C] * 70 + [77],                 # more shards than one header launch takes
    [2 * C, 0, C, 0],                # empty shards in the middle and at the end
    [2 * C + 5, 0, 0],               # a ragged shard followed by empty ones
]


@pytest.mark.parametrize("kind", ["bf16", "e5m2"])
@pytest.mark.parametrize("split", range(len(SPLITS)))
def test_joined_gpu_shards_equal_the_whole_stream(orc, kind, split):
    from lossless_kv_cache_bf16_gb300 import splitzip as S

    dt, ns = G.DT[kind], SPLITS[split]
    n = sum(ns)
    x = _tensor(kind, n, 40 + split)
    want = orc.encode(ODT[kind], CB[kind], G.as_bytes(x))
    streams, sizes, at = [], [], 0
    for m in ns:
        out = torch.empty(S.sz_encoded_size(dt, m, m), dtype=torch.uint8, device="cuda")
        ws = torch.empty(S.sz_workspace_size(dt, m), dtype=torch.uint8, device="cuda")
        ob = torch.zeros(1, dtype=torch.int64, device="cuda")
        st = torch.full((1,), -1, dtype=torch.int32, device="cuda")
        S.sz_encode(dt, CB[kind], x[at:at + m], out, ob, st, ws)
        torch.cuda.synchronize()
        assert int(st.item()) == 0
        streams.append(out)
        sizes.append(int(ob.item()))
        at += m
    out, total, st = _join(kind, streams, sizes, ns, n)
    assert st == 0 and total == want.size
    assert np.array_equal(out[:total].cpu().numpy(), want)
    y = torch.empty_like(x)
    dst = torch.full((1,), -1, dtype=torch.int32, device="cuda")
    S.sz_decode(dt, out, total, n, y, dst)
    torch.cuda.synchronize()
    assert int(dst.item()) == 0 and torch.equal(y.view(torch.uint8), x.view(torch.uint8))


@pytest.mark.parametrize("kind", ["bf16", "e5m2"])
def test_joined_oracle_shards_equal_the_whole_stream(orc, kind):
    ns = [3 * C, C, 5 * C + 999]
    n = sum(ns)
    x = _tensor(kind, n, 77)
    xb = G.as_bytes(x)
    esize = 2 if kind == "bf16" else 1
    parts, at = [], 0
    for m in ns:
        parts.append(orc.encode(ODT[kind], CB[kind], xb[at * esize:(at + m) * esize]))
        at += m
    streams = [torch.from_numpy(p).cuda() for p in parts]
    out, total, st = _join(kind, streams, [p.size for p in parts], ns, n)
    want = orc.encode(ODT[kind], CB[kind], xb)
    assert st == 0 and total == want.size
    assert np.array_equal(out[:total].cpu().numpy(), want)
    assert np.all(out[total:].cpu().numpy() == 0xA5)  # nothing written past the stream


@pytest.mark.parametrize("kind", ["bf16", "e5m2"])
def test_a_shard_with_another_codebook_is_reported(orc, kind):
    from lossless_kv_cache_bf16_gb300 import splitzip as S

    ns = [C, C + 3]
    x = _tensor(kind, sum(ns), 5)
    xb = G.as_bytes(x)
    esize = 2 if kind == "bf16" else 1
    other = np.array(CB[kind], dtype=np.uint8) + 1
    parts = [orc.encode(ODT[kind], CB[kind], xb[: C * esize]), orc.encode(ODT[kind], other, xb[C * esize:])]
    streams = [torch.from_numpy(p).cuda() for p in parts]
    _, _, st = _join(kind, streams, [p.size for p in parts], ns, sum(ns))
    assert st == S.SZ_ERR_INVALID_ARG
