"""Paged KV tensors: encode straight from a page pool through a block table,
decode straight back into the pages.

The logical tensor (pages gathered in block-table order) is built on the
host side of the test and encoded by the oracle; the paged encode must give
that stream byte for byte, and the paged decode must fill exactly the named
pages with the logical tensor's bytes, leaving every other byte of the pool
untouched.
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


CANARY = 0xA5


def _pool(kind, pages, page_elems, seed):
    g = torch.Generator(device="cuda")
    g.manual_seed(seed)
    if kind == "bf16":
        return (torch.randn(pages * page_elems, generator=g, device="cuda") * 20).to(torch.bfloat16)
    return torch.randint(0, 256, (pages * page_elems,), generator=g, device="cuda", dtype=torch.uint8)


def _case(kind, page_elems, used, tail, seed):
    pages = used + 3                                   # pages the table does not name
    pool = _pool(kind, pages, page_elems, seed)
    g = torch.Generator(device="cpu")
    g.manual_seed(seed + 1)
    ids = torch.randperm(pages, generator=g)[:used].to(torch.int32)
    n = used * page_elems - tail
    logical = pool.view(pages, page_elems)[ids.long().cuda()].reshape(-1)[:n].contiguous()
    return pool, ids.cuda(), n, logical


@pytest.mark.parametrize("kind,cb", [("bf16", CB_MID), ("bf16", CB_EDGES), ("e5m2", CB_E5_MID), ("e5m2", CB_E5_EDGES)])
@pytest.mark.parametrize("page_elems,used,tail", [(16, 700, 3), (1024, 40, 0), (1024, 37, 511), (16384, 9, 5),
                                                  (65536, 2, 1)])
def test_paged_roundtrip_matches_oracle(orc, kind, cb, page_elems, used, tail):
    dt = S.SZ_BF16 if kind == "bf16" else S.SZ_FP8_E5M2
    odt = O.BF16 if kind == "bf16" else O.E5M2
    pool, ids, n, logical = _case(kind, page_elems, used, tail, seed=page_elems + used)
    out = torch.empty(S.sz_encoded_size(dt, n, n), dtype=torch.uint8, device="cuda")
    ws = torch.empty(S.sz_workspace_size(dt, n), dtype=torch.uint8, device="cuda")
    ob = torch.zeros(1, dtype=torch.int64, device="cuda")
    st = torch.full((1,), -1, dtype=torch.int32, device="cuda")
    S.sz_encode_paged(dt, cb, pool, page_elems, ids, n, out, ob, st, ws)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    size = int(ob.item())
    want = orc.encode(odt, np.array(cb, dtype=np.uint8), G.as_bytes(logical))
    assert np.array_equal(out[:size].cpu().numpy(), want)

    # Decode into a pool of canary bytes: exactly the named elements change.
    target = torch.full_like(pool.view(torch.uint8), CANARY).view(pool.dtype)
    S.sz_decode_paged(dt, out, size, n, target, page_elems, ids, st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    tv = target.view(-1, page_elems)
    got = tv[ids.long()].reshape(-1)[:n]
    assert torch.equal(got.view(torch.uint8), logical.view(torch.uint8))
    mask = torch.ones(tv.shape[0], dtype=torch.bool, device="cuda")
    mask[ids.long()] = False
    untouched = tv[mask].view(torch.uint8)
    assert bool((untouched == CANARY).all())
    if tail:
        last = tv[ids[-1].long()][page_elems - tail:].contiguous().view(torch.uint8)
        assert bool((last == CANARY).all())


@pytest.mark.parametrize("kind", ["bf16", "e5m2"])
def test_paged_bad_page_id_is_reported(kind):
    dt = S.SZ_BF16 if kind == "bf16" else S.SZ_FP8_E5M2
    page_elems, used = 1024, 12
    pool, ids, n, _ = _case(kind, page_elems, used, 0, seed=3)
    ids[5] = pool.numel() // page_elems  # one past the pool
    out = torch.empty(S.sz_encoded_size(dt, n, n), dtype=torch.uint8, device="cuda")
    ws = torch.empty(S.sz_workspace_size(dt, n), dtype=torch.uint8, device="cuda")
    ob = torch.zeros(1, dtype=torch.int64, device="cuda")
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    S.sz_encode_paged(dt, CB_MID if kind == "bf16" else CB_E5_MID, pool, page_elems, ids, n, out, ob, st, ws)
    torch.cuda.synchronize()
    assert int(st.item()) == S.SZ_ERR_INVALID_ARG
    size = int(ob.item())
    S.sz_decode_paged(dt, out, size, n, pool, page_elems, ids, st)
    torch.cuda.synchronize()
    assert int(st.item()) == S.SZ_ERR_INVALID_ARG


def test_paged_host_checks():
    dt = S.SZ_BF16
    pool = torch.zeros(4096, dtype=torch.bfloat16, device="cuda")
    ids = torch.zeros(4, dtype=torch.int32, device="cuda")
    out = torch.empty(S.sz_encoded_size(dt, 4096, 4096), dtype=torch.uint8, device="cuda")
    ws = torch.empty(S.sz_workspace_size(dt, 4096), dtype=torch.uint8, device="cuda")
    ob = torch.zeros(1, dtype=torch.int64, device="cuda")
    for page_elems in (8, 1000, 0):                       # too small, not a power of two, zero
        with pytest.raises(S.SplitZipError):
            S.sz_encode_paged(dt, CB_MID, pool, page_elems, ids, 4096 if page_elems else 0, out, ob, None, ws)
    with pytest.raises(S.SplitZipError):                  # pool not 16-byte aligned
        S.sz_encode_paged(dt, CB_MID, pool[1:], 1024, ids, 2048, out, ob, None, ws)
