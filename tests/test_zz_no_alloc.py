"""sz_encode_noalloc: the encode entry point that allocates nothing (GPU).

Some callers cannot allocate device memory -- a serving engine that has given
nearly all of it to its KV-cache pool, or a latency-critical path that must
not take cudaMalloc's implicit synchronisation -- so they cannot hand
sz_encode a workspace.  sz_encode_noalloc uses a static scratch array inside
the library instead.  Its output must match sz_encode's exactly (the codec is
integer bit manipulation: tolerance zero), on two calls in a row, so the
second call must not see what the first left in the shared scratch.
"""
import numpy as np
import pytest
import torch

from lossless_kv_cache_bf16_gb300 import splitzip as S
from tests.oracle_pins import CB_E5_MID, CB_MID

pytestmark = pytest.mark.gpu


def _encode_with_workspace(dt, cb, x):
    n = x.numel() * x.element_size() // S.ELEMENT_BYTES[dt]
    out = torch.zeros(S.sz_encoded_size(dt, n, n), dtype=torch.uint8, device="cuda")
    ws = torch.empty(S.sz_workspace_size(dt, n), dtype=torch.uint8, device="cuda")
    ob = torch.zeros(1, dtype=torch.int64, device="cuda")
    st = torch.full((1,), -1, dtype=torch.int32, device="cuda")
    S.sz_encode(dt, cb, x, out, ob, st, ws)
    torch.cuda.synchronize()
    return out[: int(ob.item())].cpu().numpy(), int(st.item())


def _encode_noalloc(dt, cb, x):
    n = x.numel() * x.element_size() // S.ELEMENT_BYTES[dt]
    out = torch.zeros(S.sz_encoded_size(dt, n, n), dtype=torch.uint8, device="cuda")
    ob = torch.zeros(1, dtype=torch.int64, device="cuda")
    st = torch.full((1,), -1, dtype=torch.int32, device="cuda")
    S.sz_encode_noalloc(dt, cb, x, out, ob, st)
    torch.cuda.synchronize()
    return out[: int(ob.item())].cpu().numpy(), int(st.item())


def _inputs():
    g = torch.Generator(device="cuda")
    g.manual_seed(77)
    n1 = 9 * 65536 + 4321                     # many tiles, a partial chunk, escapes
    s = torch.exp(2 * torch.randn(n1, generator=g, device="cuda"))
    a = (torch.randn(n1, generator=g, device="cuda") * s).to(torch.bfloat16)
    b = torch.randint(0, 256, (3 * 65536 + 99,), generator=g, device="cuda", dtype=torch.uint8)
    return a, b


def test_noalloc_matches_sz_encode_on_two_calls_in_a_row():
    a, b = _inputs()
    cases = [(S.SZ_BF16, CB_MID, a), (S.SZ_FP8_E5M2, CB_E5_MID, b)]
    for dt, cb, x in cases:                  # two calls in a row on the shared scratch
        want, st_w = _encode_with_workspace(dt, cb, x)
        got, st_g = _encode_noalloc(dt, cb, x)
        assert st_w == 0 and st_g == 0
        assert got.size == want.size and np.array_equal(got, want)
    # Once more, the same input as the first call, after a different one.
    want, _ = _encode_with_workspace(S.SZ_BF16, CB_MID, a)
    got, st = _encode_noalloc(S.SZ_BF16, CB_MID, a)
    assert st == 0 and np.array_equal(got, want)


def test_noalloc_rejects_sizes_beyond_its_scratch():
    x = torch.zeros(16, dtype=torch.bfloat16, device="cuda")
    out = torch.zeros(64, dtype=torch.uint8, device="cuda")
    ob = torch.zeros(1, dtype=torch.int64, device="cuda")
    too_many = (1 << 28) + 1                  # the static scratch covers 2^28 elements
    with pytest.raises(S.SplitZipError) as e:
        S.sz_encode_noalloc(S.SZ_BF16, CB_MID, x, out, ob, None, n=too_many)
    assert e.value.status == S.SZ_ERR_CAPACITY
