"""The codebook ablation's alternative designs (Top-8; Top-15 + sentinel) as
GPU codecs, against the oracle's codecs for the same layouts.

The GPU encoder's stream must equal the oracle's byte for byte, the GPU
decoders must restore the tensor bit for bit from the oracle's stream, and a
corrupted header must be reported, not followed.
"""
import numpy as np
import pytest
import torch

from oracle import oracle as O
from tests import gpu_codec as G

pytestmark = pytest.mark.gpu

S = None


@pytest.fixture(autouse=True)
def _lib():
    global S
    from lossless_kv_cache_bf16_gb300 import splitzip

    S = splitzip


VARIANTS = [("top8", 1), ("sentinel", 2)]   # (name, variant) shared by the library and the oracle


def _roundtrip(orc, variant, x, cb, out_offset=0, y_offset=0):
    n = x.numel()
    cap = S.sz_ablation_encoded_size(variant, n, n)
    out = torch.zeros(cap + 16, dtype=torch.uint8, device="cuda")[out_offset:out_offset + cap]
    ws = torch.empty(S.sz_ablation_workspace_size(n), dtype=torch.uint8, device="cuda")
    ob = torch.zeros(1, dtype=torch.int64, device="cuda")
    S.sz_ablation_encode(variant, cb, x, out, ob, ws)
    torch.cuda.synchronize()
    size = int(ob.item())
    xb = G.as_bytes(x)
    want = orc.abl_encode(variant, np.array(cb, dtype=np.uint8), xb)
    assert size == want.size
    assert np.array_equal(out[:size].cpu().numpy(), want)
    # Decode the oracle's stream (uploaded) with the GPU decoder.
    src = torch.zeros(want.size + 32, dtype=torch.uint8, device="cuda")[out_offset:out_offset + want.size]
    src.copy_(torch.from_numpy(want))
    yb = torch.full((2 * n + 64,), 0x5A, dtype=torch.uint8, device="cuda")
    y = yb[2 * y_offset: 2 * y_offset + 2 * n]
    st = torch.full((1,), -1, dtype=torch.int32, device="cuda")
    S.sz_ablation_decode(variant, src, want.size, n, y, st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    assert np.array_equal(y.cpu().numpy(), xb)
    assert bool((yb[: 2 * y_offset] == 0x5A).all()) and bool((yb[2 * y_offset + 2 * n:] == 0x5A).all())
    return want


def _bf16(n, seed):
    g = torch.Generator(device="cuda")
    g.manual_seed(seed)
    return (torch.randn(n, generator=g, device="cuda") * 40).to(torch.bfloat16)


@pytest.mark.parametrize("name,variant", VARIANTS)
@pytest.mark.parametrize("n", [1, 7, 8, 8193, 65_536, 65_537, 3 * 65_536 + 5, 400_000])
def test_ablation_codecs_match_oracle(orc, name, variant, n):
    x = _bf16(n, seed=n)
    cb = S.sz_ablation_codebook(variant, orc.histogram(O.BF16, G.as_bytes(x)))
    _roundtrip(orc, variant, x, cb)


@pytest.mark.parametrize("name,variant", VARIANTS)
def test_ablation_codecs_every_pattern(orc, name, variant):
    x = torch.arange(65536, dtype=torch.int32, device="cuda").to(torch.int16).view(torch.bfloat16)
    k = 8 if variant == 1 else 15
    rng = np.random.default_rng(variant)
    for cb in (list(range(120, 120 + k)), sorted(rng.choice(256, k, replace=False).tolist())):
        s = _roundtrip(orc, variant, x, cb)
        assert s.size == (280592 if variant == 1 else 160023)
    perm = torch.cat([torch.randperm(65536, device="cuda") for _ in range(3)])
    _roundtrip(orc, variant, x[perm].contiguous(), list(range(100, 100 + k)))


@pytest.mark.parametrize("name,variant", VARIANTS)
def test_ablation_codecs_unaligned(orc, name, variant):
    x = _bf16(2 * 65_536 + 77, seed=3)[1:]
    cb = S.sz_ablation_codebook(variant, orc.histogram(O.BF16, G.as_bytes(x)))
    _roundtrip(orc, variant, x, cb, out_offset=3, y_offset=1)


@pytest.mark.parametrize("name,variant", VARIANTS)
def test_ablation_decoders_reject_a_bad_header(orc, name, variant):
    x = _bf16(3 * 65_536, seed=9)
    n = x.numel()
    xb = G.as_bytes(x)
    cb = S.sz_ablation_codebook(variant, orc.histogram(O.BF16, xb))
    s = orc.abl_encode(variant, np.array(cb, dtype=np.uint8), xb)
    k = 8 if variant == 1 else 15
    dense = n + (3 * ((n + 7) // 8) if variant == 1 else (n + 1) // 2)
    for field in (4, 8 + 4):           # chunk 0's count, chunk 1's count
        bad = s.copy()
        bad[dense + k + field] ^= 1
        assert orc.abl_decode(variant, bad, n)[0] == O.CORRUPT
        src = torch.from_numpy(bad).cuda()
        y = torch.empty(2 * n, dtype=torch.uint8, device="cuda")
        st = torch.zeros(1, dtype=torch.int32, device="cuda")
        S.sz_ablation_decode(variant, src, bad.size, n, y, st)
        torch.cuda.synchronize()
        assert int(st.item()) == S.SZ_ERR_CORRUPT
