"""sz_encode_noalloc: the encode entry point that allocates nothing (GPU).

Some callers cannot allocate device memory -- a serving engine that has given
nearly all of it to its KV-cache pool, or a latency-critical path that must
not take cudaMalloc's implicit synchronisation -- so they cannot hand
sz_encode a workspace.  sz_encode_noalloc uses a static scratch array inside
the library instead.  Its output must be the oracle's stream and sz_encode's
exactly (the codec is integer bit manipulation: tolerance zero), on two calls
in a row, so the second call must not see what the first left in the shared
scratch.  The scratch stages fewer escape records per scan tile (256) than
sz_encode's workspace (2,048 for BF16, 1,024 for E5M2), so inputs are
chosen to put scan tiles between 257 and the workspace's limit (where only
the no-alloc path re-derives records) and above it (where both do).
"""
import ctypes

import numpy as np
import pytest
import torch

from oracle import oracle as O
from lossless_kv_cache_bf16_gb300 import splitzip as S
from tests.oracle_pins import CB_E5_MID, CB_MID
from tests.test_gpu_max_size import _chunk_checks

pytestmark = pytest.mark.gpu

SCAN_TILE = 32768
NOALLOC_STAGED = 256      # escape records the static scratch stages per scan tile
WS_STAGED = {"bf16": 2048, "e5m2": 1024}  # ... and sz_encode's workspace
NOALLOC_MAX = 1 << 28     # elements the static scratch covers


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


def _with_escape_rate(kind, n, p, seed):
    """Elements whose exponent lies outside the codebook with probability p
    (inside it otherwise); sign and mantissa bits random."""
    g = torch.Generator(device="cuda")
    g.manual_seed(seed)
    esc = torch.rand(n, generator=g, device="cuda") < p
    r = torch.randint(0, 1 << 16, (n,), generator=g, device="cuda", dtype=torch.int32)
    if kind == "bf16":
        inside = torch.randint(120, 136, (n,), generator=g, device="cuda", dtype=torch.int32)
        outside = torch.randint(0, 110, (n,), generator=g, device="cuda", dtype=torch.int32)
        e = torch.where(esc, outside, inside)
        return ((r & 0x807F) | (e << 7)).to(torch.int16).view(torch.bfloat16)
    inside = torch.randint(14, 30, (n,), generator=g, device="cuda", dtype=torch.int32)
    outside = torch.randint(0, 14, (n,), generator=g, device="cuda", dtype=torch.int32)
    e = torch.where(esc, outside, inside)
    return ((r & 0x83) | (e << 2)).to(torch.uint8)


def _scan_tile_escapes(kind, cb, xh):
    """Escapes per 32,768-element scan tile, counted on the host."""
    if kind == "bf16":
        exps = (xh.view(np.uint16) >> 7) & 0xFF
    else:
        exps = (xh >> 2) & 0x1F
    esc = ~np.isin(exps, np.array(cb, dtype=exps.dtype))
    tiles = (esc.size + SCAN_TILE - 1) // SCAN_TILE
    padded = np.zeros(tiles * SCAN_TILE, dtype=np.int64)
    padded[: esc.size] = esc
    return padded.reshape(tiles, SCAN_TILE).sum(axis=1)


def _cases():
    n = 9 * 65536 + 4321                            # many scan tiles, a partial chunk
    return [
        ("bf16", CB_MID, _with_escape_rate("bf16", n, 0.02, 71), "band"),      # ~655 per scan tile
        ("bf16", CB_MID, _with_escape_rate("bf16", n, 0.1, 72), "heavy"),      # ~3,277 per scan tile
        ("e5m2", CB_E5_MID, _with_escape_rate("e5m2", 3 * 65536 + 99, 0.02, 73), "band"),
        ("e5m2", CB_E5_MID, _with_escape_rate("e5m2", 3 * 65536 + 99, 0.5, 74), "heavy"),
    ]


def test_noalloc_matches_oracle_and_sz_encode_on_two_calls_in_a_row(orc):
    cases = _cases()
    wants = []
    for kind, cb, x, band in cases:
        xh = x.view(torch.uint8).reshape(-1).cpu().numpy()
        per_tile = _scan_tile_escapes(kind, cb, xh)
        full = per_tile[: xh.size // (2 if kind == "bf16" else 1) // SCAN_TILE]
        if band == "band":
            # Every whole scan tile lies in the band where only the no-alloc
            # path re-derives records from the input.
            assert full.min() > NOALLOC_STAGED and full.max() <= WS_STAGED[kind], (full.min(), full.max())
        else:
            assert full.min() > WS_STAGED[kind]
        wants.append(orc.encode(O.BF16 if kind == "bf16" else O.E5M2, np.array(cb, dtype=np.uint8), xh))
    # Two passes over all cases: consecutive calls share the static scratch,
    # and each call follows one on a different input.
    for _ in range(2):
        for (kind, cb, x, _), want in zip(cases, wants):
            dt = S.SZ_BF16 if kind == "bf16" else S.SZ_FP8_E5M2
            got, st = _encode_noalloc(dt, cb, x)
            ref, st_ref = _encode_with_workspace(dt, cb, x)
            assert st == 0 and st_ref == 0
            assert np.array_equal(got, want), f"{kind}: no-alloc stream differs from the oracle"
            assert np.array_equal(ref, want), f"{kind}: sz_encode stream differs from the oracle"


def test_noalloc_at_its_largest_size(orc):
    """n = 2^28 BF16 elements, the most the static scratch covers, at a 2%
    escape rate: equal to sz_encode's stream on the device, and to the
    oracle's on sampled chunks (each encoded by the oracle on its own),
    with headers that are running sums and the closed-form size."""
    n = NOALLOC_MAX
    x = _with_escape_rate("bf16", n, 0.02, 75)
    cap = S.sz_encoded_size(S.SZ_BF16, n, n)
    ob = torch.zeros(1, dtype=torch.int64, device="cuda")
    st = torch.full((1,), -1, dtype=torch.int32, device="cuda")
    out = torch.empty(cap, dtype=torch.uint8, device="cuda")
    S.sz_encode_noalloc(S.SZ_BF16, CB_MID, x, out, ob, st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    size = int(ob.item())
    n_esc = (size - S.sz_encoded_size(S.SZ_BF16, n, 0)) // 3
    assert size == orc.encoded_size(O.BF16, n, n_esc)
    ref = torch.empty(cap, dtype=torch.uint8, device="cuda")
    ws = torch.empty(S.sz_workspace_size(S.SZ_BF16, n), dtype=torch.uint8, device="cuda")
    S.sz_encode(S.SZ_BF16, CB_MID, x, ref, ob, st, ws)
    torch.cuda.synchronize()
    assert int(st.item()) == 0 and int(ob.item()) == size
    assert torch.equal(out[:size], ref[:size])
    del ref, ws
    _chunk_checks(orc, O.BF16, CB_MID, x, out, n, n_esc)


def test_noalloc_rejects_sizes_beyond_its_scratch():
    """The C entry point refuses n above 2^28 before it launches anything
    (called directly: the binding would refuse an n beyond the tensor first)."""
    x = torch.zeros(16, dtype=torch.bfloat16, device="cuda")
    out = torch.zeros(64, dtype=torch.uint8, device="cuda")
    ob = torch.zeros(1, dtype=torch.int64, device="cuda")
    cb = S._codebook(CB_MID)
    for too_many in (NOALLOC_MAX + 1, 1 << 31):
        rc = S.LIB.sz_encode_noalloc(S.SZ_BF16, ctypes.byref(cb), x.data_ptr(), too_many, out.data_ptr(),
                                     out.numel(), ob.data_ptr(), None, None)
        assert rc == S.SZ_ERR_CAPACITY
