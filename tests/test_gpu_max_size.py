"""The largest tensor the format allows: n = 2^32 - 1 elements (BF16 with every
element an escape, so that record indices run up to 2^32 - 1 and byte
offsets pass 2^34; E5M2 with random bytes).  The oracle cannot hold these
streams comfortably, so parity is checked on sampled chunks, each encoded by
the oracle on its own, and through properties that hold at any size: the
closed-form size, headers that are running sums, and a bit-exact GPU round
trip."""
import numpy as np
import pytest
import torch

from oracle import oracle as O

pytestmark = pytest.mark.gpu

N_MAX = (1 << 32) - 1
CHUNK = 65536


def _chunk_checks(orc, odt, cb, x, out, n, n_esc):
    dense = orc.dense_bytes(odt, n)
    chunks = orc.num_chunks(n)
    hdr, rec = dense + 16, dense + 16 + 8 * chunks
    cb_dev = out[dense:dense + 16].cpu().numpy()
    assert cb_dev.tolist() == [int(v) for v in cb]
    # Headers: one read of all of them (512 KB), checked as running sums.
    h = out[hdr:hdr + 8 * chunks].cpu().numpy().view(np.uint32).reshape(chunks, 2).astype(np.uint64)
    assert h[0, 0] == 0 and np.array_equal(h[1:, 0], np.cumsum(h[:-1, 1])) and int(h[-1, 0] + h[-1, 1]) == n_esc
    for c in (0, 1, chunks // 2, chunks - 3, chunks - 2, chunks - 1):
        lo, hi = c * CHUNK, min(n, (c + 1) * CHUNK)
        xb = x[lo:hi].contiguous().view(torch.uint8).cpu().numpy()
        want = orc.encode(odt, np.array(cb, dtype=np.uint8), xb)   # the chunk as a stream of its own
        m = hi - lo
        w_dense = orc.dense_bytes(odt, m)
        count = int(h[c, 1])
        assert count == (want.size - orc.encoded_size(odt, m, 0)) // 3
        if odt == O.BF16:
            got_sm = out[lo:hi].cpu().numpy()
            got_nib = out[n + lo // 2:n + lo // 2 + (m + 1) // 2].cpu().numpy()
            assert np.array_equal(got_sm, want[:m]) and np.array_equal(got_nib, want[m:w_dense])
        else:
            p0 = 7 * (lo // 8)
            got = out[p0:p0 + w_dense].cpu().numpy()
            assert np.array_equal(got, want[:w_dense])
        r0 = rec + 3 * int(h[c, 0])
        got_rec = out[r0:r0 + 3 * count].cpu().numpy()
        assert np.array_equal(got_rec, want[w_dense + 16 + 8:])


@pytest.mark.parametrize("kind", ["bf16", "e5m2"])
def test_largest_tensor(orc, kind):
    from lossless_kv_cache_bf16_gb300 import splitzip as S

    n = N_MAX
    g = torch.Generator(device="cuda")
    g.manual_seed(41)
    if kind == "bf16":
        dt, odt = S.SZ_BF16, O.BF16
        cb = list(range(16))                       # exponents 0..15
        # Random patterns with exponent bit 4 set: every exponent is >= 16,
        # so every element is an escape.
        x = torch.randint(-32768, 32767, (n,), generator=g, device="cuda", dtype=torch.int16)
        x.bitwise_or_(0x0800)
        x = x.view(torch.bfloat16)
        n_esc = n
    else:
        dt, odt = S.SZ_FP8_E5M2, O.E5M2
        cb = list(range(8, 24))
        x = torch.randint(0, 256, (n,), generator=g, device="cuda", dtype=torch.uint8)
        n_esc = None
    cap = S.sz_encoded_size(dt, n, n)
    out = torch.empty(cap, dtype=torch.uint8, device="cuda")
    ws = torch.empty(S.sz_workspace_size(dt, n), dtype=torch.uint8, device="cuda")
    size = torch.zeros(1, dtype=torch.int64, device="cuda")
    st = torch.full((1,), -1, dtype=torch.int32, device="cuda")
    S.sz_encode(dt, cb, x, out, size, st, ws)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    s = int(size.item())
    if n_esc is None:
        n_esc = (s - S.sz_encoded_size(dt, n, 0)) // 3
    assert s == orc.encoded_size(odt, n, n_esc)
    del ws
    _chunk_checks(orc, odt, cb, x, out, n, n_esc)
    y = torch.empty_like(x)
    S.sz_decode(dt, out, s, n, y, st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    assert torch.equal(y.view(torch.uint8), x.view(torch.uint8))
