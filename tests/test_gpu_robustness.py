"""Corrupted streams, capacity limits and the bounded inter-block wait (GPU).

A corrupted stream must give SZ_ERR_CORRUPT exactly when the oracle's
validator rejects it, and decode must never write outside its output.  The
encode's waits are bounded: a test hook never issues one input copy, and the
wait for it must end in SZ_ERR_TIMEOUT with the CUDA context still usable.
Nothing here faults, traps or hangs the GPU.
"""
import time

import numpy as np
import pytest
import torch

from lossless_kv_cache_bf16_gb300 import splitzip as S
from oracle import oracle as O
from tests import gpu_codec as G
from tests.oracle_pins import CB_E5_MID, CB_MID

pytestmark = pytest.mark.gpu


def _stream(orc, n=2 * 65536 + 300, seed=31):
    rng = np.random.default_rng(seed)
    v = (rng.standard_normal(n) * np.exp(2 * rng.standard_normal(n))).astype(np.float32)
    x = (v.view(np.uint32) >> 16).astype(np.uint16)
    return x, orc.encode(O.BF16, CB_MID, x)


def _check_same_verdict(orc, dt_o, dt_g, stream, n):
    want, _ = orc.validate(dt_o, stream, n)
    try:
        st, y, guard_ok = G.decode(dt_g, stream, n)
    except S.SplitZipError as e:  # rejected on the host before any launch
        st, guard_ok = e.status, True
    assert guard_ok, "decode wrote outside its output"
    assert (st == S.SZ_OK) == (want == O.OK), f"oracle {want}, gpu {st}"
    if want != O.OK:
        assert st == S.SZ_ERR_CORRUPT


def test_targeted_corruptions(orc):
    x, s = _stream(orc)
    n = x.size
    dense = n + (n + 1) // 2
    hdr, rec = dense + 16, dense + 16 + 8 * 3
    cases = {
        "truncated byte": s[:-1],
        "missing record": s[:-3],
        "extra record": np.concatenate([s, s[-3:]]),
        "repeated codebook entry": np.concatenate([s[:dense + 1], s[dense:dense + 1], s[dense + 2:]]),
    }
    t = s.copy(); t[hdr + 8] ^= 1; cases["offset not a running sum"] = t
    t = s.copy(); t[rec:rec + 3], t[rec + 3:rec + 6] = s[rec + 3:rec + 6].copy(), s[rec:rec + 3].copy(); cases["positions out of order"] = t
    t = s.copy(); t[-3:-1] = 0xFF; cases["position past the chunk end"] = t
    t = s.copy(); t[hdr + 20:hdr + 24] = [0xFF, 0xFF, 0, 0]; cases["count larger than the chunk"] = t
    for name, stream in cases.items():
        _check_same_verdict(orc, O.BF16, S.SZ_BF16, stream, n)


def test_fuzzed_metadata_bf16(orc):
    x, s = _stream(orc, seed=32)
    n = x.size
    meta = n + (n + 1) // 2       # codebook, headers and records
    rng = np.random.default_rng(33)
    for trial in range(60):
        t = s.copy()
        for _ in range(rng.integers(1, 4)):
            i = int(rng.integers(meta, t.size))
            t[i] = rng.integers(0, 256)
        _check_same_verdict(orc, O.BF16, S.SZ_BF16, t, n)


def test_fuzzed_metadata_e5m2(orc):
    rng = np.random.default_rng(34)
    n = 3 * 65536 + 17
    x = rng.integers(0, 256, n, dtype=np.uint8)
    s = orc.encode(O.E5M2, CB_E5_MID, x)
    meta = 7 * ((n + 7) // 8)
    for trial in range(60):
        t = s.copy()
        for _ in range(rng.integers(1, 4)):
            i = int(rng.integers(meta, t.size))
            t[i] = rng.integers(0, 256)
        _check_same_verdict(orc, O.E5M2, S.SZ_FP8_E5M2, t, n)


@pytest.mark.parametrize("kind", ["bf16", "e5m2"])
def test_fuzzed_metadata_dense_escapes_many_blocks(orc, kind):
    # Uniformly random patterns (most of them escapes) over more tiles than
    # the decoder has blocks, so that blocks start inside chunks and walk
    # their records through several windows; corrupted headers and records
    # make the walk jump.
    rng = np.random.default_rng(36 if kind == "bf16" else 37)
    if kind == "bf16":
        n = 6_000_000 + 77
        x = rng.integers(0, 1 << 16, n, dtype=np.uint16)
        dt_o, dt_g, cb, dense = O.BF16, S.SZ_BF16, CB_MID, n + (n + 1) // 2
    else:
        n = 12_000_000 + 5
        x = rng.integers(0, 256, n, dtype=np.uint8)
        dt_o, dt_g, cb, dense = O.E5M2, S.SZ_FP8_E5M2, CB_E5_MID, 7 * ((n + 7) // 8)
    s = orc.encode(dt_o, cb, x)
    chunks = -(-n // 65536)
    hdr, rec = dense + 16, dense + 16 + 8 * chunks
    st, y, guard_ok = G.decode(dt_g, s, n)
    assert st == 0 and guard_ok and np.array_equal(y, x.view(np.uint8))
    for trial in range(12):
        t = s.copy()
        region = (hdr, rec) if trial % 2 == 0 else (rec, t.size)
        for _ in range(rng.integers(1, 3)):
            t[int(rng.integers(*region))] = rng.integers(0, 256)
        _check_same_verdict(orc, dt_o, dt_g, t, n)


def test_valid_stream_decodes_clean(orc):
    x, s = _stream(orc, seed=35)
    st, y, guard_ok = G.decode(S.SZ_BF16, s, x.size)
    assert st == 0 and guard_ok and np.array_equal(y, x.view(np.uint8))


def test_host_rejects_bad_arguments():
    x = torch.zeros(1000, dtype=torch.bfloat16, device="cuda")
    out = torch.empty(S.sz_encoded_size(S.SZ_BF16, 1000, 1000), dtype=torch.uint8, device="cuda")
    ws = torch.empty(S.sz_workspace_size(S.SZ_BF16, 1000), dtype=torch.uint8, device="cuda")
    ob = torch.zeros(1, dtype=torch.int64, device="cuda")
    bad = list(CB_MID)
    bad[0] = bad[1]
    with pytest.raises(S.SplitZipError) as e:
        S.sz_encode(S.SZ_BF16, bad, x, out, ob, None, ws)
    assert e.value.status == S.SZ_ERR_INVALID_ARG
    with pytest.raises(S.SplitZipError) as e:
        S.sz_encode(S.SZ_BF16, CB_MID, x, out[:100], ob, None, ws)
    assert e.value.status == S.SZ_ERR_CAPACITY
    with pytest.raises(S.SplitZipError) as e:
        S.sz_encode(S.SZ_BF16, CB_MID, x, out, ob, None, ws[:8])
    assert e.value.status == S.SZ_ERR_CAPACITY
    with pytest.raises(S.SplitZipError) as e:
        S.sz_encode(S.SZ_FP8_E5M2, CB_MID, x, out, ob, None, ws)   # 120..135 do not fit 5 bits
    assert e.value.status == S.SZ_ERR_INVALID_ARG


def test_stall_hook_refuses_e5m2():
    x = torch.zeros(64, dtype=torch.uint8, device="cuda")
    out = torch.empty(S.sz_encoded_size(S.SZ_FP8_E5M2, 64, 64), dtype=torch.uint8, device="cuda")
    ws = torch.empty(S.sz_workspace_size(S.SZ_FP8_E5M2, 64), dtype=torch.uint8, device="cuda")
    ob = torch.zeros(1, dtype=torch.int64, device="cuda")
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    with pytest.raises(S.SplitZipError) as e:
        S.sz_debug_encode_stalled(S.SZ_FP8_E5M2, CB_E5_MID, x, out, ob, st, ws, wait_limit_ns=1000)
    assert e.value.status == S.SZ_ERR_UNSUPPORTED


def test_stalled_wait_times_out(orc):
    n = 5 * 32768 + 7
    x = (torch.randn(n, device="cuda") * 100).to(torch.bfloat16)
    out = torch.empty(S.sz_encoded_size(S.SZ_BF16, n, n), dtype=torch.uint8, device="cuda")
    ws = torch.empty(S.sz_workspace_size(S.SZ_BF16, n), dtype=torch.uint8, device="cuda")
    ob = torch.zeros(1, dtype=torch.int64, device="cuda")
    st = torch.full((1,), -1, dtype=torch.int32, device="cuda")
    torch.cuda.synchronize()
    t0 = time.time()
    S.sz_debug_encode_stalled(S.SZ_BF16, CB_MID, x, out, ob, st, ws, wait_limit_ns=50_000_000)
    torch.cuda.synchronize()
    elapsed = time.time() - t0
    assert int(st.item()) == S.SZ_ERR_TIMEOUT
    assert elapsed < 10.0
    # The context is still usable: a normal encode right after is exact.
    got, status, _ = G.encode(S.SZ_BF16, CB_MID, x)
    assert status == 0
    assert np.array_equal(got, orc.encode(O.BF16, CB_MID, G.as_bytes(x)))
