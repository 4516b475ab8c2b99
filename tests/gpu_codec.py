"""Test helpers that drive the CUDA codec through its C ABI binding."""
import numpy as np
import torch

from lossless_kv_cache_bf16_gb300 import splitzip as S

DT = {"bf16": S.SZ_BF16, "e5m2": S.SZ_FP8_E5M2}


def as_bytes(t: torch.Tensor) -> np.ndarray:
    """Host copy of a tensor's raw bytes."""
    return t.contiguous().view(torch.uint8).reshape(-1).cpu().numpy()


def elements(dt, t):
    return t.numel() * t.element_size() // S.ELEMENT_BYTES[dt]


def encode(dt, cb, x, capacity=None, out_offset=0, stream=None):
    """Encode x on the GPU; returns (stream bytes on the host, status, size)."""
    n = elements(dt, x)
    cap = S.sz_encoded_size(dt, n, n) if capacity is None else capacity
    buf = torch.empty(cap + out_offset, dtype=torch.uint8, device="cuda")
    out = buf[out_offset:]
    ws = torch.empty(S.sz_workspace_size(dt, n), dtype=torch.uint8, device="cuda")
    ob = torch.zeros(1, dtype=torch.int64, device="cuda")
    st = torch.full((1,), -1, dtype=torch.int32, device="cuda")
    S.sz_encode(dt, cb, x, out, ob, st, ws, stream=stream)
    torch.cuda.synchronize()
    size = int(ob.item())
    return out[: min(size, cap)].cpu().numpy(), int(st.item()), size


def decode(dt, stream_bytes: np.ndarray, n, out_offset=0, in_offset=0, guard=64):
    """Decode a host stream on the GPU.  Returns (status, decoded bytes,
    guard_ok) where guard_ok says the bytes around the output were untouched."""
    src = torch.empty(stream_bytes.size + in_offset, dtype=torch.uint8, device="cuda")
    src[in_offset:] = torch.from_numpy(np.ascontiguousarray(stream_bytes)).to("cuda")
    nbytes = n * S.ELEMENT_BYTES[dt]
    canary = 0xA5
    buf = torch.full((guard + out_offset + nbytes + guard,), canary, dtype=torch.uint8, device="cuda")
    y = buf[guard + out_offset: guard + out_offset + nbytes]
    st = torch.full((1,), -1, dtype=torch.int32, device="cuda")
    S.sz_decode(dt, src[in_offset:], stream_bytes.size, n, y, st)
    torch.cuda.synchronize()
    host = buf.cpu().numpy()
    guard_ok = bool(np.all(host[: guard + out_offset] == canary) and np.all(host[guard + out_offset + nbytes:] == canary))
    return int(st.item()), host[guard + out_offset: guard + out_offset + nbytes], guard_ok


def calibrate(dt, sample):
    hist = torch.empty(S.sz_histogram_bins(dt), dtype=torch.int64, device="cuda")
    cb = S.sz_calibrate(dt, sample, hist)
    return np.array(cb, dtype=np.uint8), hist.cpu().numpy().astype(np.uint64)
