"""Python binding of the SplitZip C ABI (``include/splitzip.h``).

Argument marshalling only: every function forwards to ``libsplitzip.so`` with
the same name, passing device pointers of torch CUDA tensors and the current
CUDA stream.  All work runs in the library's CUDA kernels; there is no CPU
path, and importing this module fails loudly when the library is missing.
"""
from __future__ import annotations

import ctypes
import os

import torch

from . import build as _build

SZ_OK = 0
SZ_ERR_INVALID_ARG = 1
SZ_ERR_UNSUPPORTED = 2
SZ_ERR_CAPACITY = 3
SZ_ERR_CORRUPT = 4
SZ_ERR_TIMEOUT = 5
SZ_ERR_CUDA = 6

SZ_BF16 = 0
SZ_FP8_E5M2 = 1

SZ_ABL_TOP8 = 1        # codebook ablation: Top-8, 3-bit codes
SZ_ABL_SENTINEL = 2    # codebook ablation: Top-15 codes, 15 = escape sentinel
SZ_CHUNK_ELEMS = 65536
SZ_CODEBOOK_SIZE = 16

ELEMENT_BYTES = {SZ_BF16: 2, SZ_FP8_E5M2: 1}


class SplitZipError(RuntimeError):
    def __init__(self, fn: str, status: int):
        super().__init__(f"{fn} returned {sz_status_string(status)} ({status})")
        self.status = status


class sz_codebook(ctypes.Structure):
    _fields_ = [("exp", ctypes.c_uint8 * SZ_CODEBOOK_SIZE)]


def _load() -> ctypes.CDLL:
    path = _build.LIBRARY
    if not os.path.exists(path):
        raise RuntimeError(f"SplitZip CUDA library not found at {path}; build it with "
                           "`python -m lossless_kv_cache_bf16_gb300.build`")
    lib = ctypes.CDLL(path)
    vp, sz, i32, u64p = ctypes.c_void_p, ctypes.c_size_t, ctypes.c_int, ctypes.POINTER(ctypes.c_ulonglong)
    cbp = ctypes.POINTER(sz_codebook)
    sigs = {
        "sz_encoded_size": (sz, [i32, sz, sz]),
        "sz_workspace_size": (sz, [i32, sz]),
        "sz_histogram_bins": (sz, [i32]),
        "sz_histogram": (i32, [i32, vp, sz, vp, vp]),
        "sz_codebook_from_histogram": (i32, [i32, u64p, cbp]),
        "sz_calibrate": (i32, [i32, vp, sz, vp, cbp, vp]),
        "sz_encode": (i32, [i32, cbp, vp, sz, vp, sz, vp, vp, vp, sz, vp]),
        "sz_decode": (i32, [i32, vp, sz, sz, vp, vp, vp]),
        "sz_status_string": (ctypes.c_char_p, [i32]),
        "sz_debug_encode_stalled": (i32, [i32, cbp, vp, sz, vp, sz, vp, vp, vp, sz, ctypes.c_ulonglong, vp]),
        "sz_encode_noalloc": (i32, [i32, cbp, vp, sz, vp, sz, vp, vp, vp]),
        "sz_codebook_from_histogram_device": (i32, [i32, vp, vp, vp]),
        "sz_calibrate_device": (i32, [i32, vp, sz, ctypes.c_uint32, vp, vp, vp]),
        "sz_encode_dcb": (i32, [i32, vp, vp, sz, vp, sz, vp, vp, vp, sz, vp]),
        "sz_ablation_sizes": (i32, [i32, u64p, sz, u64p]),
        "sz_encode_paged": (i32, [i32, cbp, vp, sz, sz, vp, sz, vp, sz, vp, vp, vp, sz, vp]),
        "sz_ablation_encoded_size": (sz, [i32, sz, sz]),
        "sz_ablation_workspace_size": (sz, [sz]),
        "sz_ablation_codebook": (i32, [i32, u64p, vp]),
        "sz_ablation_encode": (i32, [i32, vp, vp, sz, vp, sz, vp, vp, sz, vp]),
        "sz_ablation_decode": (i32, [i32, vp, sz, sz, vp, vp, vp]),
        "sz_decode_paged": (i32, [i32, vp, sz, sz, vp, sz, sz, vp, vp, vp]),
        "sz_concat": (i32, [i32, sz, ctypes.POINTER(vp), ctypes.POINTER(sz), ctypes.POINTER(sz), vp, sz,
                            ctypes.POINTER(sz), vp, vp]),
    }
    for name, (res, args) in sigs.items():
        fn = getattr(lib, name)
        fn.restype = res
        fn.argtypes = args
    return lib


LIB = _load()


# ---- marshalling helpers -----------------------------------------------------

# Pointers and streams go to ctypes as plain ints (the argtypes are
# c_void_p), which skips building a ctypes object per argument.
def _dev_ptr(t: torch.Tensor | None, what: str):
    if t is None:
        return None
    if not t.is_cuda:
        raise ValueError(f"{what} must be a CUDA tensor")
    if not t.is_contiguous():
        raise ValueError(f"{what} must be contiguous")
    return t.data_ptr()


def _written_ptr(t: torch.Tensor, what: str):
    """A word the device writes: a CUDA tensor, or pinned host memory (mapped
    into the device's address space under unified addressing)."""
    if not t.is_cuda and not t.is_pinned():
        raise ValueError(f"{what} must be a CUDA tensor or pinned host memory")
    if not t.is_contiguous():
        raise ValueError(f"{what} must be contiguous")
    return t.data_ptr()


# The current stream's handle straight from the C++ side: building a
# torch.cuda.Stream object costs about 3 us per call on the Grace host, the
# raw handle about 0.1 us.
_raw_stream = getattr(torch._C, "_cuda_getCurrentRawStream", None)
_get_device = getattr(torch._C, "_cuda_getDevice", None)


def _stream(stream) -> int:
    if stream is not None:
        return stream.cuda_stream
    if _raw_stream is not None and _get_device is not None:
        return _raw_stream(_get_device())
    return torch.cuda.current_stream().cuda_stream


def _elements(dt: int, t: torch.Tensor) -> int:
    nbytes = t.numel() * t.element_size()
    if nbytes % ELEMENT_BYTES[dt]:
        raise ValueError("tensor size is not a whole number of elements")
    return nbytes // ELEMENT_BYTES[dt]


def _count(dt: int, x: torch.Tensor, n: int | None) -> int:
    """Elements to encode: all of x, or the first n of them.  An n beyond x
    would make the kernels read past x's allocation, so it is refused here,
    before anything is launched."""
    have = _elements(dt, x)
    if n is None:
        return have
    if n < 0 or n > have:
        raise ValueError(f"n = {n} is outside the tensor's {have} elements")
    return n


def _block_table(block_ids: torch.Tensor, n: int, page_elems: int) -> None:
    """The block table must name a page for every element of the logical
    tensor: ceil(n / page_elems) int32 ids.  The kernels index it without a
    bound, so a shorter table is refused before anything is launched."""
    if block_ids.dtype != torch.int32:
        raise ValueError("block_ids must be int32")
    if page_elems < 16 or page_elems & (page_elems - 1):
        return  # not a page size the library accepts: it refuses the call itself
    need = -(-n // page_elems)
    if block_ids.numel() < need:
        raise ValueError(f"block_ids holds {block_ids.numel()} ids; {n} elements in pages of "
                         f"{page_elems} need {need}")


_CODEBOOKS: dict = {}  # codebook values -> its C struct (read by the library during a call only)


def _codebook(cb) -> sz_codebook:
    if isinstance(cb, sz_codebook):
        return cb
    key = tuple(cb.tolist() if hasattr(cb, "tolist") else cb)
    c = _CODEBOOKS.get(key)
    if c is None:
        vals = [int(v) for v in key]
        if len(vals) != SZ_CODEBOOK_SIZE:
            raise ValueError("a codebook has 16 exponents")
        if any(v < 0 or v > 255 for v in vals):
            raise ValueError("codebook exponents are bytes (0..255)")
        c = sz_codebook()
        for k, v in enumerate(vals):
            c.exp[k] = v
        if len(_CODEBOOKS) < 1024:
            _CODEBOOKS[key] = c
    return c


def _check(fn: str, status: int):
    if status != SZ_OK:
        raise SplitZipError(fn, status)


# ---- the C ABI, same names ---------------------------------------------------

def sz_status_string(status: int) -> str:
    return LIB.sz_status_string(status).decode()


def sz_encoded_size(dt: int, n: int, n_escapes: int) -> int:
    return int(LIB.sz_encoded_size(dt, n, n_escapes))


def sz_workspace_size(dt: int, n: int) -> int:
    return int(LIB.sz_workspace_size(dt, n))


def sz_histogram_bins(dt: int) -> int:
    return int(LIB.sz_histogram_bins(dt))


def sz_histogram(dt: int, sample: torch.Tensor, hist: torch.Tensor, stream=None) -> None:
    """hist: int64/uint64 CUDA tensor of sz_histogram_bins(dt) counts (overwritten)."""
    assert hist.numel() == sz_histogram_bins(dt) and hist.element_size() == 8
    _check("sz_histogram", LIB.sz_histogram(dt, _dev_ptr(sample, "sample"), _elements(dt, sample),
                                            _dev_ptr(hist, "hist"), _stream(stream)))


def sz_codebook_from_histogram(dt: int, hist) -> list[int]:
    vals = [int(v) for v in (hist.tolist() if hasattr(hist, "tolist") else hist)]
    arr = (ctypes.c_ulonglong * len(vals))(*vals)
    cb = sz_codebook()
    _check("sz_codebook_from_histogram", LIB.sz_codebook_from_histogram(dt, arr, ctypes.byref(cb)))
    return list(cb.exp)


def sz_ablation_sizes(dt: int, hist, n: int) -> tuple[int, int, int]:
    """Stream sizes under Top-16 (this format), Top-8 and Top-15 + sentinel."""
    vals = [int(v) for v in (hist.tolist() if hasattr(hist, "tolist") else hist)]
    arr = (ctypes.c_ulonglong * len(vals))(*vals)
    out = (ctypes.c_ulonglong * 3)()
    _check("sz_ablation_sizes", LIB.sz_ablation_sizes(dt, arr, n, out))
    return int(out[0]), int(out[1]), int(out[2])


def sz_calibrate(dt: int, sample: torch.Tensor, hist: torch.Tensor, stream=None) -> list[int]:
    """Offline calibration; synchronises the stream; returns the 16 exponents."""
    cb = sz_codebook()
    _check("sz_calibrate", LIB.sz_calibrate(dt, _dev_ptr(sample, "sample"), _elements(dt, sample),
                                            _dev_ptr(hist, "hist"), ctypes.byref(cb), _stream(stream)))
    return list(cb.exp)


def sz_codebook_from_histogram_device(dt: int, hist: torch.Tensor, cb: torch.Tensor, stream=None) -> None:
    """Top-16 of a device histogram into cb (16 uint8 on the device); asynchronous."""
    assert hist.numel() == sz_histogram_bins(dt) and hist.element_size() == 8
    assert cb.numel() * cb.element_size() >= SZ_CODEBOOK_SIZE
    _check("sz_codebook_from_histogram_device",
           LIB.sz_codebook_from_histogram_device(dt, _dev_ptr(hist, "hist"), _dev_ptr(cb, "cb"), _stream(stream)))


def sz_calibrate_device(dt: int, x: torch.Tensor, hist: torch.Tensor, cb: torch.Tensor, sample_stride: int = 1,
                        stream=None, n: int | None = None) -> None:
    """Online calibration on the device (histogram of one 128-byte line per
    run of sample_stride lines, at a hashed position in the run, then top-16)
    into cb (16 uint8 on the device); asynchronous, no host synchronisation."""
    assert hist.numel() == sz_histogram_bins(dt) and hist.element_size() == 8
    assert cb.numel() * cb.element_size() >= SZ_CODEBOOK_SIZE
    n = _count(dt, x, n)
    _check("sz_calibrate_device",
           LIB.sz_calibrate_device(dt, _dev_ptr(x, "x"), n, sample_stride, _dev_ptr(hist, "hist"),
                                   _dev_ptr(cb, "cb"), _stream(stream)))


def sz_encode_dcb(dt: int, cb: torch.Tensor, x: torch.Tensor, out: torch.Tensor, out_bytes: torch.Tensor,
                  status: torch.Tensor | None, ws: torch.Tensor, stream=None, n: int | None = None) -> None:
    """sz_encode with the codebook in device memory (cb: 16 uint8 on the device)."""
    n = _count(dt, x, n)
    _check("sz_encode_dcb", LIB.sz_encode_dcb(dt, _dev_ptr(cb, "cb"), _dev_ptr(x, "x"), n, _dev_ptr(out, "out"),
                                              out.numel() * out.element_size(), _written_ptr(out_bytes, "out_bytes"),
                                              _dev_ptr(status, "status"), _dev_ptr(ws, "ws"),
                                              ws.numel() * ws.element_size(), _stream(stream)))


def sz_encode(dt: int, cb, x: torch.Tensor, out: torch.Tensor, out_bytes: torch.Tensor,
              status: torch.Tensor | None, ws: torch.Tensor, stream=None, n: int | None = None) -> None:
    """Asynchronous encode of x (n elements, default all of x) into out."""
    c = _codebook(cb)
    n = _count(dt, x, n)
    _check("sz_encode", LIB.sz_encode(dt, ctypes.byref(c), _dev_ptr(x, "x"), n, _dev_ptr(out, "out"),
                                      out.numel() * out.element_size(), _written_ptr(out_bytes, "out_bytes"),
                                      _dev_ptr(status, "status"), _dev_ptr(ws, "ws"),
                                      ws.numel() * ws.element_size(), _stream(stream)))


def sz_decode(dt: int, stream_bytes: torch.Tensor, in_bytes: int, n: int, y: torch.Tensor,
              status: torch.Tensor | None, stream=None) -> None:
    """Asynchronous decode of the first in_bytes bytes of stream_bytes into y."""
    if in_bytes > stream_bytes.numel() * stream_bytes.element_size():
        raise ValueError("in_bytes exceeds the stream buffer")
    if n * ELEMENT_BYTES[dt] > y.numel() * y.element_size():
        raise ValueError("output buffer too small")
    _check("sz_decode", LIB.sz_decode(dt, _dev_ptr(stream_bytes, "stream"), in_bytes, n, _dev_ptr(y, "y"),
                                      _dev_ptr(status, "status"), _stream(stream)))


def _pool_pages(dt: int, pool: torch.Tensor, page_elems: int) -> int:
    page_bytes = page_elems * ELEMENT_BYTES[dt]
    return (pool.numel() * pool.element_size()) // page_bytes if page_bytes else 0


def sz_encode_paged(dt: int, cb, pool: torch.Tensor, page_elems: int, block_ids: torch.Tensor, n: int,
                    out: torch.Tensor, out_bytes: torch.Tensor, status: torch.Tensor | None, ws: torch.Tensor,
                    stream=None) -> None:
    """Encode the n-element tensor whose element e is element e % page_elems
    of page block_ids[e // page_elems] of `pool` (pages of page_elems)."""
    _block_table(block_ids, n, page_elems)
    c = _codebook(cb)
    _check("sz_encode_paged",
           LIB.sz_encode_paged(dt, ctypes.byref(c), _dev_ptr(pool, "pool"), _pool_pages(dt, pool, page_elems),
                               page_elems, _dev_ptr(block_ids, "block_ids"), n, _dev_ptr(out, "out"),
                               out.numel() * out.element_size(), _written_ptr(out_bytes, "out_bytes"),
                               _dev_ptr(status, "status"), _dev_ptr(ws, "ws"), ws.numel() * ws.element_size(),
                               _stream(stream)))


def sz_decode_paged(dt: int, stream_bytes: torch.Tensor, in_bytes: int, n: int, pool: torch.Tensor, page_elems: int,
                    block_ids: torch.Tensor, status: torch.Tensor | None, stream=None) -> None:
    """Decode into the pages of `pool` that block_ids names (see sz_encode_paged)."""
    _block_table(block_ids, n, page_elems)
    if in_bytes > stream_bytes.numel() * stream_bytes.element_size():
        raise ValueError("in_bytes exceeds the stream buffer")
    _check("sz_decode_paged",
           LIB.sz_decode_paged(dt, _dev_ptr(stream_bytes, "stream"), in_bytes, n, _dev_ptr(pool, "pool"),
                               _pool_pages(dt, pool, page_elems), page_elems, _dev_ptr(block_ids, "block_ids"),
                               _dev_ptr(status, "status"), _stream(stream)))


def sz_concat(dt: int, streams, sizes, ns, out: torch.Tensor, status: torch.Tensor | None = None,
              stream=None) -> int:
    """Join shard streams (device tensors in tensor order; sizes[k] bytes of
    streams[k] encode ns[k] elements) into the stream of the whole tensor in
    `out`.  Returns the joined stream's size (known on the host at once)."""
    k = len(streams)
    if len(sizes) != k or len(ns) != k:
        raise ValueError("streams, sizes and ns must have the same length")
    for t, b in zip(streams, sizes):
        if b > t.numel() * t.element_size():
            raise ValueError("a shard size exceeds its buffer")
    ptrs = (ctypes.c_void_p * k)(*[_dev_ptr(t, "stream") for t in streams])
    nbytes = (ctypes.c_size_t * k)(*sizes)
    counts = (ctypes.c_size_t * k)(*ns)
    total = ctypes.c_size_t(0)
    _check("sz_concat", LIB.sz_concat(dt, k, ptrs, nbytes, counts, _dev_ptr(out, "out"),
                                      out.numel() * out.element_size(), ctypes.byref(total),
                                      _dev_ptr(status, "status"), _stream(stream)))
    return total.value


def sz_ablation_encoded_size(variant: int, n: int, n_escapes: int) -> int:
    return int(LIB.sz_ablation_encoded_size(variant, n, n_escapes))


def sz_ablation_workspace_size(n: int) -> int:
    return int(LIB.sz_ablation_workspace_size(n))


def sz_ablation_codebook(variant: int, hist) -> list[int]:
    vals = [int(v) for v in (hist.tolist() if hasattr(hist, "tolist") else hist)]
    assert len(vals) == 256
    arr = (ctypes.c_ulonglong * 256)(*vals)
    cb = (ctypes.c_uint8 * 15)()
    _check("sz_ablation_codebook", LIB.sz_ablation_codebook(variant, arr, cb))
    return list(cb)[: 8 if variant == SZ_ABL_TOP8 else 15]


def sz_ablation_encode(variant: int, cb, x: torch.Tensor, out: torch.Tensor, out_bytes: torch.Tensor,
                       ws: torch.Tensor, stream=None) -> None:
    """Encode BF16 x in one of the ablation's alternative layouts (cb: 8 or 15 exponents)."""
    vals = [int(v) for v in (cb.tolist() if hasattr(cb, "tolist") else cb)]
    arr = (ctypes.c_uint8 * 16)(*vals)
    _check("sz_ablation_encode",
           LIB.sz_ablation_encode(variant, arr, _dev_ptr(x, "x"), _elements(SZ_BF16, x), _dev_ptr(out, "out"),
                                  out.numel() * out.element_size(), _written_ptr(out_bytes, "out_bytes"),
                                  _dev_ptr(ws, "ws"), ws.numel() * ws.element_size(), _stream(stream)))


def sz_ablation_decode(variant: int, stream_bytes: torch.Tensor, in_bytes: int, n: int, y: torch.Tensor,
                       status: torch.Tensor | None, stream=None) -> None:
    if in_bytes > stream_bytes.numel() * stream_bytes.element_size():
        raise ValueError("in_bytes exceeds the stream buffer")
    if 2 * n > y.numel() * y.element_size():
        raise ValueError("output buffer too small")
    _check("sz_ablation_decode", LIB.sz_ablation_decode(variant, _dev_ptr(stream_bytes, "stream"), in_bytes, n,
                                                        _dev_ptr(y, "y"), _dev_ptr(status, "status"), _stream(stream)))


def sz_encode_noalloc(dt: int, cb, x: torch.Tensor, out: torch.Tensor, out_bytes: torch.Tensor,
                      status: torch.Tensor | None, stream=None, n: int | None = None) -> None:
    """sz_encode without a caller workspace (the library's static scratch is
    used instead), for callers that cannot allocate device memory."""
    c = _codebook(cb)
    n = _count(dt, x, n)
    _check("sz_encode_noalloc", LIB.sz_encode_noalloc(dt, ctypes.byref(c), _dev_ptr(x, "x"), n, _dev_ptr(out, "out"),
                                                      out.numel() * out.element_size(),
                                                      _written_ptr(out_bytes, "out_bytes"), _dev_ptr(status, "status"),
                                                      _stream(stream)))


def sz_debug_encode_stalled(dt: int, cb, x: torch.Tensor, out: torch.Tensor, out_bytes: torch.Tensor,
                            status: torch.Tensor, ws: torch.Tensor, wait_limit_ns: int, stream=None) -> None:
    c = _codebook(cb)
    _check("sz_debug_encode_stalled",
           LIB.sz_debug_encode_stalled(dt, ctypes.byref(c), _dev_ptr(x, "x"), _elements(dt, x), _dev_ptr(out, "out"),
                                       out.numel() * out.element_size(), _written_ptr(out_bytes, "out_bytes"),
                                       _dev_ptr(status, "status"), _dev_ptr(ws, "ws"),
                                       ws.numel() * ws.element_size(), wait_limit_ns, _stream(stream)))
