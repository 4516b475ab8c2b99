"""Python view of the SplitZip CPU oracle (``splitzip_oracle.c``).

TEST INFRASTRUCTURE ONLY.  The oracle is the parity reference for the CUDA
codec.  Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg
of ``bench.py`` may import this module; the product package never does.

This module only marshals numpy buffers into the C functions and builds the
shared object with gcc; every step of the format lives in the C file.
"""
from __future__ import annotations

import ctypes
import hashlib
import os
import subprocess
import tempfile

import numpy as np

HERE = os.path.dirname(os.path.abspath(__file__))
SOURCE = os.path.join(HERE, "splitzip_oracle.c")
LIBRARY = os.path.join(HERE, "libsplitzip_oracle.so")
CFLAGS = ["-O2", "-std=c99", "-Wall", "-Wextra", "-shared", "-fPIC"]

BF16 = 0
E5M2 = 1

OK = 0
INVALID_ARG = 1
CAPACITY = 3
CORRUPT = 4

CHUNK = 65536

ABL_TOP8 = 1       # ablation codecs (BF16): Top-8 with 3-bit codes
ABL_SENTINEL = 2   # Top-15 codes with 15 as an escape sentinel


def _digest(source_text: str, flags) -> str:
    h = hashlib.sha256()
    h.update(source_text.encode())
    h.update(" ".join(flags).encode())
    return h.hexdigest()


def compile_source(source_text: str, out_path: str, extra_flags=()) -> str:
    """Compile oracle C source text into a shared object at ``out_path``."""
    flags = CFLAGS + list(extra_flags)
    stamp = out_path + ".stamp"
    want = _digest(source_text, flags)
    if os.path.exists(out_path) and os.path.exists(stamp):
        with open(stamp) as f:
            if f.read().strip() == want:
                return out_path
    with tempfile.TemporaryDirectory() as tmp:
        src = os.path.join(tmp, "oracle.c")
        with open(src, "w") as f:
            f.write(source_text)
        part = out_path + f".{os.getpid()}.part"
        subprocess.run(["gcc", *flags, "-o", part, src], check=True)
        os.replace(part, out_path)  # atomic: concurrent loaders see old or new
    with open(stamp, "w") as f:
        f.write(want)
    return out_path


def build() -> str:
    """Compile the oracle next to its source (no-op when up to date)."""
    with open(SOURCE) as f:
        return compile_source(f.read(), LIBRARY)


def _u8(a: np.ndarray) -> np.ndarray:
    a = np.ascontiguousarray(a)
    return a.view(np.uint8).reshape(-1)


def _ptr(a: np.ndarray):
    return a.ctypes.data_as(ctypes.c_void_p)


class Oracle:
    """ctypes wrapper around one build of the oracle shared object."""

    def __init__(self, path: str | None = None):
        if path is None:
            path = build()
        lib = ctypes.CDLL(path)
        u64, i32, vp = ctypes.c_uint64, ctypes.c_int, ctypes.c_void_p
        sig = {
            "orc_dense_bytes": (u64, [i32, u64]),
            "orc_num_chunks": (u64, [u64]),
            "orc_encoded_size": (u64, [i32, u64, u64]),
            "orc_histogram": (None, [i32, vp, u64, vp]),
            "orc_codebook_from_histogram": (i32, [i32, vp, vp]),
            "orc_codebook_valid": (i32, [i32, vp]),
            "orc_count_escapes": (u64, [i32, vp, vp, u64]),
            "orc_encode": (i32, [i32, vp, vp, u64, vp, u64, ctypes.POINTER(u64)]),
            "orc_validate": (i32, [i32, vp, u64, u64, ctypes.POINTER(u64)]),
            "orc_decode": (i32, [i32, vp, u64, u64, vp]),
            "orc_ablation_sizes": (i32, [i32, vp, u64, vp]),
            "orc_abl_size": (u64, [i32, u64, u64]),
            "orc_abl_codebook": (i32, [i32, vp, vp]),
            "orc_abl_encode": (i32, [i32, vp, vp, u64, vp, u64, ctypes.POINTER(u64)]),
            "orc_abl_decode": (i32, [i32, vp, u64, u64, vp]),
        }
        for name, (res, args) in sig.items():
            fn = getattr(lib, name)
            fn.restype = res
            fn.argtypes = args
        self.lib = lib
        self.path = path

    # -- sizes ---------------------------------------------------------------
    def dense_bytes(self, dt: int, n: int) -> int:
        return int(self.lib.orc_dense_bytes(dt, n))

    def num_chunks(self, n: int) -> int:
        return int(self.lib.orc_num_chunks(n))

    def encoded_size(self, dt: int, n: int, n_escapes: int) -> int:
        return int(self.lib.orc_encoded_size(dt, n, n_escapes))

    # -- calibration -----------------------------------------------------------
    @staticmethod
    def element_count(dt: int, x: np.ndarray) -> int:
        nbytes = _u8(x).size
        return nbytes // 2 if dt == BF16 else nbytes

    def histogram(self, dt: int, x: np.ndarray) -> np.ndarray:
        xb = _u8(x)
        hist = np.zeros(256 if dt == BF16 else 32, dtype=np.uint64)
        self.lib.orc_histogram(dt, _ptr(xb), self.element_count(dt, xb), _ptr(hist))
        return hist

    def codebook_from_histogram(self, dt: int, hist: np.ndarray) -> np.ndarray:
        h = np.ascontiguousarray(hist, dtype=np.uint64)
        assert h.size == (256 if dt == BF16 else 32)
        cb = np.zeros(16, dtype=np.uint8)
        self.lib.orc_codebook_from_histogram(dt, _ptr(h), _ptr(cb))
        return cb

    def calibrate(self, dt: int, x: np.ndarray) -> np.ndarray:
        return self.codebook_from_histogram(dt, self.histogram(dt, x))

    def codebook_valid(self, dt: int, cb) -> bool:
        c = np.ascontiguousarray(cb, dtype=np.uint8)
        return bool(self.lib.orc_codebook_valid(dt, _ptr(c)))

    def count_escapes(self, dt: int, cb, x: np.ndarray) -> int:
        c = np.ascontiguousarray(cb, dtype=np.uint8)
        xb = _u8(x)
        return int(self.lib.orc_count_escapes(dt, _ptr(c), _ptr(xb), self.element_count(dt, xb)))

    # -- codec ---------------------------------------------------------------
    def encode(self, dt: int, cb, x: np.ndarray) -> np.ndarray:
        """Return the encoded stream as a uint8 array (raises on failure)."""
        c = np.ascontiguousarray(cb, dtype=np.uint8)
        xb = _u8(x)
        n = self.element_count(dt, xb)
        if not self.lib.orc_codebook_valid(dt, _ptr(c)):
            raise ValueError("invalid codebook")
        size = self.encoded_size(dt, n, self.count_escapes(dt, c, xb))
        out = np.empty(max(size, 1), dtype=np.uint8)
        got = ctypes.c_uint64(0)
        st = self.lib.orc_encode(dt, _ptr(c), _ptr(xb), n, _ptr(out), size, ctypes.byref(got))
        if st != OK:
            raise RuntimeError(f"oracle encode failed with status {st}")
        assert got.value == size
        return out[:size]

    def validate(self, dt: int, stream: np.ndarray, n: int):
        s = _u8(stream)
        e = ctypes.c_uint64(0)
        st = self.lib.orc_validate(dt, _ptr(s), s.size, n, ctypes.byref(e))
        return int(st), int(e.value)

    def decode(self, dt: int, stream: np.ndarray, n: int):
        """Return (status, decoded bytes); the bytes are all zero on failure."""
        s = _u8(stream)
        y = np.zeros(max(2 * n if dt == BF16 else n, 1), dtype=np.uint8)
        st = self.lib.orc_decode(dt, _ptr(s), s.size, n, _ptr(y))
        return int(st), y[: (2 * n if dt == BF16 else n)]


    # -- ablation ------------------------------------------------------------
    def ablation_sizes(self, dt: int, hist: np.ndarray, n: int) -> tuple[int, int, int]:
        """Stream sizes under Top-16 (this format), Top-8 and Top-15 + sentinel."""
        h = np.ascontiguousarray(hist, dtype=np.uint64)
        assert h.size == (256 if dt == BF16 else 32)
        out = np.zeros(3, dtype=np.uint64)
        self.lib.orc_ablation_sizes(dt, _ptr(h), n, _ptr(out))
        return int(out[0]), int(out[1]), int(out[2])


    # -- ablation codecs (BF16): ABL_TOP8, ABL_SENTINEL ------------------------
    def abl_size(self, variant: int, n: int, n_escapes: int) -> int:
        return int(self.lib.orc_abl_size(variant, n, n_escapes))

    def abl_codebook(self, variant: int, hist: np.ndarray) -> np.ndarray:
        h = np.ascontiguousarray(hist, dtype=np.uint64)
        assert h.size == 256
        cb = np.zeros(8 if variant == ABL_TOP8 else 15, dtype=np.uint8)
        assert self.lib.orc_abl_codebook(variant, _ptr(h), _ptr(cb)) == OK
        return cb

    def abl_encode(self, variant: int, cb, x: np.ndarray) -> np.ndarray:
        c = np.ascontiguousarray(cb, dtype=np.uint8)
        xb = _u8(x)
        n = xb.size // 2
        size = ctypes.c_uint64(0)
        st = self.lib.orc_abl_encode(variant, _ptr(c), _ptr(xb), n, None, 0, ctypes.byref(size))
        if st not in (OK, CAPACITY):
            raise ValueError(f"ablation encode failed ({st})")
        out = np.empty(max(size.value, 1), dtype=np.uint8)
        st = self.lib.orc_abl_encode(variant, _ptr(c), _ptr(xb), n, _ptr(out), out.size, ctypes.byref(size))
        assert st == OK
        return out[: size.value]

    def abl_decode(self, variant: int, stream: np.ndarray, n: int):
        s = _u8(stream)
        y = np.zeros(max(2 * n, 1), dtype=np.uint8)
        st = self.lib.orc_abl_decode(variant, _ptr(s), s.size, n, _ptr(y))
        return int(st), y[: 2 * n]


_DEFAULT: Oracle | None = None


def default() -> Oracle:
    """The oracle built from ``splitzip_oracle.c`` (built on first use)."""
    global _DEFAULT
    if _DEFAULT is None:
        _DEFAULT = Oracle()
    return _DEFAULT
