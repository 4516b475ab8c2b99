"""The C ABI library on a host without a GPU: it loads, exports every symbol
that include/splitzip.h declares, and its host-only logic (closed-form sizes,
top-16 selection, argument checks that return before any CUDA call) agrees
with the oracle and the header's contract.  No compute runs here."""
import ctypes
import os
import re

import numpy as np
import pytest

from oracle import oracle as O

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "splitzip.h")


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(sz_[a-z_]+)\s*\(", text)))


@pytest.fixture(scope="module")
def S():
    from lossless_kv_cache_bf16_gb300 import splitzip

    return splitzip


def test_exports_every_declared_symbol(S):
    names = declared_functions()
    assert len(names) >= 9
    for name in names:
        assert hasattr(S.LIB, name), f"{name} declared but not exported"
        assert callable(getattr(S, name)), f"binding lacks {name}"


def test_encoded_size_matches_oracle(S, orc):
    for dt in (O.BF16, O.E5M2):
        for n in (0, 1, 2, 7, 8, 9, 65535, 65536, 65537, 536870912, 4294967295):
            for e in (0, 1, n // 3, n):
                assert S.sz_encoded_size(dt, n, e) == orc.encoded_size(dt, n, e)
    assert S.sz_encoded_size(7, 10, 0) == 0


def test_workspace_size(S):
    # Per 32,768-element scan tile: a u32 count and an i32 error word (each
    # a 16-byte aligned block), 32 u16 unit counts, and 2,048 (BF16) or 1,024
    # (E5M2) staged 3-byte records.
    for dt, staged in ((S.SZ_BF16, 2048), (S.SZ_FP8_E5M2, 1024)):
        ws = lambda tiles: 2 * (((4 * tiles + 15) // 16) * 16) + 64 * tiles + 3 * staged * tiles
        assert S.sz_workspace_size(dt, 0) == ws(1)
        assert S.sz_workspace_size(dt, 32768) == ws(1)
        assert S.sz_workspace_size(dt, 32769) == ws(2)
        assert S.sz_workspace_size(dt, 939524096) == ws(939524096 // 32768)


def test_codebook_selection_matches_oracle(S, orc):
    rng = np.random.default_rng(1)
    for dt, bins in ((O.BF16, 256), (O.E5M2, 32)):
        for trial in range(200):
            hist = rng.integers(0, 4, bins).astype(np.uint64) * rng.integers(0, 3, bins).astype(np.uint64)
            if trial % 3 == 0:
                hist[:] = 0
                hist[rng.integers(0, bins, 5)] = 7  # ties and fewer than 16 seen
            assert S.sz_codebook_from_histogram(dt, hist) == orc.codebook_from_histogram(dt, hist).tolist()


def test_host_argument_checks_return_before_launching(S):
    """Invalid arguments return at once; the fake device pointers are never used."""
    lib = S.LIB
    fake = ctypes.c_void_p(0x10000)
    cb = S._codebook(list(range(120, 136)))
    dup = S._codebook([120] * 16)
    n = 1000
    cap = S.sz_encoded_size(0, n, n)
    ws = S.sz_workspace_size(0, n)
    enc = lambda dt, c, cap_, ws_, n_=n, out=fake: lib.sz_encode(dt, ctypes.byref(c), fake, n_, out, cap_, fake, None, fake, ws_, None)
    assert enc(0, dup, cap, ws) == S.SZ_ERR_INVALID_ARG
    assert enc(1, cb, cap, ws) == S.SZ_ERR_INVALID_ARG            # exponents >= 32 for E5M2
    assert enc(5, cb, cap, ws) == S.SZ_ERR_INVALID_ARG
    assert enc(0, cb, 10, ws) == S.SZ_ERR_CAPACITY
    assert enc(0, cb, cap, 8) == S.SZ_ERR_CAPACITY
    assert enc(0, cb, cap, ws, n_=1 << 32) == S.SZ_ERR_INVALID_ARG
    assert enc(0, cb, cap, ws, out=None) == S.SZ_ERR_INVALID_ARG
    fixed = S.sz_encoded_size(0, n, 0)
    dec = lambda size, n_=n: lib.sz_decode(0, fake, size, n_, fake, None, None)
    assert dec(fixed - 1) == S.SZ_ERR_CORRUPT
    assert dec(fixed + 1) == S.SZ_ERR_CORRUPT
    assert dec(fixed + 3 * (n + 1)) == S.SZ_ERR_CORRUPT         # more escapes than elements
    assert lib.sz_decode(0, None, fixed, n, fake, None, None) == S.SZ_ERR_INVALID_ARG
    assert lib.sz_debug_encode_stalled(0, ctypes.byref(cb), fake, n, fake, cap, fake, None, fake, ws, 1000, None) == S.SZ_ERR_INVALID_ARG


def test_concat_host_checks_return_before_launching(S):
    """sz_concat refuses bad shard lists before it touches a device pointer."""
    lib = S.LIB
    fake = 0x10000
    C = S.SZ_CHUNK_ELEMS

    def call(dt, ns, sizes, cap=1 << 40, out=fake, ptr=fake):
        k = len(ns)
        ptrs = (ctypes.c_void_p * k)(*([ptr] * k))
        b = (ctypes.c_size_t * k)(*sizes)
        n = (ctypes.c_size_t * k)(*ns)
        total = ctypes.c_size_t(0)
        return lib.sz_concat(dt, k, ptrs, b, n, out, cap, ctypes.byref(total), None, None), total.value

    size = lambda n, e=0: S.sz_encoded_size(0, n, e)
    assert call(0, [], [])[0] == S.SZ_ERR_INVALID_ARG                       # no shards
    assert call(5, [C], [size(C)])[0] == S.SZ_ERR_INVALID_ARG               # unknown dtype
    assert call(0, [C + 1, C], [size(C + 1), size(C)])[0] == S.SZ_ERR_INVALID_ARG  # not whole chunks
    assert call(0, [C], [size(C)], out=None)[0] == S.SZ_ERR_INVALID_ARG
    assert call(0, [C], [size(C)], ptr=None)[0] == S.SZ_ERR_INVALID_ARG
    assert call(0, [C, 7], [size(C) + 1, size(7)])[0] == S.SZ_ERR_CORRUPT   # not the closed form
    assert call(0, [C, 7], [size(C), size(7, 8)])[0] == S.SZ_ERR_CORRUPT    # more escapes than elements
    want = size(2 * C + 7, 5)
    assert call(0, [C, C, 7], [size(C, 2), size(C), size(7, 3)], cap=want - 1) == (S.SZ_ERR_CAPACITY, 0)
    assert call(1, [1 << 31, 1 << 31], [S.sz_encoded_size(1, 1 << 31, 0)] * 2)[0] == S.SZ_ERR_INVALID_ARG  # n >= 2^32


def test_status_strings(S):
    assert S.sz_status_string(0) == "SZ_OK"
    assert S.sz_status_string(5) == "SZ_ERR_TIMEOUT"
    assert S.sz_status_string(99) == "SZ_ERR_UNKNOWN"


def test_ablation_sizes_match_oracle(S, orc):
    """The library's ablation arithmetic is written independently of the
    oracle's; they must agree on every histogram, ties and zeros included."""
    from oracle import oracle as O

    rng = np.random.default_rng(9)
    for dt, odt in ((S.SZ_BF16, O.BF16), (S.SZ_FP8_E5M2, O.E5M2)):
        bins = S.sz_histogram_bins(dt)
        for trial in range(60):
            if trial % 3 == 0:
                h = rng.integers(0, 3, size=bins)
            elif trial % 3 == 1:
                h = rng.integers(0, 1 << 30, size=bins)
            else:
                h = np.zeros(bins, dtype=np.int64)
                h[rng.integers(0, bins, size=5)] = rng.integers(1, 100, size=5)
            h = h.astype(np.uint64)
            n = int(h.sum())
            assert S.sz_ablation_sizes(dt, h, n) == orc.ablation_sizes(odt, h, n)


def test_ablation_codebook_and_sizes_match_oracle(S, orc):
    """Top-8 / Top-15 selection and the alternative layouts' closed-form
    sizes, written independently in the library and in the oracle."""
    from oracle import oracle as O

    rng = np.random.default_rng(17)
    for variant, ov in ((S.SZ_ABL_TOP8, O.ABL_TOP8), (S.SZ_ABL_SENTINEL, O.ABL_SENTINEL)):
        for trial in range(40):
            h = (rng.integers(0, 3, size=256) if trial % 2 else rng.integers(0, 1 << 30, size=256)).astype(np.uint64)
            assert S.sz_ablation_codebook(variant, h) == [int(v) for v in orc.abl_codebook(ov, h)]
        for n, e in ((0, 0), (1, 1), (65536, 9), (65537, 65537), (10 ** 6, 123)):
            assert S.sz_ablation_encoded_size(variant, n, e) == orc.abl_size(ov, n, e)


def test_codebook_marshalling(S):
    import numpy as np

    cb = list(range(120, 136))
    c = S._codebook(cb)
    assert list(c.exp) == cb
    assert S._codebook(np.arange(120, 136, dtype=np.uint8)) is c   # cached by value
    assert S._codebook(c) is c
    for bad in ([1, 2, 3], [300] + list(range(15)), [-1] + list(range(15))):
        with pytest.raises(ValueError):
            S._codebook(bad)


def test_binding_refuses_out_of_range_counts_before_any_call(S, monkeypatch):
    """An n above the tensor's element count, or a block table shorter than
    ceil(n / page_elems), would make the kernels read (or write) past a
    caller's buffer.  The binding refuses both before it calls the library:
    the fake library below records every call, and none may happen."""
    import torch

    calls = []
    real = S.LIB
    host_only = {"sz_histogram_bins", "sz_encoded_size", "sz_workspace_size", "sz_status_string"}

    class Recorder:
        def __getattr__(self, name):
            if name in host_only:
                return getattr(real, name)

            def fn(*args):
                calls.append(name)
                return S.SZ_OK
            return fn

    monkeypatch.setattr(S, "LIB", Recorder())
    cb = list(range(120, 136))
    x = torch.zeros(1000, dtype=torch.bfloat16)
    x8 = torch.zeros(1000, dtype=torch.uint8)
    out = torch.zeros(8, dtype=torch.uint8)
    ob = torch.zeros(1, dtype=torch.int64)
    hist = torch.zeros(256, dtype=torch.int64)
    dcb = torch.zeros(16, dtype=torch.uint8)
    for dt, t in ((S.SZ_BF16, x), (S.SZ_FP8_E5M2, x8)):
        for bad in (1001, 5000, -1):
            with pytest.raises(ValueError, match="outside the tensor"):
                S.sz_encode(dt, cb, t, out, ob, None, out, n=bad)
            with pytest.raises(ValueError, match="outside the tensor"):
                S.sz_encode_dcb(dt, dcb, t, out, ob, None, out, n=bad)
            with pytest.raises(ValueError, match="outside the tensor"):
                S.sz_encode_noalloc(dt, cb, t, out, ob, None, n=bad)
            with pytest.raises(ValueError, match="outside the tensor"):
                S.sz_calibrate_device(dt, t, hist[: 256 if dt == S.SZ_BF16 else 32], dcb, n=bad)
    page = 16
    for n, ids in ((1000, 62), (1000, 0), (17, 1), (16 * 9 + 1, 9)):
        table = torch.zeros(ids, dtype=torch.int32)
        with pytest.raises(ValueError, match="block_ids holds"):
            S.sz_encode_paged(S.SZ_BF16, cb, x, page, table, n, out, ob, None, out)
        with pytest.raises(ValueError, match="block_ids holds"):
            S.sz_decode_paged(S.SZ_BF16, out, 8, n, x, page, table, None)
    with pytest.raises(ValueError, match="int32"):
        S.sz_encode_paged(S.SZ_BF16, cb, x, page, torch.zeros(63, dtype=torch.int64), 1000, out, ob, None, out)
    assert calls == []
    # A count inside the tensor and a table of exactly ceil(n / page) ids pass
    # the binding's checks and reach the library (here: the recorder, which
    # only sees host-side arguments).
    assert S._count(S.SZ_BF16, x, 1000) == 1000 and S._count(S.SZ_BF16, x, 0) == 0
    S._block_table(torch.zeros(63, dtype=torch.int32), 1000, 16)
    S._block_table(torch.zeros(0, dtype=torch.int32), 0, 16)
