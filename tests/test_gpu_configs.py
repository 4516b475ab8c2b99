"""Full-size workloads: GPU streams byte-identical to the oracle, decode
bit-exact (GPU).  These are the configurations the bench measures, at their
full sizes, in the bench's launch configuration (one encode and one decode
launch over the whole tensor)."""
import numpy as np
import pytest
import torch

from lossless_kv_cache_bf16_gb300 import workloads as W
from oracle import oracle as O
from tests import gpu_codec as G

pytestmark = pytest.mark.gpu

ODT = {"bf16": O.BF16, "e5m2": O.E5M2}


def full_parity(orc, kind, x, sample):
    dt, odt = G.DT[kind], ODT[kind]
    cb, hist = G.calibrate(dt, sample)
    sh = G.as_bytes(sample)
    assert np.array_equal(hist, orc.histogram(odt, sh))
    assert np.array_equal(cb, orc.codebook_from_histogram(odt, hist))
    del sh
    xh = G.as_bytes(x)
    n = G.elements(dt, x)
    got, status, size = G.encode(dt, cb, x)
    assert status == 0
    want = orc.encode(odt, cb, xh)
    assert size == want.size
    assert np.array_equal(got, want), "stream differs from the oracle"
    del want
    st, y, guard_ok = G.decode(dt, got, n)
    assert st == 0 and guard_ok
    assert np.array_equal(y, xh), "decode is not bit-exact"
    n_esc = (size - orc.encoded_size(odt, n, 0)) // 3
    return n_esc / max(n, 1), (2 if kind == "bf16" else 1) * n / size


def test_llama8b_prefill_full(orc):
    x = W.workload("llama8b_prefill", "cuda")
    eps, ratio = full_parity(orc, "bf16", x, W.calibration_sample("llama8b_prefill", "cuda"))
    print(f"llama8b_prefill: escape rate {eps:.5f}, ratio {ratio:.4f}")
    assert ratio > 1.3


def test_long_ctx_gqa_full(orc):
    x = W.workload("long_ctx_gqa", "cuda")
    eps, ratio = full_parity(orc, "bf16", x, W.calibration_sample("long_ctx_gqa", "cuda", full=x))
    print(f"long_ctx_gqa: escape rate {eps:.5f}, ratio {ratio:.4f}")


def test_fp8_e5m2_full(orc):
    x = W.workload("fp8_e5m2", "cuda")
    eps, ratio = full_parity(orc, "e5m2", x, W.calibration_sample("fp8_e5m2", "cuda"))
    print(f"fp8_e5m2: escape rate {eps:.5f}, ratio {ratio:.4f}")
    assert ratio <= 8 / 7


@pytest.mark.parametrize("point", [f"p={p}" for p in W.SWEEP_P] + ["adversarial", "all_escape"])
def test_escape_sweep_full(orc, point):
    sample = W.calibration_sample("escape_sweep", "cuda")
    cb, _ = G.calibrate(G.DT["bf16"], sample)
    if point == "adversarial":
        x = W.adversarial("cuda")
    elif point == "all_escape":
        x = W.all_escape(cb, "cuda")
    else:
        x = W.escape_sweep(float(point[2:]), cb, "cuda")
    eps, ratio = full_parity(orc, "bf16", x, sample)
    print(f"escape sweep {point}: escape rate {eps:.5f}, ratio {ratio:.4f}")
    if point == "all_escape":
        assert eps == 1.0
