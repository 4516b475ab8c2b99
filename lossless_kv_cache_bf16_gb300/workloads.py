"""Seeded synthetic KV-cache tensors (the workloads the codec is measured on).

This module only builds inputs.  It holds none of the codec's arithmetic and
is the one module that both the CUDA path's tests/bench and the CPU oracle's
callers share.  The pages measure on real KV activations of Qwen, Llama and
Phi models over WikiText, HumanEval and MMLU (SplitZip technical summary,
gist.science/es, "Metodologia: SplitZip" and "Resultados"); no model or
dataset is available here, so these seeded tensors with the shapes and value
structure of such KV caches stand in for them.

Every tensor is drawn with a ``torch.Generator`` on the requested device in
fp32 and rounded to nearest-even into bf16 (or float8_e5m2).  The same seed
on CUDA and on the CPU gives different numbers; a parity check always hands
both sides the same tensor.
"""
from __future__ import annotations

import math
from dataclasses import dataclass

import torch

BF16 = torch.bfloat16
E5M2 = torch.float8_e5m2


def _gen(device, seed: int) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    return g


def _lognormal(shape, sigma, g, device):
    return torch.exp(sigma * torch.randn(shape, generator=g, device=device))


# ---- configuration 1: tiny K tensor -------------------------------------------

def kv_tiny(device="cpu", seed: int = 0) -> torch.Tensor:
    """BF16 K tensor [2048 tokens, 8 kv heads, 64 head dim]: N(0,1) times a
    per-(head, dim) lognormal(0, 1) scale."""
    g = _gen(device, seed)
    scale = _lognormal((8, 64), 1.0, g, device)
    return (torch.randn((2048, 8, 64), generator=g, device=device) * scale).to(BF16)


# ---- configuration 2: Llama-3-8B-shaped prefill KV -------------------------------

def llama8b_prefill(device="cpu", seed: int = 0, layers: int = 32, tokens: int = 8192,
                    dtype=BF16) -> torch.Tensor:
    """[layers, 2 (K, V), tokens, 8 kv heads, 128 head dim].  K: N(0,1) times a
    lognormal(0, 1) scale per (layer, head, dim) channel, 2% of channels
    multiplied by 20 as outliers.  V: N(0, 0.5) (0.5 read as the standard
    deviation).  Built layer by layer in fp32, then rounded to `dtype`."""
    g = _gen(device, seed)
    out = torch.empty((layers, 2, tokens, 8, 128), dtype=dtype, device=device)
    for layer in range(layers):
        scale = _lognormal((8, 128), 1.0, g, device)
        outlier = torch.rand((8, 128), generator=g, device=device) < 0.02
        scale = torch.where(outlier, scale * 20.0, scale)
        out[layer, 0] = (torch.randn((tokens, 8, 128), generator=g, device=device) * scale).to(dtype)
        out[layer, 1] = (torch.randn((tokens, 8, 128), generator=g, device=device) * 0.5).to(dtype)
    return out


# ---- configuration 3: long-context GQA KV ------------------------------------------

def long_ctx_gqa(device="cpu", seed: int = 0, layers: int = 28, tokens: int = 32768) -> torch.Tensor:
    """[layers, 2, tokens, 4 kv heads, 128 head dim]: Student-t (nu = 4) times a
    lognormal(0, 1.5) scale per (layer, K/V, head, dim) channel times a
    per-layer scale uniform in [0.25, 4], so exponents drift across layers.
    Student-t(4) = Z / sqrt(W / 4) with W chi-square(4) = -2 ln(U1 U2)."""
    g = _gen(device, seed)
    out = torch.empty((layers, 2, tokens, 4, 128), dtype=BF16, device=device)
    for layer in range(layers):
        layer_scale = 0.25 + 3.75 * torch.rand((), generator=g, device=device)
        for kv in range(2):
            scale = _lognormal((4, 128), 1.5, g, device) * layer_scale
            z = torch.randn((tokens, 4, 128), generator=g, device=device)
            u1 = torch.rand((tokens, 4, 128), generator=g, device=device).clamp_min_(1e-30)
            u2 = torch.rand((tokens, 4, 128), generator=g, device=device).clamp_min_(1e-30)
            w = -2.0 * torch.log(u1 * u2)
            out[layer, kv] = (z / torch.sqrt(w / 4.0) * scale).to(BF16)
    return out


# ---- configuration 4: escape-rate sweep ----------------------------------------------

SWEEP_N = 134_217_728
SWEEP_P = (0.0, 0.001, 0.01, 0.05)


def gaussian_flat(device="cpu", seed: int = 0, n: int = SWEEP_N, scale: float = 1.0) -> torch.Tensor:
    g = _gen(device, seed)
    return (torch.randn((n,), generator=g, device=device) * scale).to(BF16)


def _allowed_exponents(codebook) -> torch.Tensor:
    cb = {int(v) for v in codebook}
    return torch.tensor([e for e in range(1, 255) if e not in cb], dtype=torch.int32)


def _with_exponents(x: torch.Tensor, idx: torch.Tensor, exps: torch.Tensor) -> torch.Tensor:
    """Copy of bf16 x whose elements at idx get the biased exponents exps (sign
    and mantissa kept): input construction for the escape sweep."""
    bits = x.view(torch.int16).to(torch.int32) & 0xFFFF
    sel = bits[idx]
    bits[idx] = (sel & 0x807F) | (exps.to(torch.int32) << 7)
    return bits.to(torch.int16).view(BF16)


def escape_sweep(p: float, codebook, device="cpu", n: int = SWEEP_N) -> torch.Tensor:
    """N(0,1) bf16 (seed 0) where exactly round(p n) positions, drawn without
    replacement (seed 2), get an exponent drawn uniformly from {1..254} minus
    the codebook; sign and mantissa are kept."""
    x = gaussian_flat(device, 0, n)
    k = int(round(p * n))
    if k == 0:
        return x
    g = _gen(device, 2)
    idx = torch.randperm(n, generator=g, device=device)[:k]
    allowed = _allowed_exponents(codebook).to(device)
    exps = allowed[torch.randint(0, allowed.numel(), (k,), generator=g, device=device)]
    return _with_exponents(x, idx, exps)


def all_escape(codebook, device="cpu", n: int = SWEEP_N, seed: int = 3) -> torch.Tensor:
    """Every element gets an exponent outside the codebook (uniform over
    {1..254} minus the codebook); sign and mantissa from N(0,1)."""
    x = gaussian_flat(device, 0, n)
    g = _gen(device, seed)
    allowed = _allowed_exponents(codebook).to(device)
    exps = allowed[torch.randint(0, allowed.numel(), (n,), generator=g, device=device)]
    return _with_exponents(x, torch.arange(n, device=device), exps)


NON_NAN_PER_SIGN = 255 * 128 + 1  # exponents 0..254 with any mantissa, plus infinity


def adversarial(device="cpu", n: int = SWEEP_N, seed: int = 4) -> torch.Tensor:
    """Uniformly random 16-bit patterns with NaNs excluded: a uniform index into
    the 2 x 32,641 non-NaN patterns (no rejection loop needed)."""
    g = _gen(device, seed)
    k = torch.randint(0, 2 * NON_NAN_PER_SIGN, (n,), generator=g, device=device, dtype=torch.int64)
    bits = (k // NON_NAN_PER_SIGN) * 32768 + (k % NON_NAN_PER_SIGN)
    return bits.to(torch.int32).to(torch.int16).view(BF16)


# ---- configuration 5: FP8 E5M2 KV ------------------------------------------------------

def fp8_e5m2_kv(device="cpu", seed: int = 0, layers: int = 32, tokens: int = 16384) -> torch.Tensor:
    """[layers, 2, tokens, 8, 128]: the Llama-3-8B recipe in fp32, rounded to
    nearest-even into float8_e5m2."""
    return llama8b_prefill(device, seed, layers, tokens, dtype=E5M2)


# ---- the configurations --------------------------------------------------------------

@dataclass(frozen=True)
class Config:
    name: str
    dtype: str            # "bf16" or "e5m2"
    numel: int
    description: str


CONFIGS = {
    "tiny": Config("tiny", "bf16", 2048 * 8 * 64, "BF16 K [2048, 8, 64], N(0,1) x lognormal(0,1) per channel"),
    "llama8b_prefill": Config("llama8b_prefill", "bf16", 32 * 2 * 8192 * 8 * 128,
                              "BF16 KV [32, 2, 8192, 8, 128], Llama-3-8B-shaped prefill"),
    "long_ctx_gqa": Config("long_ctx_gqa", "bf16", 28 * 2 * 32768 * 4 * 128,
                           "BF16 KV [28, 2, 32768, 4, 128], Student-t(4), drifting layer scales"),
    "escape_sweep": Config("escape_sweep", "bf16", SWEEP_N, "BF16 flat 128M, controlled escape fraction"),
    "fp8_e5m2": Config("fp8_e5m2", "e5m2", 32 * 2 * 16384 * 8 * 128, "E5M2 KV [32, 2, 16384, 8, 128]"),
}


def workload(name: str, device="cpu") -> torch.Tensor:
    """The full tensor of a named configuration (the sweep's p = 0 point)."""
    if name == "tiny":
        return kv_tiny(device, 0)
    if name == "llama8b_prefill":
        return llama8b_prefill(device, 0)
    if name == "long_ctx_gqa":
        return long_ctx_gqa(device, 0)
    if name == "escape_sweep":
        return gaussian_flat(device, 0)
    if name == "fp8_e5m2":
        return fp8_e5m2_kv(device, 0)
    raise KeyError(name)


def calibration_sample(name: str, device="cpu", full: torch.Tensor | None = None) -> torch.Tensor:
    """The sample each configuration calibrates its codebook on."""
    if name == "tiny":
        return kv_tiny(device, 1)
    if name == "llama8b_prefill":
        return llama8b_prefill(device, 1, layers=1)
    if name == "long_ctx_gqa":
        # Layer 0 (K and V) of the tensor itself.
        full = long_ctx_gqa(device, 0, layers=1) if full is None else full
        return full[0:1].contiguous()
    if name == "escape_sweep":
        return gaussian_flat(device, 1)
    if name == "fp8_e5m2":
        return fp8_e5m2_kv(device, 1, layers=1)
    raise KeyError(name)


def bytes_of(t: torch.Tensor) -> int:
    return t.numel() * t.element_size()


def ceil_div(a: int, b: int) -> int:
    return -(-a // b) if b else math.inf
