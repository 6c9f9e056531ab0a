"""Seeded synthetic BF16 workloads.

This module only draws random numbers and rounds them to BF16 bit patterns; it holds none
of the codec's arithmetic.  Both the CUDA path's tests and the oracle's tests feed the SAME
host arrays from here to the two sides.

The communication tensors the ZipCCL page evaluates on (Qwen3-A22B, DeepSeek-V3 and
Llama3-8B training traffic; "Evaluation" section) are not available, so each workload below
is a synthetic stand-in with the shape and value distribution of one of those buffers:

  weight_1m            1,048,576 values, N(0, 0.02^2) (weight-like), seed 0
  grad_bucket          4096 x 14336 (Llama3-8B hidden x FFN), N(0, 1e-3^2); exactly 0.1% of
                       positions, drawn without replacement, scaled by 100 in fp32, seed 1
  moe_a2a              16384 tokens x 7168 hidden (DeepSeek-V3), |x| = exp(N(-3, 1.5^2)),
                       random sign, exactly 0.5% of positions set to +0.0, seed 2
  sweep_<k>            2^k values, N(0, 1), k = 15 .. 29, seed 3 + k
  adversarial_256m     2^28 values in 16 segments of 2^24; segment j ~ N(0, s_j^2) with
                       s_j = 10^U(-6, 2); exactly 1% of positions replaced by uniformly random
                       16-bit patterns (NaN, Inf, subnormals and -0 included), seed 4

Recipe: numpy ``default_rng(seed)`` (PCG64) draws in fp64, values are rounded to fp32, then
to BF16 with round-to-nearest-even on the fp32 bit pattern.
"""
from __future__ import annotations

import numpy as np

_BLOCK = 1 << 24


def fp32_to_bf16_bits(a: np.ndarray) -> np.ndarray:
    """Round fp32 values to BF16 (nearest, ties to even) and return the uint16 bit patterns.

    Inputs here are finite and far from the fp32 overflow threshold, so no NaN handling is
    needed."""
    b = np.ascontiguousarray(a, dtype=np.float32).view(np.uint32)
    bias = np.uint32(0x7FFF) + ((b >> np.uint32(16)) & np.uint32(1))
    return ((b + bias) >> np.uint32(16)).astype(np.uint16)


def _gaussian_bf16(rng: np.random.Generator, n: int, sigma: float) -> np.ndarray:
    out = np.empty(n, dtype=np.uint16)
    for s in range(0, n, _BLOCK):
        e = min(n, s + _BLOCK)
        out[s:e] = fp32_to_bf16_bits((rng.standard_normal(e - s) * sigma).astype(np.float32))
    return out


def weight_1m() -> np.ndarray:
    rng = np.random.default_rng(0)
    return _gaussian_bf16(rng, 1 << 20, 0.02)


def grad_bucket(rows: int = 4096, cols: int = 14336) -> np.ndarray:
    n = rows * cols
    rng = np.random.default_rng(1)
    out = np.empty(n, dtype=np.uint16)
    hot = np.sort(rng.choice(n, size=n // 1000, replace=False))
    for s in range(0, n, _BLOCK):
        e = min(n, s + _BLOCK)
        v = (rng.standard_normal(e - s) * 1e-3).astype(np.float32)
        sel = hot[(hot >= s) & (hot < e)] - s
        v[sel] = v[sel] * np.float32(100.0)
        out[s:e] = fp32_to_bf16_bits(v)
    return out


def moe_a2a(tokens: int = 16384, hidden: int = 7168) -> np.ndarray:
    n = tokens * hidden
    rng = np.random.default_rng(2)
    out = np.empty(n, dtype=np.uint16)
    for s in range(0, n, _BLOCK):
        e = min(n, s + _BLOCK)
        mag = np.exp(rng.normal(-3.0, 1.5, e - s))
        neg = rng.integers(0, 2, e - s, dtype=np.uint8).astype(bool)
        out[s:e] = fp32_to_bf16_bits(np.where(neg, -mag, mag).astype(np.float32))
    zeros = rng.choice(n, size=int(round(n * 0.005)), replace=False)
    out[zeros] = 0x0000
    return out


def sweep(k: int) -> np.ndarray:
    if not 0 <= k <= 30:
        raise ValueError("sweep sizes are 2^k values")
    rng = np.random.default_rng(3 + k)
    return _gaussian_bf16(rng, 1 << k, 1.0)


def adversarial_256m(segments: int = 16, seg_len: int = 1 << 24) -> np.ndarray:
    n = segments * seg_len
    rng = np.random.default_rng(4)
    scales = 10.0 ** rng.uniform(-6.0, 2.0, segments)
    out = np.empty(n, dtype=np.uint16)
    for j in range(segments):
        out[j * seg_len:(j + 1) * seg_len] = _gaussian_bf16(rng, seg_len, float(scales[j]))
    pos = rng.choice(n, size=int(round(n * 0.01)), replace=False)
    out[pos] = rng.integers(0, 1 << 16, pos.size, dtype=np.uint32).astype(np.uint16)
    return out


WORKLOADS = {
    "weight_1m": weight_1m,
    "grad_bucket_4096x14336": grad_bucket,
    "moe_a2a_16384x7168": moe_a2a,
    "adversarial_256m": adversarial_256m,
}
WORKLOADS.update({f"sweep_2^{k}": (lambda k=k: sweep(k)) for k in range(15, 30)})


def make(name: str) -> np.ndarray:
    """Return the uint16 BF16 bit patterns of the named workload."""
    try:
        return WORKLOADS[name]()
    except KeyError:
        raise KeyError(f"unknown workload {name!r}; known: {sorted(WORKLOADS)}") from None


def random_patterns(n: int, seed: int) -> np.ndarray:
    """n uniformly random 16-bit patterns (every class of BF16 value)."""
    return np.random.default_rng(seed).integers(0, 1 << 16, n, dtype=np.uint32).astype(np.uint16)


def all_patterns() -> np.ndarray:
    """All 65,536 BF16 bit patterns in increasing order."""
    return np.arange(1 << 16, dtype=np.uint32).astype(np.uint16)
