"""Seeded synthetic inputs for the W4A16 linear layer.

This module is the one piece shared by the CUDA path's tests/benchmark and the
CPU oracle. It holds no quantization or GEMM arithmetic: it only draws numbers.

Recipe (the workloads of the weight-only 4-bit layer on LLaMA-3-8B and
Qwen2.5-72B shapes):

* weights ``W`` float32 [N, K] ~ Normal(0, sigma), then 1 % of the *input*
  columns (indices along K, drawn without replacement) multiplied by 10 -- the
  "salient channel" outliers that activation-aware quantization is about
  (推理优化与量化算子深度技术调研, §1.3 AWQ: about 1 % of channels matter most);
* activations ``X`` [M, K] ~ Normal(0, 1), rounded to bfloat16 with
  round-to-nearest-even, returned both as raw bf16 bit patterns and as the
  exact float32 values those patterns encode;
* calibration activations for GPTQ [n, K], n = 128 samples (推理优化与量化算子深度技术调研 §1.3:
  128 calibration samples usually suffice): correlated channels -- independent
  Normal(0, 1) noise plus a shared rank-16 component Z B (Z [n, 16], B [16, K], both
  standard normal, B scaled by 1/2) -- and 1 % of the channels multiplied by 10 (the
  salient channels of the same section).

Generator: numpy ``Generator(PCG64(seed))``; draws are float32 standard normals.
"""
from __future__ import annotations

import numpy as np

__all__ = [
    "weights",
    "activations",
    "bf16_bits_from_f32",
    "f32_from_bf16_bits",
    "calibration",
    "upper_factor",
    "SEEDS",
]

# Seed of each named workload (shape index ``i`` in the order the shapes are listed).
SEEDS = {
    "decode_4096x4096_m1": 0,
    "decode_llama3_8b": 1000,     # + shape index
    "decode_llama3_8b_mxfp4": 2000,  # + shape index
    "prefill_qwen25_72b": 3000,   # + shape index
    "crossover_8192": 4000,
}


def _rng(seed: int) -> np.random.Generator:
    return np.random.Generator(np.random.PCG64(seed))


def weights(seed: int, N: int, K: int, sigma: float, outlier_frac: float = 0.01,
            outlier_gain: float = 10.0) -> np.ndarray:
    """float32 [N, K] weight matrix with outlier input columns."""
    rng = _rng(seed)
    W = rng.standard_normal((N, K), dtype=np.float32)
    W *= np.float32(sigma)
    n_out = int(round(outlier_frac * K))
    if n_out > 0:
        cols = rng.choice(K, size=n_out, replace=False)
        W[:, cols] *= np.float32(outlier_gain)
    return W


def bf16_bits_from_f32(x: np.ndarray) -> np.ndarray:
    """Round float32 to bfloat16 (nearest, ties to even); returns uint16 bit patterns.

    Inputs here are finite draws, so NaN handling is not needed.
    """
    u = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32)
    lsb = (u >> np.uint32(16)) & np.uint32(1)
    r = (u + np.uint32(0x7FFF) + lsb) >> np.uint32(16)
    return r.astype(np.uint16)


def f32_from_bf16_bits(b: np.ndarray) -> np.ndarray:
    """The exact float32 value of each bfloat16 bit pattern."""
    return (np.ascontiguousarray(b, dtype=np.uint16).astype(np.uint32) << np.uint32(16)).view(np.float32)


def activations(seed: int, M: int, K: int, scale: float = 1.0):
    """bf16 activations [M, K]: (uint16 bit patterns, float32 exact values)."""
    rng = _rng(seed + 7919)  # a stream distinct from the weights drawn with the same seed
    x = rng.standard_normal((M, K), dtype=np.float32)
    if scale != 1.0:
        x *= np.float32(scale)
    bits = bf16_bits_from_f32(x)
    return bits, f32_from_bf16_bits(bits)


def calibration(seed: int, n: int, K: int, rank: int = 16, outlier_frac: float = 0.01,
                outlier_gain: float = 10.0) -> np.ndarray:
    """float32 [n, K] calibration activations with correlated and salient channels."""
    rng = _rng(seed + 104729)
    X = rng.standard_normal((n, K), dtype=np.float32)
    Z = rng.standard_normal((n, rank), dtype=np.float32)
    B = rng.standard_normal((rank, K), dtype=np.float32) * np.float32(0.5)
    X += Z @ B
    n_out = int(round(outlier_frac * K))
    if n_out > 0:
        cols = rng.choice(K, size=n_out, replace=False)
        X[:, cols] *= np.float32(outlier_gain)
    return X


def upper_factor(seed: int, K: int, off_sigma: float = 0.3) -> np.ndarray:
    """float32 [K, K] upper-triangular matrix with diagonal ~ Uniform(0.5, 1) and strictly
    upper entries ~ Normal(0, off_sigma / sqrt(K)): a stand-in for an inverse-Hessian Cholesky
    factor at sizes where computing one from calibration data would take minutes."""
    rng = _rng(seed + 130363)
    U = rng.standard_normal((K, K), dtype=np.float32) * np.float32(off_sigma / np.sqrt(K))
    U = np.triu(U, 1)
    U[np.arange(K), np.arange(K)] = rng.uniform(0.5, 1.0, K).astype(np.float32)
    return U
