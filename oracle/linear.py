"""The dequant-fused linear layer, as its plain definition: ``Y = X · w_hat^T`` in float64.

TEST INFRASTRUCTURE ONLY (see ``oracle/__init__.py``).

推理优化与量化算子深度技术调研 §1.2 (dequantization fused into the GEMM:
``x_deq = (q - zp) * scale`` before the multiply) and 第 6 课：量化源码走读
(W4A16: weights stored as INT4, expanded back to 16-bit inside the GEMM, activations
kept in 16-bit).  The oracle expands the weights explicitly (``int4_g128.dequantize``
/ ``mxfp4.dequantize``) and multiplies in float64; X holds the exact values of the
bf16 activations.
"""
from __future__ import annotations

import numpy as np

from . import int4_g128, mxfp4


def linear(X: np.ndarray, W_hat: np.ndarray) -> np.ndarray:
    """``Y[m, n] = sum_k X[m, k] * W_hat[n, k]`` in float64."""
    X = np.asarray(X, dtype=np.float64)
    W_hat = np.asarray(W_hat, dtype=np.float64)
    if X.shape[1] != W_hat.shape[1]:
        raise ValueError("inner dimensions differ")
    return X @ W_hat.T


def dequantize(fmt: str, Wq, scales, zeros=None) -> np.ndarray:
    """Expanded weights of either format, float64 [N, K]."""
    if fmt == "int4_g128":
        return int4_g128.dequantize(Wq, scales, zeros)
    if fmt == "mxfp4":
        return mxfp4.dequantize(Wq, scales)
    raise ValueError("unknown format " + repr(fmt))


def linear_w4a16(fmt: str, X: np.ndarray, Wq, scales, zeros=None) -> np.ndarray:
    """``Y = X · dequant(Wq)^T`` in float64."""
    return linear(X, dequantize(fmt, Wq, scales, zeros))


def qkv_split(Y: np.ndarray, Nq: int, Nkv: int):
    """The fused QKV projection's output split into its three parts (推理优化与量化算子深度技术调研
    §4.2: one GEMM over the stacked [W_Q; W_K; W_V], then the result split into Q, K and V):
    ``(Y[:, :Nq], Y[:, Nq:Nq+Nkv], Y[:, Nq+Nkv:])`` for ``Y`` [M, Nq + 2 Nkv]."""
    Y = np.asarray(Y)
    if Nq < 1 or Nkv < 1 or Y.shape[1] != Nq + 2 * Nkv:
        raise ValueError("Y must be [M, Nq + 2 Nkv] with Nq, Nkv >= 1")
    return Y[:, :Nq], Y[:, Nq:Nq + Nkv], Y[:, Nq + Nkv:]


def linear_rows(fmt: str, X: np.ndarray, Wq, scales, zeros, rows) -> np.ndarray:
    """Only the output columns ``rows`` (weight rows) of ``Y``: float64 [M, len(rows)].

    For full-size checks on a sample of outputs: dequantizes only the sampled rows.
    """
    rows = np.asarray(rows)
    z = None if zeros is None else np.asarray(zeros)[rows]
    W_hat = dequantize(fmt, np.asarray(Wq)[rows], np.asarray(scales)[rows], z)
    return linear(X, W_hat)
