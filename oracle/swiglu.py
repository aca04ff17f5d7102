"""The fused gate+up projection with its SwiGLU activation, as its plain definition.

TEST INFRASTRUCTURE ONLY (see ``oracle/__init__.py``).

推理优化与量化算子深度技术调研 §4.6 (GEMM + Activation + Bias fusion): the SwiGLU FFN
computes ``gate = x W_gate^T`` and ``up = x W_up^T``, fused into one GEMM over the
stacked weight ``[W_gate; W_up]``, then ``hidden = SiLU(gate) * up`` element-wise.

* ``silu``               -- SiLU(x) = x * sigmoid(x) = x / (1 + e^-x).  The page names the
  function without defining it; this is its standard definition.
* ``swiglu_w4a16``       -- ``Y = SiLU(X Wg^T) * (X Wu^T)`` in float64, where the fused
  packed weight holds the F gate rows first, then the F up rows (the page's
  ``[W_gate; W_up]``), each expanded by ``linear.dequantize``.
* ``interleave_gate_up`` -- the row order the CUDA kernels read the fused weight in:
  gate and up rows alternate in blocks of 8, interleaved row ``16 q + 8 h + i`` being
  stacked row ``h F + 8 q + i`` (h = 0 gate, 1 up).  A pure permutation of rows, applied
  offline once, like the weight re-layout step of 第 6 课：量化源码走读 §2
  (权重重排 in ``process_weights_after_loading``).  Row-wise quantization commutes with it.
"""
from __future__ import annotations

import numpy as np

from . import linear


def silu(x) -> np.ndarray:
    """SiLU(x) = x / (1 + exp(-x)) in float64 (evaluated without overflow for x << 0)."""
    x = np.asarray(x, dtype=np.float64)
    out = np.empty_like(x)
    pos = x >= 0
    out[pos] = x[pos] / (1.0 + np.exp(-x[pos]))
    e = np.exp(x[~pos])                       # x < 0: x e^x / (1 + e^x), e^x <= 1
    out[~pos] = x[~pos] * e / (1.0 + e)
    return out


def swiglu(gate, up) -> np.ndarray:
    """``SiLU(gate) * up`` element-wise, float64."""
    return silu(gate) * np.asarray(up, dtype=np.float64)


def swiglu_w4a16(fmt: str, X: np.ndarray, Wq, scales, zeros=None) -> np.ndarray:
    """``Y[M, F] = SiLU(X Wg^T) * (X Wu^T)`` for the stacked packed weight ``[Wg; Wu]``
    of 2F rows (gate rows first), float64."""
    H = linear.linear_w4a16(fmt, X, Wq, scales, zeros)   # [M, 2F]
    if H.shape[1] % 2:
        raise ValueError("the stacked gate+up weight needs an even number of rows")
    F = H.shape[1] // 2
    return swiglu(H[:, :F], H[:, F:])


def swiglu_rows(fmt: str, X: np.ndarray, Wq, scales, zeros, F: int, cols) -> np.ndarray:
    """Only the output columns ``cols`` of ``swiglu_w4a16`` (stacked layout, 2F rows):
    float64 [M, len(cols)].  Dequantizes just the gate rows ``cols`` and up rows ``F + cols``."""
    cols = np.asarray(cols)
    g = linear.linear_rows(fmt, X, Wq, scales, zeros, cols)
    u = linear.linear_rows(fmt, X, Wq, scales, zeros, cols + F)
    return swiglu(g, u)


def interleave_index(F: int) -> np.ndarray:
    """``src[r]``: the stacked row that interleaved row r holds (F % 8 == 0)."""
    if F < 0 or F % 8:
        raise ValueError("F must be a non-negative multiple of 8")
    src = np.empty(2 * F, dtype=np.int64)
    for r in range(2 * F):
        q, h, i = r // 16, (r // 8) % 2, r % 8
        src[r] = h * F + 8 * q + i
    return src


def interleave_gate_up(A, F: int) -> np.ndarray:
    """Rows of the stacked ``[gate; up]`` array ``A`` (2F rows, any row width) in the
    interleaved order."""
    A = np.asarray(A)
    if A.shape[0] != 2 * F:
        raise ValueError("expected 2F rows")
    return A[interleave_index(F)]
