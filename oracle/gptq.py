"""GPTQ: INT4 g128 quantization column by column, each column's error compensated on the
columns not yet quantized through the inverse Hessian.

TEST INFRASTRUCTURE ONLY (see ``oracle/__init__.py``).

第 1 章：推理加速全景 §4.2 (GPTQ), with 推理优化与量化算子深度技术调研 §1.3 and
量化与加速 (GPTQ):
* objective  min_Q ||W X - Q(W) X||^2 = sum over rows of (w - q(w)) H (w - q(w))^T with
  H = 2 X^T X + lambda I from calibration activations X [n, K];
* for column i = 0 .. K-1: quantize it, e_i = w_i - q(w_i), and for every later column j
  w_j := w_j - (e_i / H^-1[i, i]) * H^-1[i, j];
* H^-1 through its Cholesky factor, H^-1 = L L^T: the ratio H^-1[i, j] / H^-1[i, i] of the
  update is read from the factor.

Readings (where the pages leave a step open):
* G1  The factor is the upper one, U = L^T (H^-1 = U^T U).  In the sequential update the
      inverse Hessian of the columns still to be quantized has row i proportional to row i of
      U, so the update is  w_j := w_j - (e_i / U[i, i]) * U[i, j]  (j > i).
* G2  lambda = 0.01 * mean(diag(2 X^T X)).
* G3  Group parameters (s, z) of group g follow the INT4 g128 rules (``int4_g128``), computed
      from the current -- already compensated -- values of the group's 128 columns when the
      sweep reaches the group's first column; each column's codes use that column's current
      values.
* G4  The sweep runs in float32, every quotient, product and difference rounded on its own,
      in the order above, so the codes (integer decisions) are taken in the kernel's
      precision.  H, H^-1 and U are float64; U is handed to the sweep as float32.
* G5  The pages' block-of-128 "lazy batch" update is a memory-traffic optimisation of the
      same sweep; this oracle applies each update at once (the exact-arithmetic result is
      the same).
"""
from __future__ import annotations

import numpy as np

from . import int4_g128

GROUP = int4_g128.GROUP
DAMP = 0.01


def hessian(X: np.ndarray, damp: float = DAMP) -> np.ndarray:
    """``H = 2 X^T X + lambda I`` in float64, lambda = damp * mean(diag(2 X^T X)) (G2)."""
    X = np.asarray(X, dtype=np.float64)
    H = 2.0 * (X.T @ X)
    lam = damp * float(np.mean(np.diag(H)))
    return H + lam * np.eye(H.shape[0])


def inverse_cholesky_upper(H: np.ndarray) -> np.ndarray:
    """Upper-triangular ``U`` with ``H^-1 = U^T U`` (G1), float64."""
    H = np.asarray(H, dtype=np.float64)
    L = np.linalg.cholesky(H)                       # H = L L^T
    Li = np.linalg.solve(L, np.eye(H.shape[0]))     # L^-1
    Hinv = Li.T @ Li                                # H^-1
    Hinv = 0.5 * (Hinv + Hinv.T)
    return np.ascontiguousarray(np.linalg.cholesky(Hinv).T)   # H^-1 = (L')(L')^T = U^T U, U = L'^T


def sweep(W: np.ndarray, U: np.ndarray, return_trace: bool = False):
    """The GPTQ sweep over the columns of ``W`` float32 [N, K] with ``U`` float32 [K, K].

    Returns ``(Wq, scales, zeros)`` in the ``int4_g128`` packed format; with
    ``return_trace`` also ``e`` float32 [N, K] (the scaled errors e_i / U[i, i]) and the
    float32 [N, K/128, 128] values each group's parameters were computed from.
    """
    W = np.array(W, dtype=np.float32, copy=True)
    U = np.asarray(U, dtype=np.float32)
    N, K = W.shape
    if K % GROUP != 0 or U.shape != (K, K):
        raise ValueError("K must be a multiple of 128 and U must be [K, K]")
    G = K // GROUP
    q = np.zeros((N, K), dtype=np.uint32)
    s16 = np.zeros((N, G), dtype=np.float16)
    z = np.zeros((N, G), dtype=np.int32)
    e = np.zeros((N, K), dtype=np.float32)
    seen = np.zeros((N, G, GROUP), dtype=np.float32)
    for i in range(K):
        g = i // GROUP
        if i % GROUP == 0:                                   # G3
            seen[:, g, :] = W[:, i:i + GROUP]
            s16[:, g], z[:, g] = int4_g128.group_params(W[:, i:i + GROUP])
        qi = int4_g128.codes(W[:, i:i + 1], s16[:, g], z[:, g])[:, 0]
        q[:, i] = qi
        w_hat = (qi.astype(np.float32) - z[:, g].astype(np.float32)) * s16[:, g].astype(np.float32)
        ei = (W[:, i] - w_hat) / U[i, i]                     # e_i / U[i, i]      (G1, G4)
        e[:, i] = ei
        if i + 1 < K:
            W[:, i + 1:] = W[:, i + 1:] - ei[:, None] * U[i, i + 1:][None, :]
    out = (int4_g128.pack(q), s16, z.astype(np.float16))
    if return_trace:
        return out + (e, seen)
    return out


def quantize(W: np.ndarray, X: np.ndarray, damp: float = DAMP):
    """GPTQ of ``W`` [N, K] with calibration activations ``X`` [n, K]: ``(Wq, scales, zeros)``."""
    U = inverse_cholesky_upper(hessian(X, damp)).astype(np.float32)
    return sweep(W, U)
