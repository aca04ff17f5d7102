"""AWQ: activation-aware per-channel scaling of the salient input channels before INT4 g128
quantization.

TEST INFRASTRUCTURE ONLY (see ``oracle/__init__.py``).

第 1 章：推理加速全景 §4.4 (AWQ), 推理优化与量化算子深度技术调研 §1.3 (AWQ) and 量化与加速 (AWQ):
1. importance_j = mean over the calibration samples of |X_j| (input channel j);
2. the salient channels are the top 1 % by importance;
3. s_j = importance_j ^ alpha, alpha chosen by a grid search in [0, 1] minimising the output
   error || Q(W diag(s)) (X diag(s)^-1)^T - W X^T ||;
4. the packed weight is Q(W diag(s)) (INT4 g128); at run time the activations are divided
   by s (folded into the producer of X), so Q(W s) (x / s) ~ W x.

Readings:
* A1  Weights are multiplied by s and activations divided by it (推理优化与量化算子深度技术调研
      §1.3: W'' = W * s, x'' = x / s; 量化与加速: Q(w s)(x / s) ~ w x).  第 1 章 §4.4 writes
      W diag(s)^-1 and X diag(s) while its comments say the salient weights are enlarged and
      the activations shrunk; its formulas are read as garbled.
* A2  Only the top ceil(K / 100) channels by importance are scaled (量化与加速: only the top
      1 % most important channels; 第 1 章 step 1 selects them); s_j = 1 elsewhere, and also
      on a selected channel whose importance is 0 (all its calibration values are 0, so any
      scale leaves the loss unchanged; s = 0 would not be invertible).  Equal importances: the
      lower channel index ranks first.
* A3  The grid is alpha = a / 20, a = 0 .. 20 (第 1 章 gives [0, 1] without a step).  alpha = 0
      is plain round-to-nearest.  Among equal losses the smallest alpha wins.
* A4  The loss is || X (W_hat - W)^T ||_F^2 with W_hat = dequant(Q(W diag(s))) diag(s)^-1,
      float64, over the calibration set.
* A5  importance in float64, summed over the samples in order; s_j = float32(importance_j **
      alpha) computed in float64; W diag(s) in float32 (one rounding each), which is the
      quantizer's input.
"""
from __future__ import annotations

import numpy as np

from . import int4_g128

GRID = 20          # alpha = a / GRID, a = 0 .. GRID
SALIENT_FRAC = 0.01


def importance(X: np.ndarray) -> np.ndarray:
    """mean_n |X[n, j]| in float64, the samples added in order (A5)."""
    X = np.asarray(X, dtype=np.float32)
    acc = np.zeros(X.shape[1], dtype=np.float64)
    for n in range(X.shape[0]):
        acc = acc + np.abs(X[n]).astype(np.float64)
    return acc / float(X.shape[0])


def salient(imp: np.ndarray) -> np.ndarray:
    """Boolean mask of the top ceil(K / 100) channels by importance (A2)."""
    K = imp.shape[0]
    n_sal = int(np.ceil(SALIENT_FRAC * K))
    order = np.lexsort((np.arange(K), -imp))     # importance descending, index ascending
    mask = np.zeros(K, dtype=bool)
    mask[order[:n_sal]] = True
    return mask


def scales(imp: np.ndarray, mask: np.ndarray, a: int) -> np.ndarray:
    """float32 s for alpha = a / GRID (A2, A5)."""
    alpha = a / float(GRID)
    s = np.ones(imp.shape[0], dtype=np.float64)
    sel = mask & (imp > 0)
    s[sel] = imp[sel] ** alpha
    return s.astype(np.float32)


def quantize_scaled(W: np.ndarray, s: np.ndarray):
    """INT4 g128 of W diag(s), the product rounded to float32 (A5)."""
    Ws = np.asarray(W, dtype=np.float32) * np.asarray(s, dtype=np.float32)[None, :]
    return int4_g128.quantize(Ws)


def loss(W: np.ndarray, X: np.ndarray, s: np.ndarray) -> float:
    """|| X (W_hat - W)^T ||_F^2 in float64 (A4)."""
    Wq, sc, z = quantize_scaled(W, s)
    W_hat = int4_g128.dequantize(Wq, sc, z) / np.asarray(s, dtype=np.float64)[None, :]
    E = np.asarray(X, dtype=np.float64) @ (W_hat - np.asarray(W, dtype=np.float64)).T
    return float(np.sum(E * E))


def search(W: np.ndarray, X: np.ndarray):
    """Returns ``(a_best, s float32 [K], losses float64 [GRID + 1], (Wq, scales, zeros))``."""
    imp = importance(X)
    mask = salient(imp)
    losses = np.array([loss(W, X, scales(imp, mask, a)) for a in range(GRID + 1)])
    a_best = int(np.argmin(losses))               # first minimum: the smallest alpha (A3)
    s = scales(imp, mask, a_best)
    return a_best, s, losses, quantize_scaled(W, s)
