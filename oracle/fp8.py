"""FP8 E4M3 W8A8: per-output-channel weight scales, per-token activation scales, and the
linear layer on the quantized operands.

TEST INFRASTRUCTURE ONLY (see ``oracle/__init__.py``).

Format (推理优化与量化算子深度技术调研 §1.4: FP8 E4M3 for weights and activations, a floating
point format rather than an integer one, the tensor stored as ``torch.float8_e4m3fn`` with
its FP32 scale kept beside it; 量化与加速, 数值格式谱系: E4M3 spans +-448):
* a code is 1 sign bit, 4 exponent bits (bias 7) and 3 mantissa bits: exponent field e > 0
  gives (1 + m/8) 2^(e-7), e = 0 gives the subnormals (m/8) 2^-6; e = 15 with m = 7 is NaN
  and there is no infinity, so the largest finite value is 1.75 * 2^8 = 448 (reading F1);
* rows of the weight W [N, K] (output channels) and of the activations X [M, K] (tokens)
  each get one float32 scale ``s = amax / 448`` (a zero row gets 1), and each element the
  E4M3 code of ``x / s`` (float32 division), rounded to the nearest value, ties to the even
  code, saturating at +-448, sign kept on a zero (readings F2, F3);
* the layer is ``Y[m, n] = s_x[m] s_w[n] sum_k q_x[m, k] q_w[n, k]`` (reading F4; computed
  here in float64: every product of two E4M3 values is exact).
"""
from __future__ import annotations

import numpy as np

E4M3_MAX = 448.0
NAN_CODES = (0x7F, 0xFF)


def e4m3_values() -> np.ndarray:
    """float64 value of each of the 256 codes (NaN for the two NaN codes)."""
    v = np.empty(256, dtype=np.float64)
    for c in range(256):
        s, e, m = c >> 7, (c >> 3) & 0xF, c & 0x7
        if e == 15 and m == 7:
            v[c] = np.nan
            continue
        mag = (m / 8.0) * 2.0 ** -6 if e == 0 else (1.0 + m / 8.0) * 2.0 ** (e - 7)
        v[c] = -mag if s else mag
    return v


_VALUES = e4m3_values()
_MAG = _VALUES[:127]          # codes 0x00 .. 0x7E: 0 .. 448, strictly increasing


def e4m3_round(v: np.ndarray) -> np.ndarray:
    """E4M3 codes (uint8) of float32 values: nearest finite value, ties to the even code,
    |v| >= 448 saturating to 448; the sign bit of v is kept (so -0.0 gives 0x80)."""
    v = np.asarray(v, dtype=np.float32)
    a = np.abs(v).astype(np.float64)
    hi = np.clip(np.searchsorted(_MAG, a, side="left"), 1, 126)   # _MAG[hi-1] < a <= _MAG[hi], inside
    lo = hi - 1
    dl, dh = a - _MAG[lo], _MAG[hi] - a
    code = np.where(dl < dh, lo, hi)
    tie = dl == dh
    code = np.where(tie, np.where(lo % 2 == 0, lo, hi), code)
    code = np.where(a >= E4M3_MAX, 126, code)
    code = np.where(a == 0.0, 0, code)
    sign = (v.view(np.uint32) >> np.uint32(31)).astype(np.uint8)
    return ((sign << np.uint8(7)) | code.astype(np.uint8)).astype(np.uint8)


def quantize_rows(A: np.ndarray):
    """Per-row E4M3 quantization of float32 [R, K]: ``(codes uint8 [R, K], scales float32 [R])``."""
    A = np.ascontiguousarray(A, dtype=np.float32)
    if A.ndim != 2:
        raise ValueError("expected a 2-D array")
    amax = np.abs(A).max(axis=1) if A.shape[1] else np.zeros(A.shape[0], np.float32)
    s = (amax / np.float32(E4M3_MAX)).astype(np.float32)          # float32, round to nearest
    s[s == 0] = np.float32(1)                                      # zero row (F3)
    codes = e4m3_round(A / s[:, None])                             # float32 division
    return codes, s


def quantize_weights(W: np.ndarray):
    """W float32 [N, K] -> (Wq uint8 [N, K], s_w float32 [N]): one scale per output channel."""
    return quantize_rows(W)


def quantize_activations(X: np.ndarray):
    """X [M, K] (the exact values of bf16 activations) -> (Xq uint8 [M, K], s_x float32 [M]):
    one scale per token."""
    return quantize_rows(X)


def dequantize_rows(codes: np.ndarray, scales: np.ndarray) -> np.ndarray:
    """float64 ``E4M3(code) * scale`` per row."""
    return _VALUES[np.asarray(codes, dtype=np.uint8)] * np.asarray(scales, dtype=np.float64)[:, None]


def linear_w8a8(Xq: np.ndarray, s_x: np.ndarray, Wq: np.ndarray, s_w: np.ndarray) -> np.ndarray:
    """``Y[m, n] = s_x[m] s_w[n] sum_k E4M3(Xq[m, k]) E4M3(Wq[n, k])`` in float64 [M, N]."""
    x = _VALUES[np.asarray(Xq, dtype=np.uint8)]
    w = _VALUES[np.asarray(Wq, dtype=np.uint8)]
    return (x @ w.T) * np.asarray(s_x, dtype=np.float64)[:, None] * np.asarray(s_w, dtype=np.float64)[None, :]


def linear_w8a8_rows(Xq, s_x, Wq, s_w, rows) -> np.ndarray:
    """Only the output columns ``rows``: float64 [M, len(rows)]."""
    rows = np.asarray(rows)
    return linear_w8a8(Xq, s_x, np.asarray(Wq)[rows], np.asarray(s_w)[rows])
