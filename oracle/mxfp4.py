"""OCP MXFP4: E2M1 elements, one E8M0 power-of-two scale per 32 elements along K.

TEST INFRASTRUCTURE ONLY (see ``oracle/__init__.py``).

Sources
-------
* 大模型量化推理引擎全景大复盘 (里程碑六 and 方程 3 "OCP MXFP4 向量化硬件吞吐密度"):
  32 four-bit elements share one E8M0 (pure exponent) scale.
* The same page, §三 simulator: the scale is ``2 ** ceil(log2(amax / 6))``,
  computed on float32 values (6 is the largest E2M1 magnitude).
* 第 6 课：量化源码走读 (量化范式与精度矩阵; 3. 正确性条件): micro-blocks of 32;
  K must be a multiple of the block.

Format
------
``W`` float32 [N, K] (K % 32 == 0) becomes
* ``Wq``     int32 [N, K/8]  -- the bytes [N, K/2]; byte ``j`` holds element ``2j``
  in its low nibble and ``2j+1`` in its high nibble; nibble = sign<<3 | magnitude code;
* ``scales`` uint8 [N, K/32] -- E8M0 byte ``e + 127``.

Steps for row n, block b, x = W[n, 32b : 32b + 32]:
1. ``amax = max |x|`` (float32).
2. ``r = amax / 6`` in float32; ``e = ceil(log2 r)`` exactly (from the float32
   value r), clamped to [-127, 127]; ``e = -127`` when r is 0.         (R6)
3. ``v = x * 2**-e`` (exact).
4. ``|v|`` rounds to the nearest of {0, .5, 1, 1.5, 2, 3, 4, 6}; a tie goes to the
   value whose magnitude code (its index in that list) is even; above 6
   saturates at 6.                                                       (R7)
5. code = sign(x)<<3 | magnitude code, the sign taken from the sign bit of x, so
   that -0 and negatives rounding to 0 give code 8.                      (R8)
   An all-zero block (amax == 0) gives E8M0 byte 0 and all codes 0.     (R6)
6. pack two codes per byte, element 2j in the low nibble.

Dequantization: ``w_hat = (-1)^sign * E2M1[mag] * 2**(byte - 127)``.
"""
from __future__ import annotations

import math

import numpy as np

BLOCK = 32
E2M1_GRID = np.array([0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0], dtype=np.float64)
E8M0_BIAS = 127


def e8m0_exponent(r: float) -> int:
    """``ceil(log2 r)`` for a non-negative float (exact), clamped to the E8M0 range; 0 maps to -127."""
    r = float(r)
    if r == 0.0:
        return -E8M0_BIAS
    m, ex = math.frexp(r)          # r = m * 2**ex, 0.5 <= m < 1, exact
    e = ex - 1 if m == 0.5 else ex
    return max(-E8M0_BIAS, min(E8M0_BIAS, e))


def e8m0_exponents(r: np.ndarray) -> np.ndarray:
    """Array form of :func:`e8m0_exponent` (``np.frexp`` is exact)."""
    r = np.asarray(r, dtype=np.float64)
    m, ex = np.frexp(r)
    e = np.where(m == 0.5, ex - 1, ex).astype(np.int64)
    e = np.where(r == 0.0, -E8M0_BIAS, e)
    return np.clip(e, -E8M0_BIAS, E8M0_BIAS)


def e2m1_round_magnitude(a: np.ndarray) -> np.ndarray:
    """Magnitude codes (0..7) of non-negative values: nearest grid value, ties to even code."""
    a = np.asarray(a, dtype=np.float64)
    d = np.abs(a[..., None] - E2M1_GRID)              # distance to every grid value
    best = np.argmin(d, axis=-1)                        # first (lowest) index among minima
    dmin = np.take_along_axis(d, best[..., None], axis=-1)[..., 0]
    nxt = np.minimum(best + 1, 7)
    d_next = np.take_along_axis(d, nxt[..., None], axis=-1)[..., 0]
    tie = (nxt != best) & (d_next == dmin)
    best = np.where(tie & (best % 2 == 1), nxt, best)
    return best.astype(np.uint8)


def quantize(W: np.ndarray):
    """Quantize and pack. Returns ``(Wq int32 [N,K/8], scales uint8 [N,K/32])``."""
    W = np.ascontiguousarray(W, dtype=np.float32)
    if W.ndim != 2:
        raise ValueError("W must be 2-D [N, K]")
    N, K = W.shape
    if K % BLOCK != 0:
        raise ValueError("K must be a multiple of 32")
    x = W.reshape(N, K // BLOCK, BLOCK)
    amax = np.abs(x).max(axis=-1)                                  # float32
    r = amax / np.float32(6.0)                                     # float32, round to nearest
    e = e8m0_exponents(r)
    v = x.astype(np.float64) * np.exp2(-e.astype(np.float64))[..., None]
    mag = e2m1_round_magnitude(np.abs(v))
    sign = (x.view(np.uint32) >> np.uint32(31)).astype(np.uint8)
    codes = (sign << np.uint8(3)) | mag
    codes[amax == 0] = 0
    scales = np.where(amax == 0, 0, e + E8M0_BIAS).astype(np.uint8)
    return pack(codes.reshape(N, K)), scales


def pack(codes: np.ndarray) -> np.ndarray:
    """Codes uint8 [N, K] -> int32 [N, K/8]: byte j = codes[2j] | codes[2j+1] << 4."""
    c = np.asarray(codes, dtype=np.uint8)
    N, K = c.shape
    b = (c[:, 0::2] & 0xF) | ((c[:, 1::2] & 0xF) << 4)
    return np.ascontiguousarray(b.astype(np.uint8)).view(np.int32).reshape(N, K // 8)


def unpack(Wq: np.ndarray) -> np.ndarray:
    """int32 [N, K/8] -> codes uint8 [N, K]."""
    b = np.ascontiguousarray(Wq).view(np.uint8)
    N, KB = b.shape
    out = np.empty((N, KB, 2), dtype=np.uint8)
    out[:, :, 0] = b & 0xF
    out[:, :, 1] = b >> 4
    return out.reshape(N, KB * 2)


def decode_e2m1(codes: np.ndarray) -> np.ndarray:
    """E2M1 code -> float64 value."""
    c = np.asarray(codes, dtype=np.uint8)
    val = E2M1_GRID[c & 7]
    return np.where(c & 8, -val, val)


def dequantize(Wq: np.ndarray, scales: np.ndarray) -> np.ndarray:
    """``w_hat = E2M1(code) * 2**(scale_byte - 127)`` in float64, shape [N, K]."""
    c = unpack(Wq)
    N, K = c.shape
    v = decode_e2m1(c).reshape(N, K // BLOCK, BLOCK)
    f = np.exp2(np.asarray(scales, dtype=np.float64) - E8M0_BIAS)
    return (v * f[..., None]).reshape(N, K)
