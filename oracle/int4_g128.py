"""Asymmetric INT4, group size 128 along K: quantize, pack, unpack, dequantize.

TEST INFRASTRUCTURE ONLY (see ``oracle/__init__.py``).

Format
------
``W`` float32 [N, K] (N output rows, K input columns, K % 128 == 0) becomes
* ``Wq``     int32   [N, K/8]   -- eight 4-bit codes per word (第 6 课：量化源码走读,
  源码分层架构与生命周期: "8 个 INT4 紧凑打包为一个 int32" plus Scale/Zero-Point tensors);
* ``scales`` float16 [N, K/128] -- one scale per (row, group);
* ``zeros``  float16 [N, K/128] -- one zero point per (row, group), a small
  non-negative integer.

Steps for row n, group g, x = W[n, 128g : 128g + 128] (float32 arithmetic):
1. ``x_min = min(min x, 0)``, ``x_max = max(max x, 0)``                (reading R1)
2. ``s32 = (x_max - x_min) / 15``  (推理优化与量化算子深度技术调研 §1.2 with 2^4 - 1 levels;
   第 1 章：推理加速全景 §4.1)
3. ``s = fp16(min(s32, 65504))`` rounded to nearest even and stored; if that is 0,
   ``s = 1`` (readings R3, R2; the ``min`` saturates a scale that would round past the
   largest finite fp16 value to +inf at that value, reading R16)
4. ``z = min(round(-x_min / s), 15)`` with ``s`` the stored scale, round half to even
   (R4); the ``min`` keeps the zero point a code when the stored scale is far below
   ``s32`` (fp16-subnormal or saturated scales, reading R16)
5. ``q = clamp(round(x / s) + z, 0, 15)``
6. pack: word ``j`` holds ``q[8j + i]`` in bits ``4i .. 4i+3`` (low nibble first, R5)

Dequantization ``w_hat = (q - z) * s`` (推理优化与量化算子深度技术调研 §1.2, "x_deq = (q - zp) * scale").
"""
from __future__ import annotations

import numpy as np

GROUP = 128
LEVELS = 15
FP16_MAX = 65504.0   # largest finite IEEE binary16 value, (2 - 2^-10) * 2^15


def quantize(W: np.ndarray):
    """Quantize and pack. Returns ``(Wq int32 [N,K/8], scales fp16 [N,K/128], zeros fp16 [N,K/128])``."""
    W = np.ascontiguousarray(W, dtype=np.float32)
    if W.ndim != 2:
        raise ValueError("W must be 2-D [N, K]")
    N, K = W.shape
    if K % GROUP != 0:
        raise ValueError("K must be a multiple of 128")
    x = W.reshape(N, K // GROUP, GROUP)
    s16, z = group_params(x)
    q = codes(x, s16, z)
    return pack(q.reshape(N, K)), s16, z.astype(np.float16)


def group_params(x: np.ndarray):
    """Steps 1-4 for groups ``x`` float32 [..., 128]: ``(s fp16 [...], z int32 [...])``."""
    x = np.asarray(x, dtype=np.float32)
    x_min = np.minimum(x.min(axis=-1), np.float32(0))
    x_max = np.maximum(x.max(axis=-1), np.float32(0))
    s32 = (x_max - x_min) / np.float32(LEVELS)                 # float32, round to nearest
    s32 = np.minimum(s32, np.float32(FP16_MAX))                 # saturate (R16)
    s16 = np.asarray(s32.astype(np.float16))                    # stored scale
    s16[s16 == 0] = np.float16(1)
    s = s16.astype(np.float32)
    z = np.minimum(np.rint((-x_min) / s), np.float32(LEVELS))   # a code: 0 .. 15 (R16)
    return s16, z.astype(np.int32)


def codes(x: np.ndarray, s16: np.ndarray, z: np.ndarray) -> np.ndarray:
    """Step 5 for values ``x`` float32 [..., n] of groups with scale ``s16`` / zero ``z`` [...]:
    ``q = clamp(round(x / s) + z, 0, 15)`` (uint32)."""
    s = np.asarray(s16).astype(np.float32)[..., None]
    zf = np.asarray(z).astype(np.float32)[..., None]
    q = np.clip(np.rint(np.asarray(x, dtype=np.float32) / s) + zf, 0, LEVELS)
    return q.astype(np.uint32)


def pack(q: np.ndarray) -> np.ndarray:
    """Codes [N, K] (0..15) -> int32 [N, K/8], code ``8j + i`` in bits ``4i..4i+3`` of word ``j``."""
    q = np.asarray(q).astype(np.uint32)
    N, K = q.shape
    q8 = q.reshape(N, K // 8, 8)
    word = np.zeros((N, K // 8), dtype=np.uint32)
    for i in range(8):
        word |= (q8[:, :, i] & np.uint32(0xF)) << np.uint32(4 * i)
    return word.view(np.int32)


def unpack(Wq: np.ndarray) -> np.ndarray:
    """int32 [N, K/8] -> codes uint8 [N, K]."""
    w = np.ascontiguousarray(Wq).view(np.uint32)
    N, KW = w.shape
    out = np.empty((N, KW, 8), dtype=np.uint8)
    for i in range(8):
        out[:, :, i] = (w >> np.uint32(4 * i)) & np.uint32(0xF)
    return out.reshape(N, KW * 8)


def dequantize(Wq: np.ndarray, scales: np.ndarray, zeros: np.ndarray) -> np.ndarray:
    """``w_hat[n, k] = (q[n, k] - z[n, k//128]) * s[n, k//128]`` in float64, shape [N, K]."""
    q = unpack(Wq).astype(np.float64)
    N, K = q.shape
    s = np.asarray(scales, dtype=np.float64)
    z = np.asarray(zeros, dtype=np.float64)
    qg = q.reshape(N, K // GROUP, GROUP)
    return ((qg - z[..., None]) * s[..., None]).reshape(N, K)
