"""Uniform (linear) quantizers, written from the pages' formulas.

TEST INFRASTRUCTURE ONLY (see ``oracle/__init__.py``).

Sources
-------
* 推理优化与量化算子深度技术调研, §1.2 INT8 对称/非对称量化:
  symmetric ``scale = max|x| / 127``, ``q = clamp(round(x/scale), -127, 127)``;
  asymmetric ``scale = (x_max - x_min)/255``, ``zero_point = round(-x_min/scale)``,
  ``q = clamp(round(x/scale) + zero_point, 0, 255)``; dequant ``(q - zp) * scale``.
* 第 1 章：推理加速全景, §4.1 均匀量化的数学基础: the same for b bits,
  ``s = (x_max - x_min)/(2^b - 1)``, ``z = round(-x_min/s)``, codes in ``[0, 2^b - 1]``,
  ``x_hat = (x_q - z)·s``; quantization error per step ``Δ = s``.
* 第 6 课：量化源码走读, 实践任务 (answer branch): block-wise symmetric fake
  quantization with a zero block mapped to scale 1 and Python ``round``
  (ties to even); invalid geometry raises ``ValueError``.

Readings taken where the pages are silent:
* R1 the asymmetric range always contains 0 (``x_min <= 0 <= x_max``);
* R2 a zero range uses scale 1 (the lesson's zero-block rule);
* R4 ``round`` is round-half-to-even (Python ``round`` / ``torch.round``).
"""
from __future__ import annotations

import numpy as np


def blockwise_symmetric_fake_quant(values, block_size, qmax):
    """Symmetric fake quantization per block of ``block_size`` values (plain Python floats).

    Per block: ``scale = max|x| / qmax`` (1.0 for an all-zero block), codes
    ``clamp(round(x/scale), -qmax, qmax)``, restored ``code * scale``.
    Returns ``(restored, scales)`` as Python lists.
    """
    if block_size <= 0 or qmax <= 0:
        raise ValueError("invalid quantization geometry")
    restored, scales = [], []
    n = len(values)
    start = 0
    while start < n:
        block = values[start:start + block_size]
        peak = 0.0
        for v in block:
            if abs(v) > peak:
                peak = abs(v)
        scale = (peak / qmax) if peak != 0.0 else 1.0
        scales.append(scale)
        for v in block:
            code = round(v / scale)  # Python round: half to even
            if code > qmax:
                code = qmax
            if code < -qmax:
                code = -qmax
            restored.append(code * scale)
        start += block_size
    return restored, scales


def symmetric_quantize(x: np.ndarray, bits: int = 8):
    """Per-tensor symmetric quantization in float32: ``scale = max|x| / (2^(b-1)-1)``.

    Returns ``(codes int32, scale float32)``; a zero tensor gets scale 1.
    """
    x = np.asarray(x, dtype=np.float32)
    qmax = (1 << (bits - 1)) - 1
    peak = np.float32(np.max(np.abs(x))) if x.size else np.float32(0)
    scale = np.float32(peak / np.float32(qmax)) if peak != 0 else np.float32(1)
    codes = np.clip(np.rint(x / scale), -qmax, qmax).astype(np.int32)
    return codes, scale


def asymmetric_params(x: np.ndarray, bits: int, scale_dtype=np.float32):
    """Scale and zero point of one asymmetric group, float32 arithmetic.

    ``x_min = min(min x, 0)``, ``x_max = max(max x, 0)`` (R1);
    ``s32 = (x_max - x_min) / (2^b - 1)``; the stored scale is ``s32`` rounded to
    ``scale_dtype`` (fp16 for the INT4 format), and a stored scale of 0 becomes 1
    (R2); ``z = round(-x_min / s)`` with the stored ``s``.
    Returns ``(s, z)`` as float32 scalars (``s`` exactly representable in ``scale_dtype``).
    """
    x = np.asarray(x, dtype=np.float32)
    levels = np.float32((1 << bits) - 1)
    x_min = np.minimum(np.float32(x.min()), np.float32(0))
    x_max = np.maximum(np.float32(x.max()), np.float32(0))
    s32 = np.float32(np.float32(x_max - x_min) / levels)
    s = np.float32(np.asarray(s32, dtype=np.float32).astype(scale_dtype))
    if s == 0:
        s = np.float32(1)
    z = np.float32(np.rint(np.float32(-x_min) / s))
    return s, z


def asymmetric_quantize(x: np.ndarray, bits: int, scale_dtype=np.float32):
    """Asymmetric quantization of one group: ``q = clamp(round(x/s) + z, 0, 2^b - 1)``.

    Returns ``(codes int32, s, z)``.
    """
    x = np.asarray(x, dtype=np.float32)
    s, z = asymmetric_params(x, bits, scale_dtype)
    qmax = (1 << bits) - 1
    q = np.clip(np.rint(x / s) + z, 0, qmax).astype(np.int32)
    return q, s, z


def asymmetric_dequantize(q, s, z) -> np.ndarray:
    """``x_hat = (q - z) * s`` in float64 (exact for these operands)."""
    return (np.asarray(q, dtype=np.float64) - np.float64(z)) * np.float64(s)
