"""W4A4 in MXFP4: weights and activations both quantized to OCP MXFP4, the layer on the two
dequantized operands.

TEST INFRASTRUCTURE ONLY (see ``oracle/__init__.py``).

第 6 课：量化源码走读 (量化范式与精度矩阵: NVFP4/MXFP4 micro-scaling quantizes weights and
activations to 4 bits with a shared scale per small block; Q2 answer: the activations are
quantized on the fly, with the accuracy caveats that brings) and 大模型量化推理引擎全景大复盘
(里程碑六 / 方程 3: 32 elements share one E8M0 power-of-two scale).  The activations follow
exactly the weights' MXFP4 rules of ``mxfp4.quantize`` (reading W1: one 32-element block
along K per scale, the same E8M0 exponent and E2M1 rounding), applied per token row.

``Y[m, n] = sum_k deq(Xq)[m, k] * deq(Wq)[n, k]`` in float64: every product of two
E2M1 x 2^e values is exact.
"""
from __future__ import annotations

import numpy as np

from . import mxfp4


def quantize_activations(X: np.ndarray):
    """X [M, K] (the exact values of bf16 activations, K % 32 == 0) -> (Xq int32 [M, K/8],
    scales uint8 [M, K/32]): the MXFP4 quantizer of the weights, per token row."""
    return mxfp4.quantize(X)


def linear_w4a4(Xq, xs, Wq, ws) -> np.ndarray:
    """``Y = deq(Xq, xs) · deq(Wq, ws)^T`` in float64 [M, N]."""
    return mxfp4.dequantize(Xq, xs) @ mxfp4.dequantize(Wq, ws).T


def linear_w4a4_rows(Xq, xs, Wq, ws, rows) -> np.ndarray:
    """Only the output columns ``rows``: float64 [M, len(rows)]."""
    rows = np.asarray(rows)
    return linear_w4a4(Xq, xs, np.asarray(Wq)[rows], np.asarray(ws)[rows])
