"""CPU oracle for the weight-only 4-bit quantized linear layer (W4A16).

TEST INFRASTRUCTURE ONLY.  Nothing in the product path imports, calls or links
this package; only ``tests/``, ``__graft_entry__.smoke()`` and the
``cpu_baseline`` / ``--impl reference`` legs of ``bench.py`` use it.  It shares
no code, tables or constants with the CUDA library.

What it computes, step by step in the pages' order (citations are page title +
section):

* ``uniform``   -- the symmetric and asymmetric uniform quantizers of
  推理优化与量化算子深度技术调研 §1.2 and 第 1 章：推理加速全景 §4.1 (均匀量化的数学基础),
  and the block-wise symmetric fake-quant exercise of 第 6 课：量化源码走读 (实践任务).
* ``int4_g128`` -- asymmetric INT4, group size 128 along K, eight codes per
  int32, fp16 scale and zero point per group.
* ``mxfp4``     -- OCP MXFP4: E2M1 codes two per byte, one E8M0 power-of-two
  scale per 32 elements along K (大模型量化推理引擎全景大复盘, 里程碑六 / 方程 3).
* ``linear``    -- Y = X · dequant(Wq)^T in float64.
* ``swiglu``    -- the fused gate+up projection with SiLU(gate) * up
  (推理优化与量化算子深度技术调研 §4.6), and the row interleave of the stacked
  gate+up weight that the kernels read.
* ``gptq``      -- GPTQ: INT4 g128 quantization column by column with the
  inverse-Hessian error compensation of 第 1 章：推理加速全景 §4.2.
* ``awq``       -- AWQ: per-channel scaling of the salient input channels, its exponent
  found by a grid search, before INT4 g128 quantization (第 1 章 §4.4).
* ``fp8``       -- W8A8 in FP8 E4M3 (推理优化与量化算子深度技术调研 §1.4): per-output-channel
  weight scales, per-token activation scales, the layer on the quantized operands.
* ``w4a4``      -- W4A4 in MXFP4 (第 6 课：量化源码走读, micro-scaling formats): the activations
  quantized by the weights' MXFP4 rules, the layer on both dequantized operands.

Quantization arithmetic runs in float32 (the precision the pages' torch code
works in) so that integer decisions -- codes, zero points, exponents -- are
taken in the same precision as the kernels; dequantization and the matmul are
float64.

Pins (tests/test_oracle_pins.py, tests/golden/): the pages' worked example and
asserts, closed forms, brute force on tiny inputs, invariants and special
cases.  Every function here is pinned; none is "parity unpinned".
"""
from . import uniform, int4_g128, mxfp4, linear, swiglu, gptq, awq, fp8, w4a4  # noqa: F401
