"""CPU-only checks of the C-ABI library: it loads, exports every entry point the header
declares, and its host-side logic (argument validation, dispatch table, workspace size)
behaves as documented.  No kernel is launched."""
import ctypes
import os
import re

import pytest

from bit_weight_quantized_wq_gb300 import binding
from bit_weight_quantized_wq_gb300 import build as wqbuild

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "wq.h")


def _stale():
    lib = binding.LIB_PATH
    if not os.path.exists(lib):
        return True
    t = os.path.getmtime(lib)
    srcs = [os.path.join(wqbuild.CSRC, f) for f in os.listdir(wqbuild.CSRC)] + [HEADER]
    return any(os.path.getmtime(s) > t for s in srcs)


@pytest.fixture(scope="module")
def lib():
    if _stale():
        wqbuild.build()
    return binding.load_library()


def _declared():
    text = open(HEADER).read()
    return sorted(set(re.findall(r"\b(wq_[a-z0-9_]+)\s*\(", text)))


def test_header_declares_the_entry_points():
    names = _declared()
    for n in ("wq_quantize_int4_g128", "wq_quantize_mxfp4", "wq_gemm_w4a16", "wq_gemm_workspace_bytes",
              "wq_status_str", "wq_set_dispatch_threshold"):
        assert n in names
    assert set(names) == set(binding.EXPORTED)


def test_library_exports_every_declared_symbol(lib):
    for name in _declared():
        assert hasattr(lib, name), name


def test_status_strings(lib):
    for s in range(8):
        assert binding.status_str(s).startswith("WQ_")
    assert "unknown" in binding.status_str(99)


FAKE = ctypes.c_void_p(0x10000)       # aligned, never dereferenced: validation fails first
ODD = ctypes.c_void_p(0x10008)


def _gemm(lib, fmt=0, X=FAKE, M=1, K=128, N=8, Wq=FAKE, s=FAKE, z=FAKE, Y=FAKE, ws=None, wsb=0):
    return lib.wq_gemm_w4a16(fmt, X, M, K, N, Wq, s, z, Y, ws, wsb, None)


def test_validation_errors(lib):
    assert _gemm(lib, X=None) == 1                      # NULL
    assert _gemm(lib, z=None) == 1                      # INT4 needs zeros
    assert _gemm(lib, fmt=1) == 7                       # MXFP4 must not get zeros
    assert _gemm(lib, fmt=5) == 7                       # bad format
    assert _gemm(lib, M=0) == 2
    assert _gemm(lib, N=0) == 2
    assert _gemm(lib, K=64) == 2                        # INT4: K % 128
    assert _gemm(lib, fmt=1, z=None, K=48) == 2         # MXFP4: K % 32
    assert _gemm(lib, X=ODD) == 3                       # alignment
    assert _gemm(lib, Y=ODD) == 3
    assert lib.wq_gemv_w4a16(0, FAKE, 65, 128, 8, FAKE, FAKE, FAKE, FAKE, None, 0, None) == 2  # decode: M <= 64
    assert lib.wq_quantize_int4_g128(None, 4, 128, FAKE, FAKE, FAKE, None) == 1
    assert lib.wq_quantize_int4_g128(FAKE, 4, 96, FAKE, FAKE, FAKE, None) == 2
    assert lib.wq_quantize_mxfp4(FAKE, 4, 48, FAKE, FAKE, None) == 2
    assert lib.wq_quantize_mxfp4(FAKE, 0, 64, FAKE, FAKE, None) == 2
    assert lib.wq_quantize_mxfp4(ODD, 4, 64, FAKE, FAKE, None) == 3


def test_workspace_checked_before_launch(lib):
    need = lib.wq_gemm_workspace_bytes(0, 1, 4096, 4096)
    assert need > 0
    r = lib.wq_gemv_w4a16(0, FAKE, 1, 4096, 4096, FAKE, FAKE, FAKE, FAKE, None, 0, None)
    assert r == 4
    r = lib.wq_gemv_w4a16(0, FAKE, 1, 4096, 4096, FAKE, FAKE, FAKE, FAKE, FAKE, 4096, None)
    assert r == 4                      # far below what the shape needs
    assert lib.wq_gemm_workspace_bytes(9, 1, 128, 128) == 0
    assert lib.wq_gemm_workspace_bytes(0, 0, 128, 128) == 0


def test_dispatch_threshold_table(lib):
    assert binding.dispatch_threshold("int4_g128", 4096, 4096) == 32
    binding.set_dispatch_threshold("int4_g128", 4096, 4096, 4)
    assert binding.dispatch_threshold("int4_g128", 4096, 4096) == 4
    assert binding.dispatch_threshold("int4_g128", 4096, 8192) == 32
    assert binding.dispatch_threshold("mxfp4", 4096, 4096) == 32
    binding.set_dispatch_threshold("int4_g128", 4096, 4096, 32)
    with pytest.raises(ValueError):
        binding.set_dispatch_threshold("int4_g128", 4096, 4096, 65)
    assert lib.wq_set_dispatch_threshold(3, 0, 0, 1) == 7


def test_validation_errors_swiglu_interleave_gptq_awq(lib):
    # SwiGLU: F % 8, F >= 8, and the decode-only M bound
    sw = lambda fn, M=1, K=128, F=8, **kw: getattr(lib, fn)(0, FAKE, M, K, F, FAKE, FAKE, FAKE, FAKE,
                                                            kw.get("ws"), kw.get("wsb", 0), None)
    assert sw("wq_gemm_w4a16_swiglu", F=12) == 2
    assert sw("wq_gemm_w4a16_swiglu", F=0) == 2
    assert sw("wq_gemv_w4a16_swiglu", M=65, F=16) == 2
    assert sw("wq_gemm_tc_w4a16_swiglu", K=64, F=16) == 2
    assert sw("wq_gemv_w4a16_swiglu", F=4096) == 4          # workspace missing
    # interleave: NULL, F, row bytes, overlap (src == dst)
    assert lib.wq_interleave_gate_up(None, FAKE, 8, 16, None) == 1
    assert lib.wq_interleave_gate_up(FAKE, ctypes.c_void_p(0x900000), 12, 16, None) == 2
    assert lib.wq_interleave_gate_up(FAKE, ctypes.c_void_p(0x900000), 8, 0, None) == 2
    assert lib.wq_interleave_gate_up(FAKE, FAKE, 8, 16, None) == 7
    assert lib.wq_interleave_gate_up(FAKE, ctypes.c_void_p(0x10000 + 8 * 16), 8, 16, None) == 7   # overlaps
    # GPTQ: NULL factor, K % 128, K beyond one CTA's shared memory, alignment
    assert lib.wq_gptq_int4_g128(FAKE, 4, 128, None, FAKE, FAKE, FAKE, None) == 1
    assert lib.wq_gptq_int4_g128(FAKE, 4, 200, FAKE, FAKE, FAKE, FAKE, None) == 2
    assert lib.wq_gptq_int4_g128(FAKE, 4, 46336, FAKE, FAKE, FAKE, FAKE, None) == 2
    assert lib.wq_gptq_int4_g128(ODD, 4, 128, FAKE, FAKE, FAKE, FAKE, None) == 3
    # AWQ: workspace size, shapes, NULLs, alignment
    assert lib.wq_awq_workspace_bytes(4096, 4096, 128) >= 4096 * 4096 * 4
    assert lib.wq_awq_workspace_bytes(4096, 100, 128) == 0
    aw = lambda W=FAKE, N=4, K=128, X=FAKE, n=8, s=FAKE, ws=FAKE, wsb=1 << 30: lib.wq_awq_int4_g128(
        W, N, K, X, n, FAKE, FAKE, FAKE, s, None, None, ws, wsb, None)
    assert aw(X=None) == 1
    assert aw(s=None) == 1
    assert aw(n=0) == 2
    assert aw(K=96) == 2
    assert aw(X=ODD) == 3
    assert aw(ws=None) == 4
    assert aw(wsb=16) == 4


def test_selftest_argument_checks(lib):
    v = ctypes.c_uint32(0)
    assert lib.wq_selftest_wait_timeout(1000, None, None) == 1
    assert lib.wq_selftest_wait_timeout(0, ctypes.byref(v), None) == 7
    assert lib.wq_selftest_wait_timeout(2000001, ctypes.byref(v), None) == 7


def test_validation_errors_fp8(lib):
    # quantizers: NULLs, K % 16, rows, alignment (arrays 16-byte, scales 4-byte)
    assert lib.wq_quantize_fp8_weights(None, 4, 64, FAKE, FAKE, None) == 1
    assert lib.wq_quantize_fp8_weights(FAKE, 4, 24, FAKE, FAKE, None) == 2
    assert lib.wq_quantize_fp8_weights(FAKE, 0, 64, FAKE, FAKE, None) == 2
    assert lib.wq_quantize_fp8_weights(ODD, 4, 64, FAKE, FAKE, None) == 3
    assert lib.wq_quantize_fp8_activations(FAKE, 4, 64, FAKE, ctypes.c_void_p(0x10002), None) == 3
    assert lib.wq_quantize_fp8_activations(FAKE, 4, 8, FAKE, FAKE, None) == 2
    # GEMM: NULLs, shapes, alignment
    g = lambda Xq=FAKE, sx=FAKE, M=4, K=64, N=8, Wq=FAKE, sw=FAKE, Y=FAKE: lib.wq_gemm_fp8(Xq, sx, M, K, N, Wq, sw, Y, None)
    assert g(Xq=None) == 1 and g(sw=None) == 1 and g(Y=None) == 1
    assert g(K=40) == 2 and g(M=0) == 2 and g(N=0) == 2
    assert g(Wq=ODD) == 3 and g(Xq=ODD) == 3
    # fused entry: workspace size and presence
    assert lib.wq_gemm_w8a8_fp8_workspace_bytes(300, 1024) >= 300 * 1024 + 300 * 4
    assert lib.wq_gemm_w8a8_fp8_workspace_bytes(0, 1024) == 0
    f = lambda ws=FAKE, wsb=1 << 30, K=64: lib.wq_gemm_w8a8_fp8(FAKE, 4, K, 8, FAKE, FAKE, FAKE, ws, wsb, None)
    assert f(ws=None) == 4 and f(wsb=16) == 4 and f(K=40) == 2


def test_validation_errors_w4a4(lib):
    assert lib.wq_mxfp4_weights_to_e4m3(None, FAKE, 4, 64, FAKE, FAKE, None) == 1
    assert lib.wq_mxfp4_weights_to_e4m3(FAKE, FAKE, 4, 48, FAKE, FAKE, None) == 2
    assert lib.wq_mxfp4_weights_to_e4m3(ODD, FAKE, 4, 64, FAKE, FAKE, None) == 3
    assert lib.wq_quantize_w4a4_activations(FAKE, 4, 48, FAKE, FAKE, None) == 2
    assert lib.wq_quantize_w4a4_activations(FAKE, 4, 131104, FAKE, FAKE, None) == 2
    f = lambda ws=FAKE, wsb=1 << 30, K=64: lib.wq_gemm_w4a4_mxfp4(FAKE, 4, K, 8, FAKE, FAKE, FAKE, ws, wsb, None)
    assert f(ws=None) == 4 and f(K=48) == 2
