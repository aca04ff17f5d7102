"""The workspace contract of the layer entry points: a workspace zeroed once serves calls of
any shape and either kernel, because every call that completes leaves the workspace header
at zero again: the tensor-core kernel's split-K counters (64 KiB) and the decode kernel's
split-K exchange area after them (10 MiB of tagged partial sums, where 0 means "not posted").
Checked after calls whose bands or tiles are split between CTAs (decode split-K,
tensor-core split tiles), with every epilogue, and with one workspace shared by consecutive
calls of different shapes; each output against the float64 oracle, so a counter or a
partial sum left behind (which would make a later call skip, double or mix up a reduction)
shows up as a wrong result too."""
import numpy as np
import pytest

from bit_weight_quantized_wq_gb300 import inputs
from oracle import int4_g128, linear, mxfp4, swiglu
from tests._util import assert_close, to_dev, x_to_dev, y_to_host

pytestmark = pytest.mark.gpu

HEADER = 64 * 1024 + 2 * 160 * 32 * 256 * 4   # counters + the decode exchange area


@pytest.fixture(scope="module")
def B():
    import torch
    from bit_weight_quantized_wq_gb300 import binding
    binding.check_device()
    torch.cuda.init()
    return binding


def _pack(fmt, W):
    return int4_g128.quantize(W) if fmt == "int4_g128" else mxfp4.quantize(W)


def _dev(fmt, pk):
    d = [to_dev(a) for a in pk]
    return d[0], d[1], (d[2] if fmt == "int4_g128" else None)


def _header_zero(ws):
    import torch
    torch.cuda.synchronize()
    head = ws[:HEADER].cpu().numpy()
    return int(np.count_nonzero(head))


# (fmt, M, K, N, entry): decode with bands shared between CTAs (M = 1, 16, 40 -- two row
# slices), the tensor-core kernel with every tile split along K (M = 64) and with a split
# last wave (M = 300).
CASES = [("int4_g128", 1, 4096, 4096, "gemv"), ("mxfp4", 16, 4096, 6144, "gemv"), ("int4_g128", 40, 2048, 3072, "gemv"),
         ("int4_g128", 64, 4096, 256, "tc"), ("mxfp4", 300, 1024, 1024, "tc")]


@pytest.mark.parametrize("fmt,M,K,N,entry", CASES)
def test_counters_back_at_zero_after_a_call(B, fmt, M, K, N, entry):
    import torch
    pk = _pack(fmt, inputs.weights(M + K + N, N, K, 0.05))
    xb, xf = inputs.activations(M * 3 + K, M, K)
    ws = torch.zeros(max(B.gemm_workspace_bytes(fmt, M, K, N), HEADER), dtype=torch.uint8, device="cuda")
    fn = B.gemv_w4a16 if entry == "gemv" else B.gemm_tc_w4a16
    Y = fn(fmt, x_to_dev(xb), *_dev(fmt, pk), workspace=ws)
    assert _header_zero(ws) == 0, "split-K counters or partial sums left non-zero"
    assert_close(y_to_host(Y), linear.linear_w4a16(fmt, xf, *pk), "%s %s M=%d" % (entry, fmt, M))
    assert B.read_error_flags() == 0


def test_one_workspace_across_shapes_and_epilogues(B):
    """Decode, tensor-core, SwiGLU and QKV calls in a row on one workspace, zeroed once."""
    import torch
    calls = [("gemv", "int4_g128", 1, 4096, 4096), ("tc", "int4_g128", 64, 4096, 256), ("gemv", "mxfp4", 16, 4096, 2048),
             ("swiglu", "int4_g128", 4, 4096, 2048), ("qkv", "int4_g128", 300, 1024, 1536), ("gemv", "int4_g128", 1, 4096, 4096)]
    need = max(B.gemm_workspace_bytes(f, M, K, N) for _, f, M, K, N in calls)
    ws = torch.zeros(max(need, HEADER), dtype=torch.uint8, device="cuda")
    for i, (kind, fmt, M, K, N) in enumerate(calls):
        pk = _pack(fmt, inputs.weights(900 + i, N, K, 0.05))
        xb, xf = inputs.activations(950 + i, M, K)
        X = x_to_dev(xb)
        ref = linear.linear_w4a16(fmt, xf, *pk)
        if kind == "gemv":
            got = y_to_host(B.gemv_w4a16(fmt, X, *_dev(fmt, pk), workspace=ws))
            assert_close(got, ref, "call %d" % i)
        elif kind == "tc":
            got = y_to_host(B.gemm_tc_w4a16(fmt, X, *_dev(fmt, pk), workspace=ws))
            assert_close(got, ref, "call %d" % i)
        elif kind == "swiglu":
            # the fused gate+up weight in the interleaved row order; SiLU(gate) * up against
            # the float64 product of the same rows
            d = [B.interleave_gate_up(t) for t in (to_dev(a) for a in pk)]
            got = y_to_host(B.gemv_w4a16_swiglu(fmt, X, d[0], d[1], d[2], workspace=ws))
            assert_close(got, swiglu.swiglu_w4a16(fmt, xf, *pk), "call %d (SwiGLU)" % i)
        else:
            Nkv = (N - 1024) // 2
            q, k, v = B.gemm_w4a16_qkv(fmt, X, *_dev(fmt, pk), Nq=1024, Nkv=Nkv, workspace=ws)
            for t, (lo, hi) in zip((q, k, v), ((0, 1024), (1024, 1024 + Nkv), (1024 + Nkv, N))):
                assert_close(y_to_host(t), ref[:, lo:hi], "call %d (QKV)" % i)
        assert _header_zero(ws) == 0, "call %d left split-K counters or partial sums non-zero" % i
    assert B.read_error_flags() == 0
