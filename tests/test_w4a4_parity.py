"""W4A4 in MXFP4 (第 6 课：量化源码走读, micro-scaling: weights and activations in MXFP4, the
activations quantized on the fly) on the FP8 tensor-core path: the weights' and the
activations' E4M3 re-encodings reproduce the oracle's dequantized MXFP4 values exactly, and
the layer matches the oracle's float64 W4A4 product."""
import numpy as np
import pytest

from bit_weight_quantized_wq_gb300 import inputs
from oracle import fp8, mxfp4, w4a4
from tests._util import assert_close, to_dev, x_to_dev, y_to_host

pytestmark = pytest.mark.gpu

E4M3 = fp8.e4m3_values()


@pytest.fixture(scope="module")
def B():
    import torch
    from bit_weight_quantized_wq_gb300 import binding
    binding.check_device()
    torch.cuda.init()
    return binding


def _decoded(q, s):
    return E4M3[q.cpu().numpy().astype(np.uint8)] * s.cpu().numpy().astype(np.float64)[:, None]


@pytest.mark.parametrize("N,K", [(64, 256), (300, 1024), (5, 4128)])
def test_w4a4_weights_reencode_exactly(B, N, K):
    W = inputs.weights(N + K, N, K, 0.05)
    W[1] *= 1e-3                                          # rows of very different magnitude
    W[2, :] = 0.0
    pk = mxfp4.quantize(W)
    W8, sw = B.mxfp4_weights_to_e4m3(to_dev(pk[0]), to_dev(pk[1]))
    assert np.array_equal(_decoded(W8, sw), mxfp4.dequantize(*pk))


@pytest.mark.parametrize("M,K", [(1, 128), (40, 1024), (257, 4096)])
def test_w4a4_activations_quantize_and_reencode_exactly(B, M, K):
    xb, xf = inputs.activations(M * 3 + K, M, K)
    Xq, sx = B.quantize_w4a4_activations(x_to_dev(xb))
    assert np.array_equal(_decoded(Xq, sx), mxfp4.dequantize(*w4a4.quantize_activations(xf)))


def test_w4a4_blocks_far_below_the_row_max_are_bounded(B):
    # one block 2^24 above the others: the small blocks fall outside the E4M3 window; their
    # error stays below 2^-12 of the row's largest magnitude (beyond 2^-13 they become zero)
    K = 256
    rng = np.random.default_rng(5)
    x = (rng.standard_normal((1, K)) * 1e-4).astype(np.float32)
    x[0, :32] *= 2.0 ** 24
    xb = (x.view(np.uint32) >> 16).astype(np.uint16)
    xf = (xb.astype(np.uint32) << 16).view(np.float32)
    Xq, sx = B.quantize_w4a4_activations(x_to_dev(xb))
    ref = mxfp4.dequantize(*w4a4.quantize_activations(xf))
    err = np.abs(_decoded(Xq, sx) - ref)
    assert err.max() <= 2.0 ** -12 * np.abs(ref).max()
    assert np.array_equal(_decoded(Xq, sx)[:, :32], ref[:, :32])


@pytest.mark.parametrize("M,K,N", [(1, 128, 128), (17, 256, 200), (300, 1056, 384), (600, 2048, 1000)])
def test_w4a4_layer(B, M, K, N):
    W = inputs.weights(N * 3 + K, N, K, 0.05)
    xb, xf = inputs.activations(M + N, M, K)
    pk = mxfp4.quantize(W)
    W8, sw = B.mxfp4_weights_to_e4m3(to_dev(pk[0]), to_dev(pk[1]))
    Y = y_to_host(B.gemm_w4a4_mxfp4(x_to_dev(xb), W8, sw))
    Xq, xs = w4a4.quantize_activations(xf)
    assert_close(Y, w4a4.linear_w4a4(Xq, xs, *pk), "w4a4 M=%d K=%d N=%d" % (M, K, N))
    assert B.read_error_flags() == 0


def test_w4a4_full_size_sampled(B):
    # a Qwen2.5-72B prefill shape at M = 2048, 256 sampled output columns
    M, K, N = 2048, 8192, 8192
    W = inputs.weights(3001, N, K, 0.015)
    xb, xf = inputs.activations(3002, M, K)
    pk = mxfp4.quantize(W)
    W8, sw = B.mxfp4_weights_to_e4m3(to_dev(pk[0]), to_dev(pk[1]))
    Y = y_to_host(B.gemm_w4a4_mxfp4(x_to_dev(xb), W8, sw))
    rows = np.sort(np.random.default_rng(3).choice(N, 256, replace=False))
    Xq, xs = w4a4.quantize_activations(xf)
    assert_close(Y[:, rows], w4a4.linear_w4a4_rows(Xq, xs, pk[0], pk[1], rows), "w4a4 full size")
    assert B.read_error_flags() == 0
