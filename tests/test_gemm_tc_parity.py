"""tcgen05 tensor-core kernel against the float64 oracle on the same dequantized weights."""
import numpy as np
import pytest

from bit_weight_quantized_wq_gb300 import inputs
from oracle import int4_g128, linear, mxfp4
from tests._util import assert_close, to_dev, x_to_dev, y_to_host

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def B():
    import torch
    from bit_weight_quantized_wq_gb300 import binding
    binding.check_device()
    torch.cuda.init()
    return binding


def _pack(fmt, W):
    return int4_g128.quantize(W) if fmt == "int4_g128" else mxfp4.quantize(W)


def _run(fn, fmt, xbits, pk):
    X = x_to_dev(xbits)
    d = [to_dev(a) for a in pk]
    if fmt == "int4_g128":
        return fn(fmt, X, d[0], d[1], d[2])
    return fn(fmt, X, d[0], d[1])


# (M, N, K): single tile, ragged M/N, several tiles in both directions, long K.
CASES = [(1, 128, 128), (256, 128, 128), (17, 200, 256), (300, 384, 512), (513, 1000, 1024),
         (64, 256, 4096), (1024, 512, 2048)]


@pytest.mark.parametrize("fmt", ["int4_g128", "mxfp4"])
@pytest.mark.parametrize("M,N,K", CASES)
def test_gemm_tc_small(B, fmt, M, N, K):
    W = inputs.weights(N * 3 + K, N, K, 0.05)
    pk = _pack(fmt, W)
    xb, xf = inputs.activations(M + K, M, K)
    Y = _run(B.gemm_tc_w4a16, fmt, xb, pk)
    assert_close(y_to_host(Y), linear.linear_w4a16(fmt, xf, *pk), "%s M=%d N=%d K=%d" % (fmt, M, N, K))


# Mid-sized M: the activation tile is 64, 128 or 256 rows (M <= 64, <= 128, above), and
# layers with few tiles split every tile along K over up to 8 CTAs; (M, N, K) straddle the
# tile boundaries and give 2-, 4- and 8-way splits.
MID = [(33, 1024, 2048), (64, 256, 4096), (65, 512, 4096), (128, 384, 1024), (129, 256, 2048), (200, 640, 8192)]


@pytest.mark.parametrize("fmt", ["int4_g128", "mxfp4"])
@pytest.mark.parametrize("M,N,K", MID)
def test_gemm_tc_mid_m(B, fmt, M, N, K):
    W = inputs.weights(N * 11 + K + M, N, K, 0.05)
    pk = _pack(fmt, W)
    xb, xf = inputs.activations(M * 7 + K, M, K)
    Y = _run(B.gemm_tc_w4a16, fmt, xb, pk)
    assert_close(y_to_host(Y), linear.linear_w4a16(fmt, xf, *pk), "%s M=%d N=%d K=%d" % (fmt, M, N, K))
    assert B.read_error_flags() == 0


def test_gemm_tc_split_k_deterministic(B):
    # every tile split 8 ways along K: the last CTA adds the parts in part order, so two calls
    # give the same bits whichever part finishes last
    M, N, K = 64, 256, 4096
    W = inputs.weights(21, N, K, 0.05)
    pk = int4_g128.quantize(W)
    xb, xf = inputs.activations(22, M, K)
    y1 = y_to_host(_run(B.gemm_tc_w4a16, "int4_g128", xb, pk))
    y2 = y_to_host(_run(B.gemm_tc_w4a16, "int4_g128", xb, pk))
    assert np.array_equal(y1, y2)
    assert_close(y1, linear.linear_w4a16("int4_g128", xf, *pk), "split-K")


@pytest.mark.parametrize("K", [32, 96, 160])
def test_gemm_tc_mxfp4_k_tail(B, K):
    M, N = 100, 300
    W = inputs.weights(K + 5, N, K, 0.05)
    pk = mxfp4.quantize(W)
    xb, xf = inputs.activations(K + 6, M, K)
    Y = _run(B.gemm_tc_w4a16, "mxfp4", xb, pk)
    assert_close(y_to_host(Y), linear.linear_w4a16("mxfp4", xf, *pk), "mxfp4 K=%d" % K)


def test_gemm_tc_int4_large_activations(B):
    # Activations beyond the fp16 range (|x| up to ~1e6): the per-row power-of-two scaling
    # keeps them exact and finite.  The fp16 operand rounding of the dequantized weights is
    # relative to |x|, so the criterion is applied to Y / scale (the same test on a layer
    # whose activations are divided by the scale).
    M, N, K = 64, 256, 512
    scale = 2.0e5
    W = inputs.weights(7, N, K, 0.05)
    pk = int4_g128.quantize(W)
    xb, xf = inputs.activations(8, M, K, scale=scale)
    y = y_to_host(_run(B.gemm_tc_w4a16, "int4_g128", xb, pk))
    ref = linear.linear_w4a16("int4_g128", xf, *pk)
    assert np.isfinite(y).all()
    assert_close(y / scale, ref / scale, "int4 big X (scaled)")


# Activation rows of very different magnitudes in one call: unit rows, rows of ~1e-6 (fp16
# subnormals if converted unscaled), ~1e-20 and ~1e-30 (below fp16's range altogether).
ROW_SCALES = (1.0, 1e-6, 1e-20, 1e-30)


def _scaled_rows(seed, M, K):
    xb, xf = inputs.activations(seed, M, K)
    c = np.array([ROW_SCALES[m % len(ROW_SCALES)] for m in range(M)], np.float32)
    xf = xf * c[:, None]
    xb = inputs.bf16_bits_from_f32(xf)
    return xb, inputs.f32_from_bf16_bits(xb), c.astype(np.float64)


def check_small_rows(y, ref, c, what):
    """Each row m scaled back by its magnitude c_m meets the unit-scale tolerance, and every
    output with |ref| >= c_m is within 2 % of ref: relative accuracy independent of |x|."""
    y = np.asarray(y, np.float64)
    assert np.isfinite(y).all(), what + ": non-finite outputs"
    assert_close(y / c[:, None], ref / c[:, None], what + " (rows / c_m)")
    big = np.abs(ref) >= c[:, None]
    rel = np.abs(y - ref)[big] / np.abs(ref)[big]
    assert rel.size and rel.max() <= 2e-2, "%s: worst relative error %.3g" % (what, rel.max())


@pytest.mark.parametrize("fmt", ["int4_g128", "mxfp4"])
def test_gemm_tc_small_magnitude_activations(B, fmt):
    # The INT4 path converts X to fp16 with a per-row power of two; small rows must be scaled
    # up (not only large rows down), else their values become fp16 subnormals or zeros.
    M, N, K = 40, 384, 1024
    W = inputs.weights(17, N, K, 0.05)
    pk = _pack(fmt, W)
    xb, xf, c = _scaled_rows(18, M, K)
    y = y_to_host(_run(B.gemm_tc_w4a16, fmt, xb, pk))
    check_small_rows(y, linear.linear_w4a16(fmt, xf, *pk), c, "%s small |x|" % fmt)


def test_dispatch_routes_by_m(B):
    # both sides of the default threshold (32): decode at M <= 32, tensor core above
    N, K = 256, 512
    W = inputs.weights(2, N, K, 0.05)
    pk = int4_g128.quantize(W)
    for m in (1, 16, 17, 20, 32, 33, 40):
        xb, xf = inputs.activations(m, m, K)
        Y = _run(B.gemm_w4a16, "int4_g128", xb, pk)
        assert_close(y_to_host(Y), linear.linear_w4a16("int4_g128", xf, *pk), "dispatch M=%d" % m)


# Full-size prefill shapes (K, N) at M = 2048 (and one at 8192): 256 sampled output columns.
PREFILL = [(8192, 10240), (8192, 8192), (8192, 59136), (29568, 8192)]


@pytest.mark.parametrize("K,N", PREFILL)
def test_gemm_tc_full_size_sampled(B, K, N):
    W = inputs.weights(3000 + K % 97 + N % 89, N, K, 0.015)
    pk = int4_g128.quantize(W)
    rows = np.sort(np.random.default_rng(K * 7 + N).choice(N, 256, replace=False))
    M = 2048
    xb, xf = inputs.activations(K + N, M, K)
    Y = y_to_host(_run(B.gemm_tc_w4a16, "int4_g128", xb, pk))
    ref = linear.linear_rows("int4_g128", xf, pk[0], pk[1], pk[2], rows)
    assert_close(Y[:, rows], ref, "int4 K=%d N=%d M=%d" % (K, N, M))
    assert B.read_error_flags() == 0


def test_gemm_tc_full_size_m8192_sampled(B):
    K, N, M = 8192, 8192, 8192
    W = inputs.weights(3001, N, K, 0.015)
    pk = int4_g128.quantize(W)
    rows = np.sort(np.random.default_rng(5).choice(N, 128, replace=False))
    xb, xf = inputs.activations(3002, M, K)
    Y = y_to_host(_run(B.gemm_tc_w4a16, "int4_g128", xb, pk))
    ref = linear.linear_rows("int4_g128", xf, pk[0], pk[1], pk[2], rows)
    assert_close(Y[:, rows], ref, "int4 M=8192")


@pytest.mark.parametrize("M", [64, 512, 2048])
def test_gemm_tc_mxfp4_crossover_shape(B, M):
    K = N = 8192
    W = inputs.weights(4000, N, K, 0.02)
    pk = mxfp4.quantize(W)
    rows = np.sort(np.random.default_rng(M).choice(N, 256, replace=False))
    xb, xf = inputs.activations(4000 + M, M, K)
    Y = y_to_host(_run(B.gemm_tc_w4a16, "mxfp4", xb, pk))
    ref = linear.linear_rows("mxfp4", xf, pk[0], pk[1], None, rows)
    assert_close(Y[:, rows], ref, "mxfp4 M=%d" % M)


# Wide layers with short K: more tiles than SMs (a partial last wave), ragged M, N and K
# tails, and an odd number of weight tiles; the result is also the same on a second run.
WIDE_CASES = [("int4_g128", 256, 256, 10240), ("int4_g128", 300, 384, 10152), ("mxfp4", 256, 352, 10240),
            ("mxfp4", 1000, 224, 3968)]


@pytest.mark.parametrize("fmt,M,K,N", WIDE_CASES)
def test_gemm_tc_wide_short_k(B, fmt, M, K, N):
    W = inputs.weights(M + K + N, N, K, 0.05)
    pk = _pack(fmt, W)
    xb, xf = inputs.activations(M * 5 + K, M, K)
    y1 = y_to_host(_run(B.gemm_tc_w4a16, fmt, xb, pk))
    assert_close(y1, linear.linear_w4a16(fmt, xf, *pk), "wide %s M=%d K=%d N=%d" % (fmt, M, K, N))
    y2 = y_to_host(_run(B.gemm_tc_w4a16, fmt, xb, pk))
    assert np.array_equal(y1, y2), "result differs between runs"
    assert B.read_error_flags() == 0
