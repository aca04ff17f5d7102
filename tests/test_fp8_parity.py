"""W8A8 in FP8 E4M3 (推理优化与量化算子深度技术调研 §1.4; 第 6 课：量化源码走读 §4: FP8 for
large-batch prefill): the per-row quantizers bit-exact against the oracle (codes and scales),
the tcgen05 kind::f8f6f4 GEMM element-wise against the oracle's float64 layer on the same
codes, and the fused bf16-in entry point."""
import numpy as np
import pytest

from bit_weight_quantized_wq_gb300 import inputs
from oracle import fp8
from tests._util import assert_close, to_dev, x_to_dev, y_to_host

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def B():
    import torch
    from bit_weight_quantized_wq_gb300 import binding
    binding.check_device()
    torch.cuda.init()
    return binding


def _u8(t):
    return t.cpu().numpy().astype(np.uint8)


def _adversarial_rows(K, seed):
    """Rows that exercise the rounding rules: exact ties between neighbouring E4M3 values,
    saturation, -0.0, values in the subnormal range of the scaled grid, a zero row."""
    rng = np.random.default_rng(seed)
    grid = fp8.e4m3_values()[:127]
    mids = (grid[:-1] + grid[1:]) / 2.0                         # exact halfway points
    rows = []
    r = rng.choice(mids, K) * rng.choice([-1.0, 1.0], K)        # ties (scale 1: max is 448)
    r[0] = 448.0
    rows.append(r)
    r = rng.standard_normal(K) * 1e-3
    r[1] = -0.0
    r[2] = 1e3                                                   # one outlier: the rest land in subnormals
    rows.append(r)
    rows.append(np.zeros(K))
    r = rng.standard_normal(K)
    r[::7] = -0.0
    rows.append(r)
    rows.append(rng.standard_normal(K) * 3e4)
    return np.array(rows, dtype=np.float32)


@pytest.mark.parametrize("N,K", [(64, 256), (300, 1024), (17, 16), (5, 4112)])
def test_fp8_quantize_weights_bit_exact(B, N, K):
    W = inputs.weights(N + K, N, K, 0.05)
    W = np.concatenate([W, _adversarial_rows(K, N * 3 + K)])
    Wq, sw = B.quantize_fp8_weights(to_dev(W))
    ref_q, ref_s = fp8.quantize_weights(W)
    assert np.array_equal(sw.cpu().numpy(), ref_s), "scales"
    got = _u8(Wq)
    bad = np.argwhere(got != ref_q)
    assert bad.size == 0, "%d codes differ, first at %s: %#x vs %#x (value %r, scale %r)" % (
        len(bad), bad[0], got[tuple(bad[0])], ref_q[tuple(bad[0])], W[tuple(bad[0])], ref_s[bad[0][0]])
    assert B.read_error_flags() == 0


@pytest.mark.parametrize("M,K", [(1, 128), (40, 1024), (300, 4096)])
def test_fp8_quantize_activations_bit_exact(B, M, K):
    xb, xf = inputs.activations(M + K, M, K)
    adv = _adversarial_rows(K, M + 2 * K)
    # the adversarial rows as bf16 (truncate to bf16 bits: the oracle sees the same values)
    adv_b = (adv.view(np.uint32) >> 16).astype(np.uint16)
    xb = np.concatenate([xb, adv_b])
    xf = np.concatenate([xf, (adv_b.astype(np.uint32) << 16).view(np.float32)])
    Xq, sx = B.quantize_fp8_activations(x_to_dev(xb))
    ref_q, ref_s = fp8.quantize_activations(xf)
    assert np.array_equal(sx.cpu().numpy(), ref_s), "scales"
    assert np.array_equal(_u8(Xq), ref_q), "codes"


def _gemm_case(M, K, N, seed):
    W = inputs.weights(seed, N, K, 0.05)
    xb, xf = inputs.activations(seed + 1, M, K)
    Wq, sw = fp8.quantize_weights(W)
    Xq, sx = fp8.quantize_activations(xf)
    return xb, (Xq, sx, Wq, sw)


@pytest.mark.parametrize("M,K,N", [(1, 128, 128), (17, 256, 200), (256, 512, 256), (300, 1040, 384),
                                   (513, 2048, 1000), (1000, 256, 130)])
def test_fp8_gemm_small(B, M, K, N):
    _, (Xq, sx, Wq, sw) = _gemm_case(M, K, N, M * 7 + N)
    Y = B.gemm_fp8(to_dev(Xq), to_dev(sx), to_dev(Wq), to_dev(sw))
    assert_close(y_to_host(Y), fp8.linear_w8a8(Xq, sx, Wq, sw), "fp8 M=%d K=%d N=%d" % (M, K, N))
    assert B.read_error_flags() == 0


def test_fp8_fused_equals_two_steps_and_is_deterministic(B):
    M, K, N = 700, 1536, 640
    xb, (Xq, sx, Wq, sw) = _gemm_case(M, K, N, 91)
    X = x_to_dev(xb)
    Wd, swd = to_dev(Wq), to_dev(sw)
    y1 = y_to_host(B.gemm_w8a8_fp8(X, Wd, swd))
    xq, s = B.quantize_fp8_activations(X)
    y2 = y_to_host(B.gemm_fp8(xq, s, Wd, swd))
    y3 = y_to_host(B.gemm_w8a8_fp8(X, Wd, swd))
    assert np.array_equal(y1, y2) and np.array_equal(y1, y3)
    assert_close(y1, fp8.linear_w8a8(Xq, sx, Wq, sw), "fused")


# Full-size prefill shapes (Qwen2.5-72B, K, N) at M = 2048: 256 sampled output columns.
@pytest.mark.parametrize("K,N", [(8192, 10240), (8192, 8192), (8192, 59136), (29568, 8192)])
def test_fp8_full_size_sampled(B, K, N):
    M = 2048
    W = inputs.weights(3000 + K % 97 + N % 89, N, K, 0.015)
    xb, xf = inputs.activations(K + N, M, K)
    Wq, sw = B.quantize_fp8_weights(to_dev(W))
    Y = y_to_host(B.gemm_w8a8_fp8(x_to_dev(xb), Wq, sw))
    rows = np.sort(np.random.default_rng(K + N).choice(N, 256, replace=False))
    rq, rs = fp8.quantize_weights(W[rows])
    assert np.array_equal(_u8(Wq)[rows], rq) and np.array_equal(sw.cpu().numpy()[rows], rs)
    Xq, sx = fp8.quantize_activations(xf)
    assert_close(Y[:, rows], fp8.linear_w8a8(Xq, sx, rq, rs), "fp8 K=%d N=%d" % (K, N))
    assert B.read_error_flags() == 0


def test_fp8_rejects_bad_arguments(B):
    import torch
    W = torch.zeros((8, 24), dtype=torch.float32, device="cuda")           # K % 16 != 0
    with pytest.raises(ValueError):
        B.quantize_fp8_weights(W)
    Xq = torch.zeros((4, 64), dtype=torch.uint8, device="cuda")
    sx = torch.ones((4,), dtype=torch.float32, device="cuda")
    Wq = torch.zeros((8, 64), dtype=torch.uint8, device="cuda")
    with pytest.raises(ValueError):
        B.gemm_fp8(Xq, sx, Wq, torch.ones((7,), dtype=torch.float32, device="cuda"))   # s_w not [N]
    with pytest.raises(ValueError):
        B.gemm_fp8(Xq, sx[:3], Wq, torch.ones((8,), dtype=torch.float32, device="cuda"))
    with pytest.raises(ValueError):
        B.gemm_fp8(Xq, sx, Wq[:, :32].contiguous(), torch.ones((8,), dtype=torch.float32, device="cuda"))
