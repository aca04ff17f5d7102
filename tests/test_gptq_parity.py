"""GPTQ sweep on the GPU against the oracle's sweep (第 1 章：推理加速全景 §4.2): codes, scales
and zero points bit-exact.  Both sides take every decision in float32 with each operation
rounded on its own, from the same inputs: W and the float32 inverse-Hessian factor U that the
oracle computes from seeded calibration activations."""
import numpy as np
import pytest

from bit_weight_quantized_wq_gb300 import inputs
from oracle import gptq, int4_g128
from tests._util import to_dev

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def B():
    import torch
    from bit_weight_quantized_wq_gb300 import binding
    binding.check_device()
    torch.cuda.init()
    return binding


def _factor(K, seed, n=128):
    """The oracle's inverse-Hessian factor of seeded calibration activations; above K = 6144,
    where that takes minutes on the host, a seeded stand-in upper-triangular factor."""
    if K > 6144:
        return inputs.upper_factor(seed, K)
    return gptq.inverse_cholesky_upper(gptq.hessian(inputs.calibration(seed, n, K))).astype(np.float32)


def _same(got, ref, what):
    for name, a, b in zip(("Wq", "scales", "zeros"), got, ref):
        a = a.cpu().numpy() if hasattr(a, "cpu") else np.asarray(a)
        bad = np.asarray(a).view(np.uint8) != np.asarray(b).view(np.uint8)
        assert not bad.any(), "%s %s: %d of %d bytes differ" % (what, name, int(bad.sum()), bad.size)


# (N, K): one case per kernel variant -- registers with 8/8/8/8/5/2 rows per CTA for K up to
# 512/1024/2048/4096/8192/16384, shared memory above -- N ragged against the rows per CTA
@pytest.mark.parametrize("N,K", [(1, 128), (16, 128), (37, 384), (64, 1024), (19, 2048), (15, 4096), (9, 6144),
                                 (5, 10240), (2, 16896)])
def test_gptq_bit_exact(B, N, K):
    W = inputs.weights(N * 31 + K, N, K, 0.05)
    U = _factor(K, K + 3)
    got = B.gptq_int4_g128(to_dev(W), to_dev(U))
    _same(got, gptq.sweep(W, U), "N=%d K=%d" % (N, K))
    assert B.read_error_flags() == 0


def test_gptq_diagonal_factor_equals_the_plain_quantizer(B):
    # With U diagonal there is no compensation: the GPU sweep must reproduce the plain INT4
    # quantizer (the GPU's and the oracle's).
    N, K = 40, 512
    W = inputs.weights(71, N, K, 0.05)
    U = np.diag(np.random.default_rng(72).uniform(0.5, 2.0, K)).astype(np.float32)
    got = B.gptq_int4_g128(to_dev(W), to_dev(U))
    _same(got, int4_g128.quantize(W), "diagonal")
    _same(got, [t.cpu().numpy() for t in B.quantize_int4_g128(to_dev(W))], "diagonal vs GPU quantizer")


def test_gptq_full_size_sampled_rows(B):
    # LLaMA-3-8B o_proj shape (K = N = 4096): every row on the GPU, 8 sampled rows on the
    # oracle (rows are independent).
    N = K = 4096
    W = inputs.weights(73, N, K, 0.02)
    U = _factor(K, 74)
    got = [t.cpu().numpy() for t in B.gptq_int4_g128(to_dev(W), to_dev(U))]
    rows = np.sort(np.random.default_rng(75).choice(N, 8, replace=False))
    ref = gptq.sweep(W[rows], U)
    _same([g[rows] for g in got], ref, "sampled rows")


def test_gptq_rejects_bad_shapes(B):
    import torch
    W = torch.zeros((4, 200), dtype=torch.float32, device="cuda")
    U = torch.zeros((200, 200), dtype=torch.float32, device="cuda")
    with pytest.raises(ValueError):
        B.gptq_int4_g128(W, U)                  # K % 128 != 0
    W = torch.zeros((4, 256), dtype=torch.float32, device="cuda")
    with pytest.raises(ValueError):
        B.gptq_int4_g128(W, U)                  # U not [K, K]


# ------------------------------------------------------------------ the factor on the device

@pytest.mark.parametrize("n,K", [(128, 128), (64, 384), (128, 1024), (1, 512), (128, 2048)])
def test_gptq_factor_matches_the_oracle(B, n, K):
    # U with H^-1 = U^T U, H = 2 X^T X + lambda I: the device's float64 factorisation rounded to
    # float32 once, against the oracle's float64 factor rounded to float32 (within one float32
    # rounding of it plus float64 noise amplified by the conditioning of H).
    X = inputs.calibration(K + n, n, K)
    U = B.gptq_factor(to_dev(X)).cpu().numpy().astype(np.float64)
    ref = gptq.inverse_cholesky_upper(gptq.hessian(X))
    assert (np.tril(U, -1) == 0).all(), "U must be upper triangular"
    assert (np.diag(U) > 0).all(), "U must have a positive diagonal"
    err = np.abs(U - ref)
    lim = 2.0 ** -23 * np.abs(ref) + 1e-6 * np.abs(ref).max()
    assert (err <= lim).all(), "max |U - ref| = %g (%d entries outside)" % (err.max(), int((err > lim).sum()))
    # and U is a factor of H^-1 in its own right: U^T U H = I
    H = gptq.hessian(X)
    R = (U.T @ U) @ H - np.eye(K)
    assert np.abs(R).max() < 1e-3, "||U^T U H - I||_max = %g" % np.abs(R).max()
    assert B.read_error_flags() == 0


def test_gptq_factor_rejects_a_singular_hessian(B):
    # All-zero calibration activations: H = 0 (lambda = 0), no Cholesky factor; the device
    # reports it in the error word instead of faulting
    import torch
    X = torch.zeros((16, 256), dtype=torch.float32, device="cuda")
    U = B.gptq_factor(X)
    torch.cuda.synchronize()
    assert B.read_error_flags() & (1 << 6)
    assert not torch.isfinite(U).all()
    assert B.read_error_flags() == 0


@pytest.mark.parametrize("N,n,K", [(64, 128, 512), (40, 128, 2048)])
def test_gptq_end_to_end_from_calibration(B, N, n, K):
    # GPTQ with the factor computed on the device: the sweep is bit-exact against the oracle's
    # sweep fed the same (device) factor, and the layer's calibration objective
    # ||X (W_hat - W)^T||^2 is within 0.1 % of the oracle's end-to-end result.
    W = inputs.weights(N + K, N, K, 0.05)
    X = inputs.calibration(K + 7, n, K)
    got = [t.cpu().numpy() for t in B.gptq_int4_g128_calib(to_dev(W), to_dev(X))]
    U_dev = B.gptq_factor(to_dev(X)).cpu().numpy()
    _same(got, gptq.sweep(W, U_dev), "sweep with the device factor")
    ref = gptq.quantize(W, X)

    def objective(pk):
        W_hat = int4_g128.dequantize(*pk)
        D = np.asarray(X, np.float64) @ (W_hat - W.astype(np.float64)).T
        return float((D * D).sum())

    assert objective(got) <= objective(ref) * (1 + 1e-3)
    codes = int4_g128.unpack(got[0]) == int4_g128.unpack(ref[0])
    assert codes.mean() > 0.99
    assert B.read_error_flags() == 0
