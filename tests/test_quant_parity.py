"""GPU quantize + pack kernels against the CPU oracle: bit-exact codes, scales, zero points."""
import numpy as np
import pytest

from bit_weight_quantized_wq_gb300 import inputs
from oracle import int4_g128, mxfp4
from tests._util import to_dev

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def B():
    import torch
    from bit_weight_quantized_wq_gb300 import binding
    binding.check_device()
    torch.cuda.init()
    return binding


def _adversarial(K, seed=3):
    """Rows of special groups: constant, all +, all -, one outlier, exact ties, tiny, zeros, -0."""
    rng = np.random.default_rng(seed)
    rows = []
    rows.append(np.full(K, 0.37, np.float32))
    rows.append(np.abs(rng.standard_normal(K)).astype(np.float32))
    rows.append(-np.abs(rng.standard_normal(K)).astype(np.float32))
    o = (rng.standard_normal(K) * 0.02).astype(np.float32); o[::97] = 3.0; rows.append(o)
    rows.append(((np.arange(K) % 64) - 20).astype(np.float32) * np.float32(0.25))      # ties (INT4 and E2M1)
    rows.append(((np.arange(K) % 16) - 6).astype(np.float32) * np.float32(0.375))      # E2M1 midpoints
    rows.append((rng.standard_normal(K) * 1e-7).astype(np.float32))                    # fp16-subnormal scales
    rows.append((rng.standard_normal(K) * 1e-9).astype(np.float32))                    # scale underflow -> 1
    rows.append((rng.standard_normal(K) * 1e-39).astype(np.float32))                   # fp32 subnormals
    rows.append((rng.standard_normal(K) * 1e30).astype(np.float32))                    # large exponents (MXFP4)
    z = np.zeros(K, np.float32); z[::2] = -0.0; z[K // 2 + 5] = -1e-3; rows.append(z)
    rows.append(np.zeros(K, np.float32))
    return np.stack(rows)


def _check_int4(B, W, rows=None):
    Wd = to_dev(W)
    Wq, s, z = [t.cpu().numpy() for t in B.quantize_int4_g128(Wd)]
    sub = W if rows is None else W[rows]
    rq, rs, rz = int4_g128.quantize(sub)
    if rows is not None:
        Wq, s, z = Wq[rows], s[rows], z[rows]
    assert (Wq == rq).all(), "codes differ"
    assert (s.view(np.uint16) == rs.view(np.uint16)).all(), "scales differ"
    assert (z.view(np.uint16) == rz.view(np.uint16)).all(), "zeros differ"


def _check_mxfp4(B, W, rows=None):
    Wd = to_dev(W)
    Wq, s = [t.cpu().numpy() for t in B.quantize_mxfp4(Wd)]
    sub = W if rows is None else W[rows]
    rq, rs = mxfp4.quantize(sub)
    if rows is not None:
        Wq, s = Wq[rows], s[rows]
    assert (s == rs).all(), "E8M0 scales differ"
    assert (Wq == rq).all(), "codes differ"


@pytest.mark.parametrize("K", [128, 256, 1152])
def test_int4_adversarial(B, K):
    _check_int4(B, _adversarial(K))


@pytest.mark.parametrize("K", [32, 96, 256, 1056])
def test_mxfp4_adversarial(B, K):
    _check_mxfp4(B, _adversarial(K))


@pytest.mark.parametrize("N,K", [(1, 128), (3, 384), (257, 640), (4096, 4096)])
def test_int4_random(B, N, K):
    _check_int4(B, inputs.weights(N + K, N, K, 0.02))


@pytest.mark.parametrize("N,K", [(1, 32), (5, 160), (257, 640), (4096, 4096)])
def test_mxfp4_random(B, N, K):
    _check_mxfp4(B, inputs.weights(N + K + 1, N, K, 0.02))


# The weight shapes of the decode and prefill workloads (W is [N, K]); the oracle checks a
# seeded sample of rows on the largest ones (quantization is independent per row).
SHAPES = [(6144, 4096), (4096, 4096), (28672, 4096), (4096, 14336), (8192, 8192), (10240, 8192),
          (8192, 29568)]


@pytest.mark.parametrize("N,K", SHAPES)
def test_int4_config_shapes(B, N, K):
    W = inputs.weights(3000 + N % 97, N, K, 0.02)
    rows = None if N * K <= 4096 * 4096 else np.sort(np.random.default_rng(N).choice(N, 512, replace=False))
    _check_int4(B, W, rows)


@pytest.mark.parametrize("N,K", SHAPES[:4])
def test_mxfp4_config_shapes(B, N, K):
    W = inputs.weights(2000 + N % 97, N, K, 0.02)
    rows = None if N * K <= 4096 * 4096 else np.sort(np.random.default_rng(N).choice(N, 512, replace=False))
    _check_mxfp4(B, W, rows)
