"""AWQ on the GPU against the oracle's search (第 1 章：推理加速全景 §4.4).

What is unique is compared exactly: the scales s for the chosen exponent and the packed
Q(W diag(s)) are bit-exact.  The losses are fp32 products with fp64 sums on the GPU against
float64 in the oracle: within 1e-4 relative.  The chosen exponent is an arg-min over those
losses; when two grid points lie within that tolerance either is correct, so the GPU's choice
is accepted if its oracle loss is within the tolerance of the oracle's minimum."""
import numpy as np
import pytest

from bit_weight_quantized_wq_gb300 import inputs
from oracle import awq, int4_g128
from tests._util import to_dev

pytestmark = pytest.mark.gpu

LOSS_RTOL = 1e-4


@pytest.fixture(scope="module")
def B():
    import torch
    from bit_weight_quantized_wq_gb300 import binding
    binding.check_device()
    torch.cuda.init()
    return binding


def _check(B, N, K, n, seed):
    W = inputs.weights(seed, N, K, 0.05)
    X = inputs.calibration(seed + 1, n, K)
    Wq, sc, z, s, a, losses = [t.cpu().numpy() for t in B.awq_int4_g128(to_dev(W), to_dev(X))]
    a_gpu = int(a[0])
    a_ref, s_ref, l_ref, _ = awq.search(W, X)
    rel = np.abs(losses - l_ref) / l_ref
    assert rel.max() <= LOSS_RTOL, (rel.max(), int(rel.argmax()))
    assert l_ref[a_gpu] <= l_ref[a_ref] * (1 + LOSS_RTOL), (a_gpu, a_ref)
    imp = awq.importance(X)
    s_exp = awq.scales(imp, awq.salient(imp), a_gpu)
    assert (s.view(np.uint32) == s_exp.view(np.uint32)).all()
    ref = awq.quantize_scaled(W, s_exp)
    for name, g, r in zip(("Wq", "scales", "zeros"), (Wq, sc, z), ref):
        assert (np.asarray(g).view(np.uint8) == np.asarray(r).view(np.uint8)).all(), name
    return a_gpu, l_ref


@pytest.mark.parametrize("N,K,n,seed", [(37, 128, 5, 1), (64, 1024, 128, 3), (100, 2048, 64, 5), (256, 4096, 128, 7)])
def test_awq_matches_oracle(B, N, K, n, seed):
    _check(B, N, K, n, seed)


def test_awq_full_size_llama3_8b_o_proj(B):
    a, losses = _check(B, 4096, 4096, 128, 9)
    assert 0 < a < awq.GRID and losses[a] < 0.8 * losses[0]


def test_awq_lowers_the_deployed_layer_error(B):
    # The packed result through the decode kernel, activations divided by s and rounded to bf16
    # as at run time: its error against X W^T is below round-to-nearest's through the same kernel.
    import torch
    N, K, n = 512, 2048, 16
    W = inputs.weights(11, N, K, 0.05)
    Xall = inputs.calibration(12, 128 + n, K)              # one draw: the same salient channels
    Xc, X = np.ascontiguousarray(Xall[:128]), np.ascontiguousarray(Xall[128:])   # calibrate / held out
    Wq, sc, z, s, a, losses = B.awq_int4_g128(to_dev(W), to_dev(Xc))
    Xs = torch.from_numpy(X).cuda() / s
    y_awq = B.gemm_w4a16("int4_g128", Xs.to(torch.bfloat16), Wq, sc, z).float().cpu().numpy()
    r = [to_dev(t) for t in int4_g128.quantize(W)]
    y_rtn = B.gemm_w4a16("int4_g128", torch.from_numpy(X).cuda().to(torch.bfloat16), *r).float().cpu().numpy()
    y = X.astype(np.float64) @ W.astype(np.float64).T
    assert ((y_awq - y) ** 2).sum() < 0.9 * ((y_rtn - y) ** 2).sum()
    assert B.read_error_flags() == 0
