"""The fused QKV projection with its output split into Q, K and V by the kernels' epilogue
(推理优化与量化算子深度技术调研 §4.2), against the float64 oracle's column blocks of the fused
product, on both paths: the decode kernel and the tensor-core kernel."""
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


def _qkv(B, fmt, xb, pk, Nq, Nkv, path=None):
    """path: "decode" or "tc" pins the dispatch for this (fmt, K, N); None keeps the default."""
    d = [to_dev(a) for a in pk]
    X = x_to_dev(xb)
    z = d[2] if fmt == "int4_g128" else None
    K, N = X.shape[1], Nq + 2 * Nkv
    old = B.dispatch_threshold(fmt, K, N)
    if path is not None:
        B.set_dispatch_threshold(fmt, K, N, 64 if path == "decode" else 0)
    try:
        return [y_to_host(t) for t in B.gemm_w4a16_qkv(fmt, X, d[0], d[1], z, Nq=Nq, Nkv=Nkv)]
    finally:
        B.set_dispatch_threshold(fmt, K, N, old)


def _check(got, ref_full, Nq, Nkv, what, rows=None):
    parts = linear.qkv_split(ref_full, Nq, Nkv) if rows is None else None
    names = ("Q", "K", "V")
    if rows is None:
        for g, r, nm in zip(got, parts, names):
            assert g.shape == r.shape
            assert_close(g, r, "%s %s" % (what, nm))
        return
    # sampled columns of the fused product: map each sampled column to its part
    cuts = (0, Nq, Nq + Nkv, Nq + 2 * Nkv)
    for i, nm in enumerate(names):
        sel = (rows >= cuts[i]) & (rows < cuts[i + 1])
        assert_close(got[i][:, rows[sel] - cuts[i]], ref_full[:, sel], "%s %s" % (what, nm))


# (Nq, Nkv, K): GQA 4/1 with d_head 64; a ragged split (the parts' boundaries inside a 16-row
# tile and inside a 256-row band); a 64/8-head-like ratio
SMALL = [(256, 64, 512), (200, 36, 384), (1024, 128, 1024)]


@pytest.mark.parametrize("fmt", ["int4_g128", "mxfp4"])
@pytest.mark.parametrize("M", [1, 5, 16, 40])
@pytest.mark.parametrize("Nq,Nkv,K", SMALL)
def test_qkv_decode(B, fmt, M, Nq, Nkv, K):
    N = Nq + 2 * Nkv
    pk = _pack(fmt, inputs.weights(Nq + K, N, K, 0.05))
    xb, xf = inputs.activations(M + Nq, M, K)
    got = _qkv(B, fmt, xb, pk, Nq, Nkv, path="decode")
    _check(got, linear.linear_w4a16(fmt, xf, *pk), Nq, Nkv, "%s M=%d" % (fmt, M))


@pytest.mark.parametrize("fmt", ["int4_g128", "mxfp4"])
@pytest.mark.parametrize("M", [17, 300])
@pytest.mark.parametrize("Nq,Nkv,K", SMALL)
def test_qkv_tensor_core(B, fmt, M, Nq, Nkv, K):
    N = Nq + 2 * Nkv
    pk = _pack(fmt, inputs.weights(Nq + K + 1, N, K, 0.05))
    xb, xf = inputs.activations(M + Nq + 1, M, K)
    got = _qkv(B, fmt, xb, pk, Nq, Nkv, path="tc")
    _check(got, linear.linear_w4a16(fmt, xf, *pk), Nq, Nkv, "%s M=%d" % (fmt, M))


def test_qkv_full_size_llama3_8b(B):
    # LLaMA-3-8B fused QKV: K = 4096, 32 query and 8 key/value heads of 128 (Nq 4096, Nkv 1024)
    Nq, Nkv, K = 4096, 1024, 4096
    N = Nq + 2 * Nkv
    pk = int4_g128.quantize(inputs.weights(1000, N, K, 0.02))
    rows = np.sort(np.random.default_rng(7).choice(N, 384, replace=False))
    for M in (1, 4, 16):
        xb, xf = inputs.activations(M * 13 + K, M, K)
        got = _qkv(B, "int4_g128", xb, pk, Nq, Nkv)
        _check(got, linear.linear_rows("int4_g128", xf, pk[0], pk[1], pk[2], rows), Nq, Nkv, "M=%d" % M, rows)
    assert B.read_error_flags() == 0


def test_qkv_full_size_qwen25_72b_prefill(B):
    # Qwen2.5-72B fused QKV: K = 8192, 64 query and 8 key/value heads of 128 (Nq 8192, Nkv 1024)
    Nq, Nkv, K, M = 8192, 1024, 8192, 2048
    N = Nq + 2 * Nkv
    pk = int4_g128.quantize(inputs.weights(3000, N, K, 0.015))
    rows = np.sort(np.random.default_rng(8).choice(N, 192, replace=False))
    xb, xf = inputs.activations(3100 + K, M, K)
    got = _qkv(B, "int4_g128", xb, pk, Nq, Nkv)
    _check(got, linear.linear_rows("int4_g128", xf, pk[0], pk[1], pk[2], rows), Nq, Nkv, "M=2048", rows)
    assert B.read_error_flags() == 0


def test_qkv_rejects_bad_arguments(B):
    import torch
    pk = [to_dev(a) for a in int4_g128.quantize(inputs.weights(1, 384, 256, 0.05))]
    X = torch.zeros((2, 256), dtype=torch.bfloat16, device="cuda")
    with pytest.raises(ValueError):
        B.gemm_w4a16_qkv("int4_g128", X, *pk, Nq=256, Nkv=32)            # 256 + 64 != 384
    with pytest.raises(ValueError):
        B.gemm_w4a16_qkv("int4_g128", X, *pk, Nq=256, Nkv=64,
                         out=(torch.empty((2, 256), dtype=torch.bfloat16, device="cuda"),) * 2)


@pytest.mark.parametrize("fmt", ["int4_g128", "mxfp4"])
def test_qkv_tensor_core_wide_short_k(B, fmt):
    # M = 256, Nq + 2 Nkv = 10240 rows (more tiles than SMs), short K = 256
    M, Nq, Nkv, K = 256, 8192, 1024, 256
    N = Nq + 2 * Nkv
    pk = _pack(fmt, inputs.weights(777, N, K, 0.05))
    xb, xf = inputs.activations(778, M, K)
    got = _qkv(B, fmt, xb, pk, Nq, Nkv, path="tc")
    _check(got, linear.linear_w4a16(fmt, xf, *pk), Nq, Nkv, "wide QKV %s" % fmt)
