"""Decode kernel (M <= 64) against the float64 oracle on the same dequantized weights."""
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


def _run(B, fn, fmt, xbits, pk):
    X = x_to_dev(xbits)
    d = [to_dev(a) for a in pk]
    if fmt == "int4_g128":
        return fn(fmt, X, d[0], d[1], d[2])
    return fn(fmt, X, d[0], d[1])


CASES = [(16, 128), (1, 128), (256, 256), (1000, 512), (300, 1152), (777, 2048)]


@pytest.mark.parametrize("fmt", ["int4_g128", "mxfp4"])
@pytest.mark.parametrize("M", [1, 2, 3, 8, 9, 16])
@pytest.mark.parametrize("N,K", CASES)
def test_gemv_small(B, fmt, M, N, K):
    W = inputs.weights(N * 7 + K, N, K, 0.05)
    pk = _pack(fmt, W)
    xb, xf = inputs.activations(M + N, M, K)
    Y = _run(B, B.gemv_w4a16, fmt, xb, pk)
    ref = linear.linear_w4a16(fmt, xf, *pk)
    assert_close(y_to_host(Y), ref, "%s M=%d N=%d K=%d" % (fmt, M, N, K))


# One or two 256-row bands over a long K: every band is shared by 28-64 CTAs.  8-row tiles:
# the band's first CTA reads the others' posted sums in several chunks of 12; 16- and 32-row
# tiles: more CTAs share the band than it has 32-slot chunks, so some reduce nothing.  Run
# twice on one workspace: the exchange area is back at zero after each call.
@pytest.mark.parametrize("fmt", ["int4_g128", "mxfp4"])
@pytest.mark.parametrize("M", [1, 4, 16, 24])
@pytest.mark.parametrize("N,K", [(256, 14336), (300, 7168), (512, 32768)])
def test_gemv_band_shared_by_many_ctas(B, fmt, M, N, K):
    import torch
    W = inputs.weights(N + 3 * K, N, K, 0.05)
    pk = _pack(fmt, W)
    xb, xf = inputs.activations(M * 5 + K, M, K)
    ref = linear.linear_w4a16(fmt, xf, *pk)
    ws = torch.zeros(B.gemm_workspace_bytes(fmt, M, K, N), dtype=torch.uint8, device="cuda")
    X = x_to_dev(xb)
    d = [to_dev(a) for a in pk]
    for rep in range(2):
        Y = B.gemv_w4a16(fmt, X, d[0], d[1], d[2] if fmt == "int4_g128" else None, workspace=ws)
        assert_close(y_to_host(Y), ref, "%s M=%d N=%d K=%d call %d" % (fmt, M, N, K, rep))
    torch.cuda.synchronize()
    assert int(torch.count_nonzero(ws)) == 0, "split-K exchange words left behind"
    assert B.read_error_flags() == 0


@pytest.mark.parametrize("M", [1, 5, 16])
@pytest.mark.parametrize("K", [32, 96, 160, 1056])
def test_gemv_mxfp4_k_tail(B, M, K):
    # MXFP4 only needs K % 32 == 0: the last 128-k unit is partial.
    N = 300
    W = inputs.weights(K + 11, N, K, 0.05)
    pk = mxfp4.quantize(W)
    xb, xf = inputs.activations(K, M, K)
    Y = _run(B, B.gemv_w4a16, "mxfp4", xb, pk)
    assert_close(y_to_host(Y), linear.linear_w4a16("mxfp4", xf, *pk), "mxfp4 K=%d" % K)


def test_gemv_mxfp4_large_activations(B):
    # Activations beyond the fp16 range: the per-row power-of-two scaling keeps them exact.
    M, N, K = 4, 512, 1024
    W = inputs.weights(5, N, K, 0.05)
    pk = mxfp4.quantize(W)
    xb, xf = inputs.activations(6, M, K, scale=3.0e5)
    Y = _run(B, B.gemv_w4a16, "mxfp4", xb, pk)
    assert_close(y_to_host(Y), linear.linear_w4a16("mxfp4", xf, *pk), "mxfp4 big X")


@pytest.mark.parametrize("fmt", ["int4_g128", "mxfp4"])
@pytest.mark.parametrize("M", [4, 16])
def test_gemv_small_magnitude_activations(B, fmt, M):
    # Rows of ~1, 1e-6, 1e-20 and 1e-30 in one call (the MXFP4 decode path converts X to fp16
    # with a power of two per 8-row tile and stage); accuracy relative to each row's magnitude.
    from tests.test_gemm_tc_parity import _scaled_rows, check_small_rows
    N, K = 512, 1024
    W = inputs.weights(19, N, K, 0.05)
    pk = _pack(fmt, W)
    xb, xf, c = _scaled_rows(20 + M, M, K)
    y = y_to_host(_run(B, B.gemv_w4a16, fmt, xb, pk))
    check_small_rows(y, linear.linear_w4a16(fmt, xf, *pk), c, "%s M=%d small |x|" % (fmt, M))


def test_gemv_workspace_shared_across_shapes_and_kernels(B):
    # One workspace, zeroed once, serves calls of different shapes and both kernels.
    import torch
    shapes = [(4, 4096, 6144), (256, 4096, 512), (1, 4096, 28672), (16, 14336, 4096), (1, 4096, 28672)]
    nbytes = max(B.gemm_workspace_bytes("int4_g128", M, K, N) for M, K, N in shapes)
    ws = torch.zeros(nbytes, dtype=torch.uint8, device="cuda")
    for (M, K, N) in shapes:
        W = inputs.weights(N + K, N, K, 0.02)
        pk = int4_g128.quantize(W)
        xb, xf = inputs.activations(M, M, K)
        d = [to_dev(a) for a in pk]
        Y = y_to_host(B.gemm_w4a16("int4_g128", x_to_dev(xb), d[0], d[1], d[2], workspace=ws))
        rows = np.arange(0, N, max(1, N // 300))
        assert_close(Y[:, rows], linear.linear_rows("int4_g128", xf, pk[0], pk[1], pk[2], rows), "M=%d N=%d" % (M, N))


def test_gemv_deterministic_and_workspace_reusable(B):
    M, N, K = 4, 4096, 4096
    W = inputs.weights(9, N, K, 0.02)
    pk = int4_g128.quantize(W)
    xb, _ = inputs.activations(9, M, K)
    y1 = y_to_host(_run(B, B.gemv_w4a16, "int4_g128", xb, pk))
    y2 = y_to_host(_run(B, B.gemv_w4a16, "int4_g128", xb, pk))
    assert (y1 == y2).all()
    assert B.read_error_flags() == 0


# Full-size decode shapes (K, N) at M in {1, 4, 16}; the oracle checks 384 sampled output
# columns (all M rows) by dequantizing only those weight rows.
DECODE = [(4096, 4096), (4096, 6144), (4096, 28672), (14336, 4096), (8192, 8192)]


@pytest.mark.parametrize("fmt", ["int4_g128", "mxfp4"])
@pytest.mark.parametrize("K,N", DECODE)
def test_gemv_full_size_sampled(B, fmt, K, N):
    W = inputs.weights(1000 + K % 91 + N % 89, N, K, 0.02)
    pk = _pack(fmt, W)
    rows = np.sort(np.random.default_rng(K + N).choice(N, 384, replace=False))
    for M in (1, 4, 16):
        xb, xf = inputs.activations(M * 13 + K, M, K)
        Y = y_to_host(_run(B, B.gemv_w4a16, fmt, xb, pk))
        ref = linear.linear_rows(fmt, xf, pk[0], pk[1], pk[2] if fmt == "int4_g128" else None, rows)
        assert_close(Y[:, rows], ref, "%s K=%d N=%d M=%d" % (fmt, K, N, M))


def _layers(fmt, n_layers, K, seed):
    return [_pack(fmt, inputs.weights(seed + i, K, K, 0.03)) for i in range(n_layers)]


@pytest.mark.parametrize("fmt", ["int4_g128", "mxfp4"])
@pytest.mark.parametrize("graph", [False, True])
def test_gemv_chained_layers_read_the_previous_output(B, fmt, graph):
    # Each call's activations are the previous call's output, enqueued back to back with no
    # host synchronisation (and, with graph=True, replayed from one captured graph): every
    # call must read its input only after the previous kernel finished writing it.
    import torch
    M, K, L = 4, 1024, 8
    pks = _layers(fmt, L, K, 700)
    dev = [[to_dev(a) for a in pk] for pk in pks]
    xb, _ = inputs.activations(701, M, K)
    X0 = x_to_dev(xb)
    outs = [torch.empty((M, K), dtype=torch.bfloat16, device="cuda") for _ in range(L)]
    ws = torch.zeros(B.gemm_workspace_bytes(fmt, M, K, K), dtype=torch.uint8, device="cuda")

    def chain():
        x = X0
        for i in range(L):
            d = dev[i]
            B.gemv_w4a16(fmt, x, d[0], d[1], d[2] if fmt == "int4_g128" else None, out=outs[i], workspace=ws)
            x = outs[i]

    if graph:
        s = torch.cuda.Stream()
        with torch.cuda.stream(s):
            chain()
            torch.cuda.synchronize()
            for o in outs:
                o.zero_()
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, stream=s):
                chain()
            g.replay()
        torch.cuda.synchronize()
    else:
        chain()
    prev = np.asarray(inputs.activations(701, M, K)[1], dtype=np.float64)
    for i in range(L):
        y = y_to_host(outs[i])
        pk = pks[i]
        ref = linear.linear_w4a16(fmt, prev, *pk)
        assert_close(y, ref, "%s layer %d graph=%s" % (fmt, i, graph))
        prev = y.astype(np.float64)   # the next layer's reference starts from what the GPU produced
    assert B.read_error_flags() == 0


@pytest.mark.parametrize("fmt", ["int4_g128", "mxfp4"])
def test_gpu_quantize_then_decode_without_sync(B, fmt):
    # The decode call is enqueued right behind the quantize kernel that writes its weights.
    import torch
    M, N, K = 4, 2048, 2048
    W = inputs.weights(702, N, K, 0.02)
    Wd = torch.from_numpy(W).cuda()
    xb, xf = inputs.activations(703, M, K)
    X = x_to_dev(xb)
    if fmt == "int4_g128":
        Wq, s, z = B.quantize_int4_g128(Wd)
        Y = B.gemv_w4a16(fmt, X, Wq, s, z)
    else:
        Wq, s = B.quantize_mxfp4(Wd)
        Y = B.gemv_w4a16(fmt, X, Wq, s)
    ref = linear.linear_w4a16(fmt, xf, *_pack(fmt, W))
    assert_close(y_to_host(Y), ref, "%s quantize -> decode" % fmt)


# 17..64 activation rows: 32-row tiles (n-tiles in chunks of four), and M > 32 as consecutive
# 32-row launches on row slices of X and Y; bands shared by several CTAs and ragged tails.
@pytest.mark.parametrize("fmt", ["int4_g128", "mxfp4"])
@pytest.mark.parametrize("M", [17, 24, 32, 33, 40, 64])
@pytest.mark.parametrize("N,K", [(300, 1152), (1000, 512), (2048, 4096)])
def test_gemv_wide_tiles(B, fmt, M, N, K):
    W = inputs.weights(N * 5 + K + M, N, K, 0.05)
    pk = _pack(fmt, W)
    xb, xf = inputs.activations(M * 3 + N, M, K)
    Y = _run(B, B.gemv_w4a16, fmt, xb, pk)
    assert_close(y_to_host(Y), linear.linear_w4a16(fmt, xf, *pk), "%s M=%d N=%d K=%d" % (fmt, M, N, K))


@pytest.mark.parametrize("fmt", ["int4_g128", "mxfp4"])
def test_gemv_wide_tiles_full_size(B, fmt):
    # a decode-shaped layer at M = 48 (two slices), sampled output columns
    M, K, N = 48, 4096, 6144
    W = inputs.weights(77, N, K, 0.02)
    pk = _pack(fmt, W)
    xb, xf = inputs.activations(78, M, K)
    y = y_to_host(_run(B, B.gemv_w4a16, fmt, xb, pk))
    rows = np.sort(np.random.default_rng(79).choice(N, 256, replace=False))
    z = pk[2] if fmt == "int4_g128" else None
    assert_close(y[:, rows], linear.linear_rows(fmt, xf, pk[0], pk[1], z, rows), "%s M=48 sampled" % fmt)
