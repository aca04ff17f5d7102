"""The decode kernel's no-allocation entry point, wq_gemv_w4a16_noalloc, called through the C
ABI.  It is for callers that cannot allocate device memory when they run the layer (a host
framework that owns every allocation, a latency-critical loop that cannot afford the
synchronisation of cudaMalloc); its scratch is one library-owned device array.

Each call is checked element by element against the float64 oracle on the same dequantized
weights (sampled output columns on the large shapes), and bit for bit against the workspace
entry point wq_gemv_w4a16 (the same kernel with a deterministic split-K reduction), on calls
in a row of different formats and shapes, so that each reuses the array the previous one
left behind.  One call goes through the Python wrapper on a non-default stream.  Kept in a
file collected last so that a run stopping at the first failure has already run every
other test."""
import ctypes

import numpy as np
import pytest

from bit_weight_quantized_wq_gb300 import inputs
from oracle import int4_g128, linear, mxfp4
from tests._util import assert_close, to_dev, x_to_dev, y_to_host

pytestmark = pytest.mark.gpu

FMT_NAME = {0: "int4_g128", 1: "mxfp4"}


@pytest.fixture(scope="module")
def lib():
    import torch
    from bit_weight_quantized_wq_gb300 import binding
    binding.check_device()
    torch.cuda.init()
    return binding.load_library()


def _p(t):
    return ctypes.c_void_p(0 if t is None else t.data_ptr())


def _case(fmt, M, K, N, seed):
    import torch
    W = inputs.weights(seed, N, K, 0.02)
    pk = int4_g128.quantize(W) if fmt == 0 else mxfp4.quantize(W)
    d = [to_dev(a) for a in pk]
    Wq, s = d[0], d[1]
    z = d[2] if fmt == 0 else None
    xb, xf = inputs.activations(seed + 1, M, K)
    X = x_to_dev(xb)
    return (X, Wq, s, z, torch.empty((M, N), dtype=torch.bfloat16, device="cuda")), pk, xf


def _with_workspace(lib, fmt, X, Wq, s, z, M, K, N):
    import torch
    ws = torch.zeros(lib.wq_gemm_workspace_bytes(fmt, M, K, N), dtype=torch.uint8, device="cuda")
    Y = torch.empty((M, N), dtype=torch.bfloat16, device="cuda")
    st = lib.wq_gemv_w4a16(fmt, _p(X), M, K, N, _p(Wq), _p(s), _p(z), _p(Y), _p(ws), ws.numel(), None)
    assert st == 0
    return Y


def _oracle(fmt, xf, pk, N, seed):
    """float64 oracle for all columns (N <= 4096) or for 384 seeded sample columns."""
    if N <= 4096:
        return np.arange(N), linear.linear_w4a16(FMT_NAME[fmt], xf, *pk)
    rows = np.sort(np.random.default_rng(seed).choice(N, 384, replace=False))
    z = pk[2] if fmt == 0 else None
    return rows, linear.linear_rows(FMT_NAME[fmt], xf, pk[0], pk[1], z, rows)


def test_noalloc_matches_oracle_and_workspace_entry_calls_in_a_row(lib):
    import torch
    # (fmt, M, K, N, seed): a wide INT4 layer, an MXFP4 down projection, a small INT4 layer
    # and the wide one again, so every call follows a call of another shape
    cases = [(0, 4, 4096, 28672, 11), (1, 16, 14336, 4096, 12), (0, 3, 1024, 640, 13), (0, 4, 4096, 28672, 14)]
    for fmt, M, K, N, seed in cases:
        (X, Wq, s, z, Y), pk, xf = _case(fmt, M, K, N, seed)
        st = lib.wq_gemv_w4a16_noalloc(fmt, _p(X), M, K, N, _p(Wq), _p(s), _p(z), _p(Y), None)
        assert st == 0, lib.wq_status_str(st)
        torch.cuda.synchronize()
        y = y_to_host(Y)
        rows, ref = _oracle(fmt, xf, pk, N, seed)
        assert_close(y[:, rows], ref, "noalloc vs oracle fmt=%d M=%d N=%d" % (fmt, M, N))
        y_ws = y_to_host(_with_workspace(lib, fmt, X, Wq, s, z, M, K, N))
        assert np.array_equal(y, y_ws), "noalloc and workspace entry differ (fmt=%d M=%d N=%d)" % (fmt, M, N)


def test_noalloc_python_wrapper_on_a_side_stream(lib):
    import torch
    from bit_weight_quantized_wq_gb300 import binding
    M, K, N, seed = 9, 2048, 3000, 21
    (X, Wq, s, z, _), pk, xf = _case(0, M, K, N, seed)
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        Y1 = binding.gemv_w4a16_noalloc("int4_g128", X, Wq, s, z)
        Y2 = binding.gemv_w4a16_noalloc("int4_g128", X, Wq, s, z, stream=side)
    side.synchronize()
    rows, ref = _oracle(0, xf, pk, N, seed)
    assert_close(y_to_host(Y1)[:, rows], ref, "noalloc wrapper, side stream")
    assert np.array_equal(y_to_host(Y1), y_to_host(Y2))
    # the wrapper's argument checks run before any pointer reaches the library
    with pytest.raises(ValueError):
        binding.gemv_w4a16_noalloc("int4_g128", X, Wq[:, :-1].contiguous(), s, z)     # Wq not [N, K/8]
    with pytest.raises(ValueError):
        binding.gemv_w4a16_noalloc("int4_g128", X, Wq, s[:-1], z)                     # scales too short
    with pytest.raises(ValueError):
        binding.gemv_w4a16_noalloc("int4_g128", X, Wq, s, z,
                                   out=torch.empty((M, N - 1), dtype=torch.bfloat16, device="cuda"))
    with pytest.raises(ValueError):
        binding.gemv_w4a16_noalloc("int4_g128", X, Wq.cpu(), s, z)                    # not on the GPU


def test_noalloc_rejects_sizes_beyond_its_array(lib):
    fake = ctypes.c_void_p(0x10000)       # never dereferenced: refused before any launch
    assert lib.wq_gemv_w4a16_noalloc(0, fake, 1, 128, 2097152 + 128, fake, fake, fake, fake, None) == 2
    assert lib.wq_gemv_w4a16_noalloc(0, fake, 17, 128, 256, fake, fake, fake, fake, None) == 2
    assert lib.wq_gemv_w4a16_noalloc(0, None, 1, 128, 256, fake, fake, fake, fake, None) == 1
