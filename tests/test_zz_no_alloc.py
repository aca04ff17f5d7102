"""The decode kernel's no-allocation entry point, wq_gemv_w4a16_noalloc, called through the C
ABI.  It is for callers that cannot allocate device memory when they run the layer (a host
framework that owns every allocation, a latency-critical loop that cannot afford the
synchronisation of cudaMalloc); its scratch is one library-owned device array.

Checked against the workspace entry point wq_gemv_w4a16 on two calls in a row (different
formats and shapes, so the second call reuses the array the first one left behind), within
the tests' tolerance.  Kept in a file collected last so that a run stopping at the first
failure has already run every other test."""
import ctypes

import numpy as np
import pytest

from bit_weight_quantized_wq_gb300 import inputs
from oracle import int4_g128, mxfp4
from tests._util import assert_close, to_dev, x_to_dev, y_to_host

pytestmark = pytest.mark.gpu


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
    X = x_to_dev(inputs.activations(seed + 1, M, K)[0])
    return X, Wq, s, z, torch.empty((M, N), dtype=torch.bfloat16, device="cuda")


def _with_workspace(lib, fmt, X, Wq, s, z, M, K, N):
    import torch
    ws = torch.zeros(lib.wq_gemm_workspace_bytes(fmt, M, K, N), dtype=torch.uint8, device="cuda")
    Y = torch.empty((M, N), dtype=torch.bfloat16, device="cuda")
    st = lib.wq_gemv_w4a16(fmt, _p(X), M, K, N, _p(Wq), _p(s), _p(z), _p(Y), _p(ws), ws.numel(), None)
    assert st == 0
    return Y


def test_noalloc_matches_workspace_entry_two_calls_in_a_row(lib):
    import torch
    cases = [(0, 4, 4096, 28672, 11), (1, 16, 14336, 4096, 12)]   # (fmt, M, K, N, seed)
    for fmt, M, K, N, seed in cases:
        X, Wq, s, z, Y = _case(fmt, M, K, N, seed)
        st = lib.wq_gemv_w4a16_noalloc(fmt, _p(X), M, K, N, _p(Wq), _p(s), _p(z), _p(Y), None)
        assert st == 0, lib.wq_status_str(st)
        ref = y_to_host(_with_workspace(lib, fmt, X, Wq, s, z, M, K, N))
        torch.cuda.synchronize()
        assert_close(y_to_host(Y), ref, "noalloc fmt=%d M=%d N=%d" % (fmt, M, N))
    # and the same shape twice more: the array keeps the previous call's contents
    for _ in range(2):
        fmt, M, K, N, seed = cases[0]
        X, Wq, s, z, Y = _case(fmt, M, K, N, seed + 7)
        assert lib.wq_gemv_w4a16_noalloc(fmt, _p(X), M, K, N, _p(Wq), _p(s), _p(z), _p(Y), None) == 0
        assert_close(y_to_host(Y), y_to_host(_with_workspace(lib, fmt, X, Wq, s, z, M, K, N)), "repeat")


def test_noalloc_rejects_sizes_beyond_its_array(lib):
    fake = ctypes.c_void_p(0x10000)       # never dereferenced: refused before any launch
    assert lib.wq_gemv_w4a16_noalloc(0, fake, 1, 128, 2097152 + 128, fake, fake, fake, fake, None) == 2
    assert lib.wq_gemv_w4a16_noalloc(0, fake, 17, 128, 256, fake, fake, fake, fake, None) == 2
    assert lib.wq_gemv_w4a16_noalloc(0, None, 1, 128, 256, fake, fake, fake, fake, None) == 1
