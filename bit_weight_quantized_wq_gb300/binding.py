"""Thin ctypes binding of libwq.so (include/wq.h): argument marshalling only.

Every step of the quantized layer runs in the library's CUDA kernels; this module only
turns torch CUDA tensors into raw device pointers and the current torch stream into a
``cudaStream_t``.  PyTorch supplies device memory and streams.  There is no CPU fallback:
if the library is missing or the device is not a GB300-class part, calls raise.

Function names follow the C ABI (``wq_quantize_int4_g128`` -> ``quantize_int4_g128`` ...).
A non-OK status raises ``ValueError`` (argument errors, as the lesson's
``blockwise_symmetric_fake_quant`` does for invalid geometry) or ``RuntimeError``.
"""
from __future__ import annotations

import ctypes
import os

import torch

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libwq.so")

FMT_INT4_G128 = 0
FMT_MXFP4 = 1
_FMT_NAMES = {"int4_g128": FMT_INT4_G128, "mxfp4": FMT_MXFP4}

_STATUS = {0: "WQ_OK", 1: "WQ_ERR_NULL", 2: "WQ_ERR_SHAPE", 3: "WQ_ERR_ALIGN", 4: "WQ_ERR_WORKSPACE",
           5: "WQ_ERR_UNSUPPORTED_ARCH", 6: "WQ_ERR_CUDA", 7: "WQ_ERR_ARG"}

EXPORTED = [
    "wq_quantize_int4_g128", "wq_quantize_mxfp4", "wq_gemm_workspace_bytes", "wq_gemm_w4a16",
    "wq_gemv_w4a16", "wq_gemm_tc_w4a16", "wq_dispatch_threshold", "wq_set_dispatch_threshold",
    "wq_status_str", "wq_read_error_flags", "wq_check_device", "wq_gemv_w4a16_noalloc",
    "wq_gemm_w4a16_swiglu", "wq_gemv_w4a16_swiglu", "wq_gemm_tc_w4a16_swiglu", "wq_interleave_gate_up",
    "wq_gptq_int4_g128", "wq_awq_workspace_bytes", "wq_awq_int4_g128", "wq_selftest_wait_timeout",
    "wq_gemm_w4a16_qkv", "wq_gptq_workspace_bytes", "wq_gptq_factor", "wq_gptq_int4_g128_calib",
    "wq_quantize_fp8_weights", "wq_quantize_fp8_activations", "wq_gemm_fp8", "wq_gemm_w8a8_fp8_workspace_bytes",
    "wq_gemm_w8a8_fp8", "wq_mxfp4_weights_to_e4m3", "wq_quantize_w4a4_activations", "wq_gemm_w4a4_mxfp4",
]

_lib = None


def load_library(path: str = LIB_PATH) -> ctypes.CDLL:
    """Loads libwq.so and declares the C signatures.  Raises if it is missing."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(path):
        raise RuntimeError("libwq.so not built: run `python -c 'import __graft_entry__ as g; g.build()'` "
                           "(or python -m bit_weight_quantized_wq_gb300.build)")
    lib = ctypes.CDLL(path)
    P, I64, SZ, I32, U32 = ctypes.c_void_p, ctypes.c_int64, ctypes.c_size_t, ctypes.c_int, ctypes.c_uint32
    sig = {
        "wq_quantize_int4_g128": (I32, [P, I64, I64, P, P, P, P]),
        "wq_quantize_mxfp4": (I32, [P, I64, I64, P, P, P]),
        "wq_gemm_workspace_bytes": (SZ, [I32, I64, I64, I64]),
        "wq_gemm_w4a16": (I32, [I32, P, I64, I64, I64, P, P, P, P, P, SZ, P]),
        "wq_gemv_w4a16": (I32, [I32, P, I64, I64, I64, P, P, P, P, P, SZ, P]),
        "wq_gemm_tc_w4a16": (I32, [I32, P, I64, I64, I64, P, P, P, P, P, SZ, P]),
        "wq_dispatch_threshold": (I64, [I32, I64, I64]),
        "wq_set_dispatch_threshold": (I32, [I32, I64, I64, I64]),
        "wq_status_str": (ctypes.c_char_p, [I32]),
        "wq_read_error_flags": (I32, [ctypes.POINTER(U32)]),
        "wq_check_device": (I32, []),
        "wq_gemv_w4a16_noalloc": (I32, [I32, P, I64, I64, I64, P, P, P, P, P]),
        "wq_gemm_w4a16_swiglu": (I32, [I32, P, I64, I64, I64, P, P, P, P, P, SZ, P]),
        "wq_gemv_w4a16_swiglu": (I32, [I32, P, I64, I64, I64, P, P, P, P, P, SZ, P]),
        "wq_gemm_tc_w4a16_swiglu": (I32, [I32, P, I64, I64, I64, P, P, P, P, P, SZ, P]),
        "wq_interleave_gate_up": (I32, [P, P, I64, I64, P]),
        "wq_gptq_int4_g128": (I32, [P, I64, I64, P, P, P, P, P]),
        "wq_awq_workspace_bytes": (SZ, [I64, I64, I64]),
        "wq_awq_int4_g128": (I32, [P, I64, I64, P, I64, P, P, P, P, P, P, P, SZ, P]),
        "wq_selftest_wait_timeout": (I32, [U32, ctypes.POINTER(U32), P]),
        "wq_gemm_w4a16_qkv": (I32, [I32, P, I64, I64, I64, I64, P, P, P, P, P, P, P, SZ, P]),
        "wq_gptq_workspace_bytes": (SZ, [I64]),
        "wq_gptq_factor": (I32, [P, I64, I64, P, P, SZ, P]),
        "wq_gptq_int4_g128_calib": (I32, [P, I64, I64, P, I64, P, P, P, P, SZ, P]),
        "wq_quantize_fp8_weights": (I32, [P, I64, I64, P, P, P]),
        "wq_quantize_fp8_activations": (I32, [P, I64, I64, P, P, P]),
        "wq_gemm_fp8": (I32, [P, P, I64, I64, I64, P, P, P, P]),
        "wq_gemm_w8a8_fp8_workspace_bytes": (SZ, [I64, I64]),
        "wq_gemm_w8a8_fp8": (I32, [P, I64, I64, I64, P, P, P, P, SZ, P]),
        "wq_mxfp4_weights_to_e4m3": (I32, [P, P, I64, I64, P, P, P]),
        "wq_quantize_w4a4_activations": (I32, [P, I64, I64, P, P, P]),
        "wq_gemm_w4a4_mxfp4": (I32, [P, I64, I64, I64, P, P, P, P, SZ, P]),
    }
    for name, (res, args) in sig.items():
        f = getattr(lib, name)
        f.restype = res
        f.argtypes = args
    _lib = lib
    return lib


def status_str(status: int) -> str:
    return load_library().wq_status_str(int(status)).decode()


def _check(status: int, what: str) -> None:
    if status == 0:
        return
    msg = "%s failed: %s" % (what, status_str(status))
    if status in (1, 2, 3, 4, 7):
        raise ValueError(msg)
    raise RuntimeError(msg)


def _fmt(fmt) -> int:
    if isinstance(fmt, str):
        return _FMT_NAMES[fmt]
    return int(fmt)


def _ptr(t):
    return None if t is None else t.data_ptr()


# The current stream's raw handle without building a Stream object (a few microseconds per
# call otherwise, which dominates small decode calls issued from Python).
_raw_current_stream = getattr(torch._C, "_cuda_getCurrentRawStream", None)


def _stream(stream=None, device=None):
    if stream is not None:
        return stream.cuda_stream
    if _raw_current_stream is not None:
        idx = device.index if device is not None and device.index is not None else torch.cuda.current_device()
        return _raw_current_stream(idx)
    return torch.cuda.current_stream(device).cuda_stream


def _need(t: torch.Tensor, dtype, name: str) -> None:
    if not t.is_cuda:
        raise ValueError("%s must be a CUDA tensor" % name)
    if t.dtype != dtype:
        raise ValueError("%s must be %s, got %s" % (name, dtype, t.dtype))
    if not t.is_contiguous():
        raise ValueError("%s must be contiguous" % name)


def check_device() -> None:
    _check(load_library().wq_check_device(), "wq_check_device")


def quantize_int4_g128(W: torch.Tensor, stream=None):
    """W float32 [N, K] (CUDA) -> (Wq int32 [N, K/8], scales fp16 [N, K/128], zeros fp16 [N, K/128])."""
    _need(W, torch.float32, "W")
    N, K = W.shape
    Wq = torch.empty((N, K // 8), dtype=torch.int32, device=W.device)
    scales = torch.empty((N, K // 128), dtype=torch.float16, device=W.device)
    zeros = torch.empty((N, K // 128), dtype=torch.float16, device=W.device)
    _check(load_library().wq_quantize_int4_g128(_ptr(W), N, K, _ptr(Wq), _ptr(scales), _ptr(zeros),
                                                     _stream(stream, W.device)), "wq_quantize_int4_g128")
    return Wq, scales, zeros


def quantize_mxfp4(W: torch.Tensor, stream=None):
    """W float32 [N, K] (CUDA) -> (Wq int32 [N, K/8], scales uint8 [N, K/32])."""
    _need(W, torch.float32, "W")
    N, K = W.shape
    Wq = torch.empty((N, K // 8), dtype=torch.int32, device=W.device)
    scales = torch.empty((N, K // 32), dtype=torch.uint8, device=W.device)
    _check(load_library().wq_quantize_mxfp4(_ptr(W), N, K, _ptr(Wq), _ptr(scales), _stream(stream, W.device)),
           "wq_quantize_mxfp4")
    return Wq, scales


def gptq_int4_g128(W: torch.Tensor, U: torch.Tensor, stream=None):
    """GPTQ of W float32 [N, K] (CUDA) with U float32 [K, K], the upper Cholesky factor of the
    inverse Hessian (H^-1 = U^T U) -> (Wq int32 [N, K/8], scales fp16 [N, K/128], zeros fp16)."""
    _need(W, torch.float32, "W")
    _need(U, torch.float32, "U")
    N, K = W.shape
    if tuple(U.shape) != (K, K):
        raise ValueError("U must be [K, K]")
    Wq = torch.empty((N, K // 8), dtype=torch.int32, device=W.device)
    scales = torch.empty((N, K // 128), dtype=torch.float16, device=W.device)
    zeros = torch.empty((N, K // 128), dtype=torch.float16, device=W.device)
    _check(load_library().wq_gptq_int4_g128(_ptr(W), N, K, _ptr(U), _ptr(Wq), _ptr(scales), _ptr(zeros),
                                            _stream(stream, W.device)), "wq_gptq_int4_g128")
    return Wq, scales, zeros


def _gptq_workspace(K, dev, workspace):
    need = int(load_library().wq_gptq_workspace_bytes(K))
    if workspace is None:
        return torch.empty((need,), dtype=torch.uint8, device=dev)
    if not workspace.is_cuda or workspace.device != dev or not workspace.is_contiguous():
        raise ValueError("workspace must be a contiguous CUDA tensor on X's device")
    return workspace


def gptq_factor(X: torch.Tensor, workspace=None, stream=None):
    """The upper factor U float32 [K, K] of H^-1 = U^T U, H = 2 X^T X + lambda I, from calibration
    activations X float32 [n, K] (CUDA), computed on the device in float64."""
    _need(X, torch.float32, "X")
    n, K = X.shape
    ws = _gptq_workspace(K, X.device, workspace)
    U = torch.empty((K, K), dtype=torch.float32, device=X.device)
    _check(load_library().wq_gptq_factor(_ptr(X), n, K, _ptr(U), _ptr(ws), ws.numel(), _stream(stream, X.device)),
           "wq_gptq_factor")
    return U


def gptq_int4_g128_calib(W: torch.Tensor, X: torch.Tensor, workspace=None, stream=None):
    """GPTQ of W float32 [N, K] from calibration activations X float32 [n, K] (both CUDA), the
    factor and the sweep on the device -> (Wq int32 [N, K/8], scales fp16, zeros fp16)."""
    _need(W, torch.float32, "W")
    _need(X, torch.float32, "X")
    N, K = W.shape
    if X.dim() != 2 or X.shape[1] != K or X.device != W.device:
        raise ValueError("X must be [n, K] on W's device")
    n = X.shape[0]
    ws = _gptq_workspace(K, W.device, workspace)
    Wq = torch.empty((N, K // 8), dtype=torch.int32, device=W.device)
    scales = torch.empty((N, K // 128), dtype=torch.float16, device=W.device)
    zeros = torch.empty((N, K // 128), dtype=torch.float16, device=W.device)
    _check(load_library().wq_gptq_int4_g128_calib(_ptr(W), N, K, _ptr(X), n, _ptr(Wq), _ptr(scales), _ptr(zeros),
                                                  _ptr(ws), ws.numel(), _stream(stream, W.device)),
           "wq_gptq_int4_g128_calib")
    return Wq, scales, zeros


def awq_int4_g128(W: torch.Tensor, X: torch.Tensor, workspace=None, stream=None):
    """AWQ of W float32 [N, K] with calibration activations X float32 [n, K] (both CUDA) ->
    (Wq, scales, zeros, s float32 [K], alpha_index int32 [1], losses float64 [21]); the layer's
    activations are divided by s at run time."""
    _need(W, torch.float32, "W")
    _need(X, torch.float32, "X")
    N, K = W.shape
    n = X.shape[0]
    if X.shape[1] != K:
        raise ValueError("X must be [n, K]")
    dev = W.device
    Wq = torch.empty((N, K // 8), dtype=torch.int32, device=dev)
    scales = torch.empty((N, K // 128), dtype=torch.float16, device=dev)
    zeros = torch.empty((N, K // 128), dtype=torch.float16, device=dev)
    s = torch.empty((K,), dtype=torch.float32, device=dev)
    a = torch.empty((1,), dtype=torch.int32, device=dev)
    losses = torch.empty((21,), dtype=torch.float64, device=dev)
    lib = load_library()
    if workspace is None:
        workspace = torch.empty((int(lib.wq_awq_workspace_bytes(N, K, n)),), dtype=torch.uint8, device=dev)
    _check(lib.wq_awq_int4_g128(_ptr(W), N, K, _ptr(X), n, _ptr(Wq), _ptr(scales), _ptr(zeros), _ptr(s), _ptr(a),
                                _ptr(losses), _ptr(workspace), workspace.numel() * workspace.element_size(),
                                _stream(stream, dev)), "wq_awq_int4_g128")
    return Wq, scales, zeros, s, a, losses


def gemm_workspace_bytes(fmt, M: int, K: int, N: int) -> int:
    return int(load_library().wq_gemm_workspace_bytes(_fmt(fmt), M, K, N))


class Workspace:
    """A zero-initialised device scratch buffer that grows on demand (one per stream)."""

    def __init__(self, device=None):
        self.device = torch.device("cuda") if device is None else torch.device(device)
        self.buf = None

    def get(self, nbytes: int):
        if nbytes == 0:
            return None
        if self.buf is None or self.buf.numel() < nbytes:
            self.buf = torch.zeros(((nbytes + 255) // 256) * 256, dtype=torch.uint8, device=self.device)
        return self.buf


_default_ws = {}


def _workspace_for(device, nbytes, workspace):
    if workspace is not None:
        return workspace
    key = (str(device), torch.cuda.current_stream(device).cuda_stream)
    ws = _default_ws.get(key)
    if ws is None:
        ws = _default_ws[key] = Workspace(device)
    return ws.get(nbytes)


_fns = {}
_BF16, _F16, _I32, _U8 = torch.bfloat16, torch.float16, torch.int32, torch.uint8


def _fn(cname: str):
    f = _fns.get(cname)
    if f is None:
        f = _fns[cname] = getattr(load_library(), cname)
    return f


def _inputs(f, X, Wq, scales, zeros):
    """The checks every layer call makes on its inputs before their pointers reach the library,
    which sees only raw addresses and sizes: dtypes, devices, contiguity, and the shapes of Wq,
    scales and zeros against X.  Returns (M, K, N, CUDA device index).  Device checks use
    ``get_device()`` (an int, -1 on the CPU), cheaper per call than comparing device objects."""
    int4 = f == FMT_INT4_G128
    if (X.dtype is not _BF16 or Wq.dtype is not _I32 or scales.dtype is not (_F16 if int4 else _U8)
            or (zeros is not None and (not int4 or zeros.dtype is not _F16)) or (int4 and zeros is None)):
        _linear_explain(f, X, Wq, scales, zeros)
    d = X.get_device()
    if d < 0 or not (X.is_contiguous() and Wq.is_contiguous() and scales.is_contiguous()
                     and (zeros is None or zeros.is_contiguous())):
        _linear_explain(f, X, Wq, scales, zeros)
    if X.dim() != 2 or Wq.dim() != 2:
        raise ValueError("X must be [M, K] and Wq [N, K/8]")
    M, K = X.shape
    N = Wq.shape[0]
    if Wq.shape[1] * 8 != K:
        raise ValueError("Wq must be [N, K/8]")
    meta = (N, K // 128) if int4 else (N, K // 32)
    if scales.shape != meta or (zeros is not None and zeros.shape != meta):
        raise ValueError("scales%s must be [N, K/%d]" % (" and zeros" if int4 else "", 128 if int4 else 32))
    if Wq.get_device() != d or scales.get_device() != d or (zeros is not None and zeros.get_device() != d):
        if not (Wq.is_cuda and scales.is_cuda and (zeros is None or zeros.is_cuda)):
            _linear_explain(f, X, Wq, scales, zeros)
        raise ValueError("X, Wq, scales and zeros must be on the same device")
    return M, K, N, d


def _output(out, M, ncol, d, name="out"):
    """A bf16 [M, ncol] output on CUDA device ``d``: ``out`` checked, or a new tensor when None."""
    if out is None:
        return torch.empty((M, ncol), dtype=_BF16, device=torch.device("cuda", d))
    if out.dtype is not _BF16 or not out.is_contiguous() or out.get_device() < 0:
        _need(out, _BF16, name)
    if out.shape != (M, ncol) or out.get_device() != d:
        raise ValueError("%s must be [%d, %d] on X's device" % (name, M, ncol))
    return out


def _prepare(f, X, Wq, scales, zeros, out, swiglu):
    M, K, N, d = _inputs(f, X, Wq, scales, zeros)
    return M, K, N, _output(out, M, N // 2 if swiglu else N, d)


def _linear(cname: str, fmt, X, Wq, scales, zeros, out, workspace, stream, swiglu=False):
    # Marshalling for every layer call, kept lean: a decode layer runs in a few microseconds,
    # so the host side of the call must not be the slower one.  Types, devices, contiguity and
    # shapes are checked here (the library sees raw pointers); alignment, size limits and the
    # workspace size in C.
    f = fmt if fmt.__class__ is int else _FMT_NAMES[fmt]
    M, K, N, d = _inputs(f, X, Wq, scales, zeros)
    out = _output(out, M, N // 2 if swiglu else N, d)
    # a caller's workspace is checked by the library itself (WQ_ERR_WORKSPACE when too small)
    if workspace is not None and (workspace.get_device() != d or not workspace.is_contiguous()):
        raise ValueError("workspace must be a contiguous CUDA tensor on X's device")
    ws = workspace if workspace is not None else _workspace_for(X.device, gemm_workspace_bytes(f, M, K, N), None)
    ws_bytes = 0 if ws is None else ws.numel() * ws.element_size()
    if stream is not None:
        sh = stream.cuda_stream
    elif _raw_current_stream is not None:
        sh = _raw_current_stream(d)
    else:
        sh = torch.cuda.current_stream(X.device).cuda_stream
    st = _fn(cname)(f, X.data_ptr(), M, K, N // 2 if swiglu else N, Wq.data_ptr(), scales.data_ptr(),
                    None if zeros is None else zeros.data_ptr(), out.data_ptr(),
                    None if ws is None else ws.data_ptr(), ws_bytes, sh)
    if st:
        _check(st, cname)
    return out


def _linear_explain(f, X, Wq, scales, zeros):
    """Raises the precise error for a call that failed the fast type/device checks."""
    _need(X, _BF16, "X")
    _need(Wq, _I32, "Wq")
    if f == FMT_INT4_G128:
        _need(scales, _F16, "scales")
        if zeros is None:
            raise ValueError("zeros is required for INT4 g128")
        _need(zeros, _F16, "zeros")
    else:
        _need(scales, _U8, "scales")
        if zeros is not None:
            raise ValueError("zeros must be None for MXFP4")
    raise ValueError("invalid arguments")


def gemm_w4a16(fmt, X, Wq, scales, zeros=None, out=None, workspace=None, stream=None):
    """Y = X * dequant(Wq)^T (bf16 [M, N]); dispatches between the decode and tensor-core kernels."""
    return _linear("wq_gemm_w4a16", fmt, X, Wq, scales, zeros, out, workspace, stream)


def gemv_w4a16(fmt, X, Wq, scales, zeros=None, out=None, workspace=None, stream=None):
    """The decode kernel alone (M <= 64)."""
    return _linear("wq_gemv_w4a16", fmt, X, Wq, scales, zeros, out, workspace, stream)


def gemm_tc_w4a16(fmt, X, Wq, scales, zeros=None, out=None, workspace=None, stream=None):
    """The tcgen05 tensor-core kernel alone (any M)."""
    return _linear("wq_gemm_tc_w4a16", fmt, X, Wq, scales, zeros, out, workspace, stream)


def gemm_w4a16_swiglu(fmt, X, Wq, scales, zeros=None, out=None, workspace=None, stream=None):
    """Y = SiLU(X Wg^T) * (X Wu^T), bf16 [M, F], for the fused gate+up weight of 2F rows in the
    interleaved row order of ``interleave_gate_up``; dispatches like ``gemm_w4a16``."""
    return _linear("wq_gemm_w4a16_swiglu", fmt, X, Wq, scales, zeros, out, workspace, stream, swiglu=True)


def gemv_w4a16_swiglu(fmt, X, Wq, scales, zeros=None, out=None, workspace=None, stream=None):
    """The decode kernel alone with the SwiGLU epilogue (M <= 64)."""
    return _linear("wq_gemv_w4a16_swiglu", fmt, X, Wq, scales, zeros, out, workspace, stream, swiglu=True)


def gemm_tc_w4a16_swiglu(fmt, X, Wq, scales, zeros=None, out=None, workspace=None, stream=None):
    """The tensor-core kernel alone with the SwiGLU epilogue (any M)."""
    return _linear("wq_gemm_tc_w4a16_swiglu", fmt, X, Wq, scales, zeros, out, workspace, stream, swiglu=True)


def interleave_gate_up(src: torch.Tensor, out=None, stream=None):
    """Rows of the stacked [gate; up] tensor ``src`` (2F rows, any dtype, contiguous) in the
    order the SwiGLU entry points read: blocks of 8 gate rows and the matching 8 up rows."""
    if not src.is_cuda or not src.is_contiguous() or src.dim() < 1:
        raise ValueError("src must be a contiguous CUDA tensor")
    F = src.shape[0] // 2
    if src.shape[0] != 2 * F:
        raise ValueError("src needs an even number of rows")
    if out is None:
        out = torch.empty_like(src)
    elif out.shape != src.shape or out.dtype != src.dtype or not out.is_contiguous():
        raise ValueError("out must be a contiguous tensor of src's shape and dtype")
    row_bytes = (src.numel() // max(src.shape[0], 1)) * src.element_size()
    _check(load_library().wq_interleave_gate_up(_ptr(src), _ptr(out), F, row_bytes, _stream(stream, src.device)),
           "wq_interleave_gate_up")
    return out


def gemv_w4a16_noalloc(fmt, X, Wq, scales, zeros=None, out=None, stream=None):
    """The decode kernel with the library's own fixed scratch: no workspace, no allocation
    inside the library (``out`` is allocated here with torch when it is not given).  Same
    argument checks as ``gemv_w4a16``."""
    f = fmt if fmt.__class__ is int else _FMT_NAMES[fmt]
    M, K, N, out = _prepare(f, X, Wq, scales, zeros, out, False)
    st = _fn("wq_gemv_w4a16_noalloc")(f, X.data_ptr(), M, K, N, Wq.data_ptr(), scales.data_ptr(),
                                       None if zeros is None else zeros.data_ptr(), out.data_ptr(),
                                       _stream(stream, X.device))
    if st:
        _check(st, "wq_gemv_w4a16_noalloc")
    return out


def gemm_w4a16_qkv(fmt, X, Wq, scales, zeros=None, Nq=None, Nkv=None, out=None, workspace=None, stream=None):
    """The fused QKV projection split in the epilogue: (Q [M, Nq], K [M, Nkv], V [M, Nkv]) from the
    stacked packed weight [W_Q; W_K; W_V] of Nq + 2 Nkv rows; dispatches like ``gemm_w4a16``.
    ``out`` may be a tuple of three preallocated bf16 tensors."""
    f = fmt if fmt.__class__ is int else _FMT_NAMES[fmt]
    M, K, N, d = _inputs(f, X, Wq, scales, zeros)
    if Nq is None or Nkv is None or Nq < 1 or Nkv < 1 or Nq + 2 * Nkv != N:
        raise ValueError("Nq, Nkv >= 1 with Nq + 2 Nkv == Wq.shape[0] required")
    dev = X.device
    if out is not None and len(out) != 3:
        raise ValueError("out must be three tensors (Q, K, V)")
    out = tuple(_output(None if out is None else out[i], M, n, d, "out " + nm)
                for i, (n, nm) in enumerate(((Nq, "Q"), (Nkv, "K"), (Nkv, "V"))))
    if workspace is not None and (workspace.get_device() != d or not workspace.is_contiguous()):
        raise ValueError("workspace must be a contiguous CUDA tensor on X's device")
    ws = workspace if workspace is not None else _workspace_for(dev, gemm_workspace_bytes(f, M, K, N), None)
    ws_bytes = 0 if ws is None else ws.numel() * ws.element_size()
    st = _fn("wq_gemm_w4a16_qkv")(f, X.data_ptr(), M, K, Nq, Nkv, Wq.data_ptr(), scales.data_ptr(),
                                   None if zeros is None else zeros.data_ptr(), out[0].data_ptr(), out[1].data_ptr(),
                                   out[2].data_ptr(), None if ws is None else ws.data_ptr(), ws_bytes,
                                   _stream(stream, dev))
    if st:
        _check(st, "wq_gemm_w4a16_qkv")
    return out


def dispatch_threshold(fmt, K: int, N: int) -> int:
    return int(load_library().wq_dispatch_threshold(_fmt(fmt), K, N))


def set_dispatch_threshold(fmt, K: int, N: int, T: int) -> None:
    _check(load_library().wq_set_dispatch_threshold(_fmt(fmt), K, N, T), "wq_set_dispatch_threshold")


def selftest_wait_timeout(limit_us: int = 10000, stream=None) -> int:
    """Runs the bounded-wait diagnostic; returns 1 when the wait ran out (the expected result)."""
    v = ctypes.c_uint32(0)
    _check(load_library().wq_selftest_wait_timeout(limit_us, ctypes.byref(v), _stream(stream)),
           "wq_selftest_wait_timeout")
    return int(v.value)


def read_error_flags() -> int:
    v = ctypes.c_uint32(0)
    _check(load_library().wq_read_error_flags(ctypes.byref(v)), "wq_read_error_flags")
    return int(v.value)


# ------------------------------------------------------------------ FP8 E4M3 W8A8
def quantize_fp8_weights(W: torch.Tensor, stream=None):
    """W float32 [N, K] (CUDA) -> (Wq uint8 [N, K] E4M3 codes, s_w float32 [N]), one scale per
    output channel."""
    _need(W, torch.float32, "W")
    if W.dim() != 2:
        raise ValueError("W must be [N, K]")
    N, K = W.shape
    Wq = torch.empty((N, K), dtype=torch.uint8, device=W.device)
    sw = torch.empty((N,), dtype=torch.float32, device=W.device)
    _check(load_library().wq_quantize_fp8_weights(_ptr(W), N, K, _ptr(Wq), _ptr(sw), _stream(stream, W.device)),
           "wq_quantize_fp8_weights")
    return Wq, sw


def quantize_fp8_activations(X: torch.Tensor, stream=None):
    """X bf16 [M, K] (CUDA) -> (Xq uint8 [M, K] E4M3 codes, s_x float32 [M]), one scale per token."""
    _need(X, _BF16, "X")
    if X.dim() != 2:
        raise ValueError("X must be [M, K]")
    M, K = X.shape
    Xq = torch.empty((M, K), dtype=torch.uint8, device=X.device)
    sx = torch.empty((M,), dtype=torch.float32, device=X.device)
    _check(load_library().wq_quantize_fp8_activations(_ptr(X), M, K, _ptr(Xq), _ptr(sx), _stream(stream, X.device)),
           "wq_quantize_fp8_activations")
    return Xq, sx


def _fp8_operands(Wq, sw, K, dev):
    _need(Wq, torch.uint8, "Wq")
    _need(sw, torch.float32, "s_w")
    if Wq.dim() != 2 or Wq.shape[1] != K or Wq.device != dev:
        raise ValueError("Wq must be [N, K] on the activations' device")
    if sw.shape != (Wq.shape[0],) or sw.device != dev:
        raise ValueError("s_w must be [N] on the activations' device")
    return Wq.shape[0]


def gemm_fp8(Xq, sx, Wq, sw, out=None, stream=None):
    """Y bf16 [M, N] = s_x s_w^T * (E4M3(Xq) E4M3(Wq)^T) on the tensor cores."""
    _need(Xq, torch.uint8, "Xq")
    _need(sx, torch.float32, "s_x")
    M, K = Xq.shape
    if sx.shape != (M,) or sx.device != Xq.device:
        raise ValueError("s_x must be [M] on Xq's device")
    N = _fp8_operands(Wq, sw, K, Xq.device)
    Y = _output(out, M, N, Xq.get_device(), "out")
    _check(load_library().wq_gemm_fp8(_ptr(Xq), _ptr(sx), M, K, N, _ptr(Wq), _ptr(sw), _ptr(Y), _stream(stream, Xq.device)),
           "wq_gemm_fp8")
    return Y


def gemm_w8a8_fp8(X, Wq, sw, out=None, workspace=None, stream=None):
    """The W8A8 FP8 layer from bf16 activations: per-token quantization of X, then the GEMM."""
    _need(X, _BF16, "X")
    M, K = X.shape
    N = _fp8_operands(Wq, sw, K, X.device)
    Y = _output(out, M, N, X.get_device(), "out")
    lib = load_library()
    need = lib.wq_gemm_w8a8_fp8_workspace_bytes(M, K)
    ws = workspace if workspace is not None else Workspace(X.device).get(need)
    _check(lib.wq_gemm_w8a8_fp8(_ptr(X), M, K, N, _ptr(Wq), _ptr(sw), _ptr(Y), _ptr(ws), ws.numel(),
                                _stream(stream, X.device)), "wq_gemm_w8a8_fp8")
    return Y


# ------------------------------------------------------------------ W4A4 MXFP4 (FP8 tensor-core path)
def mxfp4_weights_to_e4m3(Wq: torch.Tensor, scales: torch.Tensor, stream=None):
    """MXFP4-packed weights (Wq int32 [N, K/8], E8M0 scales uint8 [N, K/32]) -> (Wq8 uint8 [N, K]
    E4M3 codes, s_w float32 [N] powers of two): E4M3(Wq8) * s_w equals the dequantized MXFP4
    weight exactly for every block within 14 binades of its row's largest."""
    _need(Wq, _I32, "Wq")
    _need(scales, _U8, "scales")
    N, K8 = Wq.shape
    K = 8 * K8
    if scales.shape != (N, K // 32) or scales.device != Wq.device:
        raise ValueError("scales must be [N, K/32] on Wq's device")
    W8 = torch.empty((N, K), dtype=torch.uint8, device=Wq.device)
    sw = torch.empty((N,), dtype=torch.float32, device=Wq.device)
    _check(load_library().wq_mxfp4_weights_to_e4m3(_ptr(Wq), _ptr(scales), N, K, _ptr(W8), _ptr(sw),
                                                    _stream(stream, Wq.device)), "wq_mxfp4_weights_to_e4m3")
    return W8, sw


def quantize_w4a4_activations(X: torch.Tensor, stream=None):
    """bf16 X [M, K] -> MXFP4 per token (the weights' rules), re-encoded: (Xq8 uint8 [M, K] E4M3,
    s_x float32 [M] powers of two)."""
    _need(X, _BF16, "X")
    M, K = X.shape
    Xq = torch.empty((M, K), dtype=torch.uint8, device=X.device)
    sx = torch.empty((M,), dtype=torch.float32, device=X.device)
    _check(load_library().wq_quantize_w4a4_activations(_ptr(X), M, K, _ptr(Xq), _ptr(sx), _stream(stream, X.device)),
           "wq_quantize_w4a4_activations")
    return Xq, sx


def gemm_w4a4_mxfp4(X, Wq8, sw, out=None, workspace=None, stream=None):
    """The W4A4 MXFP4 layer from bf16 activations (weights from ``mxfp4_weights_to_e4m3``)."""
    _need(X, _BF16, "X")
    M, K = X.shape
    N = _fp8_operands(Wq8, sw, K, X.device)
    Y = _output(out, M, N, X.get_device(), "out")
    lib = load_library()
    need = lib.wq_gemm_w8a8_fp8_workspace_bytes(M, K)
    ws = workspace if workspace is not None else Workspace(X.device).get(need)
    _check(lib.wq_gemm_w4a4_mxfp4(_ptr(X), M, K, N, _ptr(Wq8), _ptr(sw), _ptr(Y), _ptr(ws), ws.numel(),
                                  _stream(stream, X.device)), "wq_gemm_w4a4_mxfp4")
    return Y
