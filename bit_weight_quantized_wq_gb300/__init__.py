"""GB300-native weight-only 4-bit quantized linear layer (W4A16).

The compute path is the C-ABI library ``libwq.so`` (hand-written sm_103a CUDA
kernels) built from ``csrc/``; ``binding`` is its thin ctypes wrapper.  The
binding is imported lazily so that ``inputs`` can be used without a GPU.
"""
import importlib

__all__ = ["binding", "inputs"]


def __getattr__(name):
    if name in ("binding", "inputs", "build"):
        return importlib.import_module(__name__ + "." + name)
    raise AttributeError(name)
