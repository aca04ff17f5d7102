"""GB300-native weight-only 4-bit quantized linear layer (W4A16).

The compute path is the C-ABI library ``libwq.so`` (hand-written sm_103a CUDA
kernels) built from ``csrc/``; ``binding`` is its thin ctypes wrapper.  The
binding is imported lazily so that ``inputs`` can be used without a GPU.
"""
__all__ = ["binding", "inputs"]


def __getattr__(name):
    if name == "binding":
        from . import binding
        return binding
    raise AttributeError(name)
