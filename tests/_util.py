"""Helpers shared by the tests: device transfer and the tolerance check."""
import numpy as np

TOL = 1e-2  # max |y - ref| <= TOL * (1 + |ref|), elementwise (float64 oracle, same dequantized weights)


def to_dev(a, dev="cuda"):
    import torch
    return torch.from_numpy(np.ascontiguousarray(a)).to(dev)


def x_to_dev(xbits, dev="cuda"):
    import torch
    return torch.from_numpy(np.ascontiguousarray(xbits).view(np.int16)).to(dev).view(torch.bfloat16)


def y_to_host(Y):
    return Y.float().cpu().numpy().astype(np.float64)


def assert_close(y, ref, what="", extra=None):
    """|y - ref| <= TOL (1 + |ref|) (+ ``extra``, an elementwise allowance derived by the caller)."""
    y = np.asarray(y, np.float64)
    err = np.abs(y - ref)
    lim = TOL * (1 + np.abs(ref))
    if extra is not None:
        lim = lim + extra
    bad = ~(err <= lim)
    if bad.any():
        i = np.unravel_index(np.argmax(np.where(bad, err / lim, 0)), err.shape)
        raise AssertionError("%s: %d of %d outputs outside tolerance; worst at %s: y=%r ref=%r"
                             % (what, int(bad.sum()), bad.size, i, y[i], ref[i]))
    return float((err / lim).max()) if err.size else 0.0
