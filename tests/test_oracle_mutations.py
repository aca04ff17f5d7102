"""Mutation check of the oracle's pins (CPU).

Each case plants one plausible mistake in an oracle function -- a dropped term, a wrong sign
or index, a transposed operand, a missing rounding or special-case rule -- by replacing that
function (or constant) in its module, and requires that at least one pin of
``tests/test_oracle_pins.py`` then fails.  A pin set that let a planted mistake through would
not pin the oracle.  The control case (no mistake) requires every pin to pass.
"""
import inspect

import numpy as np
import pytest

from oracle import awq, fp8, gptq, int4_g128, linear, mxfp4, swiglu, w4a4
from tests import test_oracle_pins as pins

PINS = [f for n, f in inspect.getmembers(pins, inspect.isfunction)
        if n.startswith("test_") and not inspect.signature(f).parameters]


def _failing_pins():
    failed = []
    with np.errstate(all="ignore"):
        for f in PINS:
            try:
                f()
            except Exception:   # an assertion, or an error a mutated function provokes
                failed.append(f.__name__)
    return failed


# ------------------------------------------------------------------ planted mistakes
def _group_params(zero_in_range=True, z_sign=1.0, zero_rule=True, clamp_z=True):
    def gp(x):
        x = np.asarray(x, dtype=np.float32)
        lo, hi = x.min(axis=-1), x.max(axis=-1)
        if zero_in_range:
            lo, hi = np.minimum(lo, np.float32(0)), np.maximum(hi, np.float32(0))
        s32 = np.minimum((hi - lo) / np.float32(15), np.float32(int4_g128.FP16_MAX))
        s16 = np.asarray(s32.astype(np.float16))
        if zero_rule:
            s16[s16 == 0] = np.float16(1)
        s = s16.astype(np.float32)
        z = np.rint(np.float32(z_sign) * (-lo) / s)
        if clamp_z:
            z = np.minimum(z, np.float32(15))
        return s16, z.astype(np.int32)
    return gp


def _codes_floor(x, s16, z):
    s = np.asarray(s16).astype(np.float32)[..., None]
    zf = np.asarray(z).astype(np.float32)[..., None]
    return np.clip(np.floor(np.asarray(x, dtype=np.float32) / s) + zf, 0, 15).astype(np.uint32)


def _pack_int4_reversed(q):
    q = np.asarray(q).astype(np.uint32)
    N, K = q.shape
    q8 = q.reshape(N, K // 8, 8)
    word = np.zeros((N, K // 8), dtype=np.uint32)
    for i in range(8):
        word |= (q8[:, :, i] & np.uint32(0xF)) << np.uint32(4 * (7 - i))
    return word.view(np.int32)


def _unpack_int4_reversed(Wq):
    w = np.ascontiguousarray(Wq).view(np.uint32)
    N, KW = w.shape
    out = np.empty((N, KW, 8), dtype=np.uint8)
    for i in range(8):
        out[:, :, i] = (w >> np.uint32(4 * (7 - i))) & np.uint32(0xF)
    return out.reshape(N, KW * 8)


def _dequant_plus_z(Wq, scales, zeros):
    q = int4_g128.unpack(Wq).astype(np.float64)
    N, K = q.shape
    s = np.asarray(scales, dtype=np.float64)
    z = np.asarray(zeros, dtype=np.float64)
    return ((q.reshape(N, K // 128, 128) + z[..., None]) * s[..., None]).reshape(N, K)


def _e8m0_no_exact_power(r):
    r = np.asarray(r, dtype=np.float64)
    m, ex = np.frexp(r)
    e = np.where(r == 0.0, -127, ex).astype(np.int64)   # ceil wrong on exact powers of two
    return np.clip(e, -127, 127)


def _e2m1_ties_down(a):
    a = np.asarray(a, dtype=np.float64)
    return np.argmin(np.abs(a[..., None] - mxfp4.E2M1_GRID), axis=-1).astype(np.uint8)


def _mx_pack_swapped(codes):
    c = np.asarray(codes, dtype=np.uint8)
    N, K = c.shape
    b = ((c[:, 0::2] & 0xF) << 4) | (c[:, 1::2] & 0xF)
    return np.ascontiguousarray(b.astype(np.uint8)).view(np.int32).reshape(N, K // 8)


def _mx_unpack_swapped(Wq):
    b = np.ascontiguousarray(Wq).view(np.uint8)
    N, KB = b.shape
    out = np.empty((N, KB, 2), dtype=np.uint8)
    out[:, :, 0] = b >> 4
    out[:, :, 1] = b & 0xF
    return out.reshape(N, KB * 2)


def _mx_quantize(keep_sign=True, zero_block_byte=True):
    real = mxfp4.quantize

    def q(W):
        Wq, sc = real(W)
        W = np.ascontiguousarray(W, dtype=np.float32)
        N, K = W.shape
        if not keep_sign:
            c = mxfp4.unpack(Wq)
            c = np.where((c & 7) == 0, 0, c).astype(np.uint8)   # -0 written as +0
            Wq = mxfp4.pack(c)
        if not zero_block_byte:
            amax = np.abs(W.reshape(N, K // 32, 32)).max(axis=-1)
            sc = np.where(amax == 0, np.uint8(127), sc).astype(np.uint8)   # e = 0, not the E8M0 minimum
        return Wq, sc
    return q


def _linear_k_shifted(X, W_hat):
    X = np.asarray(X, dtype=np.float64)
    W_hat = np.asarray(W_hat, dtype=np.float64)
    if X.shape[1] != W_hat.shape[1]:
        raise ValueError("inner dimensions differ")
    return X @ np.roll(W_hat, 1, axis=1).T          # X[m, k] paired with W[n, k - 1]


def _linear_rows_swapped(X, W_hat):
    X = np.asarray(X, dtype=np.float64)
    W_hat = np.asarray(W_hat, dtype=np.float64)
    return X @ W_hat[::-1].T                           # output column n from weight row N-1-n


def _dequant_no_scale(Wq, scales, zeros):
    q = int4_g128.unpack(Wq).astype(np.float64)
    N, K = q.shape
    z = np.asarray(zeros, dtype=np.float64)
    return (q.reshape(N, K // 128, 128) - z[..., None]).reshape(N, K)


def _silu_no_sigmoid(x):
    return np.asarray(x, dtype=np.float64)


def _swiglu_swapped(gate, up):
    return swiglu.silu(up) * np.asarray(gate, dtype=np.float64)


def _interleave_halves_swapped(F):
    if F < 0 or F % 8:
        raise ValueError("F must be a non-negative multiple of 8")
    src = np.empty(2 * F, dtype=np.int64)
    for r in range(2 * F):
        q, h, i = r // 16, (r // 8) % 2, r % 8
        src[r] = (1 - h) * F + 8 * q + i          # up rows where the gate rows belong
    return src


def _hessian_no_factor_two(X, damp=gptq.DAMP):
    X = np.asarray(X, dtype=np.float64)
    H = X.T @ X
    return H + damp * float(np.mean(np.diag(H))) * np.eye(H.shape[0])


def _awq_scales_inverted(imp, mask, a):
    alpha = a / float(awq.GRID)
    s = np.ones(imp.shape[0], dtype=np.float64)
    sel = mask & (imp > 0)
    s[sel] = imp[sel] ** (-alpha)
    return s.astype(np.float32)


def _awq_loss_multiplied(W, X, s):
    Wq, sc, z = awq.quantize_scaled(W, s)
    W_hat = int4_g128.dequantize(Wq, sc, z) * np.asarray(s, dtype=np.float64)[None, :]
    E = np.asarray(X, dtype=np.float64) @ (W_hat - np.asarray(W, dtype=np.float64)).T
    return float(np.sum(E * E))


def _e4m3_round_variant(ties_even=True, saturate=True, keep_sign=True):
    mag = fp8.e4m3_values()[:127]

    def rnd(v):
        v = np.asarray(v, dtype=np.float32)
        a = np.abs(v).astype(np.float64)
        hi = np.clip(np.searchsorted(mag, a, side="left"), 1, 126)
        lo = hi - 1
        dl, dh = a - mag[lo], mag[hi] - a
        code = np.where(dl < dh, lo, hi)
        if ties_even:
            code = np.where(dl == dh, np.where(lo % 2 == 0, lo, hi), code)
        else:
            code = np.where(dl == dh, lo, code)
        code = np.where(a >= 448.0, 126 if saturate else 127, code)
        code = np.where(a == 0.0, 0, code)
        sign = (v.view(np.uint32) >> np.uint32(31)).astype(np.uint8)
        if not keep_sign:
            sign = np.where(code == 0, 0, sign).astype(np.uint8)
        return ((sign << np.uint8(7)) | code.astype(np.uint8)).astype(np.uint8)
    return rnd


def _fp8_quantize_rows(fmax=448.0, zero_rule=True):
    def q(A):
        A = np.ascontiguousarray(A, dtype=np.float32)
        amax = np.abs(A).max(axis=1)
        s = (amax / np.float32(fmax)).astype(np.float32)
        if zero_rule:
            s[s == 0] = np.float32(1)
        with np.errstate(all="ignore"):
            return fp8.e4m3_round(A / s[:, None]), s
    return q


def _fp8_linear_one_scale(Xq, s_x, Wq, s_w):
    v = fp8.e4m3_values()
    return (v[np.asarray(Xq)] @ v[np.asarray(Wq)].T) * np.asarray(s_x, dtype=np.float64)[:, None]


def _w4a4_activation_scales_dropped(Xq, xs, Wq, ws):
    return mxfp4.decode_e2m1(mxfp4.unpack(Xq)) @ mxfp4.dequantize(Wq, ws).T


MUTATIONS = {
    "int4: zero not in the range": (int4_g128, "group_params", _group_params(zero_in_range=False)),
    "int4: sign of the zero point": (int4_g128, "group_params", _group_params(z_sign=-1.0)),
    "int4: no zero-scale rule": (int4_g128, "group_params", _group_params(zero_rule=False)),
    "int4: zero point not clamped": (int4_g128, "group_params", _group_params(clamp_z=False)),
    "int4: no fp16 saturation": (int4_g128, "FP16_MAX", float("inf")),
    "int4: 16 levels": (int4_g128, "LEVELS", 16),
    "int4: floor instead of rint": (int4_g128, "codes", _codes_floor),
    "int4: nibble order reversed (pack)": (int4_g128, "pack", _pack_int4_reversed),
    "int4: nibble order reversed (unpack)": (int4_g128, "unpack", _unpack_int4_reversed),
    "int4: + z in dequant": (int4_g128, "dequantize", _dequant_plus_z),
    "int4: scale dropped in dequant": (int4_g128, "dequantize", _dequant_no_scale),
    "mxfp4: E8M0 off by one on powers of two": (mxfp4, "e8m0_exponents", _e8m0_no_exact_power),
    "mxfp4: ties to the lower code": (mxfp4, "e2m1_round_magnitude", _e2m1_ties_down),
    "mxfp4: nibbles swapped (pack)": (mxfp4, "pack", _mx_pack_swapped),
    "mxfp4: nibbles swapped (unpack)": (mxfp4, "unpack", _mx_unpack_swapped),
    "mxfp4: sign of -0 dropped": (mxfp4, "quantize", _mx_quantize(keep_sign=False)),
    "mxfp4: zero block scale byte": (mxfp4, "quantize", _mx_quantize(zero_block_byte=False)),
    "linear: k index off by one": (linear, "linear", _linear_k_shifted),
    "linear: weight rows reversed": (linear, "linear", _linear_rows_swapped),
    "swiglu: sigmoid dropped": (swiglu, "silu", _silu_no_sigmoid),
    "swiglu: gate and up swapped": (swiglu, "swiglu", _swiglu_swapped),
    "swiglu: interleave halves swapped": (swiglu, "interleave_index", _interleave_halves_swapped),
    "gptq: Hessian without the factor 2": (gptq, "hessian", _hessian_no_factor_two),
    "awq: exponent sign (activations scaled up)": (awq, "scales", _awq_scales_inverted),
    "awq: loss multiplies instead of dividing": (awq, "loss", _awq_loss_multiplied),
    "fp8: ties to the lower code": (fp8, "e4m3_round", _e4m3_round_variant(ties_even=False)),
    "fp8: no saturation (NaN code)": (fp8, "e4m3_round", _e4m3_round_variant(saturate=False)),
    "fp8: sign of -0 dropped": (fp8, "e4m3_round", _e4m3_round_variant(keep_sign=False)),
    "fp8: E4M3 maximum taken as 240": (fp8, "quantize_rows", _fp8_quantize_rows(fmax=240.0)),
    "fp8: no zero-row scale rule": (fp8, "quantize_rows", _fp8_quantize_rows(zero_rule=False)),
    "fp8: weight scale dropped in the layer": (fp8, "linear_w8a8", _fp8_linear_one_scale),
    "w4a4: activation block scales dropped": (w4a4, "linear_w4a4", _w4a4_activation_scales_dropped),
}


def test_control_every_pin_passes():
    assert _failing_pins() == []


@pytest.mark.parametrize("name", sorted(MUTATIONS))
def test_planted_mistake_fails_a_pin(name, monkeypatch):
    mod, attr, repl = MUTATIONS[name]
    monkeypatch.setattr(mod, attr, repl)
    assert _failing_pins(), "no pin caught: " + name
