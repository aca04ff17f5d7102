"""Pins of the CPU oracle against what the pages and the mathematics fix (CPU only).

Every oracle function is checked against something other than itself: the
pages' worked example and asserts (tests/golden/), hand-derived closed forms,
brute force on tiny inputs, exact rational arithmetic, invariants and special
cases.  A plausible mistake (dropped term, wrong sign, wrong rounding, wrong
nibble order, transposed operand) fails at least one of these.
"""
import json
import math
import os
from fractions import Fraction

import numpy as np
import pytest

from oracle import awq, gptq, int4_g128, linear, mxfp4, swiglu, uniform
from bit_weight_quantized_wq_gb300 import inputs

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _golden(name):
    with open(os.path.join(GOLDEN, name)) as f:
        return json.load(f)


# ---------------------------------------------------------------------------
# Symmetric routine: the lesson's worked example and asserts
# ---------------------------------------------------------------------------

def test_lesson6_worked_example():
    g = _golden("lesson6_blockwise_symmetric.json")["worked_example"]
    restored, scales = uniform.blockwise_symmetric_fake_quant(g["values"], g["block_size"], g["qmax"])
    assert scales == [g["scale_num"] / g["scale_den"]]
    s = scales[0]
    codes = [round(r / s) for r in restored]
    assert codes == g["codes"]
    assert [round(r, 3) for r in restored] == g["restored_printed_3dp"]
    assert restored[-1] == 8.0  # the block maximum is restored exactly


def test_lesson6_asserts():
    g = _golden("lesson6_blockwise_symmetric.json")
    a = g["asserts"][0]
    restored, scales = uniform.blockwise_symmetric_fake_quant(a["values"], a["block_size"], a["qmax"])
    assert scales == [n / d for n, d in a["scales_exact"]]
    assert abs(restored[1] - a["restored_index_1"]) < a["abs_tol"]
    assert abs(restored[-1] - a["restored_index_last"]) < a["abs_tol"]
    b = g["asserts"][1]
    assert uniform.blockwise_symmetric_fake_quant(b["values"], b["block_size"], b["qmax"]) == (
        b["restored_exact"], b["scales_exact_float"])
    for bad in g["invalid_geometry"]:
        with pytest.raises(ValueError):
            uniform.blockwise_symmetric_fake_quant([1.0], bad["block_size"], bad["qmax"])


def test_lesson6_finer_blocks_do_not_increase_error():
    # 第 6 课 "检查方法": compare error and scale count for block size 2 vs 4.
    vals = [0.0, 1.0, -2.0, 8.0]
    r2, s2 = uniform.blockwise_symmetric_fake_quant(vals, 2, 7)
    r4, s4 = uniform.blockwise_symmetric_fake_quant(vals, 4, 7)
    e2 = sum(abs(a - b) for a, b in zip(vals, r2))
    e4 = sum(abs(a - b) for a, b in zip(vals, r4))
    assert len(s2) == 2 and len(s4) == 1
    # by hand: size 2 -> blocks [0,1] (exact) and [-2,8] (s=8/7, |-2+16/7| = 2/7);
    # size 4 -> s = 8/7 for all: errors 1/7 (x=1) and 2/7 (x=-2)
    assert abs(e2 - 2 / 7) < 1e-12 and abs(e4 - 3 / 7) < 1e-12


def test_symmetric_int8_scale_and_ties():
    # scale = max|x| / 127 (推理优化与量化算子深度技术调研 §1.2); max 127 -> scale 1, so
    # the codes are the values rounded half to even: 0.5 -> 0, 1.5 -> 2.
    codes, scale = uniform.symmetric_quantize(np.array([-127.0, 0.5, 1.5, 2.5], np.float32), 8)
    assert scale == 1.0
    assert codes.tolist() == [-127, 0, 2, 2]
    codes, scale = uniform.symmetric_quantize(np.array([0.0, 0.0], np.float32), 8)
    assert scale == 1.0 and codes.tolist() == [0, 0]


# ---------------------------------------------------------------------------
# Asymmetric INT4 g128
# ---------------------------------------------------------------------------

def test_int4_linspace_closed_form():
    g = _golden("hand_derived_int4.json")["linspace_group"]
    x = np.linspace(-1, 2, 128, dtype=np.float32)[None, :]
    Wq, s, z = int4_g128.quantize(x)
    assert s.view(np.uint16)[0, 0] == int(g["scale_fp16_hex"], 16)
    assert float(s[0, 0]) == g["scale"]
    assert float(z[0, 0]) == g["zero"]
    q = int4_g128.unpack(Wq)[0]
    assert q[0] == g["code_first"] and q[-1] == g["code_last"]


def test_int4_constant_positive_group_includes_zero_in_range():
    g = _golden("hand_derived_int4.json")["constant_positive_group"]
    x = np.full((1, 128), 0.3, np.float32)
    Wq, s, z = int4_g128.quantize(x)
    assert s.view(np.uint16)[0, 0] == int(g["scale_fp16_hex"], 16)
    assert float(z[0, 0]) == g["zero"]
    assert (int4_g128.unpack(Wq) == g["code"]).all()


def test_int4_scale_saturates_at_fp16_max():
    # Reading R16: a group range above 15 * 65504 stores the largest finite fp16 scale
    # (not +inf), and the zero point stays a code; the dequantized group stays finite and
    # 0 stays exact.
    g = _golden("hand_derived_int4.json")["saturated_scale"]
    x = np.zeros((1, 128), np.float32)
    x[0, 0] = -2e6
    Wq, s, z = int4_g128.quantize(x)
    assert s.view(np.uint16)[0, 0] == int(g["scale_fp16_hex"], 16)
    assert float(z[0, 0]) == g["zero"]
    q = int4_g128.unpack(Wq)[0]
    assert q[0] == g["code_min"] and (q[1:] == g["code_zero"]).all()
    deq = int4_g128.dequantize(Wq, s, z)[0]
    assert deq[0] == g["deq_min"] and (deq[1:] == 0).all()
    # just inside the fp16 range the rounding itself gives 65504: saturation changes nothing
    g2 = _golden("hand_derived_int4.json")["scale_rounds_to_fp16_max"]
    x[0, 0] = -982650.0
    _, s, z = int4_g128.quantize(x)
    assert s.view(np.uint16)[0, 0] == int(g2["scale_fp16_hex"], 16) and float(z[0, 0]) == g2["zero"]
    # huge ranges (the 1e30 rows of the adversarial tests) give no overflow and finite values
    with np.errstate(over="raise", invalid="raise"):
        big = np.array([[-1e30, 3e38] + [0.0] * 126], np.float32)
        Wq, s, z = int4_g128.quantize(big)
        assert np.isfinite(int4_g128.dequantize(Wq, s, z)).all()
    assert s.view(np.uint16)[0, 0] == 0x7BFF and 0 <= float(z[0, 0]) <= 15


def test_int4_zero_point_clamped_to_code_range():
    # Reading R16: an fp16-subnormal scale can sit far below s32; the zero point is then
    # clamped to 15 so that 0.0 still dequantizes to exactly 0.
    g = _golden("hand_derived_int4.json")["subnormal_scale_zero_clamp"]
    x = np.zeros((1, 128), np.float32)
    x[0, 0] = np.float32(21 * 2.0 ** -24)
    x[0, 0] = -x[0, 0]
    Wq, s, z = int4_g128.quantize(x)
    assert s.view(np.uint16)[0, 0] == int(g["scale_fp16_hex"], 16)
    assert float(z[0, 0]) == g["zero"]
    q = int4_g128.unpack(Wq)[0]
    assert q[0] == g["code_min"] and (q[1:] == g["code_zero"]).all()
    assert (int4_g128.dequantize(Wq, s, z)[0, 1:] == 0).all()


def test_int4_packing_order():
    g = _golden("hand_derived_int4.json")["packing"]
    q = np.array([g["codes"]], dtype=np.uint32)
    w = int4_g128.pack(q)
    assert int(w.view(np.uint32)[0, 0]) == int(g["word_hex"], 16)
    assert int4_g128.unpack(w).tolist() == [g["codes"]]


def test_int4_zero_group_and_negative_zero():
    x = np.zeros((2, 256), np.float32)
    x[1, :128] = -0.0
    Wq, s, z = int4_g128.quantize(x)
    assert (s == 1).all() and (z == 0).all() and (z.view(np.uint16) == 0).all()
    assert (int4_g128.unpack(Wq) == 0).all()


def _special_groups(rng):
    """Adversarial groups: constant, all positive, all negative, one outlier, ties, tiny, +-0."""
    g = []
    g.append(np.full(128, 0.37, np.float32))
    g.append(np.abs(rng.standard_normal(128).astype(np.float32)))
    g.append(-np.abs(rng.standard_normal(128).astype(np.float32)))
    o = (rng.standard_normal(128) * 0.02).astype(np.float32); o[17] = 3.0; g.append(o)
    t = (np.arange(128, dtype=np.float32) - 40) * np.float32(0.25); g.append(t)  # many exact ties
    g.append((rng.standard_normal(128) * 1e-7).astype(np.float32))                  # fp16-subnormal scale
    g.append((rng.standard_normal(128) * 1e-9).astype(np.float32))                  # scale underflows -> 1
    z = np.zeros(128, np.float32); z[::2] = -0.0; z[5] = 1e-3; g.append(z)
    return np.stack(g)


def test_int4_matches_per_group_generic_routine():
    # The vectorised quantizer equals the plain per-group asymmetric routine with
    # b = 4 and fp16 scale storage, run group by group (brute force on small inputs).
    rng = np.random.default_rng(5)
    W = np.concatenate([_special_groups(rng).reshape(-1, 256),
                        (rng.standard_normal((3, 256)) * 0.05).astype(np.float32)])
    Wq, s, z = int4_g128.quantize(W)
    q = int4_g128.unpack(Wq)
    for n in range(W.shape[0]):
        for gi in range(W.shape[1] // 128):
            qq, ss, zz = uniform.asymmetric_quantize(W[n, 128 * gi:128 * gi + 128], 4, np.float16)
            assert ss == np.float32(s[n, gi]) and zz == np.float32(z[n, gi])
            assert (qq == q[n, 128 * gi:128 * gi + 128]).all()


def test_int4_code_is_nearest_grid_point():
    # Brute force: each code's dequantized value is the nearest of the 16 grid
    # points (j - z)*s, j = 0..15 (clamping included).
    rng = np.random.default_rng(7)
    W = np.concatenate([_special_groups(rng)[:6].reshape(-1, 128),
                        inputs.weights(11, 8, 256, 0.02).reshape(-1, 128)])
    Wq, s, z = int4_g128.quantize(W)
    q = int4_g128.unpack(Wq).astype(np.int64)
    for n in range(W.shape[0]):
        sv, zv = float(s[n, 0]), float(z[n, 0])
        grid = (np.arange(16) - zv) * sv
        for k in range(128):
            x = float(W[n, k])
            d = np.abs(grid - x)
            assert d[q[n, k]] == d.min(), (n, k, x, q[n, k])


def test_int4_error_bound_and_codes_in_range():
    # 第 1 章 §4.1: step Δ = s, so inside the grid's range |x - x_hat| <= s/2.
    W = inputs.weights(3, 64, 1024, 0.02)
    Wq, s, z = int4_g128.quantize(W)
    q = int4_g128.unpack(Wq)
    assert q.max() <= 15 and (z >= 0).all() and (z <= 15).all()
    W_hat = int4_g128.dequantize(Wq, s, z)
    sg = np.repeat(s.astype(np.float64), 128, axis=1)
    zg = np.repeat(z.astype(np.float64), 128, axis=1)
    lo, hi = -zg * sg, (15 - zg) * sg
    inside = (W >= lo) & (W <= hi)
    assert inside.mean() > 0.95   # group extremes may sit just outside when fp16 shrinks s
    err = np.abs(W.astype(np.float64) - W_hat)
    assert (err[inside] <= sg[inside] / 2 * (1 + 1e-12)).all()
    # outside the grid (fp16 rounding of s shrank it) the excess is at most 15*|s32 - s|
    x = W.reshape(64, 8, 128)
    s32 = (np.maximum(x.max(-1), 0) - np.minimum(x.min(-1), 0)) / np.float32(15)
    slack = np.repeat(np.abs(s32.astype(np.float64) - s.astype(np.float64)) * 16, 128, axis=1)
    assert (err <= sg / 2 + slack + 1e-12).all()


def test_int4_on_grid_weights_roundtrip_exactly():
    # Weights already on a grid (j - z)*s with j spanning 0..15 quantize without error.
    rng = np.random.default_rng(9)
    N, K = 4, 256
    W = np.empty((N, K), np.float32)
    for n in range(N):
        for gi in range(K // 128):
            sv = float(np.float16(rng.uniform(0.001, 0.1)))
            zv = int(rng.integers(0, 16))
            j = rng.integers(0, 16, 128); j[0], j[1] = 0, 15
            W[n, 128 * gi:128 * gi + 128] = (j - zv) * sv
    Wq, s, z = int4_g128.quantize(W)
    assert (int4_g128.dequantize(Wq, s, z) == W.astype(np.float64)).all()


def test_int4_group_size_sweep_error_monotone():
    # 第 6 课 "检查方法" analogue for the asymmetric routine: smaller groups, no larger error.
    W = inputs.weights(21, 32, 1024, 0.02)
    errs = []
    for gs in (32, 64, 128):
        e = 0.0
        for n in range(W.shape[0]):
            for g0 in range(0, W.shape[1], gs):
                x = W[n, g0:g0 + gs]
                q, s, z = uniform.asymmetric_quantize(x, 4, np.float16)
                e += float(np.sum((x - uniform.asymmetric_dequantize(q, s, z)) ** 2))
        errs.append(e)
    assert errs[0] <= errs[1] <= errs[2]


def test_asymmetric_int8_roundtrip():
    # b = 8 instance of the same formula (推理优化与量化算子深度技术调研 §1.2).
    x = np.array([-1.0, -0.5, 0.0, 0.25, 3.0], np.float32)
    q, s, z = uniform.asymmetric_quantize(x, 8)
    assert s == np.float32(np.float32(4.0) / np.float32(255))
    assert z == 64.0           # rint(1/s) = rint(63.75) = 64
    assert q[0] == 0 and q[-1] == 255 and q[2] == 64
    assert np.abs(x - uniform.asymmetric_dequantize(q, s, z)).max() <= s / 2 + 1e-9


# ---------------------------------------------------------------------------
# MXFP4
# ---------------------------------------------------------------------------

def test_e2m1_value_set_and_decode():
    g = _golden("mxfp4_e2m1_ties.json")
    vals = mxfp4.decode_e2m1(np.arange(16, dtype=np.uint8))
    assert vals[:8].tolist() == g["grid"]
    assert vals[8:].tolist() == [-v for v in g["grid"]]


def test_e2m1_ties_to_even_code():
    g = _golden("mxfp4_e2m1_ties.json")
    a = np.array([c[0] for c in g["cases"]])
    assert mxfp4.e2m1_round_magnitude(a).tolist() == [c[1] for c in g["cases"]]


def test_e8m0_exponent_exact():
    # amax / 2^e in (3, 6] for amax > 0 (exact rationals), boundary 6*2^j -> e = j.
    rng = np.random.default_rng(13)
    amax = np.concatenate([np.abs(rng.standard_normal(2000)).astype(np.float32) * np.float32(0.05),
                           np.float32(2.0) ** rng.integers(-60, 60, 500).astype(np.float32)])
    for a in amax:
        r = np.float32(a) / np.float32(6)
        e = mxfp4.e8m0_exponent(r)
        ratio = Fraction(float(a)) / (Fraction(2) ** e)
        assert Fraction(3) < ratio <= Fraction(6), (a, e)
    for j in range(-100, 100, 7):
        a = np.float32(6.0 * 2.0 ** j)
        assert mxfp4.e8m0_exponent(a / np.float32(6)) == j
        a_up = np.nextafter(a, np.float32(np.inf))
        assert mxfp4.e8m0_exponent(a_up / np.float32(6)) == j + 1
    assert (mxfp4.e8m0_exponents(np.array([0.0, 1.0, 1.5, 2.0 ** -140])) == [-127, 0, 1, -127]).all()


def test_mxfp4_packing_order():
    g = _golden("mxfp4_e2m1_ties.json")["packing"]
    c = np.array([g["codes"] + [0] * 6], dtype=np.uint8)
    w = mxfp4.pack(c)
    assert w.view(np.uint8)[0, 0] == int(g["byte_hex"], 16)
    assert mxfp4.unpack(w).tolist() == c.tolist()


def test_mxfp4_zero_block_and_signed_zero():
    W = np.zeros((1, 64), np.float32)
    W[0, 33] = 1.0
    W[0, 34] = -0.0
    W[0, 35] = -1e-30       # rounds to magnitude 0 but keeps its sign
    W[0, 0] = -0.0          # inside an all-zero block
    Wq, sc = mxfp4.quantize(W)
    codes = mxfp4.unpack(Wq)[0]
    assert sc[0, 0] == 0 and (codes[:32] == 0).all()
    assert codes[34] == 8 and codes[35] == 8 and codes[36] == 0
    assert sc[0, 1] == 127 - 2     # amax 1: r = 1/6, ceil(log2 r) = -2
    assert codes[33] == 6          # 1 * 2^2 = 4.0 -> magnitude code 6


def test_mxfp4_code_is_nearest_representable():
    # Brute force over the 16 signed values times 2^e: the chosen code is a nearest
    # one, and on a tie the magnitude code is even.
    W = inputs.weights(17, 4, 256, 0.02)
    Wq, sc = mxfp4.quantize(W)
    codes = mxfp4.unpack(Wq)
    cand = mxfp4.decode_e2m1(np.arange(16, dtype=np.uint8))
    for n in range(4):
        for k in range(256):
            f = 2.0 ** (int(sc[n, k // 32]) - 127)
            x = float(W[n, k])
            d = np.abs(cand * f - x)
            c = int(codes[n, k])
            assert d[c] == d.min()
            ties = np.flatnonzero(d == d.min())
            if len({int(t) & 7 for t in ties}) > 1:
                assert (c & 7) % 2 == 0


def test_mxfp4_error_bound_and_grid_roundtrip():
    W = inputs.weights(19, 16, 512, 0.02)
    Wq, sc = mxfp4.quantize(W)
    W_hat = mxfp4.dequantize(Wq, sc)
    f = np.repeat(np.exp2(sc.astype(np.float64) - 127), 32, axis=1)
    assert (np.abs(W - W_hat) <= f + 1e-300).all()        # half the widest spacing (2) times 2^e
    assert (np.abs(W_hat) <= 6 * f).all()
    # on-grid blocks (grid value * 2^e, block max 6 * 2^e) round-trip exactly
    rng = np.random.default_rng(23)
    e = rng.integers(-20, 5, (3, 4))
    idx = rng.integers(0, 16, (3, 128))
    G = mxfp4.decode_e2m1(idx.astype(np.uint8)).reshape(3, 4, 32)
    G[:, :, 0] = 6.0
    Wg = (G * np.exp2(e)[..., None]).reshape(3, 128).astype(np.float32)
    Wq, sc = mxfp4.quantize(Wg)
    assert (sc.astype(np.int64) - 127 == e).all()
    assert (mxfp4.dequantize(Wq, sc) == Wg.astype(np.float64)).all()


# ---------------------------------------------------------------------------
# The linear layer
# ---------------------------------------------------------------------------

def test_linear_brute_force_fractions():
    rng = np.random.default_rng(29)
    for fmt in ("int4_g128", "mxfp4"):
        M, K, N = 3, 256, 5
        W = inputs.weights(31, N, K, 0.05)
        _, X = inputs.activations(37, M, K)
        if fmt == "int4_g128":
            Wq, s, z = int4_g128.quantize(W)
            W_hat = int4_g128.dequantize(Wq, s, z)
            Y = linear.linear_w4a16(fmt, X, Wq, s, z)
        else:
            Wq, s = mxfp4.quantize(W)
            W_hat = mxfp4.dequantize(Wq, s)
            Y = linear.linear_w4a16(fmt, X, Wq, s)
        assert Y.shape == (M, N)
        for m in range(M):
            for n in range(N):
                exact = sum(Fraction(float(X[m, k])) * Fraction(float(W_hat[n, k])) for k in range(K))
                assert abs(Fraction(float(Y[m, n])) - exact) <= Fraction(1, 10 ** 12) * (1 + abs(exact))


def test_qkv_split_definition():
    # 推理优化与量化算子深度技术调研 §4.2: Q, K, V are the column blocks of the fused projection,
    # W_Q rows first.  A hand-built weight whose rows are one-hot (row n selects input n) makes
    # the fused output the input itself, so each part is a known slice of X.
    X = np.arange(2 * 12, dtype=np.float64).reshape(2, 12)
    Y = linear.linear(X, np.eye(12)[[3, 1, 4, 1, 5, 9, 2, 6]])          # Nq = 4, Nkv = 2
    q, k, v = linear.qkv_split(Y, 4, 2)
    assert q.tolist() == X[:, [3, 1, 4, 1]].tolist()
    assert k.tolist() == X[:, [5, 9]].tolist() and v.tolist() == X[:, [2, 6]].tolist()
    with pytest.raises(ValueError):
        linear.qkv_split(Y, 4, 3)


def test_linear_special_cases():
    M, K, N = 4, 256, 6
    _, X = inputs.activations(41, M, K)
    Wq, s, z = int4_g128.quantize(np.zeros((N, K), np.float32))
    assert (linear.linear_w4a16("int4_g128", X, Wq, s, z) == 0).all()
    # on-grid weights: the quantized layer equals the unquantized product
    W = ((np.arange(N * K).reshape(N, K) % 16) - 3).astype(np.float32) * np.float32(0.125)
    Wq, s, z = int4_g128.quantize(W)
    assert (linear.linear_w4a16("int4_g128", X, Wq, s, z) == X.astype(np.float64) @ W.T.astype(np.float64)).all()
    rows = [5, 0, 3]
    full = linear.linear_w4a16("int4_g128", X, Wq, s, z)
    assert (linear.linear_rows("int4_g128", X, Wq, s, z, rows) == full[:, rows]).all()


@pytest.mark.parametrize("outliers,bar", [(0.0, 0.99), (0.01, 0.95)])
def test_linear_sanity_against_unquantized(outliers, bar):
    # 量化与加速 deployment checklist: no NaN/Inf, cosine similarity > 0.99 vs the fp32
    # layer.  With 1 % of input columns x10 (the salient channels of 推理优化与量化算子深度技术调研
    # §1.3), plain round-to-nearest loses more (about 0.98) -- the gap AWQ scaling closes.
    M, K, N = 4, 1024, 64
    W = inputs.weights(43, N, K, 0.02, outlier_frac=outliers)
    _, X = inputs.activations(43, M, K)
    ref = X.astype(np.float64) @ W.T.astype(np.float64)
    for fmt in ("int4_g128", "mxfp4"):
        if fmt == "int4_g128":
            Y = linear.linear_w4a16(fmt, X, *int4_g128.quantize(W))
        else:
            Y = linear.linear_w4a16(fmt, X, *mxfp4.quantize(W))
        assert np.isfinite(Y).all()
        cos = float((Y * ref).sum() / math.sqrt((Y * Y).sum() * (ref * ref).sum()))
        assert cos > bar, (fmt, cos)


# ---------------------------------------------------------------------------
# SwiGLU on the fused gate+up projection (推理优化与量化算子深度技术调研 §4.6)
# ---------------------------------------------------------------------------

def test_silu_closed_forms():
    # SiLU(x) = x sigmoid(x); sigmoid(1) = e / (1 + e), sigmoid(ln 3) = 3/4, sigmoid(0) = 1/2
    assert swiglu.silu(0.0) == 0.0
    assert abs(float(swiglu.silu(1.0)) - 0.7310585786300049) < 1e-15
    assert abs(float(swiglu.silu(-1.0)) + 0.2689414213699951) < 1e-15
    assert abs(float(swiglu.silu(math.log(3.0))) - 0.75 * math.log(3.0)) < 1e-15
    assert abs(float(swiglu.silu(-math.log(3.0))) + 0.25 * math.log(3.0)) < 1e-15
    # far tails: the identity above, zero below, no overflow
    assert float(swiglu.silu(1000.0)) == 1000.0
    assert abs(float(swiglu.silu(-1000.0))) < 1e-300
    # sigmoid(x) + sigmoid(-x) = 1  =>  SiLU(x) - SiLU(-x) = x
    x = np.linspace(-30, 30, 2001)
    assert np.allclose(swiglu.silu(x) - swiglu.silu(-x), x, rtol=0, atol=1e-13)
    # the global minimum: at x = -1 - W(1/e) = -1.27846454..., value -0.27846454...
    xs = np.linspace(-1.3, -1.25, 50001)
    v = swiglu.silu(xs)
    assert abs(xs[np.argmin(v)] + 1.2784645427610738) < 2e-6
    assert abs(v.min() + 0.2784645427610738) < 1e-10


def _one_hot_stacked_int4(F, K=128):
    """Hand-packed stacked [gate; up] INT4 weight, z = 8 everywhere: only the code at k = 0
    differs from the zero point (code k = 0 sits in bits 0..3 of word 0)."""
    Wq = np.full((2 * F, K // 8), 0x88888888, dtype=np.uint32)
    sc = np.zeros((2 * F, K // 128), dtype=np.float16)
    z = np.full((2 * F, K // 128), 8, dtype=np.float16)
    g_exp, u_exp = [], []
    for j in range(F):
        qg, qu = 4 + j % 8, 15 - j % 8              # gate (q - 8) * 0.5, up (q - 8) * 0.25
        Wq[j, 0] = 0x88888880 | qg
        Wq[F + j, 0] = 0x88888880 | qu
        sc[j, 0], sc[F + j, 0] = 0.5, 0.25
        g_exp.append((qg - 8) * 0.5)
        u_exp.append((qu - 8) * 0.25)
    return Wq.view(np.int32), sc, z, g_exp, u_exp


def test_swiglu_hand_packed_one_hot():
    # X = e_0: gate_j and up_j are the dequantized k = 0 weights of rows j and F + j.
    F, K = 16, 128
    Wq, sc, z, g_exp, u_exp = _one_hot_stacked_int4(F, K)
    X = np.zeros((1, K))
    X[0, 0] = 1.0
    Y = swiglu.swiglu_w4a16("int4_g128", X, Wq, sc, z)
    assert Y.shape == (1, F)
    for j in range(F):
        g, u = g_exp[j], u_exp[j]
        assert abs(Y[0, j] - g / (1.0 + math.exp(-g)) * u) < 1e-15, j
    # j = 5: g = 0.5, u = 0.5; gate/up swapped or the sigmoid dropped would differ
    assert abs(Y[0, 5] - 0.5 * 0.5 / (1.0 + math.exp(-0.5))) < 1e-15
    # g = 0 (j = 4) zeroes the output whatever up is; u = 0 (j = 7) too
    assert Y[0, 4] == 0.0 and Y[0, 7] == 0.0
    # row sampling agrees with the full product
    cols = np.array([3, 0, 15])
    assert (swiglu.swiglu_rows("int4_g128", X, Wq, sc, z, F, cols) == Y[:, cols]).all()


def test_interleave_order():
    # F = 8: one block of 8 gate rows then 8 up rows -- already the stacked order
    assert (swiglu.interleave_index(8) == np.arange(16)).all()
    # F = 16, written out
    assert swiglu.interleave_index(16).tolist() == (
        list(range(0, 8)) + list(range(16, 24)) + list(range(8, 16)) + list(range(24, 32)))
    for F in (8, 24, 128, 1000):
        src = swiglu.interleave_index(F)
        assert sorted(src.tolist()) == list(range(2 * F))          # a permutation
        r = np.arange(2 * F)
        gate = (r // 8) % 2 == 0
        # gate row r and row r + 8 hold gate_j and up_j of the same output j = 8 (r // 16) + r % 8
        assert (src[r[gate]] == 8 * (r[gate] // 16) + r[gate] % 8).all()
        assert (src[r[gate] + 8] == src[r[gate]] + F).all()
    with pytest.raises(ValueError):
        swiglu.interleave_index(12)


def test_interleave_commutes_with_rowwise_quantization():
    F, K = 24, 256
    W = inputs.weights(47, 2 * F, K, 0.03)
    for q in (int4_g128.quantize, mxfp4.quantize):
        a = [swiglu.interleave_gate_up(t, F) for t in q(W)]
        b = q(swiglu.interleave_gate_up(W, F))
        for x, y in zip(a, b):
            assert (np.asarray(x).view(np.uint8) == np.asarray(y).view(np.uint8)).all()


# ---------------------------------------------------------------------------
# GPTQ (第 1 章：推理加速全景 §4.2; 推理优化与量化算子深度技术调研 §1.3)
# ---------------------------------------------------------------------------

def test_gptq_hessian_closed_form():
    # X^T X = [[2, 1], [1, 5]] -> 2 X^T X = [[4, 2], [2, 10]], lambda = 0.01 * 7
    X = np.array([[1.0, 0.0], [0.0, 2.0], [1.0, 1.0]])
    H = gptq.hessian(X)
    assert np.allclose(H, [[4.07, 2.0], [2.0, 10.07]], rtol=0, atol=1e-12)


def test_gptq_inverse_cholesky_closed_form():
    # H = [[4, 2], [2, 3]]: H^-1 = [[3, -2], [-2, 4]] / 8 = U^T U with
    # U = [[sqrt(3/8), -(1/4)/sqrt(3/8)], [0, sqrt(1/3)]]
    U = gptq.inverse_cholesky_upper(np.array([[4.0, 2.0], [2.0, 3.0]]))
    u11 = math.sqrt(3.0 / 8.0)
    ref = np.array([[u11, -0.25 / u11], [0.0, math.sqrt(1.0 / 3.0)]])
    assert np.allclose(U, ref, rtol=0, atol=1e-14)
    # a larger case: upper triangular, positive diagonal, U^T U H = I
    X = inputs.calibration(5, 64, 48)
    H = gptq.hessian(X)
    U = gptq.inverse_cholesky_upper(H)
    assert np.allclose(np.tril(U, -1), 0) and (np.diag(U) > 0).all()
    assert np.allclose(U.T @ U @ H, np.eye(48), atol=1e-9)


def test_gptq_diagonal_hessian_is_round_to_nearest():
    # H diagonal -> U diagonal -> no compensation: the sweep is the plain INT4 g128 quantizer
    N, K = 24, 384
    W = inputs.weights(61, N, K, 0.05)
    d = np.random.default_rng(62).uniform(0.5, 2.0, K).astype(np.float32)
    got = gptq.sweep(W, np.diag(d))
    ref = int4_g128.quantize(W)
    for a, b in zip(got, ref):
        assert (np.asarray(a).view(np.uint8) == np.asarray(b).view(np.uint8)).all()


def _gptq_case(N=16, K=384, seed=63):
    W = inputs.weights(seed, N, K, 0.05)
    X = inputs.calibration(seed, 128, K)
    H = gptq.hessian(X)
    U64 = gptq.inverse_cholesky_upper(H)
    U = U64.astype(np.float32)
    Wq, s, z, e, seen = gptq.sweep(W, U, return_trace=True)
    W_hat = int4_g128.dequantize(Wq, s, z)
    return W, X, H, U64, U, (Wq, s, z), e, seen, W_hat


def test_gptq_error_is_e_times_u_and_the_loss_decomposes():
    # With w_j updated by -e_i U[i, j] for every i < j and w_hat_j = w_j(current) - e_j U[j, j]:
    # w - w_hat = e U exactly; with H^-1 = U^T U that gives (w - w_hat) H (w - w_hat)^T = |e|^2.
    W, X, H, U64, U, pk, e, seen, W_hat = _gptq_case()
    delta = W.astype(np.float64) - W_hat
    eU = e.astype(np.float64) @ U.astype(np.float64)
    assert np.abs(delta - eU).max() <= 1e-4 * np.abs(delta).max()
    Hf = np.linalg.inv(U.astype(np.float64).T @ U.astype(np.float64))
    loss = np.einsum("nk,kl,nl->n", delta, Hf, delta)
    assert np.allclose(loss, (e.astype(np.float64) ** 2).sum(axis=1), rtol=1e-3)


def test_gptq_group_parameters_come_from_compensated_values():
    W, X, H, U64, U, (Wq, s, z), e, seen, W_hat = _gptq_case()
    s_ref, z_ref = int4_g128.group_params(seen)
    assert (s_ref.view(np.uint16) == s.view(np.uint16)).all()
    assert (z_ref.astype(np.float16).view(np.uint16) == z.view(np.uint16)).all()
    # the first group starts from the original weights, later ones from compensated values
    assert (seen[:, 0, :] == W[:, :128]).all()
    assert not (seen[:, 1, :] == W[:, 128:256]).all()


def test_gptq_lowers_the_calibration_objective():
    # The point of the method: sum over rows of (w - w_hat) H (w - w_hat)^T falls below
    # round-to-nearest's on the calibration set.
    W, X, H, U64, U, pk, e, seen, W_hat = _gptq_case(N=32)
    rtn = int4_g128.dequantize(*int4_g128.quantize(W))
    obj = lambda Wh: float(np.einsum("nk,kl,nl->", W - Wh, H, W - Wh))
    assert obj(W_hat) < 0.8 * obj(rtn)


# ---------------------------------------------------------------------------
# AWQ (第 1 章：推理加速全景 §4.4; 推理优化与量化算子深度技术调研 §1.3; 量化与加速)
# ---------------------------------------------------------------------------

def test_awq_importance_and_salient_set():
    X = np.array([[1.0, -2.0, 0.5], [3.0, 0.0, -0.5]], dtype=np.float32)
    assert awq.importance(X).tolist() == [2.0, 1.0, 0.5]
    # ceil(K / 100) channels: 3 of 201; equal importances rank by channel index
    imp = np.ones(201)
    imp[[7, 50, 199]] = [4.0, 9.0, 4.0]
    assert np.flatnonzero(awq.salient(imp)).tolist() == [7, 50, 199]
    imp[199] = 1.0
    assert np.flatnonzero(awq.salient(imp)).tolist() == [0, 7, 50]
    assert awq.salient(np.arange(100.0)).sum() == 1


def test_awq_scales_closed_forms():
    imp = np.array([4.0, 9.0, 2.25, 1.0])
    mask = np.array([True, True, False, False])
    assert awq.scales(imp, mask, 0).tolist() == [1.0, 1.0, 1.0, 1.0]
    assert awq.scales(imp, mask, 20).tolist() == [4.0, 9.0, 1.0, 1.0]     # alpha = 1
    assert awq.scales(imp, mask, 10).tolist() == [2.0, 3.0, 1.0, 1.0]     # alpha = 1/2


def test_awq_alpha_zero_is_round_to_nearest():
    W = inputs.weights(83, 32, 512, 0.05)
    X = inputs.calibration(84, 64, 512)
    s = awq.scales(awq.importance(X), awq.salient(awq.importance(X)), 0)
    got = awq.quantize_scaled(W, s)
    ref = int4_g128.quantize(W)
    for a, b in zip(got, ref):
        assert (np.asarray(a).view(np.uint8) == np.asarray(b).view(np.uint8)).all()
    W_hat = int4_g128.dequantize(*ref)
    E = X.astype(np.float64) @ (W_hat - W.astype(np.float64)).T
    assert abs(awq.loss(W, X, s) - float((E * E).sum())) <= 1e-9 * float((E * E).sum())


def test_awq_loss_is_the_runtime_error_with_divided_activations():
    # Q(W s) applied to x / s, minus W x: the same number as the loss computed on W_hat = Q(W s) / s,
    # which pins the direction of the scaling (weights times s, activations divided by s).
    W = inputs.weights(85, 24, 384, 0.05)
    X = inputs.calibration(86, 32, 384)
    imp = awq.importance(X)
    s = awq.scales(imp, awq.salient(imp), 12)
    assert (s > 1).any()
    Qws = int4_g128.dequantize(*awq.quantize_scaled(W, s))
    Y_q = (X.astype(np.float64) / s.astype(np.float64)[None, :]) @ Qws.T
    Y = X.astype(np.float64) @ W.astype(np.float64).T
    ref = float(((Y_q - Y) ** 2).sum())
    assert abs(awq.loss(W, X, s) - ref) <= 1e-9 * ref


def test_awq_search_protects_salient_channels():
    # With 1 % of the activation channels ten times larger, scaling them lowers the output error
    # well below round-to-nearest's; alpha = 0 is in the grid, so the search never does worse.
    W = inputs.weights(87, 64, 1024, 0.05)
    X = inputs.calibration(88, 128, 1024)
    a, s, losses, pk = awq.search(W, X)
    assert losses[a] == losses.min() and 0 < a < awq.GRID
    assert losses[a] < 0.8 * losses[0]
    assert (np.asarray(pk[0]) == np.asarray(awq.quantize_scaled(W, s)[0])).all()


# ------------------------------------------------------------------ FP8 E4M3 W8A8 (oracle/fp8.py)
# 推理优化与量化算子深度技术调研 §1.4 (E4M3 weights and activations with FP32 scales beside the
# tensor) and 量化与加速's format table (E4M3: 4 exponent bits, 3 mantissa bits, +-448).

def _e4m3_by_bits(c):
    """E4M3 code -> value by moving its fields into a float32 bit pattern (an independent
    formulation of the format: normal values are 1.m x 2^(e-7), subnormals m/8 x 2^-6)."""
    import struct
    s, e, m = c >> 7, (c >> 3) & 0xF, c & 7
    if e == 15 and m == 7:
        return float("nan")
    if e == 0:
        v = m * 2.0 ** -9
    else:
        v = struct.unpack("<f", struct.pack("<I", ((e - 7 + 127) << 23) | (m << 20)))[0]
    return -v if s else v


def test_e4m3_value_set():
    from oracle import fp8
    v = fp8.e4m3_values()
    for c in range(256):
        b = _e4m3_by_bits(c)
        assert (np.isnan(b) and np.isnan(v[c])) or b == v[c], hex(c)
    # named points of the format: 1.0, 1.5, 2.0, the largest finite value 448 and the next
    # one down 416 / the value 240, the smallest normal 2^-6 and subnormal 2^-9
    assert (v[0x38], v[0x3C], v[0x40], v[0x7E], v[0x7D], v[0x77]) == (1.0, 1.5, 2.0, 448.0, 416.0, 240.0)
    assert (v[0x08], v[0x01], v[0x80]) == (2.0 ** -6, 2.0 ** -9, 0.0)
    assert np.isnan(v[0x7F]) and np.isnan(v[0xFF]) and int(np.isfinite(v).sum()) == 254
    assert np.nanmax(v) == fp8.E4M3_MAX == 448.0


def test_e4m3_rounding_ties_saturation_and_signed_zero():
    from oracle import fp8
    cases = [  # (value, code): hand-derived from the value grid
        (1.0625, 0x38),      # halfway 1 | 1.125 -> even code 0x38
        (1.1875, 0x3A),      # halfway 1.125 | 1.25 -> even code 0x3A
        (1.05, 0x38), (1.07, 0x39), (1.1, 0x39),
        (15.5, 0x58),        # halfway 15 (0x57) | 16 (0x58) -> 0x58
        (440.0, 0x7E), (420.0, 0x7D), (432.0, 0x7E),   # 432 halfway 416 | 448 -> even 0x7E
        (464.0, 0x7E), (1.0e6, 0x7E),                   # saturation at 448
        (2.0 ** -10, 0x00),  # halfway 0 | 2^-9 -> even code 0
        (3 * 2.0 ** -10, 0x02),   # halfway 2^-9 | 2^-8 -> even 0x02
        (2.0 ** -9, 0x01), (2.0 ** -6, 0x08), (0.0, 0x00),
        (-1.0, 0xB8), (-448.0, 0xFE), (-1.0e9, 0xFE),
    ]
    for x, c in cases:
        got = int(fp8.e4m3_round(np.float32(x)))
        assert got == c, "%r -> %#x, expected %#x" % (x, got, c)
    assert int(fp8.e4m3_round(np.float32(-0.0))) == 0x80                  # sign kept on zero
    assert int(fp8.e4m3_round(np.float32(-2.0 ** -11))) == 0x80            # rounds to -0


def test_e4m3_code_is_nearest_finite_value():
    from oracle import fp8
    rng = np.random.default_rng(811)
    x = np.concatenate([rng.standard_normal(4000) * 50, rng.standard_normal(2000) * 0.01,
                        rng.uniform(-470, 470, 2000)]).astype(np.float32)
    codes = fp8.e4m3_round(x)
    grid = np.array([_e4m3_by_bits(c) for c in range(256)])
    fin = np.isfinite(grid)
    for xi, ci in zip(x.astype(np.float64), codes):
        d = np.abs(grid[fin] - min(max(xi, -448.0), 448.0))
        assert abs(grid[ci] - min(max(xi, -448.0), 448.0)) == d.min()
        if np.sum(d == d.min()) > 1 and grid[ci] != 0.0:                  # a tie: the even code
            assert ci % 2 == 0


def test_fp8_row_scales_closed_forms():
    from oracle import fp8
    # a row whose largest magnitude is 448 * 2^-3 has the scale 2^-3 exactly; values on the
    # scaled grid come back exactly
    grid = np.array([_e4m3_by_bits(c) for c in range(0x7F)])
    W = (np.array([grid[[0x7E, 0x38, 0x3C, 0x01, 0x00, 0x55]], -grid[[0x40, 0x77, 0x08, 0x7D, 0x10, 0x20]]])
         * 2.0 ** -3).astype(np.float32)
    q, s = fp8.quantize_weights(W)
    assert s[0] == np.float32(2.0 ** -3)
    assert np.array_equal(fp8.dequantize_rows(q[:1], s[:1]), W[:1].astype(np.float64))
    assert int(q[0, 0]) == 0x7E                          # the row's maximum maps to 448
    # a zero row gets the scale 1 and the codes 0 (F3); -0.0 keeps its sign
    q, s = fp8.quantize_activations(np.array([[0.0, -0.0, 0.0, 0.0]], np.float32))
    assert s[0] == 1.0 and list(q[0]) == [0x00, 0x80, 0x00, 0x00]
    # the scale is amax / 448 rounded to float32, and x / s rounds per element
    x = np.array([[3.0, -1.0, 0.5, 0.0]], np.float32)
    q, s = fp8.quantize_activations(x)
    assert s[0] == np.float32(np.float32(3.0) / np.float32(448.0))
    assert int(q[0, 0]) == 0x7E and int(q[0, 1]) & 0x80


def test_fp8_error_bound():
    from oracle import fp8
    # inside the normal range the E4M3 spacing is 2^(e-3) on [2^e, 2^(e+1)): the error of a
    # value is at most half of that, i.e. relative 2^-4, plus the subnormal floor 2^-10 s
    rng = np.random.default_rng(813)
    X = (rng.standard_normal((6, 512)) * np.array([1e-3, 0.1, 1, 10, 1e3, 1e5])[:, None]).astype(np.float32)
    q, s = fp8.quantize_activations(X)
    err = np.abs(fp8.dequantize_rows(q, s) - X.astype(np.float64))
    bound = np.abs(X).astype(np.float64) * 2.0 ** -4 + s.astype(np.float64)[:, None] * 2.0 ** -10
    assert (err <= bound * (1 + 1e-6)).all()


def test_fp8_linear_brute_force_fractions():
    from oracle import fp8
    M, K, N = 3, 64, 4
    rng = np.random.default_rng(817)
    W = rng.standard_normal((N, K)).astype(np.float32) * 0.05
    _, X = inputs.activations(819, M, K)
    Wq, sw = fp8.quantize_weights(W)
    Xq, sx = fp8.quantize_activations(X)
    Y = fp8.linear_w8a8(Xq, sx, Wq, sw)
    for m in range(M):
        for n in range(N):
            exact = sum(Fraction(_e4m3_by_bits(int(Xq[m, k]))) * Fraction(_e4m3_by_bits(int(Wq[n, k])))
                        for k in range(K)) * Fraction(float(sx[m])) * Fraction(float(sw[n]))
            assert abs(Fraction(float(Y[m, n])) - exact) <= Fraction(1, 10 ** 12) * (1 + abs(exact))
    rows = np.array([2, 0])
    assert np.array_equal(fp8.linear_w8a8_rows(Xq, sx, Wq, sw, rows), Y[:, rows])


# ------------------------------------------------------------------ W4A4 MXFP4 (oracle/w4a4.py)

def test_w4a4_brute_force_fractions_and_grid_activations():
    from oracle import w4a4
    M, K, N = 2, 64, 3
    W = inputs.weights(821, N, K, 0.05)
    _, X = inputs.activations(823, M, K)
    Xq, xs = w4a4.quantize_activations(X)
    Wq, ws = mxfp4.quantize(W)
    Y = w4a4.linear_w4a4(Xq, xs, Wq, ws)
    # the layer is the exact sum of products of the two dequantized operands
    xv = mxfp4.dequantize(Xq, xs)
    wv = mxfp4.dequantize(Wq, ws)
    for m in range(M):
        for n in range(N):
            exact = sum(Fraction(float(xv[m, k])) * Fraction(float(wv[n, k])) for k in range(K))
            assert abs(Fraction(float(Y[m, n])) - exact) <= Fraction(1, 10 ** 12) * (1 + abs(exact))
    # activations already on the MXFP4 grid are quantized exactly, so the W4A4 layer then equals
    # the W4A16 MXFP4 layer on the same activations
    grid = np.array([0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0])
    rng = np.random.default_rng(827)
    Xg = (rng.choice(grid, (M, K)) * rng.choice([-1.0, 1.0], (M, K))).astype(np.float32)
    Xg[:, ::32] = 6.0                                   # every block's max: scale 2^0
    Xq, xs = w4a4.quantize_activations(Xg)
    assert np.array_equal(mxfp4.dequantize(Xq, xs), Xg.astype(np.float64))
    assert np.array_equal(w4a4.linear_w4a4(Xq, xs, Wq, ws), linear.linear_w4a16("mxfp4", Xg, Wq, ws))
    rows = np.array([2, 0])
    assert np.array_equal(w4a4.linear_w4a4_rows(Xq, xs, Wq, ws, rows), w4a4.linear_w4a4(Xq, xs, Wq, ws)[:, rows])
