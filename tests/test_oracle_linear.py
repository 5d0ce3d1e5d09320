"""Pins for the oracle's q8ta_linear / q8ta_linear_gemv (CPU only).

Source: "Add q8ta_linear op" (PR #21197), Solution paragraph -- a register
tiled i32 GEMM acc = sum_k (x[m,k] - input_zero_point) * w[n,k], dequantize
acc * input_scale * weight_scales[n] + bias, requantize
clamp(round(v * inv_output_scale) + output_zero_point, -128, 127); the M == 1
gemv has the identical schema.  Constraints paragraph: x / w are row-major
[M,K] / [N,K]; the zero-point fold sum (x - zp) w == sum x w - zp sum w.

Pins: exhaustive products for K == 1, float64 matmul (exact for these
magnitudes), the fold identity, int32 wrap-around computed with Python
integers, and the epilogue against exact rational arithmetic with a binary32
rounding after every step (which rejects a fused multiply-add, a different
association of the three-factor product, a dropped or sign-flipped bias, a
single-precision reciprocal and round-half-away).
"""
from fractions import Fraction

import numpy as np
import pytest

import oracle
import synth
from exact_fp32 import add, as_f32, clamp_i8, f32, mul, recip_in_double_then_f32, rne_int


def _exact_requant(acc, s_in, ws, b, out_scale, ozp):
    a = f32(Fraction(int(acc)))
    t1 = mul(a, as_f32(s_in))
    t2 = mul(t1, as_f32(ws))
    v = add(t2, as_f32(b))
    u = mul(v, recip_in_double_then_f32(out_scale))
    r = rne_int(u)
    if isinstance(r, float):
        return clamp_i8(r)
    return clamp_i8(f32(r + ozp))


@pytest.mark.parametrize("izp", [-128, -5, 0, 3, 127])
def test_k1_exhaustive_products(izp):
    xs = np.arange(-128, 128, dtype=np.int8).reshape(256, 1)
    ws = np.arange(-128, 128, dtype=np.int8).reshape(256, 1)
    acc = oracle.linear_acc(xs, izp, ws)
    want = (np.arange(-128, 128, dtype=np.int64)[:, None] - izp) * np.arange(-128, 128)[None, :]
    np.testing.assert_array_equal(acc.astype(np.int64), want)


@pytest.mark.parametrize("M,K,N,ldw,izp", [
    (1, 4096, 64, 4096, 0), (3, 17, 5, 20, -7), (8, 64, 32, 64, 3), (33, 130, 12, 136, 127),
    (64, 300, 48, 300, -128)])
def test_acc_equals_float64_matmul(M, K, N, ldw, izp):
    x = synth.int8_uniform(M * 7 + K, "lx", (M, K), -128, 127)
    w = synth.int8_uniform(M * 7 + K, "lw", (N, ldw), -128, 127)
    acc = oracle.linear_acc(x, izp, w)
    ref = (x.astype(np.float64) - izp) @ w[:, :K].astype(np.float64).T
    np.testing.assert_array_equal(acc.astype(np.float64), ref)


@pytest.mark.parametrize("izp", [-128, -7, 1, 127])
def test_zero_point_fold_identity(izp):
    # sum (x - zp) w == sum x w - zp sum w  (both pages' Constraints paragraphs)
    x = synth.int8_uniform(5, "fx", (9, 200), -128, 127)
    w = synth.int8_uniform(5, "fw", (16, 200), -128, 127)
    lhs = oracle.linear_acc(x, izp, w).astype(np.int64)
    raw = oracle.linear_acc(x, 0, w).astype(np.int64)
    wsum = w.astype(np.int64).sum(axis=1)
    np.testing.assert_array_equal(lhs, raw - izp * wsum[None, :])


def test_int32_accumulator_wraps():
    K = 140_000
    x = np.full((1, K), 127, np.int8)
    w = np.full((1, K), 127, np.int8)
    acc = int(oracle.linear_acc(x, -128, w)[0, 0])
    exact = 255 * 127 * K
    want = ((exact + 2 ** 31) % 2 ** 32) - 2 ** 31
    assert exact > 2 ** 31 and acc == want


def test_epilogue_exact_rational():
    n = 4000
    accs = np.concatenate([
        synth.uniform_int(31, "ea", (n // 2,), -2 ** 31, 2 ** 31 - 1),
        synth.uniform_int(32, "eb", (n // 2,), -300000, 300000)])
    s_in = synth.uniform_float(31, "es", (n,), 0.001, 0.05).astype(np.float64)
    ws = synth.uniform_float(31, "ew", (n,), 0.0005, 0.02)
    b = synth.normal(31, "eB", (n,), 0.0, 0.1)
    osc = synth.uniform_float(31, "eo", (n,), 0.01, 1.0).astype(np.float64)
    ozp = synth.uniform_int(31, "ez", (n,), -128, 127)
    for i in range(n):
        got = int(oracle.requantize(np.array([[accs[i]]], np.int32), float(s_in[i]),
                                    ws[i:i + 1], b[i:i + 1], float(osc[i]), int(ozp[i]))[0, 0])
        assert got == _exact_requant(accs[i], s_in[i], ws[i], b[i], osc[i], ozp[i]), i


def _ulp(q):
    """Unit in the last place of a nonzero normal binary32 value (exact)."""
    q = abs(q)
    e = q.numerator.bit_length() - q.denominator.bit_length()
    while Fraction(2) ** e > q:
        e -= 1
    while Fraction(2) ** (e + 1) <= q:
        e += 1
    return Fraction(2) ** (e - 23)


def test_epilogue_order_is_observable():
    """Cases built so that one ulp of t2 = (a*s_in)*ws changes the int8 result:
    the bias cancels t2 down to a few ulps (exactly, by Sterbenz) and
    inv_output_scale = 2/ulp(t2) turns each ulp into two output steps, so a
    fused multiply-add (which keeps t2's rounding error, up to half an ulp)
    and a different association (one ulp off) both move the rounded result.
    The oracle must follow the specified order on every case."""
    n, distinguishing = 600, 0
    accs = synth.uniform_int(41, "oa", (n,), -5_000_000, 5_000_000)
    s_in = synth.uniform_float(41, "os", (n,), 0.001, 0.05).astype(np.float64)
    ws = synth.uniform_float(41, "ow", (n,), 0.0005, 0.02)
    ks = synth.uniform_int(41, "ok", (n,), -40, 40)
    for i in range(n):
        if accs[i] == 0:
            continue
        a = f32(Fraction(int(accs[i])))
        si, wi = as_f32(s_in[i]), as_f32(ws[i])
        t2 = mul(mul(a, si), wi)
        ulp = _ulp(t2)
        b = f32(-t2 + int(ks[i]) * ulp)
        out_scale = float(ulp / 2)                  # a power of two: its reciprocal is exact
        want = _exact_requant(accs[i], s_in[i], ws[i], float(b), out_scale, 0)
        got = int(oracle.requantize(np.array([[accs[i]]], np.int32), float(s_in[i]),
                                    ws[i:i + 1], np.array([float(b)], np.float32), out_scale,
                                    0)[0, 0])
        assert got == want, i
        inv = 2 / ulp
        alt_assoc = clamp_i8(rne_int(mul(add(mul(a, mul(si, wi)), b), inv)))
        fused = clamp_i8(rne_int(mul(f32(mul(a, si) * wi + b), inv)))
        if alt_assoc != want or fused != want:
            distinguishing += 1
    assert distinguishing > n // 10


def test_closed_form_unit_scales():
    # s_in = ws = output_scale = 1, b = 0: q = clamp(acc + ozp, -128, 127)
    acc = np.arange(-300, 300, dtype=np.int32).reshape(1, -1)
    N = acc.shape[1]
    for ozp in (-128, -2, 0, 1, 127):
        q = oracle.requantize(acc, 1.0, np.ones(N, np.float32), np.zeros(N, np.float32), 1.0, ozp)
        np.testing.assert_array_equal(q[0].astype(int), np.clip(acc[0] + ozp, -128, 127))


def test_epilogue_ties_and_bias():
    # u = acc + 0.5 with unit scales: ties to even; bias sign matters
    acc = np.array([[0, 1, -1, 2, -2, 3]], np.int32)
    one = np.ones(6, np.float32)
    q = oracle.requantize(acc, 1.0, one, np.full(6, 0.5, np.float32), 1.0, 0)
    assert q[0].tolist() == [0, 2, 0, 2, -2, 4]
    q = oracle.requantize(acc, 1.0, one, np.full(6, -0.5, np.float32), 1.0, 0)
    assert q[0].tolist() == [0, 0, -2, 2, -2, 2]
    q = oracle.requantize(acc, 1.0, one, None, 1.0, 0)
    assert q[0].tolist() == [0, 1, -1, 2, -2, 3]


def test_epilogue_saturation():
    acc = np.array([[2 ** 31 - 1, -2 ** 31, 10 ** 6, -10 ** 6]], np.int32)
    q = oracle.requantize(acc, 0.02, np.full(4, 0.01, np.float32), np.zeros(4, np.float32),
                          1e-6, 5)
    assert q[0].tolist() == [127, -128, 127, -128]


def test_linear_is_acc_then_requantize():
    x = synth.int8_uniform(7, "cx", (5, 77), -128, 127)
    w = synth.int8_uniform(7, "cw", (12, 80), -127, 127)
    ws = synth.uniform_float(7, "cs", (12,), 0.002, 0.01)
    b = synth.normal(7, "cb", (12,), 0.0, 0.1)
    full = oracle.linear(x, 0.02, -3, w, ws, b, 0.05, 4, K=77)
    acc = oracle.linear_acc(x, -3, w)
    np.testing.assert_array_equal(full, oracle.requantize(acc, 0.02, ws, b, 0.05, 4))
    # a null bias equals an all-zero bias
    np.testing.assert_array_equal(oracle.linear(x, 0.02, -3, w, ws, None, 0.05, 4),
                                  oracle.linear(x, 0.02, -3, w, ws, np.zeros(12, np.float32),
                                                0.05, 4))
