"""Pins for the oracle's quantize_per_tensor (CPU only).

Source: "Add quantize_per_tensor op (int8 buffer path)" (PR #21187), Solution
paragraph -- q = clamp(round(x * inv_scale) + zero_point, -128, 127) with
inv_scale the reciprocal taken in double and cast to f32, matching torch's
round(input * (1.0 / scale)).

Pins, none of which re-types the oracle's C:
* torch's CPU quantized_decomposed.quantize_per_tensor (the library op the
  page says it bit-matches);
* exact rational arithmetic with binary32 rounding after each step;
* hand-derived ties, saturation and zero-point cases;
* a scale for which (float)(1.0/scale) differs from 1.0f/(float)scale, so a
  single-precision reciprocal would fail.
"""
from fractions import Fraction

import numpy as np
import pytest

import oracle
import synth
from exact_fp32 import as_f32, clamp_i8, f32, mul, recip_in_double_then_f32, rne_int


def _torch_quantize(x, scale, zp):
    torch = pytest.importorskip("torch")
    import torch.ao.quantization.fx._decomposed  # noqa: F401  registers the op
    op = torch.ops.quantized_decomposed.quantize_per_tensor.default
    return op(torch.from_numpy(x), float(scale), int(zp), -128, 127, torch.int8).numpy()


def _exact_quantize(x, scale, zp):
    inv = recip_in_double_then_f32(scale)
    t = mul(as_f32(x), inv)
    r = rne_int(t)
    if isinstance(r, float):
        return clamp_i8(r)
    return clamp_i8(f32(r + zp))


@pytest.mark.parametrize("seed,scale,zp,var", [
    (0, 0.02, 3, 1.0), (1, 0.03, -5, 3.0), (2, 1.0, 0, 4000.0), (3, 0.5, 127, 10.0),
    (4, 0.0037, -128, 0.5), (5, 7.25, 1, 1e6)])
def test_matches_torch_decomposed_op(seed, scale, zp, var):
    x = synth.normal(seed, "qx", (20000,), 0.0, var)
    ours = oracle.quantize_per_tensor(x, scale, zp)
    ref = _torch_quantize(x, scale, zp)
    np.testing.assert_array_equal(ours, ref)


def test_matches_exact_rational_arithmetic():
    rng_x = synth.normal(11, "ex", (3000,), 0.0, 30.0)
    scales = synth.uniform_float(11, "es", (3000,), 0.001, 2.0).astype(np.float64)
    zps = synth.uniform_int(11, "ez", (3000,), -128, 127)
    for x, s, zp in zip(rng_x, scales, zps):
        got = int(oracle.quantize_per_tensor(np.array([x], np.float32), float(s), int(zp))[0])
        assert got == _exact_quantize(x, float(s), int(zp)), (x, s, zp)


def test_ties_round_half_to_even():
    # scale 1 makes inv exactly 1; x = k + 0.5 is exact in binary32.
    ks = np.arange(-140, 140)
    x = (ks + 0.5).astype(np.float32)
    got = oracle.quantize_per_tensor(x, 1.0, 0).astype(int)
    want = [max(-128, min(127, round(Fraction(int(k)) + Fraction(1, 2)))) for k in ks]
    assert list(got) == want
    # spot values written out by hand
    x = np.array([0.5, 1.5, 2.5, -0.5, -1.5, -2.5, 126.5, 127.5, -128.5, -127.5], np.float32)
    assert list(oracle.quantize_per_tensor(x, 1.0, 0)) == [0, 2, 2, 0, -2, -2, 126, 127, -128, -128]
    # ties after the zero-point shift: rne(0.5)=0, +3 -> 3; rne(1.5)=2, +3 -> 5
    assert list(oracle.quantize_per_tensor(np.array([0.5, 1.5], np.float32), 1.0, 3)) == [3, 5]


def test_zero_point_and_saturation():
    for zp in (-128, -5, 0, 3, 127):
        assert oracle.quantize_per_tensor(np.zeros(4, np.float32), 0.02, zp).tolist() == [zp] * 4
    x = np.array([np.inf, -np.inf, 1e30, -1e30, 3.0e38, -3.0e38], np.float32)
    assert oracle.quantize_per_tensor(x, 0.02, 0).tolist() == [127, -128, 127, -128, 127, -128]
    # clamp happens after the zero-point add: 120 + 10 -> 127, -120 - 10 -> -128
    x = np.array([120.0, -120.0], np.float32)
    assert oracle.quantize_per_tensor(x, 1.0, 10).tolist() == [127, -110]
    assert oracle.quantize_per_tensor(x, 1.0, -10).tolist() == [110, -128]


def _find_double_vs_single_reciprocal_case():
    """A (scale, x) where the f32-of-double reciprocal and a single-precision
    reciprocal lead to different quantized values."""
    s_values = synth.uniform_float(21, "rs", (20000,), 0.001, 1.0).astype(np.float64)
    for s in s_values:
        s = float(np.float64(s) * (1 + 1e-9))      # not exactly a binary32 value
        inv_d = recip_in_double_then_f32(s)
        inv_f = f32(Fraction(1) / as_f32(s))
        if inv_d == inv_f:
            continue
        # x chosen so that x * inv lands next to a .5 boundary for one reading
        for k in range(1, 120):
            x = as_f32(float((Fraction(2 * k + 1, 2)) / inv_d))
            qd = rne_int(mul(x, inv_d))
            qf = rne_int(mul(x, inv_f))
            if qd != qf:
                return s, float(x), int(qd), int(qf)
    return None


def test_reciprocal_taken_in_double():
    case = _find_double_vs_single_reciprocal_case()
    assert case is not None, "no distinguishing scale found"
    s, x, qd, qf = case
    got = int(oracle.quantize_per_tensor(np.array([x], np.float32), s, 0)[0])
    assert got == max(-128, min(127, qd))
    assert got != max(-128, min(127, qf))


def test_full_int8_range_roundtrip():
    # every int8 value q is reproduced from x = q * scale when scale is a power of two
    q = np.arange(-128, 128)
    for scale in (1.0, 0.25, 2.0 ** -7):
        x = (q * scale).astype(np.float32)
        assert oracle.quantize_per_tensor(x, scale, 0).astype(int).tolist() == q.tolist()
