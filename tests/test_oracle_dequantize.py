"""Pins for the oracle's dequantize_per_tensor (CPU only).

Source: the quantize -> q8ta_* -> dequantize subgraph that the Problem
paragraphs of "Add q8ta_linear op" (PR #21197) and "Add
q8ta_conv2d_transposed op" (PR #21205) delegate; the closing op is named
there but its arithmetic is not printed.  The reading taken is the library
op that the quantize page bit-matches, torch's decomposed
dequantize_per_tensor: y = ((float)q - (float)zp) * (float)scale, with one
binary32 rounding per step and no fused multiply-add.

Pins, none of which re-types the oracle's C:
* torch's CPU quantized_decomposed.dequantize_per_tensor over every int8
  value, several zero points and scales that are not binary32 values;
* exact rational arithmetic with a binary32 rounding after each step;
* discriminating cases: for the scales used, each of three plausible other
  readings -- the product taken in double, q*s - zp*s, and that difference
  with a fused multiply-add -- differs from the pinned reading on at least
  one input, so an oracle computing any of them fails here.
"""
from fractions import Fraction

import numpy as np
import pytest

import oracle
from exact_fp32 import as_f32, f32

ALL_Q = np.arange(-128, 128, dtype=np.int8)
ZPS = [-128, -3, 0, 127]
# not representable in binary32, so the cast of the scale matters
SCALES = [0.1, 0.037, 0.03, 1.0 / 3.0, 0.0078125 + 1e-12, 2.0 ** -7 * 1.1, 123.456]


def _torch_dequantize(q, scale, zp):
    torch = pytest.importorskip("torch")
    import torch.ao.quantization.fx._decomposed  # noqa: F401  registers the op
    op = torch.ops.quantized_decomposed.dequantize_per_tensor.default
    return op(torch.from_numpy(q), float(scale), int(zp), -128, 127, torch.int8).numpy()


def _exact(q, scale, zp):
    """((float)q - (float)zp) * (float)scale, each step rounded to binary32."""
    d = f32(Fraction(int(q)) - Fraction(int(zp)))
    return f32(d * as_f32(scale))


def _in_double(q, scale, zp):
    """The product taken in double, rounded to binary32 once."""
    return f32((Fraction(int(q)) - Fraction(int(zp))) * Fraction(float(scale)))


def _distributed(q, scale, zp):
    """q*s - zp*s, each product and the difference rounded to binary32."""
    s = as_f32(scale)
    return f32(f32(Fraction(int(q)) * s) - f32(Fraction(int(zp)) * s))


def _distributed_fma(q, scale, zp):
    """fma(q, s, -(zp*s)): one rounding after the exact q*s - f32(zp*s)."""
    s = as_f32(scale)
    return f32(Fraction(int(q)) * s - f32(Fraction(int(zp)) * s))


def _as_fraction(v):
    return Fraction(float(v))


@pytest.mark.parametrize("zp", ZPS)
@pytest.mark.parametrize("scale", SCALES)
def test_matches_torch_decomposed_op(scale, zp):
    ours = oracle.dequantize_per_tensor(ALL_Q, scale, zp)
    ref = _torch_dequantize(ALL_Q, scale, zp)
    assert ours.dtype == np.float32
    np.testing.assert_array_equal(ours.view(np.uint32), ref.view(np.uint32))


@pytest.mark.parametrize("zp", ZPS)
@pytest.mark.parametrize("scale", SCALES)
def test_matches_exact_rational_arithmetic(scale, zp):
    ours = oracle.dequantize_per_tensor(ALL_Q, scale, zp)
    for q, y in zip(ALL_Q, ours):
        assert _as_fraction(y) == _exact(q, scale, zp), (int(q), scale, zp)


@pytest.mark.parametrize("other", [_in_double, _distributed, _distributed_fma])
def test_other_readings_are_distinguished(other):
    """Each alternative reading disagrees with the oracle somewhere in the
    pinned grid (so the two tests above would catch an oracle using it)."""
    diffs = 0
    for scale in SCALES:
        for zp in ZPS:
            ours = oracle.dequantize_per_tensor(ALL_Q, scale, zp)
            for q, y in zip(ALL_Q, ours):
                if _as_fraction(y) != other(q, scale, zp):
                    diffs += 1
    assert diffs > 0


def test_closed_forms():
    """Unit scale returns q - zp exactly; q == zp gives +0; a power-of-two
    scale is exact; the extremes of the range."""
    q = ALL_Q
    np.testing.assert_array_equal(oracle.dequantize_per_tensor(q, 1.0, 0), q.astype(np.float32))
    np.testing.assert_array_equal(oracle.dequantize_per_tensor(q, 1.0, -128),
                                  q.astype(np.float32) + 128.0)
    y = oracle.dequantize_per_tensor(np.array([5, -7], np.int8), 0.3, 5)
    assert y[0] == 0.0 and not np.signbit(y[0])
    np.testing.assert_array_equal(oracle.dequantize_per_tensor(q, 0.25, 3),
                                  (q.astype(np.float32) - 3.0) * np.float32(0.25))
    ext = oracle.dequantize_per_tensor(np.array([127, -128], np.int8), 1.0, -128)
    np.testing.assert_array_equal(ext, np.array([255.0, 0.0], np.float32))
    ext = oracle.dequantize_per_tensor(np.array([127, -128], np.int8), 1.0, 127)
    np.testing.assert_array_equal(ext, np.array([0.0, -255.0], np.float32))


def test_empty_and_shape():
    assert oracle.dequantize_per_tensor(np.zeros(0, np.int8), 0.5, 0).size == 0
    q = ALL_Q.reshape(16, 16)
    y = oracle.dequantize_per_tensor(q, 0.5, 1)
    assert y.shape == (16, 16)
    np.testing.assert_array_equal(y.ravel(), oracle.dequantize_per_tensor(ALL_Q, 0.5, 1))
