"""The CUDA epilogue's conversion-free rounding equals the plain one (CPU).

The kernels compute clamp(rint(u) + zp, lo, 127) (lo = -128, or zp under
relu) without a float->int conversion instruction, in two forms:
  * the quantize kernels raise u to at least -2^22, add 1.5 * 2^23 in f32
    (round to nearest even), read the integer from the sum's encoding and
    clamp it as an integer;
  * the GEMM and gemv epilogues clamp u first, to [lo - zp, 127 - zp], then
    add 1.5 * 2^23 and read the integer, already in range;
  * the exchanged-operand convolution epilogue takes only the floor on the
    float (u raised to lo - zp), adds 1.5 * 2^23, reads the integer and
    leaves the upper clamp to a saturating conversion to int8.
This test replays the forms in numpy float32 -- whose
addition rounds to nearest even like the GPU's __fadd_rn -- over every
rounding tie near the int8 range, their float neighbours, random bit
patterns (NaN, infinities, subnormals included) and every zero point.
"""
import numpy as np

F = np.float32


def plain(u, zp):
    """rint half-to-even, + zp in f32, clamp, truncate (NaN -> -128 through
    fmaxf's choice of the non-NaN operand)."""
    r = np.rint(u).astype(F)
    t = (r + F(zp)).astype(F)
    t = np.where(np.isnan(t), F(-128.0), t)
    t = np.minimum(np.maximum(t, F(-128.0)), F(127.0))
    return t.astype(np.int32)


def alu_only(u, zp):
    c = np.where(np.isnan(u), F(-4194304.0), u).astype(F)      # fmaxf(NaN, c) = c
    c = np.maximum(c, F(-4194304.0)).astype(F)
    y = (c + F(12582912.0)).astype(F)
    bits = y.view(np.int32).astype(np.int32)
    assert (bits > 0).all()                                     # y stays positive
    q = (bits - np.int32(0x4B400000 - zp)).astype(np.int64)    # int32 arithmetic, no overflow
    assert (q < 2 ** 31).all() and (q >= -2 ** 31).all()
    return np.clip(q, -128, 127).astype(np.int32)


def plain_lo(u, zp, lo):
    """plain() with the floor lo (relu: lo = zp, the clamp of max(v, 0)
    after the requantization; NaN -> the floor)."""
    return np.maximum(plain(u, zp), np.int32(lo)).astype(np.int32)


def clamp_first(u, zp, lo):
    c = np.where(np.isnan(u), F(lo - zp), u).astype(F)            # fmaxf(NaN, c) = c
    c = np.minimum(np.maximum(c, F(lo - zp)), F(127 - zp)).astype(F)
    y = (c + F(12582912.0)).astype(F)
    q = y.view(np.int32).astype(np.int64) - (0x4B400000 - zp)
    assert (q >= lo).all() and (q <= 127).all()
    return q.astype(np.int32)


def floor_first(u, zp, lo):
    c = np.where(np.isnan(u), F(lo - zp), u).astype(F)            # fmaxf(NaN, c) = c
    c = np.maximum(c, F(lo - zp)).astype(F)
    y = (c + F(12582912.0)).astype(F)
    bits = y.view(np.int32).astype(np.int64)
    assert (bits > 0).all()                                         # y stays positive
    q = bits - (0x4B400000 - zp)
    assert (q >= lo).all() and (q < 2 ** 31).all()                  # an int32, at least lo
    return np.clip(q, -128, 127).astype(np.int32)                   # the saturating pack


def _samples():
    ties = np.arange(-400, 400, dtype=np.float64) + 0.5
    ints = np.arange(-400, 400, dtype=np.float64)
    base = np.concatenate([ties, ints]).astype(F)
    up = np.nextafter(base, F(np.inf))
    down = np.nextafter(base, F(-np.inf))
    big = np.array([2.0 ** 21, 2.0 ** 21 + 0.5, 2.0 ** 22, 2.0 ** 22 - 0.5, 2.0 ** 22 + 1,
                    2.0 ** 23, 2.0 ** 24, 3.4e38, 1e30, 4194303.5, 8388607.5, 12582912.0,
                    12582911.5, 16777215.0], dtype=np.float64)
    big = np.concatenate([big, -big]).astype(F)
    special = np.array([np.inf, -np.inf, np.nan, 0.0, -0.0, 1e-45, -1e-45, 1e-38], dtype=F)
    rng = np.random.default_rng(7)
    bits = rng.integers(0, 2 ** 32, size=200_000, dtype=np.uint64).astype(np.uint32).view(F)
    scaled = (rng.standard_normal(200_000) * 150.0).astype(F)
    return np.concatenate([base, up, down, big, special, bits, scaled])


def test_alu_rounding_matches_rint_add_clamp_for_every_zero_point():
    u = _samples()
    with np.errstate(invalid="ignore", over="ignore"):
        for zp in range(-128, 128):
            np.testing.assert_array_equal(alu_only(u, zp), plain(u, zp), err_msg=f"zp={zp}")


def test_clamp_first_matches_rint_add_clamp_for_every_zero_point_and_floor():
    u = _samples()
    with np.errstate(invalid="ignore", over="ignore"):
        for zp in range(-128, 128):
            np.testing.assert_array_equal(clamp_first(u, zp, -128), plain(u, zp),
                                          err_msg=f"zp={zp}")
            np.testing.assert_array_equal(clamp_first(u, zp, zp), plain_lo(u, zp, zp),
                                          err_msg=f"relu zp={zp}")


def test_floor_first_with_saturation_matches_rint_add_clamp():
    u = _samples()
    with np.errstate(invalid="ignore", over="ignore"):
        for zp in range(-128, 128):
            np.testing.assert_array_equal(floor_first(u, zp, -128), plain(u, zp),
                                          err_msg=f"zp={zp}")
            np.testing.assert_array_equal(floor_first(u, zp, zp), plain_lo(u, zp, zp),
                                          err_msg=f"relu zp={zp}")


def test_ties_round_to_even():
    u = np.array([0.5, 1.5, 2.5, -0.5, -1.5, -2.5, 126.5, -127.5], dtype=F)
    assert alu_only(u, 0).tolist() == [0, 2, 2, 0, -2, -2, 126, -128]
    assert clamp_first(u, 0, -128).tolist() == [0, 2, 2, 0, -2, -2, 126, -128]
    assert clamp_first(u, 1, -128).tolist() == [1, 3, 3, 1, -1, -1, 127, -127]


def test_bf16_of_small_integers_by_bit_pattern():
    """The operand preparation forms bf16(v) for v = x - zp in [-255, 255]
    without a conversion instruction: f = float(bits(1.5 * 2^23) + v) - 1.5 *
    2^23 (exact), and the bf16 encoding is the high half of f's encoding,
    whose low half is zero (at most 8 significant bits)."""
    v = np.arange(-255, 256, dtype=np.int64)
    f = ((np.int64(0x4B400000) + v).astype(np.int32).view(F) - F(12582912.0)).astype(F)
    np.testing.assert_array_equal(f, v.astype(F))
    bits = f.view(np.uint32)
    assert (bits & 0xFFFF == 0).all()
    # against a rounding conversion to bfloat16 of the exact float (round to nearest even)
    u = v.astype(F).view(np.uint32).astype(np.uint64)
    rne = ((u + 0x7FFF + ((u >> 16) & 1)) >> 16).astype(np.uint32)
    np.testing.assert_array_equal(bits >> 16, rne)
