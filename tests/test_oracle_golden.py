"""The oracle reproduces the committed regression fixtures (tests/golden)."""
import numpy as np

import oracle
from golden_io import load


def test_linear_chain_8x64x32_fixture():
    t, m = load("linear_chain_8x64x32.txt")
    xq = oracle.quantize_per_tensor(t["x"], m["in_scale"], m["in_zp"])
    np.testing.assert_array_equal(xq, t["xq"])
    np.testing.assert_array_equal(oracle.linear_acc(xq, m["in_zp"], t["w"]), t["acc"])
    out = oracle.linear(xq, m["in_scale"], m["in_zp"], t["w"], t["ws"], t["b"], m["out_scale"],
                        m["out_zp"])
    np.testing.assert_array_equal(out, t["out"])
    # the fixture exercises saturation of the quantize step (about 1% of x)
    assert np.count_nonzero((t["xq"] == 127) | (t["xq"] == -128)) > 0


def test_conv_t_small_fixture():
    t, m = load("conv_t_1x3x5x4_k3s2p1op1.txt")
    H, W = t["out"].shape[2:]
    acc = oracle.conv2d_transposed_acc(t["x"], m["in_zp"], t["w"], 3, 3, H, W, (2, 2), (1, 1))
    np.testing.assert_array_equal(acc, t["acc"])
    out = oracle.conv2d_transposed(t["x"], m["in_scale"], m["in_zp"], t["w"], 3, 3, t["ws"],
                                   t["b"], m["out_scale"], m["out_zp"], H, W, (2, 2), (1, 1))
    np.testing.assert_array_equal(out, t["out"])
