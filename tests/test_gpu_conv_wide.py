"""GPU parity of the convolutions with more than 64 output channels per group.

Those take the exchanged-operand tiles: 128 output channels on the MMA's M
side and 256 output pixels on its N side, one output channel per epilogue
thread writing runs of contiguous bytes.  Every case is compared with the CPU
oracle bit for bit (int8 outputs and int32 accumulators).  The shapes reach
each store form: whole 64-pixel runs inside the row (16-byte stores, the
stride-2 column phases merged through the output), runs cut by the right
edge, output columns past the natural size, narrow tiles (fewer than 64 columns per tile row), planes whose size is
not a multiple of 16 (unaligned runs), strides 1, 2 and 3, ragged channel
blocks, dilation, groups, relu, the packed weights, and tiles whose k-loop
needs several exact f32 chunks.
"""
import numpy as np
import pytest
import torch

import oracle
import synth

pytestmark = pytest.mark.gpu

q8 = pytest.importorskip("int8_quantized_q8ta_gb300")
DEV = torch.device("cuda:0")
P = dict(ws_lo=0.002, ws_hi=0.01, b_mean=0.0, b_var=0.1)


def T(a):
    return torch.from_numpy(np.ascontiguousarray(a)).to(DEV)


def H(t):
    torch.cuda.synchronize()
    return t.cpu().numpy()


@pytest.fixture(autouse=True)
def _no_device_error():
    yield
    assert q8.device_error(clear=True) == 0


def _inputs(seed, N, IC, OC, H_in, W_in, K, groups):
    x = synth.int8_uniform(seed, "x", (N, IC, H_in, W_in), -128, 127)
    w = synth.int8_uniform(seed, "w", (OC, K * K * (IC // groups)), -127, 127)
    ws = synth.uniform_float(seed, "ws", (OC,), P["ws_lo"], P["ws_hi"])
    b = synth.normal(seed, "b", (OC,), P["b_mean"], P["b_var"])
    return x, w, ws, b


def _w4(W):
    # the ops' guard W_out % 4 == 0: round the natural width up
    return (W + 3) // 4 * 4


def _not_degenerate(ref):
    # the case exercises the requantization, not only the clamp
    assert len(np.unique(ref)) > 16


# (N, IC, OC, H_in, W_in, K, stride, pad, out_pad, dil, groups, izp, ozp, act)
CONV_T = [
    # whole rows: W_out = 128 -> 64 phase columns, 16-byte runs, phases merged
    (1, 64, 128, 64, 64, 3, 2, 1, 1, 1, 1, -7, 2, "none"),
    # two channel blocks (200 = 128 + 72), phase width 37 of a 64-wide tile
    (1, 96, 200, 20, 37, 3, 2, 1, 1, 1, 1, 4, -3, "relu"),
    # W_out past the natural size (89 -> 92): the last columns lack taps
    (2, 64, 96, 18, 45, 3, 2, 1, 0, 1, 1, 0, 0, "none"),
    # stride 3: three column phases, byte stores
    (1, 64, 100, 12, 50, 4, 3, 1, 2, 1, 1, -20, 5, "none"),
    # stride 1: one phase, unaligned planes (19 * 68 % 16 != 0)
    (1, 128, 130, 19, 66, 3, 1, 1, 0, 1, 1, 11, -1, "relu"),
    # dilation 2 with groups: 96 output channels per group
    (1, 128, 192, 24, 40, 3, 2, 2, 1, 2, 2, -3, 1, "none"),
    # narrow tile rows (phase width 20 -> 32-wide tiles): generic placement
    (2, 64, 128, 24, 20, 3, 2, 1, 1, 1, 1, 1, 0, "none"),
]


@pytest.mark.parametrize("case", CONV_T, ids=[f"ct{i}" for i in range(len(CONV_T))])
def test_conv_t_wide(case):
    N, IC, OC, Hi, Wi, K, s, p, op, d, g, izp, ozp, act = case
    x, w, ws, b = _inputs(600 + CONV_T.index(case), N, IC, OC, Hi, Wi, K, g)
    Ho, Wo = synth.output_hw(Hi, Wi, K, K, s, s, p, p, op, op, d, d)
    Wo = _w4(Wo)
    ref = oracle.conv2d_transposed(x, 0.02, izp, w, K, K, ws, b, 0.12, ozp, Ho, Wo, (s, s),
                                   (p, p), (d, d), groups=g, activation=act)
    _not_degenerate(ref)
    got = H(q8.conv2d_transposed(T(x), 0.02, izp, T(w), None, T(ws), T(b), 0.12, ozp, K,
                                 stride=s, padding=p, output_padding=op, dilation=d, groups=g,
                                 activation=act, output_size=(Ho, Wo)))
    np.testing.assert_array_equal(got, ref)
    acc = H(q8.conv2d_transposed_acc32(T(x), izp, T(w), K, (Ho, Wo), stride=s, padding=p,
                                       dilation=d, groups=g))
    np.testing.assert_array_equal(acc, oracle.conv2d_transposed_acc(
        x, izp, w, K, K, Ho, Wo, (s, s), (p, p), (d, d), groups=g))
    packed = q8.pack_conv2d_transposed_weight(T(w), in_channels=IC, kernel_size=K, groups=g)
    got = H(q8.conv2d_transposed_packed(T(x), 0.02, izp, packed, T(ws), T(b), 0.12, ozp,
                                        stride=s, padding=p, output_padding=op, dilation=d,
                                        activation=act, output_size=(Ho, Wo)))
    np.testing.assert_array_equal(got, ref)
    np.testing.assert_array_equal(
        H(q8.conv2d_transposed_packed_acc32(T(x), izp, packed, (Ho, Wo), stride=s, padding=p,
                                            dilation=d)), acc)


def test_conv_t_wide_several_chunks():
    """384 input channels and the widest zero point: a 2x2-tap phase spans 24
    k-blocks against exact f32 chunks of 8, so its tiles add three chunks in
    int32 before the requantization."""
    N, IC, OC, Hi, Wi, K = 1, 384, 128, 16, 64, 3
    x, w, ws, b = _inputs(77, N, IC, OC, Hi, Wi, K, 1)
    x[..., ::3] = -128                      # reach the bound |x - zp| = 255
    izp = 127
    Ho, Wo = synth.output_hw(Hi, Wi, K, K, 2, 2, 1, 1, 1, 1)
    ref = oracle.conv2d_transposed(x, 0.004, izp, w, K, K, ws, b, 0.2, 0, Ho, Wo, (2, 2),
                                   (1, 1), (1, 1))
    _not_degenerate(ref)
    got = H(q8.conv2d_transposed(T(x), 0.004, izp, T(w), None, T(ws), T(b), 0.2, 0, K,
                                 stride=2, padding=1, output_padding=1, output_size=(Ho, Wo)))
    np.testing.assert_array_equal(got, ref)
    acc = H(q8.conv2d_transposed_acc32(T(x), izp, T(w), K, (Ho, Wo), stride=2, padding=1))
    np.testing.assert_array_equal(acc, oracle.conv2d_transposed_acc(
        x, izp, w, K, K, Ho, Wo, (2, 2), (1, 1), (1, 1)))


# (N, IC, OC, H_in, W_in, K, stride, pad, dil, groups, izp, ozp, act)
CONV2D = [
    # whole rows of 128 output columns
    (1, 64, 128, 34, 130, 3, 1, 0, 1, 1, -7, 2, "none"),
    # stride 2, ragged right edge (W_out 45 -> 48) and channel block
    (2, 96, 160, 40, 90, 3, 2, 1, 1, 1, 3, -2, "relu"),
    # dilation 2 with groups, 80 output channels per group
    (1, 128, 160, 30, 72, 3, 1, 2, 2, 2, 0, 0, "none"),
    # narrow rows (W_out = 24): generic placement
    (1, 64, 128, 40, 24, 3, 1, 1, 1, 1, -1, 1, "none"),
]


@pytest.mark.parametrize("case", CONV2D, ids=[f"c{i}" for i in range(len(CONV2D))])
def test_conv2d_wide(case):
    N, IC, OC, Hi, Wi, K, s, p, d, g, izp, ozp, act = case
    x, w, ws, b = _inputs(700 + CONV2D.index(case), N, IC, OC, Hi, Wi, K, g)
    Ho, Wo = q8.conv2d_output_size(Hi, Wi, K, s, p, d)
    Wo = _w4(Wo)
    ref = oracle.conv2d(x, 0.02, izp, w, K, K, ws, b, 0.12, ozp, Ho, Wo, (s, s), (p, p), (d, d),
                        groups=g, activation=act)
    _not_degenerate(ref)
    got = H(q8.conv2d(T(x), 0.02, izp, T(w), T(ws), T(b), 0.12, ozp, K, stride=s, padding=p,
                      dilation=d, groups=g, activation=act, output_size=(Ho, Wo)))
    np.testing.assert_array_equal(got, ref)
    acc = H(q8.conv2d_acc32(T(x), izp, T(w), K, (Ho, Wo), stride=s, padding=p, dilation=d,
                            groups=g))
    np.testing.assert_array_equal(acc, oracle.conv2d_acc(x, izp, w, K, K, Ho, Wo, (s, s), (p, p),
                                                         (d, d), groups=g))
    packed = q8.pack_conv2d_weight(T(w), in_channels=IC, kernel_size=K, groups=g)
    got = H(q8.conv2d_packed(T(x), 0.02, izp, packed, T(ws), T(b), 0.12, ozp, stride=s,
                             padding=p, dilation=d, activation=act, output_size=(Ho, Wo)))
    np.testing.assert_array_equal(got, ref)
    np.testing.assert_array_equal(
        H(q8.conv2d_packed_acc32(T(x), izp, packed, (Ho, Wo), stride=s, padding=p, dilation=d)),
        acc)
