"""Seeded random sweep of GPU parity (bit-exact against the CPU oracle).

Shapes, zero points, scales, strides, paddings, dilations, groups and the
activation are drawn from the counter-based generator within the ops'
guards, at sizes the oracle finishes quickly; each case compares the int8
output and the int32 accumulators.  The draws cover what the hand-picked
cases may miss: odd channel counts, 1-pixel images, tiny and ragged K,
zero points at both ends, every tile path (one CTA, CTA pairs and their
tile widths, both convolution modes, and the exchanged-operand tiles of
more than 64 output channels per group on images of at least 256 pixels
per stride phase).
"""
import numpy as np
import pytest
import torch

import oracle
import synth

pytestmark = pytest.mark.gpu

q8 = pytest.importorskip("int8_quantized_q8ta_gb300")
DEV = torch.device("cuda:0")


def T(a):
    return torch.from_numpy(np.ascontiguousarray(a)).to(DEV)


def H(t):
    torch.cuda.synchronize()
    return t.cpu().numpy()


@pytest.fixture(autouse=True)
def _no_device_error():
    yield
    assert q8.device_error(clear=True) == 0


def _draw(seed, name, lo, hi):
    return int(synth.uniform_int(seed, name, (1,), lo, hi)[0])


def _common(seed):
    izp = _draw(seed, "izp", -128, 127)
    ozp = _draw(seed, "ozp", -128, 127)
    act = "relu" if _draw(seed, "act", 0, 1) else "none"
    s_in = float(synth.uniform_float(seed, "sin", (1,), 0.005, 0.05)[0])
    s_out = float(synth.uniform_float(seed, "sout", (1,), 0.02, 0.5)[0])
    return izp, ozp, act, s_in, s_out


@pytest.mark.parametrize("seed", range(100, 116))
def test_linear_sweep(seed):
    M = _draw(seed, "M", 1, 600)
    N = 4 * _draw(seed, "N", 1, 300)
    K = 4 * _draw(seed, "K", 1, 400)
    izp, ozp, act, s_in, s_out = _common(seed)
    x = synth.int8_uniform(seed, "x", (M, K), -128, 127)
    w = synth.int8_uniform(seed, "w", (N, K), -128, 127)
    ws = synth.uniform_float(seed, "ws", (N,), 0.0005, 0.01)
    b = synth.normal(seed, "b", (N,), 0.0, 0.2)
    ref = oracle.linear(x, s_in, izp, w, ws, b, s_out, ozp, activation=act)
    got = H(q8.linear(T(x), s_in, izp, T(w), None, T(ws), T(b), s_out, ozp, activation=act))
    np.testing.assert_array_equal(got, ref)
    if M > 1:
        acc = H(q8.linear_packed_acc32(T(x), izp, q8.pack_weight(T(w))))
        np.testing.assert_array_equal(acc, oracle.linear_acc(x, izp, w))


def _conv_draw(seed, transposed):
    g = [1, 1, 2, 3, 4][_draw(seed, "g", 0, 4)]
    IC = g * _draw(seed, "icg", 1, 40)
    OC = g * _draw(seed, "ocg", 1, 40)
    N = _draw(seed, "n", 1, 2)
    H_in, W_in = _draw(seed, "h", 1, 12), _draw(seed, "w", 1, 12)
    K = _draw(seed, "k", 1, 4)
    s = _draw(seed, "s", 1, 3 if transposed else 4)
    p = _draw(seed, "p", 0, 2)
    d = _draw(seed, "d", 1, 2)
    return g, IC, OC, N, H_in, W_in, K, s, p, d


@pytest.mark.parametrize("seed", range(200, 214))
def test_conv_t_sweep(seed):
    g, IC, OC, N, H_in, W_in, K, s, p, d = _conv_draw(seed, True)
    izp, ozp, act, s_in, s_out = _common(seed)
    Hn, Wn = synth.output_hw(H_in, W_in, K, K, s, s, p, p, 0, 0, d, d)
    Ho = max(1, Hn + _draw(seed, "oph", 0, 1))
    Wo = max(4, (max(1, Wn) + 3) // 4 * 4)          # the W_out % 4 guard
    x = synth.int8_uniform(seed, "x", (N, IC, H_in, W_in), -128, 127)
    w = synth.int8_uniform(seed, "w", (OC, K * K * (IC // g)), -128, 127)
    ws = synth.uniform_float(seed, "ws", (OC,), 0.0005, 0.01)
    b = synth.normal(seed, "b", (OC,), 0.0, 0.2)
    ref = oracle.conv2d_transposed(x, s_in, izp, w, K, K, ws, b, s_out, ozp, Ho, Wo, (s, s),
                                   (p, p), (d, d), groups=g, activation=act)
    got = H(q8.conv2d_transposed(T(x), s_in, izp, T(w), None, T(ws), T(b), s_out, ozp, K,
                                 stride=s, padding=p, dilation=d, groups=g, activation=act,
                                 output_size=(Ho, Wo)))
    np.testing.assert_array_equal(got, ref)
    acc = H(q8.conv2d_transposed_acc32(T(x), izp, T(w), K, (Ho, Wo), stride=s, padding=p,
                                       dilation=d, groups=g))
    np.testing.assert_array_equal(acc, oracle.conv2d_transposed_acc(
        x, izp, w, K, K, Ho, Wo, (s, s), (p, p), (d, d), groups=g))


@pytest.mark.parametrize("seed", range(300, 314))
def test_conv2d_sweep(seed):
    g, IC, OC, N, H_in, W_in, K, s, p, d = _conv_draw(seed, False)
    izp, ozp, act, s_in, s_out = _common(seed)
    Hn, Wn = q8.conv2d_output_size(H_in, W_in, K, s, p, d)
    Ho = max(1, Hn)
    Wo = max(4, (max(1, Wn) + 3) // 4 * 4)          # extra columns read only padding
    x = synth.int8_uniform(seed, "x", (N, IC, H_in, W_in), -128, 127)
    w = synth.int8_uniform(seed, "w", (OC, K * K * (IC // g)), -128, 127)
    ws = synth.uniform_float(seed, "ws", (OC,), 0.0005, 0.01)
    b = synth.normal(seed, "b", (OC,), 0.0, 0.2)
    ref = oracle.conv2d(x, s_in, izp, w, K, K, ws, b, s_out, ozp, Ho, Wo, (s, s), (p, p), (d, d),
                        groups=g, activation=act)
    got = H(q8.conv2d(T(x), s_in, izp, T(w), T(ws), T(b), s_out, ozp, K, stride=s, padding=p,
                      dilation=d, groups=g, activation=act, output_size=(Ho, Wo)))
    np.testing.assert_array_equal(got, ref)
    acc = H(q8.conv2d_acc32(T(x), izp, T(w), K, (Ho, Wo), stride=s, padding=p, dilation=d,
                            groups=g))
    np.testing.assert_array_equal(acc, oracle.conv2d_acc(x, izp, w, K, K, Ho, Wo, (s, s), (p, p),
                                                         (d, d), groups=g))


def _wide_draw(seed, transposed):
    g = [1, 1, 2][_draw(seed, "g", 0, 2)]
    IC = g * _draw(seed, "icg", 1, 130)
    OC = g * _draw(seed, "ocg", 65, 200)
    N = _draw(seed, "n", 1, 2)
    s = _draw(seed, "s", 1, 3 if transposed else 2)
    H_in = _draw(seed, "h", 16, 28) if transposed else s * _draw(seed, "h", 16, 34)
    W_in = _draw(seed, "w", 16, 56) if transposed else s * _draw(seed, "w", 16, 80)
    K = _draw(seed, "k", 1, 3)
    p = _draw(seed, "p", 0, 1)
    d = _draw(seed, "d", 1, 2)
    return g, IC, OC, N, H_in, W_in, K, s, p, d


@pytest.mark.parametrize("seed", range(400, 408))
def test_conv_t_wide_sweep(seed):
    g, IC, OC, N, H_in, W_in, K, s, p, d = _wide_draw(seed, True)
    izp, ozp, act, s_in, s_out = _common(seed)
    Hn, Wn = synth.output_hw(H_in, W_in, K, K, s, s, p, p, 0, 0, d, d)
    Ho = max(1, Hn + _draw(seed, "oph", 0, 1))
    Wo = max(4, (max(1, Wn) + 3) // 4 * 4)
    x = synth.int8_uniform(seed, "x", (N, IC, H_in, W_in), -128, 127)
    w = synth.int8_uniform(seed, "w", (OC, K * K * (IC // g)), -128, 127)
    ws = synth.uniform_float(seed, "ws", (OC,), 0.0005, 0.01)
    b = synth.normal(seed, "b", (OC,), 0.0, 0.2)
    ref = oracle.conv2d_transposed(x, s_in, izp, w, K, K, ws, b, s_out, ozp, Ho, Wo, (s, s),
                                   (p, p), (d, d), groups=g, activation=act)
    packed = q8.pack_conv2d_transposed_weight(T(w), in_channels=IC, kernel_size=K, groups=g)
    got = H(q8.conv2d_transposed_packed(T(x), s_in, izp, packed, T(ws), T(b), s_out, ozp,
                                        stride=s, padding=p, dilation=d, activation=act,
                                        output_size=(Ho, Wo)))
    np.testing.assert_array_equal(got, ref)
    acc = H(q8.conv2d_transposed_packed_acc32(T(x), izp, packed, (Ho, Wo), stride=s, padding=p,
                                              dilation=d))
    np.testing.assert_array_equal(acc, oracle.conv2d_transposed_acc(
        x, izp, w, K, K, Ho, Wo, (s, s), (p, p), (d, d), groups=g))


@pytest.mark.parametrize("seed", range(500, 506))
def test_conv2d_wide_sweep(seed):
    g, IC, OC, N, H_in, W_in, K, s, p, d = _wide_draw(seed, False)
    izp, ozp, act, s_in, s_out = _common(seed)
    Hn, Wn = q8.conv2d_output_size(H_in, W_in, K, s, p, d)
    Ho, Wo = max(1, Hn), max(4, (max(1, Wn) + 3) // 4 * 4)
    x = synth.int8_uniform(seed, "x", (N, IC, H_in, W_in), -128, 127)
    w = synth.int8_uniform(seed, "w", (OC, K * K * (IC // g)), -128, 127)
    ws = synth.uniform_float(seed, "ws", (OC,), 0.0005, 0.01)
    b = synth.normal(seed, "b", (OC,), 0.0, 0.2)
    ref = oracle.conv2d(x, s_in, izp, w, K, K, ws, b, s_out, ozp, Ho, Wo, (s, s), (p, p), (d, d),
                        groups=g, activation=act)
    got = H(q8.conv2d(T(x), s_in, izp, T(w), T(ws), T(b), s_out, ozp, K, stride=s, padding=p,
                      dilation=d, groups=g, activation=act, output_size=(Ho, Wo)))
    np.testing.assert_array_equal(got, ref)
    packed = q8.pack_conv2d_weight(T(w), in_channels=IC, kernel_size=K, groups=g)
    acc = H(q8.conv2d_packed_acc32(T(x), izp, packed, (Ho, Wo), stride=s, padding=p, dilation=d))
    np.testing.assert_array_equal(acc, oracle.conv2d_acc(x, izp, w, K, K, Ho, Wo, (s, s), (p, p),
                                                         (d, d), groups=g))

