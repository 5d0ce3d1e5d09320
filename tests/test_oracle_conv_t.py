"""Pins for the oracle's q8ta_conv2d_transposed (CPU only).

Source: "Add q8ta_conv2d_transposed op (int8 transposed conv)" (PR #21205).
Solution paragraph: per output, acc = sum over (ic, kh, kw) of
(x[n,ic,ih,iw] - input_zero_point) * weight[oc, (kh*Kw+kw)*IC + ic] with
ih = (oh + pad_h - kh*dil_h) / stride_h taken only when the numerator is
non-negative, divisible by stride_h and ih < H_in (iw likewise), then the same
dequantize / requantize epilogue as q8ta_linear with per-oc scales.
Constraints paragraph: the AOT reshape maps weight[oc,(kh*Kw+kw)*IC+ic] =
original[ic,oc,kh,kw]; out-of-bounds taps contribute nothing, exactly like
filling them with the zero-point ((zp - zp) * w = 0).

Pins: torch's float64 conv_transpose2d on the reshaped weight (exact for
these integer magnitudes), the independent scatter form, a zero-point-filled
dilate-and-pad textbook form, the 1x1 case reducing to q8ta_linear, and
outputs that no tap reaches.
"""
import itertools

import numpy as np
import pytest

import oracle
import synth


def _torch_weight(w, OC, IC, Kh, Kw):
    # original[ic, oc, kh, kw] = w[oc, (kh*Kw + kw)*IC + ic]
    return w[:, :Kh * Kw * IC].reshape(OC, Kh, Kw, IC).transpose(3, 0, 1, 2).copy()


def _cases():
    out = []
    for (s, p, K, d, op) in itertools.product((1, 2, 3), (0, 1, 2), (1, 2, 3, 4), (1, 2), (0, 1)):
        if op >= max(s, d):
            continue
        H_in, W_in = 5, 4
        H, W = synth.output_hw(H_in, W_in, K, K, s, s, p, p, op, op, d, d)
        if H <= 0 or W <= 0:
            continue
        out.append((s, p, K, d, op))
    return out


CASES = _cases()


@pytest.mark.parametrize("s,p,K,d,op", CASES)
def test_gather_equals_scatter_and_torch(s, p, K, d, op):
    torch = pytest.importorskip("torch")
    N, IC, OC, H_in, W_in = 2, 3, 4, 5, 4
    seed = s * 1000 + p * 100 + K * 10 + d + op * 7
    x = synth.int8_uniform(seed, "tx", (N, IC, H_in, W_in), -128, 127)
    ldw = K * K * IC + 3
    w = synth.int8_uniform(seed, "tw", (OC, ldw), -128, 127)
    izp = int(synth.uniform_int(seed, "tz", (1,), -128, 127)[0])
    H, W = synth.output_hw(H_in, W_in, K, K, s, s, p, p, op, op, d, d)
    g = oracle.conv2d_transposed_acc(x, izp, w, K, K, H, W, (s, s), (p, p), (d, d), "gather")
    sc = oracle.conv2d_transposed_acc(x, izp, w, K, K, H, W, (s, s), (p, p), (d, d), "scatter")
    np.testing.assert_array_equal(g, sc)
    xt = torch.from_numpy(x.astype(np.float64) - izp)
    wt = torch.from_numpy(_torch_weight(w, OC, IC, K, K).astype(np.float64))
    ref = torch.nn.functional.conv_transpose2d(xt, wt, stride=s, padding=p, output_padding=op,
                                               dilation=d).numpy()
    assert ref.shape == g.shape
    np.testing.assert_array_equal(g.astype(np.float64), ref)


def _zp_filled_textbook(x, izp, w, Kh, Kw, H, W, s, p, d):
    """Transposed conv as a direct correlation over the stride-dilated input
    padded by d*(K-1)-p, where every inserted or padded position holds the
    zero-point: those positions then contribute (zp - zp) * w = 0."""
    N, IC, H_in, W_in = x.shape
    OC = w.shape[0]
    ph, pw = d[0] * (Kh - 1) - p[0], d[1] * (Kw - 1) - p[1]
    Hd, Wd = (H_in - 1) * s[0] + 1, (W_in - 1) * s[1] + 1
    big_h, big_w = Hd + 2 * abs(ph) + H + Kh * d[0], Wd + 2 * abs(pw) + W + Kw * d[1]
    filled = np.full((N, IC, big_h, big_w), izp, np.int64)
    oh0, ow0 = abs(ph) + ph, abs(pw) + pw          # where the data starts after padding
    filled[:, :, oh0:oh0 + Hd:s[0], ow0:ow0 + Wd:s[1]] = x
    filled -= izp
    base_h, base_w = abs(ph), abs(pw)
    wt = _torch_weight(w, OC, IC, Kh, Kw).astype(np.int64)    # [IC, OC, Kh, Kw]
    acc = np.zeros((N, OC, H, W), np.int64)
    for kh in range(Kh):
        for kw in range(Kw):
            # flipped kernel tap (Kh-1-kh, Kw-1-kw) reads the window shifted by (kh*d, kw*d)
            win = filled[:, :, base_h + kh * d[0]: base_h + kh * d[0] + H,
                         base_w + kw * d[1]: base_w + kw * d[1] + W]
            tap = wt[:, :, Kh - 1 - kh, Kw - 1 - kw]             # [IC, OC]
            acc += np.einsum("nihw,io->nohw", win, tap)
    return acc


@pytest.mark.parametrize("s,p,K,d,op", CASES[::3])
def test_zero_point_fill_equivalence(s, p, K, d, op):
    N, IC, OC, H_in, W_in = 1, 2, 3, 5, 4
    seed = 77 + s * 13 + p * 5 + K + d * 3 + op
    x = synth.int8_uniform(seed, "zx", (N, IC, H_in, W_in), -128, 127)
    w = synth.int8_uniform(seed, "zw", (OC, K * K * IC), -128, 127)
    izp = -7
    H, W = synth.output_hw(H_in, W_in, K, K, s, s, p, p, op, op, d, d)
    g = oracle.conv2d_transposed_acc(x, izp, w, K, K, H, W, (s, s), (p, p), (d, d))
    ref = _zp_filled_textbook(x, izp, w, K, K, H, W, (s, s), (p, p), (d, d))
    np.testing.assert_array_equal(g.astype(np.int64), ref)


def test_1x1_stride1_equals_linear():
    N, IC, OC, H, W = 2, 24, 8, 3, 5
    x = synth.int8_uniform(3, "ox", (N, IC, H, W), -128, 127)
    w = synth.int8_uniform(3, "ow", (OC, IC), -127, 127)
    ws = synth.uniform_float(3, "os", (OC,), 0.002, 0.01)
    b = synth.normal(3, "ob", (OC,), 0.0, 0.1)
    conv = oracle.conv2d_transposed(x, 0.02, 4, w, 1, 1, ws, b, 0.08, -1, H, W, (1, 1), (0, 0))
    x_rows = x.transpose(0, 2, 3, 1).reshape(N * H * W, IC)
    lin = oracle.linear(x_rows, 0.02, 4, w, ws, b, 0.08, -1)
    np.testing.assert_array_equal(conv, lin.reshape(N, H, W, OC).transpose(0, 3, 1, 2))


def test_outputs_without_taps_equal_requantized_bias():
    # stride 3, 1x1 kernel: only positions with oh % 3 == 0 and ow % 3 == 0 get a tap
    N, IC, OC, H_in, W_in = 1, 4, 2, 3, 3
    x = synth.int8_uniform(9, "nx", (N, IC, H_in, W_in), -128, 127)
    w = synth.int8_uniform(9, "nw", (OC, IC), -127, 127)
    ws = np.array([0.004, 0.009], np.float32)
    b = np.array([0.33, -0.71], np.float32)
    H, W = synth.output_hw(H_in, W_in, 1, 1, 3, 3, 0, 0, 2, 2)
    out = oracle.conv2d_transposed(x, 0.02, 4, w, 1, 1, ws, b, 0.08, 3, H, W, (3, 3), (0, 0))
    empty = oracle.requantize(np.zeros((1, OC), np.int32), 0.02, ws, b, 0.08, 3)[0]
    for oc in range(OC):
        for oh in range(H):
            for ow in range(W):
                if oh % 3 or ow % 3:
                    assert out[0, oc, oh, ow] == empty[oc]
    # hand check: rne(0.33 / 0.08) + 3 = rne(4.125) + 3 = 7; rne(-0.71 / 0.08) + 3 = -9 + 3 = -6
    assert empty.tolist() == [7, -6]


def test_full_op_equals_acc_then_requantize_and_ignores_row_padding():
    N, IC, OC, H_in, W_in, K, s, p = 2, 5, 6, 4, 4, 3, 2, 1
    H, W = synth.output_hw(H_in, W_in, K, K, s, s, p, p, 1, 1)
    x = synth.int8_uniform(4, "fx", (N, IC, H_in, W_in), -128, 127)
    w = synth.int8_uniform(4, "fw", (OC, K * K * IC), -127, 127)
    ws = synth.uniform_float(4, "fs", (OC,), 0.002, 0.01)
    b = synth.normal(4, "fb", (OC,), 0.0, 0.1)
    full = oracle.conv2d_transposed(x, 0.02, -7, w, K, K, ws, b, 0.15, 2, H, W, (s, s), (p, p))
    acc = oracle.conv2d_transposed_acc(x, -7, w, K, K, H, W, (s, s), (p, p))
    rq = oracle.requantize(acc.transpose(0, 2, 3, 1).reshape(-1, OC), 0.02, ws, b, 0.15, 2)
    np.testing.assert_array_equal(full, rq.reshape(N, H, W, OC).transpose(0, 3, 1, 2))
    # padding columns of a wider weight row are never read
    wide = np.concatenate([w, np.full((OC, 13), 99, np.int8)], axis=1)
    np.testing.assert_array_equal(
        full, oracle.conv2d_transposed(x, 0.02, -7, wide, K, K, ws, b, 0.15, 2, H, W, (s, s),
                                       (p, p)))
