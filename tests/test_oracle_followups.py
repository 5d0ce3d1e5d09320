"""Pins for the oracle's follow-up forms (CPU only).

Sources: "Add q8ta_linear op" (PR #21197) and "Add q8ta_conv2d_transposed op"
(PR #21205), Constraints paragraphs: a relu-fused activation, transposed
convolution with groups > 1 and dilation != 1 are the named fail-loud
follow-ups; the Problem paragraph of the transposed-convolution page names
the general q8ta_conv2d whose scaffold and [OC, Kh*Kw*IC] weight layout it
reuses.

Readings (the pages fix none of these details):
* relu raises the dequantized value v to 0 before requantization.  As
  v * inv_out is monotone and rint(0) = 0, that equals max(q, zp) on the
  output, which the first tests check on every element;
* groups g: output channel oc of group j = oc // (OC/g) sums over input
  channels j*(IC/g) .. (j+1)*(IC/g) - 1 with weight[oc, (kh*Kw+kw)*(IC/g) +
  icl] = original[j*(IC/g) + icl, oc - j*(OC/g), kh, kw] (PyTorch's grouped
  ConvTranspose2d weight [IC, OC/g, Kh, Kw]); checked against torch's float64
  conv_transpose2d(groups=g);
* q8ta_conv2d: ih = oh*stride - pad + kh*dil (the direct correlation),
  weight[oc, (kh*Kw+kw)*(IC/g) + icl] = original[oc, icl, kh, kw]; checked
  against torch's float64 conv2d, a zero-point-padded form without bounds
  tests, the 1x1 case reducing to q8ta_linear, and the adjoint identity
  <conv2d(x), y> = <x, conv_transpose(y)>.
"""
import itertools

import numpy as np
import pytest

import oracle
import synth


# ----------------------------------------------------------------- relu

@pytest.mark.parametrize("ozp", [-128, -7, 0, 5, 127])
def test_relu_is_max_with_the_output_zero_point(ozp):
    rows, N = 64, 48
    acc = synth.uniform_int(5, "racc", (rows, N), -2_000_000, 2_000_000).astype(np.int32)
    acc[0, :] = 0
    acc[1, :] = np.arange(-24, 24)
    ws = synth.uniform_float(5, "rws", (N,), 0.001, 0.01)
    b = synth.normal(5, "rb", (N,), 0.0, 0.3)
    none = oracle.requantize(acc, 0.05, ws, b, 0.2, ozp)
    relu = oracle.requantize(acc, 0.05, ws, b, 0.2, ozp, activation="relu")
    np.testing.assert_array_equal(relu, np.maximum(none, ozp))
    assert (relu == none).any()
    if ozp > -128:          # at -128 the output floor is the clamp's own
        assert (relu != none).any()


def test_relu_hand_values():
    # s_in = ws = output_scale = 1, no bias: v = acc exactly
    acc = np.array([[-300, -5, 0, 3, 200]], np.int32)
    ws = np.ones(5, np.float32)
    got = oracle.requantize(acc, 1.0, ws, None, 1.0, 10, activation="relu")
    assert got.tolist() == [[10, 10, 10, 13, 127]]
    got = oracle.requantize(acc, 1.0, ws, None, 1.0, -20, activation="relu")
    assert got.tolist() == [[-20, -20, -20, -17, 127]]
    assert oracle.requantize(acc, 1.0, ws, None, 1.0, -20).tolist() == [[-128, -25, -20, -17, 127]]


def test_relu_through_linear_and_conv_t():
    x, w, ws, b = synth.linear_inputs(6, 9, 40, 12, x_kind="int8",
                                      p=dict(ws_lo=0.002, ws_hi=0.01, b_mean=0.0, b_var=0.1))
    none = oracle.linear(x, 0.03, 2, w, ws, b, 0.1, -3)
    relu = oracle.linear(x, 0.03, 2, w, ws, b, 0.1, -3, activation="relu")
    np.testing.assert_array_equal(relu, np.maximum(none, -3))
    xc = synth.int8_uniform(7, "rx", (1, 3, 5, 4), -128, 127)
    wc = synth.int8_uniform(7, "rw", (4, 27), -127, 127)
    H, W = synth.output_hw(5, 4, 3, 3, 2, 2, 1, 1, 1, 1)
    args = (xc, 0.02, 4, wc, 3, 3, ws[:4], b[:4], 0.08, 1, H, W, (2, 2), (1, 1))
    np.testing.assert_array_equal(oracle.conv2d_transposed(*args, activation="relu"),
                                  np.maximum(oracle.conv2d_transposed(*args), 1))
    with pytest.raises(ValueError):
        oracle.linear(x, 0.03, 2, w, ws, b, 0.1, -3, activation="gelu")


# --------------------------------------------------------- grouped conv_t

def _torch_t_weight(w, OC, IC, Kh, Kw, g):
    """original [IC, OC/g, Kh, Kw] from the reshaped [OC, Kh*Kw*IC/g]."""
    ICg, OCg = IC // g, OC // g
    r = w[:, :Kh * Kw * ICg].reshape(OC, Kh, Kw, ICg)
    out = np.zeros((IC, OCg, Kh, Kw), np.float64)
    for oc in range(OC):
        j, ocl = divmod(oc, OCg)
        out[j * ICg:(j + 1) * ICg, ocl] = r[oc].transpose(2, 0, 1)
    return out


@pytest.mark.parametrize("g,s,p,K,d", [(2, 2, 1, 3, 1), (3, 1, 0, 2, 2), (6, 2, 0, 3, 2),
                                       (2, 3, 2, 4, 1), (1, 2, 1, 3, 3)])
def test_grouped_conv_t_equals_torch_and_scatter(g, s, p, K, d):
    torch = pytest.importorskip("torch")
    N, IC, OC, H_in, W_in = 2, 6, 12, 5, 4
    seed = 100 * g + 10 * s + K + d
    x = synth.int8_uniform(seed, "gx", (N, IC, H_in, W_in), -128, 127)
    w = synth.int8_uniform(seed, "gw", (OC, K * K * (IC // g) + 2), -128, 127)
    izp = int(synth.uniform_int(seed, "gz", (1,), -128, 127)[0])
    H, W = synth.output_hw(H_in, W_in, K, K, s, s, p, p, 0, 0, d, d)
    gat = oracle.conv2d_transposed_acc(x, izp, w, K, K, H, W, (s, s), (p, p), (d, d), groups=g)
    sca = oracle.conv2d_transposed_acc(x, izp, w, K, K, H, W, (s, s), (p, p), (d, d),
                                       form="scatter", groups=g)
    np.testing.assert_array_equal(gat, sca)
    ref = torch.nn.functional.conv_transpose2d(
        torch.from_numpy(x.astype(np.float64) - izp),
        torch.from_numpy(_torch_t_weight(w, OC, IC, K, K, g)), stride=s, padding=p, dilation=d,
        groups=g).numpy()
    np.testing.assert_array_equal(gat.astype(np.float64), ref)


# ------------------------------------------------------------- conv2d

def _torch_weight(w, OC, IC, Kh, Kw, g):
    """original [OC, IC/g, Kh, Kw] from the reshaped [OC, Kh*Kw*IC/g]."""
    ICg = IC // g
    return w[:, :Kh * Kw * ICg].reshape(OC, Kh, Kw, ICg).transpose(0, 3, 1, 2).astype(np.float64)


def _out_hw(H_in, W_in, K, s, p, d):
    return ((H_in + 2 * p - d * (K - 1) - 1) // s + 1, (W_in + 2 * p - d * (K - 1) - 1) // s + 1)


CONV2D_CASES = [c for c in itertools.product((1, 2, 3), (0, 1, 2), (1, 2, 3), (1, 2), (1, 3))
                if _out_hw(7, 6, c[2], c[0], c[1], c[3])[0] > 0 and
                _out_hw(7, 6, c[2], c[0], c[1], c[3])[1] > 0]


@pytest.mark.parametrize("s,p,K,d,g", CONV2D_CASES)
def test_conv2d_equals_torch(s, p, K, d, g):
    torch = pytest.importorskip("torch")
    N, IC, OC, H_in, W_in = 2, 6, 9, 7, 6
    seed = 1000 + 97 * s + 31 * p + 7 * K + 3 * d + g
    x = synth.int8_uniform(seed, "cx", (N, IC, H_in, W_in), -128, 127)
    w = synth.int8_uniform(seed, "cw", (OC, K * K * (IC // g) + 1), -128, 127)
    izp = int(synth.uniform_int(seed, "cz", (1,), -128, 127)[0])
    H, W = _out_hw(H_in, W_in, K, s, p, d)
    got = oracle.conv2d_acc(x, izp, w, K, K, H, W, (s, s), (p, p), (d, d), groups=g)
    ref = torch.nn.functional.conv2d(torch.from_numpy(x.astype(np.float64) - izp),
                                     torch.from_numpy(_torch_weight(w, OC, IC, K, K, g)),
                                     stride=s, padding=p, dilation=d, groups=g).numpy()
    np.testing.assert_array_equal(got.astype(np.float64), ref)


def test_conv2d_zero_point_padding_form():
    """Pad the input with the zero point and correlate with no bounds tests:
    padded positions contribute (zp - zp) * w = 0."""
    N, IC, OC, H_in, W_in, K, s, p, d = 1, 4, 5, 6, 7, 3, 2, 2, 2
    x = synth.int8_uniform(21, "px", (N, IC, H_in, W_in), -128, 127)
    w = synth.int8_uniform(21, "pw", (OC, K * K * IC), -128, 127)
    izp = -9
    H, W = _out_hw(H_in, W_in, K, s, p, d)
    xp = np.full((N, IC, H_in + 2 * p, W_in + 2 * p), izp, np.int64)
    xp[:, :, p:p + H_in, p:p + W_in] = x
    wt = w.reshape(OC, K, K, IC).astype(np.int64)
    ref = np.zeros((N, OC, H, W), np.int64)
    for oh in range(H):
        for ow in range(W):
            for kh in range(K):
                for kw in range(K):
                    col = xp[:, :, oh * s + kh * d, ow * s + kw * d] - izp     # [N, IC]
                    ref[:, :, oh, ow] += col @ wt[:, kh, kw, :].T
    got = oracle.conv2d_acc(x, izp, w, K, K, H, W, (s, s), (p, p), (d, d))
    np.testing.assert_array_equal(got.astype(np.int64), ref)


def test_conv2d_1x1_equals_linear():
    N, IC, OC, H, W = 2, 24, 8, 3, 5
    x = synth.int8_uniform(3, "lx", (N, IC, H, W), -128, 127)
    w = synth.int8_uniform(3, "lw", (OC, IC), -127, 127)
    ws = synth.uniform_float(3, "ls", (OC,), 0.002, 0.01)
    b = synth.normal(3, "lb", (OC,), 0.0, 0.1)
    conv = oracle.conv2d(x, 0.02, 4, w, 1, 1, ws, b, 0.08, -1, H, W, (1, 1), (0, 0))
    lin = oracle.linear(x.transpose(0, 2, 3, 1).reshape(N * H * W, IC), 0.02, 4, w, ws, b, 0.08, -1)
    np.testing.assert_array_equal(conv, lin.reshape(N, H, W, OC).transpose(0, 3, 1, 2))


@pytest.mark.parametrize("s,p,K,d,g", [(2, 1, 3, 1, 1), (1, 0, 2, 2, 2), (3, 2, 3, 1, 3)])
def test_conv2d_and_conv_t_are_adjoint(s, p, K, d, g):
    """With zero points 0: <conv2d(x; w), y> = <x, conv_t(y; w')>, w' being
    the same kernel seen from the output side (the roles of IC and OC swap)."""
    N, C_in, C_out, H_in, W_in = 1, 6, 3 * g, 8, 7
    x = synth.int8_uniform(50 + s, "ax", (N, C_in, H_in, W_in), -128, 127)
    w = synth.int8_uniform(50 + s, "aw", (C_out, K * K * (C_in // g)), -128, 127)
    H, W = _out_hw(H_in, W_in, K, s, p, d)
    y = synth.int8_uniform(50 + s, "ay", (N, C_out, H, W), -128, 127)
    fwd = oracle.conv2d_acc(x, 0, w, K, K, H, W, (s, s), (p, p), (d, d), groups=g)
    # conv_t weight [C_in, K*K*C_out/g]: w'[ic, (kh*K+kw)*ocg + ocl] = w[j*ocg + ocl, (kh*K+kw)*icg + icl]
    icg, ocg = C_in // g, C_out // g
    wr = w.reshape(C_out, K, K, icg)
    wt = np.zeros((C_in, K, K, ocg), np.int8)
    for ic in range(C_in):
        j, icl = divmod(ic, icg)
        wt[ic] = wr[j * ocg:(j + 1) * ocg, :, :, icl].transpose(1, 2, 0)
    back = oracle.conv2d_transposed_acc(y, 0, wt.reshape(C_in, -1), K, K, H_in, W_in, (s, s),
                                        (p, p), (d, d), groups=g)
    lhs = int((fwd.astype(np.int64) * y).sum())
    rhs = int((x.astype(np.int64) * back).sum())
    assert lhs == rhs
