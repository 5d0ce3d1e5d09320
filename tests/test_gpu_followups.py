"""GPU parity of the follow-up forms: relu, dilated and grouped transposed
convolution, the packed convolution weights and the direct q8ta_conv2d.

Every result is compared with the CPU oracle bit for bit (int8 outputs and
int32 accumulators).  Shapes span several tiles with ragged edges and cover
the degenerate cases: phases with no tap (stride above the kernel, and
dilations sharing a factor with the stride), depthwise groups (one channel
per group, padded to a 64-channel block), windows lying wholly in the
padding, the largest element stride (8).
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


# ----------------------------------------------------------------- relu

@pytest.mark.parametrize("M,K,N,izp,ozp", [(1, 4096, 256, 3, 5), (1, 100, 12, -2, -128),
                                           (64, 320, 96, 0, 7), (300, 520, 1040, -9, -3)])
def test_linear_relu(M, K, N, izp, ozp):
    x, w, ws, b = synth.linear_inputs(M + K + N, M, K, N, x_kind="int8", p=P)
    ref = oracle.linear(x, 0.03, izp, w, ws, b, 0.05, ozp, activation="relu")
    assert (ref == ozp).any() and (ref > ozp).any()
    got = H(q8.linear(T(x), 0.03, izp, T(w), None, T(ws), T(b), 0.05, ozp, activation="relu"))
    np.testing.assert_array_equal(got, ref)
    if M > 1:
        packed = q8.pack_weight(T(w))
        got = H(q8.linear_packed(T(x), 0.03, izp, packed, T(ws), T(b), 0.05, ozp,
                                 activation="relu"))
        np.testing.assert_array_equal(got, ref)


def test_conv_t_relu():
    d = dict(N=2, IC=64, H_in=9, W_in=8, OC=36, Kh=4, Kw=4)
    x, w, ws, b = synth.conv_t_inputs(31, d, dict(in_scale=0.02, **P))
    ref = oracle.conv2d_transposed(x, 0.02, 3, w, 4, 4, ws, b, 0.1, -4, 18, 16, (2, 2), (1, 1),
                                   activation="relu")
    got = H(q8.conv2d_transposed(T(x), 0.02, 3, T(w), None, T(ws), T(b), 0.1, -4, 4, stride=2,
                                 padding=1, activation="relu", output_size=(18, 16)))
    np.testing.assert_array_equal(got, ref)


# ------------------------------------------- dilated / grouped conv_t

CONV_T_CASES = [
    # seed, N, IC, H, W, OC, K, s, p, d, g, izp, ozp, (H_out, W_out)
    (41, 1, 16, 6, 7, 8, 3, 2, 1, 2, 1, -5, 1, (15, 16)),     # gcd(d, s) = 2: phases without taps
    (42, 2, 24, 5, 6, 12, 3, 3, 2, 2, 1, 7, -2, (13, 16)),    # d, s coprime
    (43, 1, 64, 8, 8, 64, 2, 2, 0, 3, 1, 0, 0, (18, 20)),
    (44, 1, 32, 7, 5, 48, 3, 2, 1, 1, 2, -128, 3, (14, 12)),  # groups 2
    (45, 2, 128, 6, 6, 128, 3, 2, 1, 1, 4, 9, -1, (12, 12)),  # groups 4, 32 channels each
    (46, 1, 16, 9, 8, 16, 3, 1, 1, 2, 16, 2, 4, (13, 12)),    # depthwise, dilated
    (47, 2, 96, 10, 12, 64, 4, 2, 1, 2, 2, -3, 0, (24, 28)),  # 48 channels per group, padded
]


@pytest.mark.parametrize("case", CONV_T_CASES)
def test_conv_t_dilated_grouped(case):
    seed, N, IC, H_in, W_in, OC, K, s, p, dil, g, izp, ozp, (Ho, Wo) = case
    x = synth.int8_uniform(seed, "x", (N, IC, H_in, W_in), -128, 127)
    w = synth.int8_uniform(seed, "w", (OC, K * K * (IC // g)), -127, 127)
    ws = synth.uniform_float(seed, "ws", (OC,), 0.002, 0.01)
    b = synth.normal(seed, "b", (OC,), 0.0, 0.1)
    ref = oracle.conv2d_transposed(x, 0.02, izp, w, K, K, ws, b, 0.15, ozp, Ho, Wo, (s, s),
                                   (p, p), (dil, dil), groups=g)
    got = H(q8.conv2d_transposed(T(x), 0.02, izp, T(w), None, T(ws), T(b), 0.15, ozp, K,
                                 stride=s, padding=p, dilation=dil, groups=g, output_size=(Ho, Wo)))
    np.testing.assert_array_equal(got, ref)
    acc_ref = oracle.conv2d_transposed_acc(x, izp, w, K, K, Ho, Wo, (s, s), (p, p), (dil, dil),
                                           groups=g)
    acc = H(q8.conv2d_transposed_acc32(T(x), izp, T(w), K, (Ho, Wo), stride=s, padding=p,
                                       dilation=dil, groups=g))
    np.testing.assert_array_equal(acc, acc_ref)
    packed = q8.pack_conv2d_transposed_weight(T(w), IC, K, groups=g)
    got = H(q8.conv2d_transposed_packed(T(x), 0.02, izp, packed, T(ws), T(b), 0.15, ozp, stride=s,
                                        padding=p, dilation=dil, output_size=(Ho, Wo)))
    np.testing.assert_array_equal(got, ref)


# ------------------------------------------------------------- conv2d

CONV2D_CASES = [
    # seed, N, IC, H, W, OC, K, s, p, d, g, izp, ozp
    (51, 1, 3, 9, 8, 4, 3, 1, 1, 1, 1, -7, 2),        # tiny, one partial tile
    (52, 2, 64, 20, 16, 36, 3, 1, 1, 1, 1, 4, 0),     # staged rows
    (53, 1, 70, 17, 18, 132, 3, 2, 1, 1, 1, -128, -3),
    (54, 1, 16, 15, 31, 8, 1, 2, 0, 1, 1, 127, 1),    # pointwise, strided
    (55, 2, 32, 24, 26, 48, 5, 2, 2, 1, 2, 0, 0),     # groups 2
    (56, 1, 64, 16, 16, 64, 3, 1, 2, 2, 64, 9, -9),   # depthwise, dilated
    (57, 1, 24, 33, 40, 16, 3, 4, 1, 1, 1, -1, 5),    # stride 4
    (58, 1, 8, 40, 72, 12, 2, 8, 0, 1, 1, 2, 2),      # stride 8 (the TMA limit)
    (59, 1, 8, 10, 10, 12, 3, 1, 4, 1, 1, 3, -1),     # windows wholly in the padding
    (60, 2, 128, 12, 300, 256, 3, 1, 1, 1, 1, -3, 3),  # W_out > 128: several w tiles
]


def _conv2d_inputs(case):
    seed, N, IC, H_in, W_in, OC, K, s, p, d, g, izp, ozp = case
    x = synth.int8_uniform(seed, "x", (N, IC, H_in, W_in), -128, 127)
    w = synth.int8_uniform(seed, "w", (OC, K * K * (IC // g)), -127, 127)
    ws = synth.uniform_float(seed, "ws", (OC,), 0.002, 0.01)
    b = synth.normal(seed, "b", (OC,), 0.0, 0.1)
    Ho, Wo = q8.conv2d_output_size(H_in, W_in, K, s, p, d)
    Wo -= Wo % 4                              # the W_out % 4 guard: drop the last columns
    return x, w, ws, b, Ho, Wo


@pytest.mark.parametrize("case", CONV2D_CASES)
def test_conv2d_matches_oracle(case):
    seed, N, IC, H_in, W_in, OC, K, s, p, d, g, izp, ozp = case
    x, w, ws, b, Ho, Wo = _conv2d_inputs(case)
    ref = oracle.conv2d(x, 0.02, izp, w, K, K, ws, b, 0.15, ozp, Ho, Wo, (s, s), (p, p), (d, d),
                        groups=g)
    got = H(q8.conv2d(T(x), 0.02, izp, T(w), T(ws), T(b), 0.15, ozp, K, stride=s, padding=p,
                      dilation=d, groups=g, output_size=(Ho, Wo)))
    np.testing.assert_array_equal(got, ref)
    acc_ref = oracle.conv2d_acc(x, izp, w, K, K, Ho, Wo, (s, s), (p, p), (d, d), groups=g)
    acc = H(q8.conv2d_acc32(T(x), izp, T(w), K, (Ho, Wo), stride=s, padding=p, dilation=d,
                            groups=g))
    np.testing.assert_array_equal(acc, acc_ref)


@pytest.mark.parametrize("case", [CONV2D_CASES[1], CONV2D_CASES[4]])
def test_conv2d_packed_and_relu(case):
    seed, N, IC, H_in, W_in, OC, K, s, p, d, g, izp, ozp = case
    x, w, ws, b, Ho, Wo = _conv2d_inputs(case)
    packed = q8.pack_conv2d_weight(T(w), IC, K, groups=g)
    for act in ("none", "relu"):
        ref = oracle.conv2d(x, 0.02, izp, w, K, K, ws, b, 0.15, ozp, Ho, Wo, (s, s), (p, p),
                            (d, d), groups=g, activation=act)
        got = H(q8.conv2d_packed(T(x), 0.02, izp, packed, T(ws), T(b), 0.15, ozp, stride=s,
                                 padding=p, dilation=d, activation=act, output_size=(Ho, Wo)))
        np.testing.assert_array_equal(got, ref)


def test_conv2d_acc32_exact_at_the_chunk_bound():
    """|x - zp| = 128 (zp = 0) and w = -128 over 9 taps x 512 channels: every
    exact chunk of 1024 products sums to 2^24."""
    N, IC, H_in, W_in, OC, K = 1, 512, 8, 8, 64, 3
    x = np.full((N, IC, H_in, W_in), -128, np.int8)
    w = np.full((OC, K * K * IC), -128, np.int8)
    w[32:, :] = synth.int8_uniform(61, "cw", (OC - 32, K * K * IC), -128, 127)
    ref = oracle.conv2d_acc(x, 0, w, K, K, 8, 8, (1, 1), (1, 1))
    got = H(q8.conv2d_acc32(T(x), 0, T(w), K, (8, 8), stride=1, padding=1))
    np.testing.assert_array_equal(got, ref)


# ------------------------------------------------- back-to-back launches

def test_dependent_launches_back_to_back():
    """Every kernel starts under the previous one's tail (programmatic
    dependent launch) and waits for it before touching global memory.  A
    chain where each op consumes the previous op's output, enqueued without
    host synchronisation, checks that ordering: quantize -> linear (reading
    the quantized activations) -> linear again (reading that output) ->
    gemv -> conv2d on the reshaped result, then the same chain again into
    the same buffers."""
    M, K, N = 256, 512, 512
    xf = synth.normal(71, "x", (M, K), 0.0, 3.0)
    w1 = synth.int8_uniform(71, "w1", (N, K), -127, 127)
    w2 = synth.int8_uniform(71, "w2", (N, N), -127, 127)
    ws1 = synth.uniform_float(71, "s1", (N,), 0.001, 0.005)
    ws2 = synth.uniform_float(71, "s2", (N,), 0.001, 0.005)
    b = synth.normal(71, "b", (N,), 0.0, 0.1)
    g_w = synth.int8_uniform(71, "gw", (64, N), -127, 127)
    cw = synth.int8_uniform(71, "cw", (8, 9 * 16), -127, 127)
    c_ws = synth.uniform_float(71, "cs", (8,), 0.002, 0.01)
    # oracle chain
    xq = oracle.quantize_per_tensor(xf, 0.03, -5)
    y1 = oracle.linear(xq, 0.03, -5, w1, ws1, b, 0.1, 1)
    y2 = oracle.linear(y1, 0.1, 1, w2, ws2, b, 0.2, -2, activation="relu")
    g = oracle.linear(y2[:1], 0.2, -2, g_w, ws1[:64], b[:64], 0.5, 0)
    ximg = y2.reshape(8, 16, 32, 32)[:1]
    c = oracle.conv2d(ximg, 0.2, -2, cw, 3, 3, c_ws, None, 0.3, 3, 32, 32, (1, 1), (1, 1))
    # GPU chain, twice into the same buffers, one stream, no host sync inside
    Txf, Tw1, Tw2, Tgw, Tcw = T(xf), T(w1), T(w2), T(g_w), T(cw)
    Tws1, Tws2, Tb, Tcws = T(ws1), T(ws2), T(b), T(c_ws)
    p1, p2 = q8.pack_weight(Tw1), q8.pack_weight(Tw2)
    q_out = torch.empty((M, K), dtype=torch.int8, device=DEV)
    y1_d = torch.empty((M, N), dtype=torch.int8, device=DEV)
    y2_d = torch.empty((M, N), dtype=torch.int8, device=DEV)
    g_d = torch.empty((1, 64), dtype=torch.int8, device=DEV)
    c_d = torch.empty((1, 8, 32, 32), dtype=torch.int8, device=DEV)
    for _ in range(2):
        q8.quantize_per_tensor(Txf, 0.03, -5, out=q_out)
        q8.linear_packed(q_out, 0.03, -5, p1, Tws1, Tb, 0.1, 1, out=y1_d)
        q8.linear_packed(y1_d, 0.1, 1, p2, Tws2, Tb, 0.2, -2, activation="relu", out=y2_d)
        q8.linear_gemv(y2_d[:1], 0.2, -2, Tgw, None, Tws1[:64], Tb[:64], 0.5, 0, out=g_d)
        q8.conv2d(y2_d.view(8, 16, 32, 32)[:1], 0.2, -2, Tcw, Tcws, None, 0.3, 3, 3, padding=1,
                  out=c_d)
    np.testing.assert_array_equal(H(q_out), xq)
    np.testing.assert_array_equal(H(y1_d), y1)
    np.testing.assert_array_equal(H(y2_d), y2)
    np.testing.assert_array_equal(H(g_d), g)
    np.testing.assert_array_equal(H(c_d), c)
