"""GPU parity: the CUDA path against the CPU oracle, element by element.

Integer results (int8 outputs, int32 accumulators) must be bit-exact.  Sizes
span several tiles with ragged tails; the five benchmark workloads run at
full size on the GPU and are compared with the oracle on every output
(the large ones with the oracle's slices run on all host cores).
"""
import numpy as np
import pytest
import torch

import oracle
import parallel_oracle
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


# --------------------------------------------------------------- quantize

@pytest.mark.parametrize("n", [4, 12, 16, 1000, 4096 + 4, (1 << 20) + 12])
@pytest.mark.parametrize("scale,zp,var", [(0.03, -5, 3.0), (0.02, 3, 1.0), (1.0, 0, 4e4)])
def test_quantize_matches_oracle(n, scale, zp, var):
    x = synth.normal(n, "gq", (n,), 0.0, var)
    got = H(q8.quantize_per_tensor(T(x), scale, zp))
    np.testing.assert_array_equal(got, oracle.quantize_per_tensor(x, scale, zp))


def test_quantize_special_values_and_unaligned_view():
    x = np.array([0.5, 1.5, 2.5, -0.5, -2.5, np.inf, -np.inf, 1e30, -1e30, 127.5, -128.5, 0.0],
                 np.float32)
    np.testing.assert_array_equal(H(q8.quantize_per_tensor(T(x), 1.0, 0)),
                                  oracle.quantize_per_tensor(x, 1.0, 0))
    # a view starting 4 bytes into an allocation takes the scalar path
    base = synth.normal(7, "gu", (4101,), 0.0, 3.0)
    xt = T(base)[1:]
    assert xt.data_ptr() % 16 != 0
    got = H(q8.quantize_per_tensor(xt, 0.03, -5))
    np.testing.assert_array_equal(got, oracle.quantize_per_tensor(base[1:], 0.03, -5))


def test_quantize_64Mi_full():
    wl = synth.CONFIGS["quantize_64Mi"]
    p = wl.params
    x = synth.normal(wl.seed, "x", (wl.dims["numel"],), p["x_mean"], p["x_var"])
    got = H(q8.quantize_per_tensor(T(x), p["in_scale"], p["in_zp"]))
    ref = oracle.quantize_per_tensor(x, p["in_scale"], p["in_zp"])
    np.testing.assert_array_equal(got, ref)
    sat = np.count_nonzero((ref == 127) | (ref == -128)) / ref.size
    assert 0.01 < sat < 0.05          # "~2% saturating"


def test_dequantize_matches_oracle():
    q = synth.int8_uniform(3, "dq", (4096 + 8,), -128, 127)
    got = H(q8.dequantize_per_tensor(T(q), 0.037, -3))
    np.testing.assert_array_equal(got.view(np.uint32),
                                  oracle.dequantize_per_tensor(q, 0.037, -3).view(np.uint32))


# --------------------------------------------------------------- gemv

def test_gemv_1x4096x4096_full():
    wl = synth.CONFIGS["gemv_1x4096x4096"]
    d, p = wl.dims, wl.params
    x, w, ws, b = synth.linear_inputs(wl.seed, 1, d["K"], d["N"], x_kind="int8", p=p)
    got = H(q8.linear_gemv(T(x), p["in_scale"], p["in_zp"], T(w), None, T(ws), T(b),
                           p["out_scale"], p["out_zp"]))
    ref = oracle.linear(x, p["in_scale"], p["in_zp"], w, ws, b, p["out_scale"], p["out_zp"])
    np.testing.assert_array_equal(got, ref)
    # the same through q8_linear, which dispatches M == 1 to the gemv kernel
    got2 = H(q8.linear(T(x), p["in_scale"], p["in_zp"], T(w), None, T(ws), T(b), p["out_scale"],
                       p["out_zp"]))
    np.testing.assert_array_equal(got2, ref)


# K % 16 == 0 takes 16-byte loads (up to K = 16384 here, N = 36 and 1004
# leaving partial blocks of four rows), K % 4 == 0 4-byte loads.
@pytest.mark.parametrize("K,N,izp", [(4, 4, 0), (20, 8, -128), (64, 36, 127), (100, 12, 5),
                                     (4096 + 16, 8, -7), (1028, 40, 3), (16, 4, 0),
                                     (2048, 1004, 3), (4096 + 64, 300, 17), (8192, 20, -100),
                                     (12288, 8, -128), (16384, 12, 127)])
def test_gemv_ragged(K, N, izp):
    p = dict(ws_lo=0.002, ws_hi=0.01, b_mean=0.0, b_var=0.1)
    x, w, ws, b = synth.linear_inputs(K + N, 1, K, N, x_kind="int8", p=p)
    got = H(q8.linear_gemv(T(x), 0.02, izp, T(w), None, T(ws), T(b), 0.07, -2))
    np.testing.assert_array_equal(got, oracle.linear(x, 0.02, izp, w, ws, b, 0.07, -2))
    got_nb = H(q8.linear_gemv(T(x), 0.02, izp, T(w), None, T(ws), None, 0.07, -2))
    np.testing.assert_array_equal(got_nb, oracle.linear(x, 0.02, izp, w, ws, None, 0.07, -2))


# The gemv from a packed weight (its first 4 KB of each row read before the
# launch dependency wait, 16 rows per block): K % 16 == 0 up to one round,
# several rounds (K > 4096, a ragged last round), N not a multiple of 16,
# and K % 16 != 0 (the host falls back to the plain kernel).
@pytest.mark.parametrize("K,N,izp", [(16, 4, 0), (4096, 4096, 0), (64, 36, 127), (1028, 40, 3),
                                     (4096 + 16, 8, -7), (8192, 20, -100), (16384, 12, 127),
                                     (2048, 1004, 3), (100, 12, 5), (3 * 4096 + 48, 36, 1)])
def test_gemv_packed_matches_oracle(K, N, izp):
    p = dict(ws_lo=0.002, ws_hi=0.01, b_mean=0.0, b_var=0.1)
    x, w, ws, b = synth.linear_inputs(2 * K + N, 1, K, N, x_kind="int8", p=p)
    packed = q8.pack_gemv_weight(T(w))
    got = H(q8.linear_gemv_packed(T(x), 0.02, izp, packed, T(ws), T(b), 0.07, -2))
    np.testing.assert_array_equal(got, oracle.linear(x, 0.02, izp, w, ws, b, 0.07, -2))
    got = H(q8.linear_gemv_packed(T(x), 0.02, izp, packed, T(ws), None, 0.07, -2,
                                  activation="relu"))
    np.testing.assert_array_equal(got, oracle.linear(x, 0.02, izp, w, ws, None, 0.07, -2,
                                                     activation="relu"))


def test_gemv_packed_chain_of_layers():
    """Layers back to back with no host sync, each reading the previous
    layer's output as its input (the decode pattern the early weight read
    serves): every layer's output equals the oracle's chain."""
    K = N = 1024
    p = dict(ws_lo=0.002, ws_hi=0.01, b_mean=0.0, b_var=0.1)
    x0 = synth.int8_uniform(90, "cx", (1, K), -128, 127)
    layers = [synth.linear_inputs(91 + i, 1, K, N, x_kind="int8", p=p)[1:] for i in range(6)]
    packs = [(q8.pack_gemv_weight(T(w)), T(ws), T(b)) for w, ws, b in layers]
    xt = T(x0)
    outs = []
    for pk, ws, b in packs:
        xt = q8.linear_gemv_packed(xt, 0.05, 1, pk, ws, b, 0.05, 1)
        outs.append(xt)
    torch.cuda.synchronize()
    x = x0
    for (w, ws, b), o in zip(layers, outs):
        x = oracle.linear(x, 0.05, 1, w, ws, b, 0.05, 1)
        np.testing.assert_array_equal(o.cpu().numpy(), x)


# --------------------------------------------------------------- linear

# The last three rows pick the 224-, 240- and 256-column pair tiles on a
# 152-SM GPU (the widths that fill the last wave best); the others use the
# 192-column pair tile or one CTA per tile.  Odd k-block counts leave a
# zero-filled half stage.
LINEAR_SHAPES = [(2, 4, 4, 0), (8, 64, 32, 3), (130, 200, 36, -128), (257, 520, 260, 127),
                 (129, 1040, 516, -5), (300, 4096, 136, 1), (64, 1536, 64, -100),
                 (257, 192, 7300, 77), (257, 136, 8516, -3), (257, 520, 9124, 0)]


@pytest.mark.parametrize("M,K,N,izp", LINEAR_SHAPES)
def test_linear_matches_oracle(M, K, N, izp):
    p = dict(ws_lo=0.001, ws_hi=0.005, b_mean=0.0, b_var=0.1)
    x, w, ws, b = synth.linear_inputs(M * 3 + K + N, M, K, N, x_kind="int8", p=p)
    ref_acc = oracle.linear_acc(x, izp, w)
    ref = oracle.linear(x, 0.03, izp, w, ws, b, 0.1, 1)
    got = H(q8.linear(T(x), 0.03, izp, T(w), None, T(ws), T(b), 0.1, 1))
    np.testing.assert_array_equal(got, ref)
    packed = q8.pack_weight(T(w))
    np.testing.assert_array_equal(H(q8.linear_packed(T(x), 0.03, izp, packed, T(ws), T(b), 0.1,
                                                     1)), ref)
    np.testing.assert_array_equal(H(q8.linear_packed_acc32(T(x), izp, packed)), ref_acc)
    operand = q8.prepare_operand(T(x), izp)
    np.testing.assert_array_equal(H(q8.linear_operand_packed(operand, 0.03, packed, T(ws), T(b),
                                                             0.1, 1)), ref)


def test_linear_chain_8x64x32():
    wl = synth.CONFIGS["linear_chain_8x64x32"]
    d, p = wl.dims, wl.params
    x, w, ws, b = synth.linear_inputs(wl.seed, d["M"], d["K"], d["N"], x_kind="fp32", p=p)
    xq_ref = oracle.quantize_per_tensor(x, p["in_scale"], p["in_zp"])
    ref = oracle.linear(xq_ref, p["in_scale"], p["in_zp"], w, ws, b, p["out_scale"], p["out_zp"])
    xq = q8.quantize_per_tensor(T(x), p["in_scale"], p["in_zp"])
    got = q8.linear(xq, p["in_scale"], p["in_zp"], T(w), None, T(ws), T(b), p["out_scale"],
                    p["out_zp"])
    np.testing.assert_array_equal(H(xq), xq_ref)
    np.testing.assert_array_equal(H(got), ref)
    packed = q8.pack_weight(T(w))
    fxq, fout = q8.quantize_linear_packed(T(x), p["in_scale"], p["in_zp"], packed, T(ws), T(b),
                                          p["out_scale"], p["out_zp"])
    np.testing.assert_array_equal(H(fxq), xq_ref)
    np.testing.assert_array_equal(H(fout), ref)


# The quantize -> operand kernel of the prefill chain on the values where a
# rounding or clamping slip would show: ties (x * inv = k + 1/2), +-0, +-inf,
# NaN, values far past the int8 range, for zero points at both ends and an
# odd one; K = 64 and 72 (8-element items from 16-byte loads; 72 also pads
# its last k-block with zeros) and K = 70 (rows not 16-byte aligned: one
# element at a time).  x_q and the GEMM's result both equal the oracle's.
@pytest.mark.parametrize("zp", [-128, -7, 0, 3, 127])
@pytest.mark.parametrize("K", [64, 72, 70])
def test_quantize_to_operand_special_values(zp, K):
    special = np.array([0.5, 1.5, 2.5, -0.5, -1.5, -2.5, 0.0, -0.0, np.inf, -np.inf, np.nan,
                        1e30, -1e30, 127.5, -128.5, 126.5, -127.5, 255.5, -255.5, 3e9],
                       np.float32)
    M = 6
    x = synth.normal(11 + K, "qs", (M, K), 0.0, 60.0)
    flat = x.reshape(-1)
    flat[: special.size] = special
    flat[-special.size:] = special[::-1]
    p = dict(ws_lo=0.002, ws_hi=0.01, b_mean=0.0, b_var=0.1)
    _, w, ws, b = synth.linear_inputs(5 + K, M, K, 8, x_kind="int8", p=p)
    packed = q8.pack_weight(T(w))
    xq, out = q8.quantize_linear_packed(T(x), 1.0, zp, packed, T(ws), T(b), 0.3, -1)
    xq_ref = oracle.quantize_per_tensor(x, 1.0, zp)
    np.testing.assert_array_equal(H(xq), xq_ref)
    np.testing.assert_array_equal(H(out), oracle.linear(xq_ref, 1.0, zp, w, ws, b, 0.3, -1))


def _mismatches(got, ref):
    """Count of differing elements and the first few (index, got, ref)."""
    bad = np.argwhere(got != ref)
    first = [(tuple(int(i) for i in ix), int(got[tuple(ix)]), int(ref[tuple(ix)]))
             for ix in bad[:5]]
    return len(bad), first


def test_linear_chain_2048x4096x11008_full():
    """Full-size prefill chain (quantize 2048x4096 -> q8ta_linear N = 11008),
    in the launch configuration the benchmark times, compared with the
    oracle on every one of the 2048 x 11008 outputs (the oracle runs on all
    host cores, row slices in parallel)."""
    wl = synth.CONFIGS["linear_chain_2048x4096x11008"]
    d, p = wl.dims, wl.params
    x, w, ws, b = synth.linear_inputs(wl.seed, d["M"], d["K"], d["N"], x_kind="fp32", p=p)
    packed = q8.pack_weight(T(w))
    xq, out = q8.quantize_linear_packed(T(x), p["in_scale"], p["in_zp"], packed, T(ws), T(b),
                                        p["out_scale"], p["out_zp"])
    xq, out = H(xq), H(out)
    xq_ref = oracle.quantize_per_tensor(x, p["in_scale"], p["in_zp"])
    np.testing.assert_array_equal(xq, xq_ref)
    ref = parallel_oracle.linear(xq_ref, p["in_scale"], p["in_zp"], w, ws, b, p["out_scale"],
                                 p["out_zp"])
    n_bad, first = _mismatches(out, ref)
    assert n_bad == 0, f"{n_bad} of {ref.size} outputs differ, first: {first}"
    # the two-phase form the benchmark step runs (operand, then the GEMM)
    operand = q8.operand_buffer(d["M"], d["K"], DEV)
    q8.quantize_to_operand(T(x), p["in_scale"], p["in_zp"], operand=operand)
    out2 = H(q8.linear_operand_packed(operand, p["in_scale"], packed, T(ws), T(b),
                                      p["out_scale"], p["out_zp"]))
    n_bad, first = _mismatches(out2, ref)
    assert n_bad == 0, f"{n_bad} of {ref.size} outputs differ, first: {first}"
    # the fused form (quantize inside the GEMM kernel, one launch)
    xq3, out3, _ = q8.quantize_linear_fused(T(x), p["in_scale"], p["in_zp"], packed, T(ws),
                                            T(b), p["out_scale"], p["out_zp"], operand=operand)
    np.testing.assert_array_equal(H(xq3), xq_ref)
    n_bad, first = _mismatches(H(out3), ref)
    assert n_bad == 0, f"{n_bad} of {ref.size} outputs differ, first: {first}"


def test_acc32_exact_at_the_chunk_bound():
    """Adversarial magnitudes: |x - zp| = 255 and |w| = 128 make each
    512-long chunk reach 512 * 32640 = 16,711,680 (just below 2^24) before it
    is drained; mixed rows check that low-order bits survive next to it."""
    M, K, N = 256, 4096 + 64, 256
    x = np.full((M, K), 127, np.int8)
    w = np.full((N, K), -128, np.int8)
    # rows 64..127: alternate +255 / -255 operands; rows 128..: max then one small term
    x[64:128, 1::2] = -128
    x[128:, :] = synth.int8_uniform(1, "ax", (M - 128, K), -128, 127)
    x[128:, ::512] = 127
    w[64:, :] = synth.int8_uniform(2, "aw", (N - 64, K), -128, 127)
    w[200:, :511] = -128
    w[200:, 511] = 1
    packed = q8.pack_weight(T(w))
    got = H(q8.linear_packed_acc32(T(x), -128, packed))
    np.testing.assert_array_equal(got, oracle.linear_acc(x, -128, w))
    got = H(q8.linear_packed_acc32(T(x), 127, packed))
    np.testing.assert_array_equal(got, oracle.linear_acc(x, 127, w))


@pytest.mark.parametrize("izp", [0, 1, -1, -5, 64, -100])
def test_acc32_exact_at_the_zero_point_chunk_bound(izp):
    """The exact f32 chunk holds floor(2048 / b) k-blocks for b = max(128 +
    zp, 127 - zp), the largest |x - zp|: with every |x - zp| = b and w = -128
    each chunk reaches its largest sum (2^24 exactly for zp = 0).  Rows past
    the first 64 mix in random values so low-order bits sit next to it."""
    M, K, N = 256, 4096 + 64, 256
    xe = -128 if izp >= 0 else 127
    x = np.full((M, K), xe, np.int8)
    w = np.full((N, K), -128, np.int8)
    x[64:, :] = synth.int8_uniform(11, "bx", (M - 64, K), -128, 127)
    x[64:, ::97] = xe
    w[128:, :] = synth.int8_uniform(12, "bw", (N - 128, K), -128, 127)
    packed = q8.pack_weight(T(w))
    ref = oracle.linear_acc(x, izp, w)
    np.testing.assert_array_equal(H(q8.linear_packed_acc32(T(x), izp, packed)), ref)
    operand = q8.prepare_operand(T(x), izp)
    ws = np.full(N, 2.0 ** -12, np.float32)
    got = H(q8.linear_operand_packed(operand, 1.0, packed, T(ws), None, 1.0, 0))
    np.testing.assert_array_equal(got, oracle.linear(x, 1.0, izp, w, ws, None, 1.0, 0))


def test_conv_t_acc32_exact_at_the_chunk_bound():
    """Transposed convolution with |x - zp| = 128 (zp = 0) and w = -128 over
    9 taps x 512 channels: every exact chunk of 1024 products sums to 2^24."""
    N, IC, H_in, W_in, OC, K = 1, 512, 8, 8, 64, 3
    x = np.full((N, IC, H_in, W_in), -128, np.int8)
    w = np.full((OC, K * K * IC), -128, np.int8)
    w[32:, :] = synth.int8_uniform(13, "cw", (OC - 32, K * K * IC), -128, 127)
    H_out, W_out = synth.output_hw(H_in, W_in, K, K, 1, 1, 1, 1, 0, 0)
    ref = oracle.conv2d_transposed_acc(x, 0, w, K, K, H_out, W_out, (1, 1), (1, 1))
    got = H(q8.conv2d_transposed_acc32(T(x), 0, T(w), K, (H_out, W_out), stride=1, padding=1))
    np.testing.assert_array_equal(got, ref)


# --------------------------------------------------------------- conv_t

def _conv_case(seed, N, IC, H_in, W_in, OC, K, s, p, op, izp, ozp, out_hw=None):
    d = dict(N=N, IC=IC, H_in=H_in, W_in=W_in, OC=OC, Kh=K, Kw=K)
    pp = dict(in_scale=0.02, ws_lo=0.002, ws_hi=0.01, b_mean=0.0, b_var=0.1)
    x, w, ws, b = synth.conv_t_inputs(seed, d, pp)
    Hn, Wn = synth.output_hw(H_in, W_in, K, K, s, s, p, p, op, op)
    H_out, W_out = out_hw if out_hw else (Hn, Wn)
    ref = oracle.conv2d_transposed(x, 0.02, izp, w, K, K, ws, b, 0.15, ozp, H_out, W_out, (s, s),
                                   (p, p))
    got = H(q8.conv2d_transposed(T(x), 0.02, izp, T(w), None, T(ws), T(b), 0.15, ozp, K,
                                 stride=s, padding=p, output_padding=op,
                                 output_size=(H_out, W_out)))
    np.testing.assert_array_equal(got, ref)
    acc_ref = oracle.conv2d_transposed_acc(x, izp, w, K, K, H_out, W_out, (s, s), (p, p))
    acc = H(q8.conv2d_transposed_acc32(T(x), izp, T(w), K, (H_out, W_out), stride=s, padding=p))
    np.testing.assert_array_equal(acc, acc_ref)


CONV_SHAPES = [
    # seed, N, IC, H, W, OC, K, s, p, op, izp, ozp, (H_out, W_out) or None
    (1, 1, 3, 5, 4, 4, 3, 2, 1, 1, -7, 2, None),
    (2, 2, 64, 7, 9, 36, 4, 2, 1, 0, 4, 0, (14, 16)),
    (3, 1, 70, 6, 6, 132, 3, 1, 0, 0, -128, -3, (8, 8)),
    (4, 1, 16, 5, 5, 8, 1, 3, 0, 2, 127, 1, (15, 16)),        # phases with no tap
    (5, 3, 8, 4, 6, 12, 5, 2, 2, 1, 0, 0, (10, 12)),
    (6, 1, 32, 40, 150, 16, 2, 2, 0, 0, 9, -9, (80, 300)),   # W' > 128: several w tiles
    (7, 2, 128, 8, 8, 256, 3, 2, 1, 1, -1, 5, (16, 16)),
    (8, 1, 8, 3, 3, 4, 3, 2, 0, 0, 2, 2, (9, 12)),           # output larger than natural
    (9, 1, 40, 9, 10, 24, 4, 2, 1, 0, -3, 3, (24, 32)),      # staged rows, ragged row tiles
    (10, 2, 64, 16, 16, 64, 3, 2, 1, 1, 11, -4, (32, 32)),   # staged, several images
]


@pytest.mark.parametrize("case", CONV_SHAPES)
def test_conv_t_matches_oracle(case):
    seed, N, IC, H_in, W_in, OC, K, s, p, op, izp, ozp, hw = case
    _conv_case(seed, N, IC, H_in, W_in, OC, K, s, p, op, izp, ozp, hw)


def _workload_conv(name):
    wl = synth.CONFIGS[name]
    d, p = wl.dims, wl.params
    x, w, ws, b = synth.conv_t_inputs(wl.seed, d, p)
    Ho, Wo = synth.output_hw(d["H_in"], d["W_in"], d["Kh"], d["Kw"], d["s"], d["s"], d["p"],
                             d["p"], d["op"], d["op"])
    got = H(q8.conv2d_transposed(T(x), p["in_scale"], p["in_zp"], T(w), None, T(ws), T(b),
                                 p["out_scale"], p["out_zp"], (d["Kh"], d["Kw"]), stride=d["s"],
                                 padding=d["p"], output_padding=d["op"]))
    return wl, d, p, x, w, ws, b, Ho, Wo, got


def test_conv_t_1x64x32x32_full():
    wl, d, p, x, w, ws, b, Ho, Wo, got = _workload_conv("conv_t_1x64x32x32_k4s2")
    assert (Ho, Wo) == (64, 64)
    ref = oracle.conv2d_transposed(x, p["in_scale"], p["in_zp"], w, 4, 4, ws, b, p["out_scale"],
                                   p["out_zp"], Ho, Wo, (2, 2), (1, 1))
    np.testing.assert_array_equal(got, ref)


def test_conv_t_8x256x64x64_full():
    """The 8x256x64x64 -> 8x128x128x128 transposed convolution (packed
    weight and caller workspace, as the benchmark runs it, and the raw-weight
    form) compared with the oracle on every output of every image and
    channel (the oracle runs on all host cores in (image, channel) blocks)."""
    wl, d, p, x, w, ws, b, Ho, Wo, got = _workload_conv("conv_t_8x256x64x64_k3s2")
    assert (Ho, Wo) == (128, 128)
    ref = parallel_oracle.conv2d_transposed(x, p["in_scale"], p["in_zp"], w, 3, 3, ws, b,
                                            p["out_scale"], p["out_zp"], Ho, Wo, (2, 2), (1, 1))
    n_bad, first = _mismatches(got, ref)
    assert n_bad == 0, f"{n_bad} of {ref.size} outputs differ, first: {first}"
    packed = q8.pack_conv2d_transposed_weight(T(w), d["IC"], (d["Kh"], d["Kw"]))
    got2 = H(q8.conv2d_transposed_packed(T(x), p["in_scale"], p["in_zp"], packed, T(ws), T(b),
                                         p["out_scale"], p["out_zp"], stride=d["s"],
                                         padding=d["p"], output_padding=d["op"]))
    n_bad, first = _mismatches(got2, ref)
    assert n_bad == 0, f"{n_bad} of {ref.size} outputs differ, first: {first}"


# ------------------------------------------------- empty and large sizes

def test_quantize_and_dequantize_empty():
    x = torch.empty(0, dtype=torch.float32, device=DEV)
    assert q8.quantize_per_tensor(x, 0.1, 0).numel() == 0
    q = torch.empty((0, 4), dtype=torch.int8, device=DEV)
    assert q8.dequantize_per_tensor(q, 0.1, 0).shape == (0, 4)


def _pattern_f32(idx):
    """x[i] = ((i mod 509) - 254) * 0.0173 in float32 (both sides compute it)."""
    return ((idx % 509) - 254).astype(np.float32) * np.float32(0.0173)


def test_quantize_beyond_2_pow_31_elements():
    """64-bit element indexing: 2^31 + 8 elements (8.6 GB of fp32), filled on
    the device with a closed-form pattern and checked at sampled indices,
    including the last ones."""
    n = (1 << 31) + 8
    x = torch.empty(n, dtype=torch.float32, device=DEV)
    blk = 1 << 26
    for b0 in range(0, n, blk):
        idx = torch.arange(b0, min(n, b0 + blk), device=DEV, dtype=torch.int64)
        x[b0:b0 + idx.numel()] = ((idx % 509) - 254).to(torch.float32) * 0.0173
    out = q8.quantize_per_tensor(x, 0.05, 3)
    rng = np.random.default_rng(0)
    sample = np.concatenate([np.arange(0, 64), np.arange(n - 64, n),
                             np.arange((1 << 31) - 32, (1 << 31) + 8),
                             rng.integers(0, n, 4096)]).astype(np.int64)
    got = H(out[torch.from_numpy(sample).to(DEV)])
    ref = oracle.quantize_per_tensor(_pattern_f32(sample), 0.05, 3)
    np.testing.assert_array_equal(got, ref)
    del x, out


def test_linear_output_beyond_2_pow_31_bytes():
    """A linear whose int8 output holds more than 2^31 bytes (M * N > 2^31):
    64-bit output addressing in the GEMM epilogue, checked on sampled rows."""
    M, K, N = 70000, 64, 32768
    x = synth.int8_uniform(81, "x", (M, K), -128, 127)
    w = synth.int8_uniform(81, "w", (N, K), -127, 127)
    ws = synth.uniform_float(81, "ws", (N,), 0.001, 0.005)
    b = synth.normal(81, "b", (N,), 0.0, 0.1)
    out = q8.linear_packed(T(x), 0.03, -1, q8.pack_weight(T(w)), T(ws), T(b), 0.1, 2)
    rows = np.array([0, 1, 255, 256, 65535, 65536, M - 2, M - 1], dtype=np.int64)
    got = H(out[torch.from_numpy(rows).to(DEV)])
    np.testing.assert_array_equal(got, oracle.linear(x[rows], 0.03, -1, w, ws, b, 0.1, 2))
    del out


def test_gemv_weight_beyond_2_pow_31_bytes():
    """A gemv whose weight holds more than 2^31 bytes (N * K > 2^31), filled
    on the device with a closed-form pattern; sampled outputs."""
    N, K = 65536 + 4, 32768
    w = torch.empty((N, K), dtype=torch.int8, device=DEV)
    kk = torch.arange(K, device=DEV, dtype=torch.int64)
    for n0 in range(0, N, 4096):
        nn = torch.arange(n0, min(N, n0 + 4096), device=DEV, dtype=torch.int64)[:, None]
        w[n0:n0 + nn.shape[0]] = ((nn * 131 + kk * 7) % 255 - 127).to(torch.int8)
    x = synth.int8_uniform(82, "x", (1, K), -128, 127)
    ws = synth.uniform_float(82, "ws", (N,), 0.002, 0.01)
    b = synth.normal(82, "b", (N,), 0.0, 0.1)
    out = q8.linear_gemv(T(x), 0.02, 5, w, None, T(ws), T(b), 0.5, -1)
    rows = np.array([0, 1, 65535, 65536, N - 1], dtype=np.int64)
    k = np.arange(K, dtype=np.int64)
    w_rows = ((rows[:, None] * 131 + k[None, :] * 7) % 255 - 127).astype(np.int8)
    ref = oracle.linear(x, 0.02, 5, w_rows, ws[rows], b[rows], 0.5, -1)
    np.testing.assert_array_equal(H(out)[:, rows], ref)
    del w, out
