"""Exact f32 chunks sized from a packed weight's k-block bound.

A packed weight records the largest sum of |w| over one k-block (64
consecutive weights of one row, per tap for a convolution); the tensor-core
kernels add that many k-blocks in f32 as can stay exact.  These cases hold one
extreme row (every weight 127) among rows of small weights, with every
|x - zp| = 255: a bound taken from anything but the largest k-block would let
the extreme row's f32 sums pass 2^24 and round, so the int32 accumulators
and the int8 outputs are compared with the oracle bit for bit.  The small
rows alone would allow chunks over the whole k range.
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


@pytest.mark.parametrize("M,K,N", [(256, 4096, 512), (100, 2048, 96)])
def test_linear_packed_bound_takes_the_largest_block(M, K, N):
    x = np.full((M, K), -128, dtype=np.int8)            # x - zp = -255 with zp = 127
    w = synth.int8_uniform(5, "w", (N, K), -2, 2)
    w[N // 3] = 127                                      # one row at the bound
    ws = synth.uniform_float(5, "ws", (N,), 1e-6, 2e-6)
    b = synth.normal(5, "b", (N,), 0.0, 0.1)
    acc_ref = oracle.linear_acc(x, 127, w)
    assert abs(int(acc_ref[:, N // 3].min())) > 1 << 24  # the row's sum is past 2^24
    packed = q8.pack_weight(T(w))
    np.testing.assert_array_equal(H(q8.linear_packed_acc32(T(x), 127, packed)), acc_ref)
    ref = oracle.linear(x, 0.01, 127, w, ws, b, 0.02, 3)
    got = H(q8.linear_packed(T(x), 0.01, 127, packed, T(ws), T(b), 0.02, 3))
    np.testing.assert_array_equal(got, ref)


@pytest.mark.parametrize("OC", [128, 40])
def test_conv_t_packed_bound_takes_the_largest_block(OC):
    N, IC, Hi, Wi, K = 1, 256, 16, 64, 3
    x = np.full((N, IC, Hi, Wi), -128, dtype=np.int8)
    w = synth.int8_uniform(6, "w", (OC, K * K * IC), -2, 2)
    w[OC // 2] = 127
    ws = synth.uniform_float(6, "ws", (OC,), 1e-6, 2e-6)
    b = synth.normal(6, "b", (OC,), 0.0, 0.1)
    Ho, Wo = synth.output_hw(Hi, Wi, K, K, 2, 2, 1, 1, 1, 1)
    acc_ref = oracle.conv2d_transposed_acc(x, 127, w, K, K, Ho, Wo, (2, 2), (1, 1), (1, 1))
    assert abs(int(acc_ref[:, OC // 2].min())) > 1 << 24
    packed = q8.pack_conv2d_transposed_weight(T(w), in_channels=IC, kernel_size=K)
    acc = H(q8.conv2d_transposed_packed_acc32(T(x), 127, packed, (Ho, Wo), stride=2, padding=1))
    np.testing.assert_array_equal(acc, acc_ref)
    ref = oracle.conv2d_transposed(x, 0.01, 127, w, K, K, ws, b, 0.02, 3, Ho, Wo, (2, 2), (1, 1),
                                   (1, 1))
    got = H(q8.conv2d_transposed_packed(T(x), 0.01, 127, packed, T(ws), T(b), 0.02, 3, stride=2,
                                        padding=1, output_padding=1, output_size=(Ho, Wo)))
    np.testing.assert_array_equal(got, ref)


def test_conv2d_packed_bound_takes_the_largest_block():
    N, IC, Hi, Wi, K, OC = 1, 256, 20, 72, 3, 96
    x = np.full((N, IC, Hi, Wi), -128, dtype=np.int8)
    w = synth.int8_uniform(8, "w", (OC, K * K * IC), -2, 2)
    w[7] = 127
    Ho, Wo = 20, 72
    acc_ref = oracle.conv2d_acc(x, 127, w, K, K, Ho, Wo, (1, 1), (1, 1), (1, 1))
    assert abs(int(acc_ref[:, 7].min())) > 1 << 24
    packed = q8.pack_conv2d_weight(T(w), in_channels=IC, kernel_size=K)
    acc = H(q8.conv2d_packed_acc32(T(x), 127, packed, (Ho, Wo), stride=1, padding=1))
    np.testing.assert_array_equal(acc, acc_ref)


def test_operand_reused_back_to_back_with_a_wider_zero_point():
    """Two acc32 calls on one workspace, back to back: the second prepares
    its operand with zero point 127 (|x - zp| bound 255, chunks of 8 k-blocks
    against all-127 weights) over the first one's (zero point 0: chunks of
    16).  The GEMM reads the operand's bound word only after the preceding
    kernel has finished (programmatic dependent launch), so it never sizes
    its chunks from the earlier zero point."""
    M, K, N = 256, 4096, 256
    x = np.full((M, K), -128, dtype=np.int8)
    w = np.full((N, K), 127, dtype=np.int8)
    packed = q8.pack_weight(T(w))
    ws = torch.empty(1 << 26, dtype=torch.uint8, device=DEV)
    xt = T(x)
    a0 = q8.linear_packed_acc32(xt, 0, packed, workspace=ws)
    a1 = q8.linear_packed_acc32(xt, 127, packed, workspace=ws)
    ref1 = oracle.linear_acc(x, 127, w)
    assert abs(int(ref1.min())) > 1 << 24
    np.testing.assert_array_equal(H(a1), ref1)
    np.testing.assert_array_equal(H(a0), oracle.linear_acc(x, 0, w))


def test_conv_packed_buffer_rewritten_after_packing_is_caught():
    """The host records a packed weight's bound when it packs it and picks
    the single-chunk kernel from that record; a buffer rewritten afterwards
    with a weight that needs shorter chunks is caught on the device: the
    kernel runs nothing and sets the error word (0x107)."""
    N, IC, Hi, Wi, K, OC = 1, 256, 16, 64, 3, 128
    x = np.full((N, IC, Hi, Wi), -128, dtype=np.int8)
    w_small = synth.int8_uniform(9, "w", (OC, K * K * IC), -2, 2)
    w_big = w_small.copy()
    w_big[5] = 127
    Ho, Wo = synth.output_hw(Hi, Wi, K, K, 2, 2, 1, 1, 1, 1)
    pa = q8.pack_conv2d_transposed_weight(T(w_small), in_channels=IC, kernel_size=K)
    pb = q8.pack_conv2d_transposed_weight(T(w_big), in_channels=IC, kernel_size=K)
    pa.data.copy_(pb.data)          # behind the library's back
    q8.conv2d_transposed_packed_acc32(T(x), 127, pa, (Ho, Wo), stride=2, padding=1)
    torch.cuda.synchronize()
    assert q8.device_error(clear=True) == 0x107
    acc = H(q8.conv2d_transposed_packed_acc32(T(x), 127, pb, (Ho, Wo), stride=2, padding=1))
    np.testing.assert_array_equal(acc, oracle.conv2d_transposed_acc(x, 127, w_big, K, K, Ho, Wo,
                                                                    (2, 2), (1, 1), (1, 1)))

