"""GPU parity of the fused quantize -> q8ta_linear kernel (one launch).

The GEMM's own warps quantize fp32 x into the bf16 operand chunk by chunk
along K, and the TMA producers of all CTAs load a chunk only once every CTA
has signalled it.  Compared element by element with the oracle's
quantize_per_tensor -> linear on the same seeded inputs: ragged M, K and N
(K % 8 != 0 takes the scalar path, K % 64 != 0 a zero-padded last k-block),
single-CTA and CTA-pair tiles, with and without x_q, relu, two calls in a
row on one operand (the chunk counters must be back at zero), reuse of the
operand by the two-phase path, and an operand whose trailer was never
initialized (nothing runs, device error 0x109).
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


P = dict(x_mean=0.0, x_var=3.0, ws_lo=0.001, ws_hi=0.005, b_mean=0.0, b_var=0.1)

# M, K, N, scale, zp: single-CTA tiles (M or N <= 128) and CTA pairs; K from
# one k-block to several chunks, ragged tails
SHAPES = [(2, 4, 4, 0.03, 0), (8, 64, 32, 0.02, 3), (130, 200, 36, 0.05, -128),
          (257, 520, 260, 0.03, 127), (129, 1036, 516, 0.01, -5), (300, 4096, 136, 0.03, 1),
          (640, 2052, 1024, 0.04, -7), (1000, 8192, 264, 0.03, 77), (256, 12, 192, 0.5, 2),
          (1, 64, 32, 0.02, 3), (3, 4, 8, 0.1, -1)]


@pytest.mark.parametrize("M,K,N,scale,zp", SHAPES)
def test_fused_matches_oracle(M, K, N, scale, zp):
    x, w, ws, b = synth.linear_inputs(M + 7 * K + N, M, K, N, x_kind="fp32", p=P)
    xq_ref = oracle.quantize_per_tensor(x, scale, zp)
    ref = oracle.linear(xq_ref, scale, zp, w, ws, b, 0.1, 1)
    packed = q8.pack_weight(T(w))
    xq, out, operand = q8.quantize_linear_fused(T(x), scale, zp, packed, T(ws), T(b), 0.1, 1)
    np.testing.assert_array_equal(H(xq), xq_ref)
    np.testing.assert_array_equal(H(out), ref)
    # the second call on the same operand, another x, no x_q, relu
    x2 = synth.normal(M + 7 * K + N + 1, "x2", (M, K), 0.0, 3.0)
    xq2_ref = oracle.quantize_per_tensor(x2, scale, zp)
    ref2 = oracle.linear(xq2_ref, scale, zp, w, ws, b, 0.1, 1, activation="relu")
    _, out2, _ = q8.quantize_linear_fused(T(x2), scale, zp, packed, T(ws), T(b), 0.1, 1,
                                          activation="relu", operand=operand, want_x_q=False)
    np.testing.assert_array_equal(H(out2), ref2)
    # the operand the fused kernel wrote serves the two-phase path as well
    out3 = q8.linear_operand_packed(operand, scale, packed, T(ws), T(b), 0.1, 1,
                                    activation="relu")
    np.testing.assert_array_equal(H(out3), ref2)


def test_fused_many_calls_in_a_row_on_one_operand():
    """Twenty launches back to back on one operand (no host sync between
    them): each launch's last CTA resets the chunk counters for the next."""
    M, K, N = 512, 1024, 512
    x, w, ws, b = synth.linear_inputs(71, M, K, N, x_kind="fp32", p=P)
    packed = q8.pack_weight(T(w))
    operand = q8.operand_buffer(M, K, DEV)
    xs = [synth.normal(100 + i, "xs", (M, K), 0.0, 3.0) for i in range(4)]
    xts = [T(a) for a in xs]
    outs = []
    for i in range(20):
        _, o, _ = q8.quantize_linear_fused(xts[i % 4], 0.03, -5, packed, T(ws), T(b), 0.1, 1,
                                           operand=operand, want_x_q=False)
        outs.append(o)
    for i in range(4):
        ref = oracle.linear(oracle.quantize_per_tensor(xs[i], 0.03, -5), 0.03, -5, w, ws, b,
                            0.1, 1)
        for j in range(i, 20, 4):
            np.testing.assert_array_equal(H(outs[j]), ref)


def test_fused_uninitialized_operand_runs_nothing():
    M, K, N = 256, 512, 256
    x, w, ws, b = synth.linear_inputs(72, M, K, N, x_kind="fp32", p=P)
    packed = q8.pack_weight(T(w))
    raw = q8.Operand(torch.zeros(q8.lib().q8_linear_operand_bytes(M, K), dtype=torch.uint8,
                                 device=DEV), M, K)
    out = torch.full((M, N), 55, dtype=torch.int8, device=DEV)
    q8.quantize_linear_fused(T(x), 0.03, 0, packed, T(ws), T(b), 0.1, 1, out=out, operand=raw,
                             want_x_q=False)
    torch.cuda.synchronize()
    assert q8.device_error(clear=True) == 0x109
    assert bool((out == 55).all())
    # initializing that buffer makes it usable
    assert q8.lib().q8_linear_operand_init(q8._ptr(raw.data), M, K, raw.data.numel(),
                                           q8._stream(raw.data)) == q8.Q8_OK
    q8.quantize_linear_fused(T(x), 0.03, 0, packed, T(ws), T(b), 0.1, 1, out=out, operand=raw,
                             want_x_q=False)
    ref = oracle.linear(oracle.quantize_per_tensor(x, 0.03, 0), 0.03, 0, w, ws, b, 0.1, 1)
    np.testing.assert_array_equal(H(out), ref)
