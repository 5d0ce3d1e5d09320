"""Failure detection on the device: a bounded pipeline wait that runs out.

Every mbarrier wait of the tensor-core GEMM gives up after a time limit; the
kernel then records a code in the library's device error word, stops issuing
work, waits (bounded) for its own copies and MMAs in flight, frees its tensor
memory and returns.  Here a test-only entry point makes the TMA producer
leave out one ring fill with a 5 ms limit, so the MMA's wait for that stage
(or the epilogue's wait for the accumulator) runs out.  No trap, no fault and
no unbounded wait is involved: the call returns within a few limits, the
error word holds the wait's code, and the same CUDA context then runs the
normal path bit-exactly against the oracle.

Single-CTA tiles (M <= 128) are used: each CTA's producer then waits for
every copy it issued on its own barriers before the CTA exits.
"""
import time

import numpy as np
import pytest
import torch

import oracle
import synth

pytestmark = pytest.mark.gpu

q8 = pytest.importorskip("int8_quantized_q8ta_gb300")
DEV = torch.device("cuda:0")
WAIT_CODES = {0x101, 0x103}   # the MMA's full-barrier wait, the epilogue's accumulator wait


def T(a):
    return torch.from_numpy(np.ascontiguousarray(a)).to(DEV)


@pytest.mark.parametrize("M,K,N,skip", [(128, 1024, 128, 2), (96, 2048, 512, 0),
                                        (128, 4096, 1024, 7)])
def test_bounded_wait_runs_out_and_context_stays_usable(M, K, N, skip):
    assert q8.device_error(clear=True) == 0
    x = synth.int8_uniform(M + K, "tx", (M, K), -128, 127)
    w = synth.int8_uniform(M + K, "tw", (N, K), -127, 127)
    packed = q8.pack_weight(T(w))
    xt = T(x)
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    q8.debug_linear_packed_stall(xt, 3, packed, wait_limit_ns=5_000_000, skip_fill=skip)
    torch.cuda.synchronize()
    elapsed = time.perf_counter() - t0
    code = q8.device_error(clear=True)
    assert code in WAIT_CODES, hex(code)
    assert elapsed < 1.0, elapsed
    # the same context runs the normal path, bit-exact
    acc = q8.linear_packed_acc32(xt, 3, packed)
    torch.cuda.synchronize()
    np.testing.assert_array_equal(acc.cpu().numpy(), oracle.linear_acc(x, 3, w))
    assert q8.device_error(clear=True) == 0


def test_stall_hook_guards():
    x = torch.zeros((128, 64), dtype=torch.int8, device=DEV)
    packed = q8.pack_weight(torch.zeros((128, 64), dtype=torch.int8, device=DEV))
    for limit, skip in ((999_999, 0), (2_000_000_000, 0), (5_000_000, -1)):
        with pytest.raises(q8.Q8Error) as e:
            q8.debug_linear_packed_stall(x, 0, packed, wait_limit_ns=limit, skip_fill=skip)
        assert e.value.status == q8.Q8_ERR_ARG
    assert q8.device_error(clear=True) == 0
