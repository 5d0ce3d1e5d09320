"""q8_linear_noalloc, the entry point for callers that cannot allocate.

Some callers cannot allocate device memory where they run a layer (a plugin
whose host runtime owns the device memory pool, a latency-critical loop that
cannot afford cudaMalloc/cudaFree, a deployment with a memory budget fixed at
start-up).  q8_linear_noalloc serves them from a fixed library-owned scratch
array.  This test calls it through the C ABI and checks its output against
q8_linear's (with a caller workspace) and against the CPU oracle on two
calls in a row with different inputs, so a second call that saw the first
call's leftover scratch contents would show up; it also checks that an
over-size problem is refused before anything is launched (real device
buffers, output left untouched).  It sits in a file of its own that pytest collects
last, and it builds the library if needed, so it also runs alone in a fresh
process.
"""
import ctypes

import numpy as np
import pytest
import torch

import oracle
import synth

pytestmark = pytest.mark.gpu

from int8_quantized_q8ta_gb300 import _build  # noqa: E402

_build.build()
import int8_quantized_q8ta_gb300 as q8  # noqa: E402

DEV = torch.device("cuda:0")


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _case(seed, M, K, N, izp):
    p = dict(ws_lo=0.001, ws_hi=0.005, b_mean=0.0, b_var=0.1)
    x, w, ws, b = synth.linear_inputs(seed, M, K, N, x_kind="int8", p=p)
    T = lambda a: torch.from_numpy(np.ascontiguousarray(a)).to(DEV)  # noqa: E731
    return T(x), T(w), T(ws), T(b), izp


def _oracle(x, w, ws, b, izp, act="none"):
    c = lambda t: t.cpu().numpy()  # noqa: E731
    return torch.from_numpy(oracle.linear(c(x), 0.03, izp, c(w), c(ws), c(b), 0.1, 1,
                                          activation=act)).to(DEV)


def _noalloc(x, w, ws, b, izp, out, act=b"none"):
    M, K = x.shape
    N = w.shape[0]
    stream = ctypes.c_void_p(torch.cuda.current_stream(DEV).cuda_stream)
    return q8.lib().q8_linear_noalloc(_ptr(x), M, K, 0.03, izp, _ptr(w), N, None, _ptr(ws),
                                      _ptr(b), 0.1, 1, act, _ptr(out), stream)


def test_noalloc_matches_q8_linear_on_two_calls():
    # two different problems in a row; the second is smaller along K and M,
    # so the scratch still holds the first call's bytes around the region the
    # second call writes and then reads
    for seed, (M, K, N, izp) in ((1, (300, 1040, 516, -5)), (2, (130, 200, 36, 127))):
        x, w, ws, b, izp = _case(seed, M, K, N, izp)
        out = torch.full((M, N), 55, dtype=torch.int8, device=DEV)
        assert _noalloc(x, w, ws, b, izp, out) == q8.Q8_OK
        ref = q8.linear(x, 0.03, izp, w, None, ws, b, 0.1, 1)
        torch.cuda.synchronize()
        assert torch.equal(out, ref)
        assert torch.equal(out, _oracle(x, w, ws, b, izp))
    # the relu activation through the same scratch
    out = torch.empty((M, N), dtype=torch.int8, device=DEV)
    assert _noalloc(x, w, ws, b, izp, out, b"relu") == q8.Q8_OK
    ref = q8.linear(x, 0.03, izp, w, None, ws, b, 0.1, 1, activation="relu")
    torch.cuda.synchronize()
    assert torch.equal(out, ref)
    assert torch.equal(out, _oracle(x, w, ws, b, izp, "relu"))
    assert q8.device_error(clear=True) == 0


def test_noalloc_refuses_oversize_and_serves_gemv():
    # 2 * (M + N) * ceil64(K) bf16 bytes = 2 * 2048 * 4160 > 16 MiB while the
    # int8 inputs hold only 8.5 MB: refused before any launch, out untouched
    M, K, N = 1024, 4160, 1024
    x, w, ws, b, izp = _case(4, M, K, N, 0)
    out = torch.full((M, N), 55, dtype=torch.int8, device=DEV)
    assert _noalloc(x, w, ws, b, izp, out) == q8.Q8_ERR_WORKSPACE
    torch.cuda.synchronize()
    assert bool((out == 55).all())
    # M == 1 needs no scratch
    x, w, ws, b, izp = _case(3, 1, 4096, 1024, 0)
    out = torch.empty((1, 1024), dtype=torch.int8, device=DEV)
    assert _noalloc(x, w, ws, b, izp, out) == q8.Q8_OK
    ref = q8.linear_gemv(x, 0.03, izp, w, None, ws, b, 0.1, 1)
    torch.cuda.synchronize()
    assert torch.equal(out, ref)
    assert torch.equal(out, _oracle(x, w, ws, b, izp))
    assert q8.device_error(clear=True) == 0
