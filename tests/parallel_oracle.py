"""Run the unchanged CPU oracle over slices of a large problem on every host
core (test infrastructure).

The oracle's ctypes calls release the GIL, so a thread pool runs one slice
per core.  Slices are independent outputs of the same definition (rows of a
linear, (image, output-channel) blocks of a convolution), so joining them
gives exactly the oracle's full result; no arithmetic happens here.
"""
from __future__ import annotations

import concurrent.futures as cf
import os

import numpy as np

import oracle


def _pool():
    return cf.ThreadPoolExecutor(max_workers=max(1, os.cpu_count() or 1))


def linear(x, input_scale, izp, w, ws, b, output_scale, ozp, rows_per_task=16):
    """oracle.linear over row slices of x; returns the int8 [M, N] output."""
    M = x.shape[0]
    out = np.empty((M, w.shape[0]), np.int8)

    def run(r0):
        r1 = min(M, r0 + rows_per_task)
        out[r0:r1] = oracle.linear(x[r0:r1], input_scale, izp, w, ws, b, output_scale, ozp)

    with _pool() as ex:
        list(ex.map(run, range(0, M, rows_per_task)))
    return out


def conv2d_transposed(x, input_scale, izp, w, Kh, Kw, ws, b, output_scale, ozp, H_out, W_out,
                      stride, pad, oc_per_task=8):
    """oracle.conv2d_transposed (groups 1) over (image, output-channel) blocks."""
    N, OC = x.shape[0], w.shape[0]
    out = np.empty((N, OC, H_out, W_out), np.int8)

    def run(task):
        n, c0 = task
        c1 = min(OC, c0 + oc_per_task)
        out[n:n + 1, c0:c1] = oracle.conv2d_transposed(
            x[n:n + 1], input_scale, izp, w[c0:c1], Kh, Kw, ws[c0:c1],
            None if b is None else b[c0:c1], output_scale, ozp, H_out, W_out, stride, pad)

    tasks = [(n, c0) for n in range(N) for c0 in range(0, OC, oc_per_task)]
    with _pool() as ex:
        list(ex.map(run, tasks))
    return out
