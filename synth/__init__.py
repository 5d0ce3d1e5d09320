"""Seeded synthetic inputs for the q8ta int8 quantized contraction.

This module is shared by the CPU oracle's tests, the CUDA parity tests and
``bench.py``.  It draws random numbers and nothing else: it holds none of the
method's arithmetic (no quantization, no contraction, no epilogue), so both
sides of every parity check see identical input bytes without sharing any
computation.

Generator: a counter-based SplitMix64.  Element ``i`` of the stream keyed by
``(seed, name)`` is ``mix64(key + (i + 1) * 0x9E3779B97F4A7C15)`` with the
SplitMix64 finaliser (Steele, Lea and Flood, "Fast splittable pseudorandom
number generators", OOPSLA 2014).  Being counter based, any sub-range of a
stream can be regenerated without producing the elements before it.

Transforms (all written here, none from ``numpy.random``):
* uniform integers on ``[lo, hi]``: Lemire's multiply-shift on the top 32 bits
  (bias below 2**-24 for the ranges used, which is irrelevant for test data);
* uniform floats on ``[a, b)``: a 24-bit mantissa draw, affine map in float64,
  cast to float32;
* normals ``N(mu, var)``: Box-Muller in float64 from two independent streams,
  scaled by ``sqrt(var)`` (the second parameter is a VARIANCE), cast to float32.

The workload recipes (``CONFIGS``) restate the five workloads of the q8ta
pages' benchmark set with their shapes and value distributions; see the
``Workload`` docstring.
"""
from __future__ import annotations

import dataclasses
import hashlib
from typing import Dict

import numpy as np

_GOLDEN = np.uint64(0x9E3779B97F4A7C15)
_M1 = np.uint64(0xBF58476D1CE4E5B9)
_M2 = np.uint64(0x94D049BB133111EB)


def _key(seed: int, name: str) -> np.uint64:
    h = hashlib.sha256(f"{seed}:{name}".encode()).digest()
    return np.uint64(int.from_bytes(h[:8], "little"))


def _mix64(z: np.ndarray) -> np.ndarray:
    z = (z ^ (z >> np.uint64(30))) * _M1
    z = (z ^ (z >> np.uint64(27))) * _M2
    return z ^ (z >> np.uint64(31))


def raw_u64(seed: int, name: str, n: int, start: int = 0) -> np.ndarray:
    """``n`` uint64 draws of stream ``(seed, name)`` starting at counter ``start``."""
    with np.errstate(over="ignore"):
        idx = np.arange(start + 1, start + n + 1, dtype=np.uint64)
        return _mix64(_key(seed, name) + idx * _GOLDEN)


def uniform_int(seed: int, name: str, shape, lo: int, hi: int) -> np.ndarray:
    """Integers uniform on the closed range ``[lo, hi]`` as int64."""
    n = int(np.prod(shape))
    span = np.uint64(hi - lo + 1)
    top = raw_u64(seed, name, n) >> np.uint64(32)
    with np.errstate(over="ignore"):
        v = ((top * span) >> np.uint64(32)).astype(np.int64) + lo
    return v.reshape(shape)


def uniform_float(seed: int, name: str, shape, a: float, b: float) -> np.ndarray:
    """float32 values uniform on ``[a, b)``."""
    n = int(np.prod(shape))
    u = (raw_u64(seed, name, n) >> np.uint64(40)).astype(np.float64) * (2.0 ** -24)
    return (a + (b - a) * u).astype(np.float32).reshape(shape)


def normal(seed: int, name: str, shape, mean: float, var: float) -> np.ndarray:
    """float32 values from N(mean, var) -- ``var`` is the variance."""
    n = int(np.prod(shape))
    u1 = ((raw_u64(seed, name + "#bm1", n) >> np.uint64(11)).astype(np.float64) + 1.0) * (2.0 ** -53)
    u2 = (raw_u64(seed, name + "#bm2", n) >> np.uint64(11)).astype(np.float64) * (2.0 ** -53)
    z = np.sqrt(-2.0 * np.log(u1)) * np.cos(2.0 * np.pi * u2)
    return (mean + np.sqrt(var) * z).astype(np.float32).reshape(shape)


def int8_uniform(seed: int, name: str, shape, lo: int, hi: int) -> np.ndarray:
    return uniform_int(seed, name, shape, lo, hi).astype(np.int8)


# --------------------------------------------------------------------------
# Workload recipes
# --------------------------------------------------------------------------

@dataclasses.dataclass(frozen=True)
class Workload:
    """One of the five benchmark workloads of the q8ta pages' op set.

    kind:
      ``chain``    fp32 x -> quantize_per_tensor -> q8ta_linear (int8 out)
      ``quantize`` quantize_per_tensor alone, fp32 x drawn normal
      ``gemv``     q8ta_linear_gemv, M == 1, int8 x drawn directly
      ``conv_t``   q8ta_conv2d_transposed, int8 x drawn directly
    ``dims`` holds the sizes and ``params`` the scales, zero-points and the
    parameters of the value distributions (normal parameters are mean and
    VARIANCE).
    """
    name: str
    kind: str
    seed: int
    dims: Dict[str, int]
    params: Dict[str, float]


def output_hw(H_in, W_in, Kh, Kw, s_h, s_w, p_h, p_w, op_h, op_w, d_h=1, d_w=1):
    """Transposed-convolution output size (the usual PyTorch formula)."""
    H = (H_in - 1) * s_h - 2 * p_h + d_h * (Kh - 1) + op_h + 1
    W = (W_in - 1) * s_w - 2 * p_w + d_w * (Kw - 1) + op_w + 1
    return H, W


CONFIGS = {
    # quantize_per_tensor -> q8ta_linear, M=8 K=64 N=32, seed 0
    "linear_chain_8x64x32": Workload(
        "linear_chain_8x64x32", "chain", 0, dict(M=8, K=64, N=32),
        dict(x_mean=0.0, x_var=1.0, in_scale=0.02, in_zp=3, ws_lo=0.002, ws_hi=0.01,
             b_mean=0.0, b_var=0.1, out_scale=0.05, out_zp=-2)),
    # q8ta_linear_gemv M=1 K=4096 N=4096
    "gemv_1x4096x4096": Workload(
        "gemv_1x4096x4096", "gemv", 1, dict(M=1, K=4096, N=4096),
        dict(in_scale=0.02, in_zp=0, ws_lo=0.002, ws_hi=0.01, b_mean=0.0, b_var=0.1,
             out_scale=0.5, out_zp=0)),
    # quantize 64Mi fp32 elements; prefill chain M=2048 K=4096 N=11008
    "quantize_64Mi": Workload(
        "quantize_64Mi", "quantize", 2, dict(numel=64 * 1024 * 1024),
        dict(x_mean=0.0, x_var=3.0, in_scale=0.03, in_zp=-5)),
    "linear_chain_2048x4096x11008": Workload(
        "linear_chain_2048x4096x11008", "chain", 2, dict(M=2048, K=4096, N=11008),
        dict(x_mean=0.0, x_var=3.0, in_scale=0.03, in_zp=-5, ws_lo=0.001, ws_hi=0.005,
             b_mean=0.0, b_var=0.1, out_scale=0.1, out_zp=1)),
    # q8ta_conv2d_transposed N=1 IC=64 32x32 OC=32 K=4 s=2 p=1 -> 64x64
    "conv_t_1x64x32x32_k4s2": Workload(
        "conv_t_1x64x32x32_k4s2", "conv_t", 3,
        dict(N=1, IC=64, H_in=32, W_in=32, OC=32, Kh=4, Kw=4, s=2, p=1, op=0),
        dict(in_scale=0.02, in_zp=4, ws_lo=0.002, ws_hi=0.01, b_mean=0.0, b_var=0.1,
             out_scale=0.08, out_zp=0)),
    # q8ta_conv2d_transposed N=8 IC=256 64x64 OC=128 K=3 s=2 p=1 op=1 -> 128x128
    "conv_t_8x256x64x64_k3s2": Workload(
        "conv_t_8x256x64x64_k3s2", "conv_t", 4,
        dict(N=8, IC=256, H_in=64, W_in=64, OC=128, Kh=3, Kw=3, s=2, p=1, op=1),
        dict(in_scale=0.02, in_zp=-7, ws_lo=0.002, ws_hi=0.01, b_mean=0.0, b_var=0.1,
             out_scale=0.15, out_zp=2)),
}


def linear_inputs(seed: int, M: int, K: int, N: int, *, x_kind: str, p: Dict[str, float]):
    """Inputs of one q8ta_linear problem.

    ``x_kind`` is ``"fp32"`` (x drawn N(x_mean, x_var), to be quantized by the
    caller) or ``"int8"`` (x drawn uniform on [-128, 127]).  The weight is int8
    uniform on [-127, 127] (row-major [N, K]); weight_scales uniform on
    [ws_lo, ws_hi); bias N(b_mean, b_var).
    """
    if x_kind == "fp32":
        x = normal(seed, "x", (M, K), p["x_mean"], p["x_var"])
    else:
        x = int8_uniform(seed, "x", (M, K), -128, 127)
    w = int8_uniform(seed, "w", (N, K), -127, 127)
    ws = uniform_float(seed, "ws", (N,), p["ws_lo"], p["ws_hi"])
    b = normal(seed, "b", (N,), p["b_mean"], p["b_var"])
    return x, w, ws, b


def conv_t_inputs(seed: int, d: Dict[str, int], p: Dict[str, float]):
    """Inputs of one q8ta_conv2d_transposed problem.

    x int8 uniform on [-128, 127] in NCHW; weight int8 uniform on [-127, 127]
    in the pages' [OC, Kh*Kw*IC] layout; weight_scales uniform; bias normal.
    """
    x = int8_uniform(seed, "x", (d["N"], d["IC"], d["H_in"], d["W_in"]), -128, 127)
    w = int8_uniform(seed, "w", (d["OC"], d["Kh"] * d["Kw"] * d["IC"]), -127, 127)
    ws = uniform_float(seed, "ws", (d["OC"],), p["ws_lo"], p["ws_hi"])
    b = normal(seed, "b", (d["OC"],), p["b_mean"], p["b_var"])
    return x, w, ws, b
