"""CPU oracle for the q8ta int8 quantized contraction -- TEST INFRASTRUCTURE.

Only ``tests/``, ``__graft_entry__.smoke()`` and ``bench.py``'s CPU-baseline
leg may import this package.  The CUDA library never loads it and shares no
code with it.

The arithmetic lives in ``q8ta_oracle.c`` (plain C, nested loops, compiled
with ``-O2 -ffp-contract=off``); this module only builds that file into a
shared library and marshals numpy arrays into it.  See the header of
``q8ta_oracle.c`` for the passages of the pages each function follows and the
readings taken where they are silent.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "q8ta_oracle.c")
_LIB = os.path.join(_HERE, "libq8ta_oracle.so")
_lock = threading.Lock()
_lib = None

_CFLAGS = ["-O2", "-std=c11", "-ffp-contract=off", "-fno-fast-math", "-fPIC", "-shared",
           "-Wall", "-Wextra"]


def build(force: bool = False) -> str:
    """Compile the oracle with gcc (no CUDA involved).  Returns the .so path."""
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + f".tmp{os.getpid()}"
        subprocess.check_call(["gcc", *_CFLAGS, _SRC, "-o", tmp, "-lm"])
        os.replace(tmp, _LIB)
    return _LIB


class ConvTShape(ctypes.Structure):
    _fields_ = [(n, ctypes.c_int64) for n in (
        "N", "IC", "H_in", "W_in", "OC", "Kh", "Kw", "ldw", "H_out", "W_out",
        "stride_h", "stride_w", "pad_h", "pad_w", "dil_h", "dil_w", "groups")]


def _load():
    global _lib
    with _lock:
        if _lib is None:
            lib = ctypes.CDLL(build())
            P = ctypes.c_void_p
            I64, I32, D = ctypes.c_int64, ctypes.c_int32, ctypes.c_double
            lib.oracle_quantize_per_tensor.argtypes = [P, I64, D, I32, P]
            lib.oracle_requantize.argtypes = [P, I64, I64, D, P, P, D, I32, ctypes.c_int, P]
            lib.oracle_linear_acc.argtypes = [P, I64, I64, I32, P, I64, I64, P]
            lib.oracle_linear.argtypes = [P, I64, I64, D, I32, P, I64, I64, P, P, D, I32,
                                          ctypes.c_int, P]
            SP = ctypes.POINTER(ConvTShape)
            lib.oracle_conv2d_transposed_acc_gather.argtypes = [P, I32, P, SP, P]
            lib.oracle_conv2d_transposed_acc_scatter.argtypes = [P, I32, P, SP, P]
            lib.oracle_conv2d_transposed_acc_scatter.restype = ctypes.c_int
            lib.oracle_conv2d_transposed.argtypes = [P, D, I32, P, SP, P, P, D, I32, ctypes.c_int,
                                                     P]
            lib.oracle_conv2d_acc.argtypes = [P, I32, P, SP, P]
            lib.oracle_conv2d.argtypes = [P, D, I32, P, SP, P, P, D, I32, ctypes.c_int, P]
            lib.oracle_dequantize_per_tensor.argtypes = [P, I64, D, I32, P]
            for f in ("oracle_quantize_per_tensor", "oracle_requantize", "oracle_linear_acc",
                      "oracle_linear", "oracle_conv2d_transposed_acc_gather",
                      "oracle_conv2d_transposed", "oracle_dequantize_per_tensor",
                      "oracle_conv2d_acc", "oracle_conv2d"):
                getattr(lib, f).restype = None
            _lib = lib
    return _lib


def _ptr(a: np.ndarray):
    return ctypes.c_void_p(a.ctypes.data)


def _c(a, dtype):
    a = np.ascontiguousarray(a, dtype=dtype)
    return a


# ---------------------------------------------------------------------------

def quantize_per_tensor(x, scale: float, zero_point: int) -> np.ndarray:
    """fp32 -> int8: clamp(rne(x * (float)(1/scale)) + zp, -128, 127)."""
    x = _c(x, np.float32)
    out = np.empty(x.shape, np.int8)
    _load().oracle_quantize_per_tensor(_ptr(x), x.size, float(scale), int(zero_point), _ptr(out))
    return out


def dequantize_per_tensor(q, scale: float, zero_point: int) -> np.ndarray:
    q = _c(q, np.int8)
    out = np.empty(q.shape, np.float32)
    _load().oracle_dequantize_per_tensor(_ptr(q), q.size, float(scale), int(zero_point), _ptr(out))
    return out


def _relu_flag(activation) -> int:
    if activation not in ("none", "relu"):
        raise ValueError(f"activation {activation!r}")
    return 1 if activation == "relu" else 0


def requantize(acc, input_scale, weight_scales, bias, output_scale, output_zero_point,
               activation="none"):
    """The dequant/requant epilogue on an int32 [rows, N] accumulator array."""
    acc = _c(acc, np.int32)
    rows, N = acc.shape
    ws = _c(weight_scales, np.float32)
    b = None if bias is None else _c(bias, np.float32)
    out = np.empty((rows, N), np.int8)
    _load().oracle_requantize(_ptr(acc), rows, N, float(input_scale), _ptr(ws),
                              None if b is None else _ptr(b), float(output_scale),
                              int(output_zero_point), _relu_flag(activation), _ptr(out))
    return out


def linear_acc(x, input_zero_point, w) -> np.ndarray:
    """int32 [M, N] accumulators sum_k (x - izp) * w (x [M,K], w [N,K] or [N, ldw])."""
    x = _c(x, np.int8)
    w = _c(w, np.int8)
    M, K = x.shape
    N, ldw = w.shape
    assert ldw >= K
    acc = np.empty((M, N), np.int32)
    _load().oracle_linear_acc(_ptr(x), M, K, int(input_zero_point), _ptr(w), N, ldw, _ptr(acc))
    return acc


def linear(x, input_scale, input_zero_point, w, weight_scales, bias, output_scale,
           output_zero_point, K=None, activation="none") -> np.ndarray:
    """q8ta_linear: int8 [M,K] x int8 [N,K] (row stride may exceed K) -> int8 [M,N]."""
    x = _c(x, np.int8)
    w = _c(w, np.int8)
    M, Kx = x.shape
    N, ldw = w.shape
    K = Kx if K is None else K
    assert K == Kx and ldw >= K
    ws = _c(weight_scales, np.float32)
    b = None if bias is None else _c(bias, np.float32)
    out = np.empty((M, N), np.int8)
    _load().oracle_linear(_ptr(x), M, K, float(input_scale), int(input_zero_point), _ptr(w), N,
                          ldw, _ptr(ws), None if b is None else _ptr(b), float(output_scale),
                          int(output_zero_point), _relu_flag(activation), _ptr(out))
    return out


def _conv_shape(x, w, Kh, Kw, H_out, W_out, stride, pad, dil, groups=1):
    N, IC, H_in, W_in = x.shape
    OC, ldw = w.shape
    assert groups >= 1 and IC % groups == 0 and OC % groups == 0
    assert ldw >= Kh * Kw * (IC // groups)
    return ConvTShape(N, IC, H_in, W_in, OC, Kh, Kw, ldw, H_out, W_out,
                      stride[0], stride[1], pad[0], pad[1], dil[0], dil[1], groups)


def conv2d_transposed_acc(x, input_zero_point, w, Kh, Kw, H_out, W_out, stride, pad,
                          dil=(1, 1), form="gather", groups=1) -> np.ndarray:
    """int32 [N, OC, H_out, W_out] accumulators of the transposed convolution."""
    x = _c(x, np.int8)
    w = _c(w, np.int8)
    s = _conv_shape(x, w, Kh, Kw, H_out, W_out, stride, pad, dil, groups)
    acc = np.empty((s.N, s.OC, H_out, W_out), np.int32)
    lib = _load()
    if form == "gather":
        lib.oracle_conv2d_transposed_acc_gather(_ptr(x), int(input_zero_point), _ptr(w),
                                                ctypes.byref(s), _ptr(acc))
    elif form == "scatter":
        rc = lib.oracle_conv2d_transposed_acc_scatter(_ptr(x), int(input_zero_point), _ptr(w),
                                                      ctypes.byref(s), _ptr(acc))
        if rc != 0:
            raise MemoryError("oracle scatter: allocation failed")
    else:
        raise ValueError(form)
    return acc


def conv2d_transposed(x, input_scale, input_zero_point, w, Kh, Kw, weight_scales, bias,
                      output_scale, output_zero_point, H_out, W_out, stride, pad,
                      dil=(1, 1), groups=1, activation="none") -> np.ndarray:
    """q8ta_conv2d_transposed: int8 NCHW x, int8 [OC, Kh*Kw*IC/groups] w -> int8 NCHW."""
    x = _c(x, np.int8)
    w = _c(w, np.int8)
    s = _conv_shape(x, w, Kh, Kw, H_out, W_out, stride, pad, dil, groups)
    ws = _c(weight_scales, np.float32)
    b = None if bias is None else _c(bias, np.float32)
    out = np.empty((s.N, s.OC, H_out, W_out), np.int8)
    _load().oracle_conv2d_transposed(_ptr(x), float(input_scale), int(input_zero_point),
                                     _ptr(w), ctypes.byref(s), _ptr(ws),
                                     None if b is None else _ptr(b), float(output_scale),
                                     int(output_zero_point), _relu_flag(activation), _ptr(out))
    return out


def conv2d_acc(x, input_zero_point, w, Kh, Kw, H_out, W_out, stride, pad, dil=(1, 1),
               groups=1) -> np.ndarray:
    """int32 [N, OC, H_out, W_out] accumulators of the direct convolution (q8ta_conv2d)."""
    x = _c(x, np.int8)
    w = _c(w, np.int8)
    s = _conv_shape(x, w, Kh, Kw, H_out, W_out, stride, pad, dil, groups)
    acc = np.empty((s.N, s.OC, H_out, W_out), np.int32)
    _load().oracle_conv2d_acc(_ptr(x), int(input_zero_point), _ptr(w), ctypes.byref(s), _ptr(acc))
    return acc


def conv2d(x, input_scale, input_zero_point, w, Kh, Kw, weight_scales, bias, output_scale,
           output_zero_point, H_out, W_out, stride, pad, dil=(1, 1), groups=1,
           activation="none") -> np.ndarray:
    """q8ta_conv2d: int8 NCHW x, int8 [OC, Kh*Kw*IC/groups] w -> int8 NCHW."""
    x = _c(x, np.int8)
    w = _c(w, np.int8)
    s = _conv_shape(x, w, Kh, Kw, H_out, W_out, stride, pad, dil, groups)
    ws = _c(weight_scales, np.float32)
    b = None if bias is None else _c(bias, np.float32)
    out = np.empty((s.N, s.OC, H_out, W_out), np.int8)
    _load().oracle_conv2d(_ptr(x), float(input_scale), int(input_zero_point), _ptr(w),
                          ctypes.byref(s), _ptr(ws), None if b is None else _ptr(b),
                          float(output_scale), int(output_zero_point), _relu_flag(activation),
                          _ptr(out))
    return out
