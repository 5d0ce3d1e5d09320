"""Python binding of the q8ta C ABI (include/q8ta.h) for GB300 (sm_103a).

Argument marshalling only: every step of every op runs in the CUDA kernels
of ``libq8ta.so``.  PyTorch supplies device memory and the current stream.
There is no CPU fallback: if the library is missing, the first call into it
raises ImportError, and every call on a tensor that is not on a CUDA device
raises.

Build the library with ``python -m int8_quantized_q8ta_gb300._build`` (or
``__graft_entry__.build()``).
"""
from __future__ import annotations

import ctypes
import dataclasses
import os
from typing import Optional, Sequence

import torch

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libq8ta.so")

Q8_OK, Q8_ERR_NULL, Q8_ERR_SHAPE, Q8_ERR_ALIGN, Q8_ERR_UNSUPPORTED = 0, 1, 2, 3, 4
Q8_ERR_WORKSPACE, Q8_ERR_CUDA, Q8_ERR_DEVICE, Q8_ERR_ARG = 5, 6, 7, 8

#: every symbol include/q8ta.h declares
EXPORTS = (
    "q8_status_string", "q8_version", "q8_device_error",
    "q8_quantize_per_tensor", "q8_dequantize_per_tensor",
    "q8_linear_workspace_bytes", "q8_linear", "q8_linear_noalloc", "q8_linear_gemv",
    "q8_linear_gemv_packed_weight_bytes", "q8_linear_gemv_pack_weight", "q8_linear_gemv_packed",
    "q8_linear_packed_weight_bytes", "q8_linear_pack_weight",
    "q8_linear_operand_bytes", "q8_linear_prepare_operand", "q8_quantize_to_linear_operand",
    "q8_linear_operand_packed", "q8_linear_packed", "q8_quantize_linear_packed",
    "q8_linear_operand_init", "q8_quantize_linear_fused",
    "q8_linear_packed_acc32", "q8_debug_linear_packed_stall",
    "q8_conv2d_transposed_workspace_bytes", "q8_conv2d_transposed",
    "q8_conv2d_transposed_acc32", "q8_conv2d_transposed_packed_weight_bytes",
    "q8_conv2d_transposed_packed_workspace_bytes", "q8_conv2d_transposed_pack_weight",
    "q8_conv2d_transposed_packed", "q8_conv2d_transposed_packed_acc32",
    "q8_conv2d_workspace_bytes", "q8_conv2d", "q8_conv2d_acc32", "q8_conv2d_packed_weight_bytes",
    "q8_conv2d_packed_workspace_bytes", "q8_conv2d_pack_weight", "q8_conv2d_packed",
    "q8_conv2d_packed_acc32",
)


class Q8Error(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        super().__init__(f"{where}: {_lib.q8_status_string(status).decode()}")


class ConvTShape(ctypes.Structure):
    """Mirror of q8_conv2d_transposed_shape."""
    _fields_ = [(n, ctypes.c_int64) for n in (
        "N", "IC", "H_in", "W_in", "OC", "Kh", "Kw", "weight_row_stride", "H_out", "W_out",
        "stride_h", "stride_w", "pad_h", "pad_w", "output_padding_h", "output_padding_w",
        "dilation_h", "dilation_w", "groups")]


class ConvShape(ctypes.Structure):
    """Mirror of q8_conv2d_shape."""
    _fields_ = [(n, ctypes.c_int64) for n in (
        "N", "IC", "H_in", "W_in", "OC", "Kh", "Kw", "weight_row_stride", "H_out", "W_out",
        "stride_h", "stride_w", "pad_h", "pad_w", "dilation_h", "dilation_w", "groups")]


def _load() -> ctypes.CDLL:
    if not os.path.exists(LIB_PATH):
        raise ImportError(
            f"{LIB_PATH} is missing: build it with `python -m int8_quantized_q8ta_gb300._build` "
            "(the q8ta ops have no CPU fallback)")
    lib = ctypes.CDLL(LIB_PATH)
    P, I64, I32, D, S = (ctypes.c_void_p, ctypes.c_int64, ctypes.c_int32, ctypes.c_double,
                         ctypes.c_size_t)
    C = ctypes.c_char_p
    SP = ctypes.POINTER(ConvTShape)
    DP = ctypes.POINTER(ConvShape)
    sig = {
        "q8_status_string": (ctypes.c_char_p, [ctypes.c_int]),
        "q8_version": (ctypes.c_int, []),
        "q8_device_error": (ctypes.c_int, [ctypes.POINTER(ctypes.c_uint32), ctypes.c_int]),
        "q8_quantize_per_tensor": (ctypes.c_int, [P, I64, D, I32, P, P]),
        "q8_dequantize_per_tensor": (ctypes.c_int, [P, I64, D, I32, P, P]),
        "q8_linear_workspace_bytes": (S, [I64, I64, I64]),
        "q8_linear": (ctypes.c_int, [P, I64, I64, D, I32, P, I64, P, P, P, D, I32, C, P, P, S, P]),
        "q8_linear_gemv": (ctypes.c_int, [P, I64, I64, D, I32, P, I64, P, P, P, D, I32, C, P, P, S,
                                          P]),
        "q8_linear_noalloc": (ctypes.c_int, [P, I64, I64, D, I32, P, I64, P, P, P, D, I32, C, P,
                                             P]),
        "q8_linear_gemv_packed_weight_bytes": (S, [I64, I64]),
        "q8_linear_gemv_pack_weight": (ctypes.c_int, [P, I64, I64, P, S, P]),
        "q8_linear_gemv_packed": (ctypes.c_int, [P, I64, D, I32, P, I64, P, P, D, I32, C, P, P]),
        "q8_linear_packed_weight_bytes": (S, [I64, I64]),
        "q8_linear_pack_weight": (ctypes.c_int, [P, I64, I64, P, S, P]),
        "q8_linear_operand_bytes": (S, [I64, I64]),
        "q8_linear_prepare_operand": (ctypes.c_int, [P, I64, I64, I32, P, S, P]),
        "q8_quantize_to_linear_operand": (ctypes.c_int, [P, I64, I64, D, I32, P, P, S, P]),
        "q8_linear_operand_packed": (ctypes.c_int, [P, I64, I64, D, P, I64, P, P, D, I32, C, P,
                                                    P]),
        "q8_linear_packed": (ctypes.c_int, [P, I64, I64, D, I32, P, I64, P, P, D, I32, C, P, P, S,
                                            P]),
        "q8_quantize_linear_packed": (ctypes.c_int, [P, I64, I64, D, I32, P, I64, P, P, D, I32, C,
                                                     P, P, P, S, P]),
        "q8_linear_packed_acc32": (ctypes.c_int, [P, I64, I64, I32, P, I64, P, P, S, P]),
        "q8_linear_operand_init": (ctypes.c_int, [P, I64, I64, S, P]),
        "q8_quantize_linear_fused": (ctypes.c_int, [P, I64, I64, D, I32, P, I64, P, P, D, I32, C,
                                                    P, P, P, S, P]),
        "q8_debug_linear_packed_stall": (ctypes.c_int, [P, I64, I64, I32, P, I64, P, P, S,
                                                        ctypes.c_uint64, I64, P]),
        "q8_conv2d_transposed_workspace_bytes": (S, [SP]),
        "q8_conv2d_transposed": (ctypes.c_int, [P, SP, D, I32, P, P, P, P, D, I32, C, P, P, S, P]),
        "q8_conv2d_transposed_acc32": (ctypes.c_int, [P, SP, I32, P, P, P, S, P]),
        "q8_conv2d_transposed_packed_weight_bytes": (S, [SP]),
        "q8_conv2d_transposed_packed_workspace_bytes": (S, [SP]),
        "q8_conv2d_transposed_pack_weight": (ctypes.c_int, [P, SP, P, S, P]),
        "q8_conv2d_transposed_packed": (ctypes.c_int, [P, SP, D, I32, P, P, P, D, I32, C, P, P, S,
                                                       P]),
        "q8_conv2d_transposed_packed_acc32": (ctypes.c_int, [P, SP, I32, P, P, P, S, P]),
        "q8_conv2d_workspace_bytes": (S, [DP]),
        "q8_conv2d": (ctypes.c_int, [P, DP, D, I32, P, P, P, D, I32, C, P, P, S, P]),
        "q8_conv2d_acc32": (ctypes.c_int, [P, DP, I32, P, P, P, S, P]),
        "q8_conv2d_packed_weight_bytes": (S, [DP]),
        "q8_conv2d_packed_workspace_bytes": (S, [DP]),
        "q8_conv2d_pack_weight": (ctypes.c_int, [P, DP, P, S, P]),
        "q8_conv2d_packed": (ctypes.c_int, [P, DP, D, I32, P, P, P, D, I32, C, P, P, S, P]),
        "q8_conv2d_packed_acc32": (ctypes.c_int, [P, DP, I32, P, P, P, S, P]),
    }
    for name, (res, args) in sig.items():
        f = getattr(lib, name)
        f.restype = res
        f.argtypes = args
    return lib


_lib_handle: Optional[ctypes.CDLL] = None


def lib() -> ctypes.CDLL:
    """The loaded C library (for callers that pass raw pointers).  Loaded on
    first use; raises ImportError if libq8ta.so has not been built."""
    global _lib_handle
    if _lib_handle is None:
        _lib_handle = _load()
    return _lib_handle


class _LazyLib:
    def __getattr__(self, name):
        return getattr(lib(), name)


_lib = _LazyLib()


# ---------------------------------------------------------------------------
# marshalling helpers
# ---------------------------------------------------------------------------

def _ptr(t: Optional[torch.Tensor]):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(t: torch.Tensor):
    return ctypes.c_void_p(torch.cuda.current_stream(t.device).cuda_stream)


def _need(t: torch.Tensor, dtype, name: str):
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor (the q8ta ops run only on the GPU)")
    if t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    return t


def _check(status: int, where: str):
    if status != Q8_OK:
        raise Q8Error(status, where)


def _workspace(nbytes: int, device, workspace: Optional[torch.Tensor]):
    if nbytes == 0:
        return None
    if workspace is not None:
        _need(workspace, torch.uint8, "workspace")
        if workspace.numel() < nbytes:
            raise ValueError(f"workspace needs {nbytes} bytes, got {workspace.numel()}")
        return workspace
    return torch.empty(nbytes, dtype=torch.uint8, device=device)


def device_error(clear: bool = True) -> int:
    """Synchronize and return the library's device error word (0 = none)."""
    code = ctypes.c_uint32(0)
    _check(_lib.q8_device_error(ctypes.byref(code), int(clear)), "q8_device_error")
    return int(code.value)


# ---------------------------------------------------------------------------
# quantize / dequantize
# ---------------------------------------------------------------------------

def quantize_per_tensor(x: torch.Tensor, scale: float, zero_point: int,
                        out: Optional[torch.Tensor] = None) -> torch.Tensor:
    _need(x, torch.float32, "x")
    out = torch.empty(x.shape, dtype=torch.int8, device=x.device) if out is None else out
    _need(out, torch.int8, "out")
    _check(_lib.q8_quantize_per_tensor(_ptr(x), x.numel(), float(scale), int(zero_point),
                                       _ptr(out), _stream(x)), "q8_quantize_per_tensor")
    return out


def dequantize_per_tensor(q: torch.Tensor, scale: float, zero_point: int,
                          out: Optional[torch.Tensor] = None) -> torch.Tensor:
    _need(q, torch.int8, "q")
    out = torch.empty(q.shape, dtype=torch.float32, device=q.device) if out is None else out
    _need(out, torch.float32, "out")
    _check(_lib.q8_dequantize_per_tensor(_ptr(q), q.numel(), float(scale), int(zero_point),
                                         _ptr(out), _stream(q)), "q8_dequantize_per_tensor")
    return out


# ---------------------------------------------------------------------------
# q8ta_linear
# ---------------------------------------------------------------------------

def _linear_common(fn_name, x, input_scale, input_zero_point, weight, weight_sums, weight_scales,
                   bias, output_scale, output_zero_point, activation, out, workspace):
    _need(x, torch.int8, "x")
    _need(weight, torch.int8, "weight")
    _need(weight_scales, torch.float32, "weight_scales")
    if bias is not None:
        _need(bias, torch.float32, "bias")
    if weight_sums is not None:
        _need(weight_sums, torch.int32, "weight_sums")
    M, K = x.shape
    N = weight.shape[0]
    out = torch.empty((M, N), dtype=torch.int8, device=x.device) if out is None else out
    _need(out, torch.int8, "out")
    nbytes = _lib.q8_linear_workspace_bytes(M, K, N) if fn_name == "q8_linear" else 0
    ws = _workspace(nbytes, x.device, workspace)
    st = getattr(_lib, fn_name)(
        _ptr(x), M, K, float(input_scale), int(input_zero_point), _ptr(weight), N,
        _ptr(weight_sums), _ptr(weight_scales), _ptr(bias), float(output_scale),
        int(output_zero_point), activation.encode(), _ptr(out), _ptr(ws), nbytes, _stream(x))
    _check(st, fn_name)
    return out


def linear(x, input_scale, input_zero_point, weight, weight_sums, weight_scales, bias,
           output_scale, output_zero_point, activation="none", out=None, workspace=None):
    """q8ta_linear: int8 x [M, K], int8 weight [N, K] -> int8 [M, N]."""
    return _linear_common("q8_linear", x, input_scale, input_zero_point, weight, weight_sums,
                          weight_scales, bias, output_scale, output_zero_point, activation, out,
                          workspace)


def linear_gemv(x, input_scale, input_zero_point, weight, weight_sums, weight_scales, bias,
                output_scale, output_zero_point, activation="none", out=None):
    """q8ta_linear_gemv: the M == 1 case."""
    return _linear_common("q8_linear_gemv", x, input_scale, input_zero_point, weight,
                          weight_sums, weight_scales, bias, output_scale, output_zero_point,
                          activation, out, None)


@dataclasses.dataclass
class PackedWeight:
    """A q8ta_linear weight in the tensor cores' bf16 layout (see
    q8_linear_pack_weight): ``data`` is a uint8 CUDA buffer."""
    data: torch.Tensor
    N: int
    K: int


def pack_weight(weight: torch.Tensor) -> PackedWeight:
    _need(weight, torch.int8, "weight")
    N, K = weight.shape
    nbytes = _lib.q8_linear_packed_weight_bytes(N, K)
    buf = torch.empty(nbytes, dtype=torch.uint8, device=weight.device)
    _check(_lib.q8_linear_pack_weight(_ptr(weight), N, K, _ptr(buf), nbytes, _stream(weight)),
           "q8_linear_pack_weight")
    return PackedWeight(buf, N, K)


@dataclasses.dataclass
class PackedGemvWeight:
    """A q8ta_linear_gemv weight packed once at load time (see
    q8_linear_gemv_pack_weight): ``data`` is a uint8 CUDA buffer."""
    data: torch.Tensor
    N: int
    K: int


def pack_gemv_weight(weight: torch.Tensor) -> PackedGemvWeight:
    _need(weight, torch.int8, "weight")
    N, K = weight.shape
    nbytes = _lib.q8_linear_gemv_packed_weight_bytes(N, K)
    buf = torch.empty(nbytes, dtype=torch.uint8, device=weight.device)
    _check(_lib.q8_linear_gemv_pack_weight(_ptr(weight), N, K, _ptr(buf), nbytes,
                                           _stream(weight)), "q8_linear_gemv_pack_weight")
    return PackedGemvWeight(buf, N, K)


def linear_gemv_packed(x, input_scale, input_zero_point, packed: PackedGemvWeight, weight_scales,
                       bias, output_scale, output_zero_point, activation="none", out=None):
    """q8ta_linear_gemv (M == 1) from a packed weight."""
    _need(x, torch.int8, "x")
    _need(weight_scales, torch.float32, "weight_scales")
    if bias is not None:
        _need(bias, torch.float32, "bias")
    if x.numel() != packed.K:
        raise ValueError(f"x has {x.numel()} elements, the packed weight K={packed.K}")
    out = torch.empty((1, packed.N), dtype=torch.int8, device=x.device) if out is None else out
    _need(out, torch.int8, "out")
    _check(_lib.q8_linear_gemv_packed(_ptr(x), packed.K, float(input_scale),
                                      int(input_zero_point), _ptr(packed.data), packed.N,
                                      _ptr(weight_scales), _ptr(bias), float(output_scale),
                                      int(output_zero_point), activation.encode(), _ptr(out),
                                      _stream(x)), "q8_linear_gemv_packed")
    return out


def linear_packed(x, input_scale, input_zero_point, packed: PackedWeight, weight_scales, bias,
                  output_scale, output_zero_point, activation="none", out=None, workspace=None):
    _need(x, torch.int8, "x")
    _need(weight_scales, torch.float32, "weight_scales")
    if bias is not None:
        _need(bias, torch.float32, "bias")
    M, K = x.shape
    if K != packed.K:
        raise ValueError(f"x has K={K}, packed weight has K={packed.K}")
    out = torch.empty((M, packed.N), dtype=torch.int8, device=x.device) if out is None else out
    _need(out, torch.int8, "out")
    nbytes = _lib.q8_linear_operand_bytes(M, K)
    ws = _workspace(nbytes, x.device, workspace)
    _check(_lib.q8_linear_packed(_ptr(x), M, K, float(input_scale), int(input_zero_point),
                                 _ptr(packed.data), packed.N, _ptr(weight_scales), _ptr(bias),
                                 float(output_scale), int(output_zero_point), activation.encode(),
                                 _ptr(out), _ptr(ws), nbytes, _stream(x)), "q8_linear_packed")
    return out


def quantize_linear_packed(x_f32, input_scale, input_zero_point, packed: PackedWeight,
                           weight_scales, bias, output_scale, output_zero_point,
                           activation="none", x_q=None, out=None, workspace=None,
                           want_x_q: bool = True):
    """fp32 x -> quantize_per_tensor -> q8ta_linear in one call.
    Returns (x_q, out); x_q is None when want_x_q is False and x_q is None."""
    _need(x_f32, torch.float32, "x_f32")
    _need(weight_scales, torch.float32, "weight_scales")
    if bias is not None:
        _need(bias, torch.float32, "bias")
    M, K = x_f32.shape
    if K != packed.K:
        raise ValueError(f"x has K={K}, packed weight has K={packed.K}")
    if x_q is None and want_x_q:
        x_q = torch.empty((M, K), dtype=torch.int8, device=x_f32.device)
    if x_q is not None:
        _need(x_q, torch.int8, "x_q")
    out = torch.empty((M, packed.N), dtype=torch.int8, device=x_f32.device) if out is None else out
    _need(out, torch.int8, "out")
    nbytes = _lib.q8_linear_operand_bytes(M, K)
    ws = _workspace(nbytes, x_f32.device, workspace)
    _check(_lib.q8_quantize_linear_packed(
        _ptr(x_f32), M, K, float(input_scale), int(input_zero_point), _ptr(packed.data), packed.N,
        _ptr(weight_scales), _ptr(bias), float(output_scale), int(output_zero_point),
        activation.encode(), _ptr(x_q), _ptr(out), _ptr(ws), nbytes, _stream(x_f32)),
        "q8_quantize_linear_packed")
    return x_q, out


@dataclasses.dataclass
class Operand:
    """A prepared q8ta_linear activation operand (bf16 of x - input_zero_point)."""
    data: torch.Tensor
    M: int
    K: int


def operand_buffer(M: int, K: int, device) -> Operand:
    """An operand buffer for M x K activations, its trailer prepared for the
    fused quantize -> linear kernel as well (q8_linear_operand_init)."""
    data = torch.empty(_lib.q8_linear_operand_bytes(M, K), dtype=torch.uint8, device=device)
    _check(_lib.q8_linear_operand_init(_ptr(data), M, K, data.numel(), _stream(data)),
           "q8_linear_operand_init")
    return Operand(data, M, K)


def quantize_linear_fused(x_f32, input_scale, input_zero_point, packed: PackedWeight,
                          weight_scales, bias, output_scale, output_zero_point, activation="none",
                          x_q=None, out=None, operand: Optional[Operand] = None,
                          want_x_q: bool = True):
    """fp32 x -> quantize_per_tensor -> q8ta_linear in one kernel (the GEMM's
    warps quantize x into the operand, chunk by chunk along K).  Returns
    (x_q, out, operand); pass the operand back in to reuse it."""
    _need(x_f32, torch.float32, "x_f32")
    _need(weight_scales, torch.float32, "weight_scales")
    if bias is not None:
        _need(bias, torch.float32, "bias")
    M, K = x_f32.shape
    if K != packed.K:
        raise ValueError(f"x has K={K}, packed weight has K={packed.K}")
    if x_q is None and want_x_q:
        x_q = torch.empty((M, K), dtype=torch.int8, device=x_f32.device)
    if x_q is not None:
        _need(x_q, torch.int8, "x_q")
    out = torch.empty((M, packed.N), dtype=torch.int8, device=x_f32.device) if out is None else out
    _need(out, torch.int8, "out")
    operand = operand_buffer(M, K, x_f32.device) if operand is None else operand
    if (operand.M, operand.K) != (M, K):
        raise ValueError(f"operand is for {operand.M}x{operand.K}, x is {M}x{K}")
    _check(_lib.q8_quantize_linear_fused(
        _ptr(x_f32), M, K, float(input_scale), int(input_zero_point), _ptr(packed.data), packed.N,
        _ptr(weight_scales), _ptr(bias), float(output_scale), int(output_zero_point),
        activation.encode(), _ptr(x_q), _ptr(out), _ptr(operand.data), operand.data.numel(),
        _stream(x_f32)), "q8_quantize_linear_fused")
    return x_q, out, operand


def prepare_operand(x, input_zero_point, operand: Optional[Operand] = None) -> Operand:
    _need(x, torch.int8, "x")
    M, K = x.shape
    operand = operand_buffer(M, K, x.device) if operand is None else operand
    _check(_lib.q8_linear_prepare_operand(_ptr(x), M, K, int(input_zero_point),
                                          _ptr(operand.data), operand.data.numel(), _stream(x)),
           "q8_linear_prepare_operand")
    return operand


def quantize_to_operand(x_f32, input_scale, input_zero_point, x_q=None,
                        operand: Optional[Operand] = None):
    """quantize_per_tensor fused with the operand preparation; returns (x_q, operand)."""
    _need(x_f32, torch.float32, "x_f32")
    M, K = x_f32.shape
    if x_q is not None:
        _need(x_q, torch.int8, "x_q")
    operand = operand_buffer(M, K, x_f32.device) if operand is None else operand
    _check(_lib.q8_quantize_to_linear_operand(_ptr(x_f32), M, K, float(input_scale),
                                              int(input_zero_point), _ptr(x_q),
                                              _ptr(operand.data), operand.data.numel(),
                                              _stream(x_f32)), "q8_quantize_to_linear_operand")
    return x_q, operand


def linear_operand_packed(operand: Operand, input_scale, packed: PackedWeight, weight_scales,
                          bias, output_scale, output_zero_point, activation="none", out=None):
    """The q8ta_linear contraction + epilogue from a prepared operand (one kernel)."""
    _need(weight_scales, torch.float32, "weight_scales")
    if bias is not None:
        _need(bias, torch.float32, "bias")
    if operand.K != packed.K:
        raise ValueError(f"operand has K={operand.K}, packed weight has K={packed.K}")
    dev = operand.data.device
    out = torch.empty((operand.M, packed.N), dtype=torch.int8, device=dev) if out is None else out
    _need(out, torch.int8, "out")
    _check(_lib.q8_linear_operand_packed(_ptr(operand.data), operand.M, operand.K,
                                         float(input_scale), _ptr(packed.data), packed.N,
                                         _ptr(weight_scales), _ptr(bias), float(output_scale),
                                         int(output_zero_point), activation.encode(), _ptr(out),
                                         _stream(operand.data)), "q8_linear_operand_packed")
    return out


def linear_packed_acc32(x, input_zero_point, packed: PackedWeight, out=None, workspace=None):
    """Exact int32 accumulators sum_k (x - zp) * w of q8ta_linear."""
    _need(x, torch.int8, "x")
    M, K = x.shape
    out = torch.empty((M, packed.N), dtype=torch.int32, device=x.device) if out is None else out
    _need(out, torch.int32, "out")
    nbytes = _lib.q8_linear_operand_bytes(M, K)
    ws = _workspace(nbytes, x.device, workspace)
    _check(_lib.q8_linear_packed_acc32(_ptr(x), M, K, int(input_zero_point), _ptr(packed.data),
                                       packed.N, _ptr(out), _ptr(ws), nbytes, _stream(x)),
           "q8_linear_packed_acc32")
    return out


def debug_linear_packed_stall(x, input_zero_point, packed: PackedWeight, wait_limit_ns,
                              skip_fill, out=None, workspace=None):
    """Failure-detection test: linear_packed_acc32 with a short barrier-wait
    limit and one TMA ring fill left out, so a bounded wait runs out (the
    device error word then holds its code).  Returns the (partly written)
    accumulator tensor."""
    _need(x, torch.int8, "x")
    M, K = x.shape
    out = torch.zeros((M, packed.N), dtype=torch.int32, device=x.device) if out is None else out
    _need(out, torch.int32, "out")
    nbytes = _lib.q8_linear_operand_bytes(M, K)
    ws = _workspace(nbytes, x.device, workspace)
    _check(_lib.q8_debug_linear_packed_stall(_ptr(x), M, K, int(input_zero_point),
                                             _ptr(packed.data), packed.N, _ptr(out), _ptr(ws),
                                             nbytes, int(wait_limit_ns), int(skip_fill),
                                             _stream(x)), "q8_debug_linear_packed_stall")
    return out


# ---------------------------------------------------------------------------
# q8ta_conv2d_transposed
# ---------------------------------------------------------------------------

def _pair(v) -> Sequence[int]:
    return (int(v), int(v)) if isinstance(v, int) else (int(v[0]), int(v[1]))


def conv_t_shape(x_shape, weight_shape, Kh, Kw, H_out, W_out, stride=1, padding=0,
                 output_padding=0, dilation=1, groups=1) -> ConvTShape:
    N, IC, H_in, W_in = x_shape
    OC, ldw = weight_shape
    sh, sw = _pair(stride)
    ph, pw = _pair(padding)
    oph, opw = _pair(output_padding)
    dh, dw = _pair(dilation)
    return ConvTShape(N, IC, H_in, W_in, OC, Kh, Kw, ldw, H_out, W_out, sh, sw, ph, pw, oph, opw,
                      dh, dw, int(groups))


def conv2d_transposed(x, input_scale, input_zero_point, weight, weight_sums, weight_scales, bias,
                      output_scale, output_zero_point, kernel_size, stride=1, padding=0,
                      output_padding=0, dilation=1, groups=1, activation="none",
                      output_size=None, out=None, workspace=None):
    """q8ta_conv2d_transposed: int8 NCHW x, int8 weight [OC, Kh*Kw*IC] -> int8 NCHW.
    ``output_size`` (H_out, W_out) defaults to the usual transposed-conv size."""
    _need(x, torch.int8, "x")
    _need(weight, torch.int8, "weight")
    _need(weight_scales, torch.float32, "weight_scales")
    if bias is not None:
        _need(bias, torch.float32, "bias")
    Kh, Kw = _pair(kernel_size)
    if output_size is None:
        sh, sw = _pair(stride)
        ph, pw = _pair(padding)
        oph, opw = _pair(output_padding)
        dh, dw = _pair(dilation)
        output_size = ((x.shape[2] - 1) * sh - 2 * ph + dh * (Kh - 1) + oph + 1,
                       (x.shape[3] - 1) * sw - 2 * pw + dw * (Kw - 1) + opw + 1)
    H_out, W_out = output_size
    shape = conv_t_shape(tuple(x.shape), tuple(weight.shape), Kh, Kw, H_out, W_out, stride,
                         padding, output_padding, dilation, groups)
    if out is None:
        out = torch.empty((x.shape[0], weight.shape[0], H_out, W_out), dtype=torch.int8,
                          device=x.device)
    _need(out, torch.int8, "out")
    nbytes = _lib.q8_conv2d_transposed_workspace_bytes(ctypes.byref(shape))
    ws = _workspace(nbytes, x.device, workspace)
    _check(_lib.q8_conv2d_transposed(
        _ptr(x), ctypes.byref(shape), float(input_scale), int(input_zero_point), _ptr(weight),
        _ptr(weight_sums), _ptr(weight_scales), _ptr(bias), float(output_scale),
        int(output_zero_point), activation.encode(), _ptr(out), _ptr(ws), nbytes, _stream(x)),
        "q8_conv2d_transposed")
    return out


def conv2d_transposed_acc32(x, input_zero_point, weight, kernel_size, output_size, stride=1,
                            padding=0, dilation=1, groups=1, out=None, workspace=None):
    """Exact int32 accumulators of q8ta_conv2d_transposed."""
    _need(x, torch.int8, "x")
    _need(weight, torch.int8, "weight")
    Kh, Kw = _pair(kernel_size)
    H_out, W_out = output_size
    shape = conv_t_shape(tuple(x.shape), tuple(weight.shape), Kh, Kw, H_out, W_out, stride,
                         padding, 0, dilation, groups)
    if out is None:
        out = torch.empty((x.shape[0], weight.shape[0], H_out, W_out), dtype=torch.int32,
                          device=x.device)
    _need(out, torch.int32, "out")
    nbytes = _lib.q8_conv2d_transposed_workspace_bytes(ctypes.byref(shape))
    ws = _workspace(nbytes, x.device, workspace)
    _check(_lib.q8_conv2d_transposed_acc32(_ptr(x), ctypes.byref(shape), int(input_zero_point),
                                           _ptr(weight), _ptr(out), _ptr(ws), nbytes, _stream(x)),
           "q8_conv2d_transposed_acc32")
    return out


@dataclasses.dataclass
class PackedConvWeight:
    """A convolution weight in the tensor cores' bf16 layout (see
    q8_conv2d_transposed_pack_weight / q8_conv2d_pack_weight)."""
    data: torch.Tensor
    transposed: bool
    OC: int
    IC: int
    Kh: int
    Kw: int
    groups: int


def _pack_shape(transposed, weight, in_channels, Kh, Kw, groups):
    # the packed layout depends on the weight only; a minimal valid problem
    # around it satisfies the shape guards
    OC, ldw = weight.shape
    if transposed:
        return ConvTShape(1, in_channels, 1, 1, OC, Kh, Kw, ldw, 1, 4, 1, 1, 0, 0, 0, 0, 1, 1,
                          int(groups))
    return ConvShape(1, in_channels, 1, 1, OC, Kh, Kw, ldw, 1, 4, 1, 1, 0, 0, 1, 1, int(groups))


def _pack_conv(transposed, weight, in_channels, kernel_size, groups):
    _need(weight, torch.int8, "weight")
    Kh, Kw = _pair(kernel_size)
    shape = _pack_shape(transposed, weight, in_channels, Kh, Kw, groups)
    pre = "q8_conv2d_transposed" if transposed else "q8_conv2d"
    nbytes = getattr(_lib, pre + "_packed_weight_bytes")(ctypes.byref(shape))
    if nbytes == 0:
        raise Q8Error(Q8_ERR_SHAPE, pre + "_packed_weight_bytes")
    data = torch.empty(nbytes, dtype=torch.uint8, device=weight.device)
    _check(getattr(_lib, pre + "_pack_weight")(_ptr(weight), ctypes.byref(shape), _ptr(data),
                                                nbytes, _stream(weight)), pre + "_pack_weight")
    return PackedConvWeight(data, transposed, weight.shape[0], in_channels, Kh, Kw, int(groups))


def pack_conv2d_transposed_weight(weight, in_channels, kernel_size, groups=1) -> PackedConvWeight:
    """Pack a q8ta_conv2d_transposed weight [OC, Kh*Kw*IC/groups] once."""
    return _pack_conv(True, weight, in_channels, kernel_size, groups)


def pack_conv2d_weight(weight, in_channels, kernel_size, groups=1) -> PackedConvWeight:
    """Pack a q8ta_conv2d weight [OC, Kh*Kw*IC/groups] once."""
    return _pack_conv(False, weight, in_channels, kernel_size, groups)


def conv2d_transposed_packed(x, input_scale, input_zero_point, packed: PackedConvWeight,
                             weight_scales, bias, output_scale, output_zero_point, stride=1,
                             padding=0, output_padding=0, dilation=1, activation="none",
                             output_size=None, out=None, workspace=None):
    """q8ta_conv2d_transposed from a packed weight."""
    if not packed.transposed:
        raise ValueError("packed weight is a q8ta_conv2d weight")
    _need(x, torch.int8, "x")
    _need(weight_scales, torch.float32, "weight_scales")
    if bias is not None:
        _need(bias, torch.float32, "bias")
    if x.shape[1] != packed.IC:
        raise ValueError(f"x has {x.shape[1]} channels, the packed weight {packed.IC}")
    Kh, Kw = packed.Kh, packed.Kw
    if output_size is None:
        sh, sw = _pair(stride)
        ph, pw = _pair(padding)
        oph, opw = _pair(output_padding)
        dh, dw = _pair(dilation)
        output_size = ((x.shape[2] - 1) * sh - 2 * ph + dh * (Kh - 1) + oph + 1,
                       (x.shape[3] - 1) * sw - 2 * pw + dw * (Kw - 1) + opw + 1)
    H_out, W_out = output_size
    ldw = Kh * Kw * (packed.IC // packed.groups)
    shape = conv_t_shape(tuple(x.shape), (packed.OC, ldw), Kh, Kw, H_out, W_out, stride, padding,
                         output_padding, dilation, packed.groups)
    if out is None:
        out = torch.empty((x.shape[0], packed.OC, H_out, W_out), dtype=torch.int8, device=x.device)
    _need(out, torch.int8, "out")
    nbytes = _lib.q8_conv2d_transposed_packed_workspace_bytes(ctypes.byref(shape))
    ws = _workspace(nbytes, x.device, workspace)
    _check(_lib.q8_conv2d_transposed_packed(
        _ptr(x), ctypes.byref(shape), float(input_scale), int(input_zero_point),
        _ptr(packed.data), _ptr(weight_scales), _ptr(bias), float(output_scale),
        int(output_zero_point), activation.encode(), _ptr(out), _ptr(ws), nbytes, _stream(x)),
        "q8_conv2d_transposed_packed")
    return out


def conv2d_transposed_packed_acc32(x, input_zero_point, packed: PackedConvWeight, output_size,
                                   stride=1, padding=0, dilation=1, out=None, workspace=None):
    """Exact int32 accumulators of q8ta_conv2d_transposed from a packed weight."""
    if not packed.transposed:
        raise ValueError("packed weight is a q8ta_conv2d weight")
    _need(x, torch.int8, "x")
    if x.shape[1] != packed.IC:
        raise ValueError(f"x has {x.shape[1]} channels, the packed weight {packed.IC}")
    H_out, W_out = output_size
    ldw = packed.Kh * packed.Kw * (packed.IC // packed.groups)
    shape = conv_t_shape(tuple(x.shape), (packed.OC, ldw), packed.Kh, packed.Kw, H_out, W_out,
                         stride, padding, 0, dilation, packed.groups)
    if out is None:
        out = torch.empty((x.shape[0], packed.OC, H_out, W_out), dtype=torch.int32,
                          device=x.device)
    _need(out, torch.int32, "out")
    nbytes = _lib.q8_conv2d_transposed_packed_workspace_bytes(ctypes.byref(shape))
    ws = _workspace(nbytes, x.device, workspace)
    _check(_lib.q8_conv2d_transposed_packed_acc32(
        _ptr(x), ctypes.byref(shape), int(input_zero_point), _ptr(packed.data), _ptr(out),
        _ptr(ws), nbytes, _stream(x)), "q8_conv2d_transposed_packed_acc32")
    return out


# ---------------------------------------------------------------------------
# q8ta_conv2d (the direct convolution)
# ---------------------------------------------------------------------------
def conv2d_shape(x_shape, weight_shape, Kh, Kw, H_out, W_out, stride=1, padding=0, dilation=1,
                 groups=1) -> ConvShape:
    N, IC, H_in, W_in = x_shape
    OC, ldw = weight_shape
    sh, sw = _pair(stride)
    ph, pw = _pair(padding)
    dh, dw = _pair(dilation)
    return ConvShape(N, IC, H_in, W_in, OC, Kh, Kw, ldw, H_out, W_out, sh, sw, ph, pw, dh, dw,
                     int(groups))


def conv2d_output_size(H_in, W_in, kernel_size, stride=1, padding=0, dilation=1):
    Kh, Kw = _pair(kernel_size)
    sh, sw = _pair(stride)
    ph, pw = _pair(padding)
    dh, dw = _pair(dilation)
    return ((H_in + 2 * ph - dh * (Kh - 1) - 1) // sh + 1,
            (W_in + 2 * pw - dw * (Kw - 1) - 1) // sw + 1)


def conv2d(x, input_scale, input_zero_point, weight, weight_scales, bias, output_scale,
           output_zero_point, kernel_size, stride=1, padding=0, dilation=1, groups=1,
           activation="none", output_size=None, out=None, workspace=None):
    """q8ta_conv2d: int8 NCHW x, int8 weight [OC, Kh*Kw*IC/groups] -> int8 NCHW."""
    _need(x, torch.int8, "x")
    _need(weight, torch.int8, "weight")
    _need(weight_scales, torch.float32, "weight_scales")
    if bias is not None:
        _need(bias, torch.float32, "bias")
    Kh, Kw = _pair(kernel_size)
    if output_size is None:
        output_size = conv2d_output_size(x.shape[2], x.shape[3], kernel_size, stride, padding,
                                         dilation)
    H_out, W_out = output_size
    shape = conv2d_shape(tuple(x.shape), tuple(weight.shape), Kh, Kw, H_out, W_out, stride,
                         padding, dilation, groups)
    if out is None:
        out = torch.empty((x.shape[0], weight.shape[0], H_out, W_out), dtype=torch.int8,
                          device=x.device)
    _need(out, torch.int8, "out")
    nbytes = _lib.q8_conv2d_workspace_bytes(ctypes.byref(shape))
    ws = _workspace(nbytes, x.device, workspace)
    _check(_lib.q8_conv2d(
        _ptr(x), ctypes.byref(shape), float(input_scale), int(input_zero_point), _ptr(weight),
        _ptr(weight_scales), _ptr(bias), float(output_scale), int(output_zero_point),
        activation.encode(), _ptr(out), _ptr(ws), nbytes, _stream(x)), "q8_conv2d")
    return out


def conv2d_acc32(x, input_zero_point, weight, kernel_size, output_size=None, stride=1, padding=0,
                 dilation=1, groups=1, out=None, workspace=None):
    """Exact int32 accumulators of q8ta_conv2d."""
    _need(x, torch.int8, "x")
    _need(weight, torch.int8, "weight")
    Kh, Kw = _pair(kernel_size)
    if output_size is None:
        output_size = conv2d_output_size(x.shape[2], x.shape[3], kernel_size, stride, padding,
                                         dilation)
    H_out, W_out = output_size
    shape = conv2d_shape(tuple(x.shape), tuple(weight.shape), Kh, Kw, H_out, W_out, stride,
                         padding, dilation, groups)
    if out is None:
        out = torch.empty((x.shape[0], weight.shape[0], H_out, W_out), dtype=torch.int32,
                          device=x.device)
    _need(out, torch.int32, "out")
    nbytes = _lib.q8_conv2d_workspace_bytes(ctypes.byref(shape))
    ws = _workspace(nbytes, x.device, workspace)
    _check(_lib.q8_conv2d_acc32(_ptr(x), ctypes.byref(shape), int(input_zero_point), _ptr(weight),
                                _ptr(out), _ptr(ws), nbytes, _stream(x)), "q8_conv2d_acc32")
    return out


def conv2d_packed(x, input_scale, input_zero_point, packed: PackedConvWeight, weight_scales, bias,
                  output_scale, output_zero_point, stride=1, padding=0, dilation=1,
                  activation="none", output_size=None, out=None, workspace=None):
    """q8ta_conv2d from a packed weight."""
    if packed.transposed:
        raise ValueError("packed weight is a q8ta_conv2d_transposed weight")
    _need(x, torch.int8, "x")
    _need(weight_scales, torch.float32, "weight_scales")
    if bias is not None:
        _need(bias, torch.float32, "bias")
    if x.shape[1] != packed.IC:
        raise ValueError(f"x has {x.shape[1]} channels, the packed weight {packed.IC}")
    Kh, Kw = packed.Kh, packed.Kw
    if output_size is None:
        output_size = conv2d_output_size(x.shape[2], x.shape[3], (Kh, Kw), stride, padding,
                                         dilation)
    H_out, W_out = output_size
    ldw = Kh * Kw * (packed.IC // packed.groups)
    shape = conv2d_shape(tuple(x.shape), (packed.OC, ldw), Kh, Kw, H_out, W_out, stride, padding,
                         dilation, packed.groups)
    if out is None:
        out = torch.empty((x.shape[0], packed.OC, H_out, W_out), dtype=torch.int8, device=x.device)
    _need(out, torch.int8, "out")
    nbytes = _lib.q8_conv2d_packed_workspace_bytes(ctypes.byref(shape))
    ws = _workspace(nbytes, x.device, workspace)
    _check(_lib.q8_conv2d_packed(
        _ptr(x), ctypes.byref(shape), float(input_scale), int(input_zero_point),
        _ptr(packed.data), _ptr(weight_scales), _ptr(bias), float(output_scale),
        int(output_zero_point), activation.encode(), _ptr(out), _ptr(ws), nbytes, _stream(x)),
        "q8_conv2d_packed")
    return out


def conv2d_packed_acc32(x, input_zero_point, packed: PackedConvWeight, output_size=None, stride=1,
                        padding=0, dilation=1, out=None, workspace=None):
    """Exact int32 accumulators of q8ta_conv2d from a packed weight."""
    if packed.transposed:
        raise ValueError("packed weight is a q8ta_conv2d_transposed weight")
    _need(x, torch.int8, "x")
    if x.shape[1] != packed.IC:
        raise ValueError(f"x has {x.shape[1]} channels, the packed weight {packed.IC}")
    Kh, Kw = packed.Kh, packed.Kw
    if output_size is None:
        output_size = conv2d_output_size(x.shape[2], x.shape[3], (Kh, Kw), stride, padding,
                                         dilation)
    H_out, W_out = output_size
    ldw = Kh * Kw * (packed.IC // packed.groups)
    shape = conv2d_shape(tuple(x.shape), (packed.OC, ldw), Kh, Kw, H_out, W_out, stride, padding,
                         dilation, packed.groups)
    if out is None:
        out = torch.empty((x.shape[0], packed.OC, H_out, W_out), dtype=torch.int32,
                          device=x.device)
    _need(out, torch.int32, "out")
    nbytes = _lib.q8_conv2d_packed_workspace_bytes(ctypes.byref(shape))
    ws = _workspace(nbytes, x.device, workspace)
    _check(_lib.q8_conv2d_packed_acc32(_ptr(x), ctypes.byref(shape), int(input_zero_point),
                                       _ptr(packed.data), _ptr(out), _ptr(ws), nbytes, _stream(x)),
           "q8_conv2d_packed_acc32")
    return out
