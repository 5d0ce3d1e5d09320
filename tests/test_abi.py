"""Host-side checks of the C ABI (no GPU needed).

The library loads, exports every function include/q8ta.h declares, and its
argument guards -- which run on the host before anything is enqueued --
return the documented status codes.  No call here reaches a kernel launch:
each passes an argument that a guard rejects first.
"""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "q8ta.h")

q8 = pytest.importorskip("int8_quantized_q8ta_gb300")
lib = q8.lib()

FAKE = ctypes.c_void_p(0x10000)  # never dereferenced: a guard fails first


def _declared():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(q8_[a-z0-9_]+)\s*\(", text)))


def test_every_declared_symbol_is_exported():
    names = _declared()
    assert len(names) >= 17
    for n in names:
        assert hasattr(lib, n), n
    assert sorted(q8.EXPORTS) == names


def test_status_strings_and_version():
    assert lib.q8_version() == 1
    for s in range(9):
        assert lib.q8_status_string(s).startswith(b"Q8_")
    assert lib.q8_status_string(99) == b"unknown q8_status"


def test_quantize_guards():
    f = lib.q8_quantize_per_tensor
    assert f(None, 4, 0.1, 0, FAKE, None) == q8.Q8_ERR_NULL
    assert f(FAKE, 4, 0.1, 0, None, None) == q8.Q8_ERR_NULL
    assert f(None, 0, 0.1, 0, None, None) == q8.Q8_OK               # empty: nothing to do
    assert lib.q8_dequantize_per_tensor(None, 0, 0.1, 0, None, None) == q8.Q8_OK
    assert f(FAKE, 6, 0.1, 0, FAKE, None) == q8.Q8_ERR_SHAPE        # numel % 4
    assert f(FAKE, -4, 0.1, 0, FAKE, None) == q8.Q8_ERR_SHAPE
    assert f(FAKE, 4, 0.0, 0, FAKE, None) == q8.Q8_ERR_ARG
    assert f(FAKE, 4, float("inf"), 0, FAKE, None) == q8.Q8_ERR_ARG
    assert f(FAKE, 4, 0.1, 128, FAKE, None) == q8.Q8_ERR_ARG
    assert lib.q8_dequantize_per_tensor(FAKE, 5, 0.1, 0, FAKE, None) == q8.Q8_ERR_SHAPE


def _lin(fn, M=8, K=64, N=32, act=b"none", izp=0, ozp=0, s_in=0.02, s_out=0.05, ws=FAKE,
         out=FAKE, workspace=None, wbytes=0):
    return fn(FAKE, M, K, s_in, izp, FAKE, N, None, ws, None, s_out, ozp, act, out, workspace,
              wbytes, None)


@pytest.mark.parametrize("name", ["q8_linear", "q8_linear_gemv"])
def test_linear_guards(name):
    f = getattr(lib, name)
    M = 1
    assert _lin(f, M=M, N=30) == q8.Q8_ERR_SHAPE                    # N % 4
    assert _lin(f, M=M, K=63) == q8.Q8_ERR_SHAPE                    # M*K % 4 with M = 1
    assert _lin(f, M=M, act=b"gelu") == q8.Q8_ERR_UNSUPPORTED
    assert _lin(f, M=M, act=b"relu", N=30) == q8.Q8_ERR_SHAPE      # relu passes the activation guard
    assert _lin(f, M=M, act=None) == q8.Q8_ERR_NULL
    assert _lin(f, M=M, ws=None) == q8.Q8_ERR_NULL
    assert _lin(f, M=M, out=None) == q8.Q8_ERR_NULL
    assert _lin(f, M=M, izp=-129) == q8.Q8_ERR_ARG
    assert _lin(f, M=M, s_out=-1.0) == q8.Q8_ERR_ARG
    assert _lin(f, M=0) == q8.Q8_ERR_SHAPE


def test_linear_workspace_and_gemv_shape_guards():
    assert _lin(lib.q8_linear_gemv, M=2) == q8.Q8_ERR_SHAPE
    assert _lin(lib.q8_linear, M=8) == q8.Q8_ERR_WORKSPACE
    need = lib.q8_linear_workspace_bytes(8, 64, 32)
    assert need > 0 and need % 256 == 0
    assert _lin(lib.q8_linear, M=8, workspace=FAKE, wbytes=need - 1) == q8.Q8_ERR_WORKSPACE
    assert _lin(lib.q8_linear, M=8, workspace=ctypes.c_void_p(0x10010), wbytes=need) == \
        q8.Q8_ERR_ALIGN
    assert lib.q8_linear_workspace_bytes(1, 4096, 4096) == 0


def test_workspace_sizes():
    # bf16 copies padded to a multiple of 64 along K, 256-byte aligned; a
    # packed weight adds a 256-byte trailer holding its per-k-block |w| bound
    assert lib.q8_linear_packed_weight_bytes(11008, 4096) == 11008 * 4096 * 2 + 256
    # operand: the bf16 data plus a 256-byte trailer holding its |x - zp| bound
    assert lib.q8_linear_operand_bytes(2048, 4096) == 2048 * 4096 * 2 + 256
    assert lib.q8_linear_packed_weight_bytes(4, 70) == (4 * 128 * 2 + 255) // 256 * 256 + 256
    s = q8.conv_t_shape((8, 256, 64, 64), (128, 2304), 3, 3, 128, 128, 2, 1, 1)
    assert lib.q8_conv2d_transposed_workspace_bytes(ctypes.byref(s)) == \
        8 * 64 * 64 * 256 * 2 + 128 * 9 * 256 * 2


def test_operand_guards():
    assert lib.q8_linear_prepare_operand(None, 8, 64, 0, FAKE, 1 << 20, None) == q8.Q8_ERR_NULL
    assert lib.q8_linear_prepare_operand(FAKE, 1, 3, 0, FAKE, 1 << 20, None) == q8.Q8_ERR_SHAPE
    assert lib.q8_linear_prepare_operand(FAKE, 8, 64, 0, FAKE, 10, None) == q8.Q8_ERR_WORKSPACE
    assert lib.q8_linear_prepare_operand(FAKE, 8, 64, 0, ctypes.c_void_p(0x10008), 1 << 20,
                                         None) == q8.Q8_ERR_ALIGN
    assert lib.q8_quantize_to_linear_operand(FAKE, 8, 64, 0.0, 0, None, FAKE, 1 << 20,
                                             None) == q8.Q8_ERR_ARG
    assert lib.q8_linear_operand_packed(FAKE, 8, 64, 0.02, FAKE, 30, FAKE, None, 0.1, 0, b"none",
                                        FAKE, None) == q8.Q8_ERR_SHAPE
    assert lib.q8_linear_operand_packed(FAKE, 8, 64, 0.02, FAKE, 32, FAKE, None, 0.1, 0, b"tanh",
                                        FAKE, None) == q8.Q8_ERR_UNSUPPORTED


def _conv(**kw):
    base = dict(x_shape=(1, 3, 5, 4), w_shape=(4, 27), Kh=3, Kw=3, H_out=10, W_out=8, stride=2,
                padding=1, output_padding=1, dilation=1, groups=1)
    base.update(kw)
    s = q8.conv_t_shape(base["x_shape"], base["w_shape"], base["Kh"], base["Kw"], base["H_out"],
                        base["W_out"], base["stride"], base["padding"], base["output_padding"],
                        base["dilation"], base["groups"])
    act = kw.get("act", b"none")
    return lib.q8_conv2d_transposed(FAKE, ctypes.byref(s), 0.02, 0, FAKE, None, FAKE, None, 0.1,
                                    0, act, FAKE, None, 0, None)


def test_conv_t_guards():
    assert _conv(groups=0) == q8.Q8_ERR_UNSUPPORTED
    assert _conv(dilation=0) == q8.Q8_ERR_UNSUPPORTED
    assert _conv(groups=2) == q8.Q8_ERR_SHAPE                      # IC = 3 is not divisible
    assert _conv(stride=0) == q8.Q8_ERR_SHAPE
    assert _conv(W_out=9) == q8.Q8_ERR_SHAPE                       # W_out % 4
    assert _conv(w_shape=(4, 26)) == q8.Q8_ERR_SHAPE               # row stride < Kh*Kw*IC
    assert _conv(padding=-1) == q8.Q8_ERR_SHAPE
    assert _conv(act=b"gelu") == q8.Q8_ERR_UNSUPPORTED
    assert _conv() == q8.Q8_ERR_WORKSPACE                          # all guards pass
    assert _conv(act=b"relu") == q8.Q8_ERR_WORKSPACE
    assert _conv(dilation=2) == q8.Q8_ERR_WORKSPACE
    # groups = 2 with IC = 4, OC = 4: rows of Kh*Kw*IC/2 = 18
    assert _conv(x_shape=(1, 4, 5, 4), w_shape=(4, 18), groups=2) == q8.Q8_ERR_WORKSPACE
    s = q8.conv_t_shape((1, 3, 5, 4), (4, 27), 3, 3, 10, 8, 2, 1, 1)
    assert lib.q8_conv2d_transposed(FAKE, None, 0.02, 0, FAKE, None, FAKE, None, 0.1, 0, b"none",
                                    FAKE, None, 0, None) == q8.Q8_ERR_NULL
    assert lib.q8_conv2d_transposed(FAKE, ctypes.byref(s), 0.02, 300, FAKE, None, FAKE, None, 0.1,
                                    0, b"none", FAKE, None, 0, None) == q8.Q8_ERR_ARG


def test_binding_refuses_cpu_tensors():
    torch = pytest.importorskip("torch")
    with pytest.raises(ValueError, match="CUDA"):
        q8.quantize_per_tensor(torch.zeros(8), 0.1, 0)


def _conv2d(**kw):
    base = dict(x_shape=(1, 3, 6, 8), w_shape=(4, 27), Kh=3, Kw=3, H_out=6, W_out=8, stride=1,
                padding=1, dilation=1, groups=1)
    base.update(kw)
    s = q8.conv2d_shape(base["x_shape"], base["w_shape"], base["Kh"], base["Kw"], base["H_out"],
                        base["W_out"], base["stride"], base["padding"], base["dilation"],
                        base["groups"])
    act = kw.get("act", b"none")
    return lib.q8_conv2d(FAKE, ctypes.byref(s), 0.02, 0, FAKE, FAKE, None, 0.1, 0, act, FAKE,
                         None, 0, None)


def test_conv2d_guards_and_sizes():
    assert _conv2d(stride=9) == q8.Q8_ERR_UNSUPPORTED              # TMA element stride <= 8
    assert _conv2d(stride=0) == q8.Q8_ERR_SHAPE
    assert _conv2d(W_out=6) == q8.Q8_ERR_SHAPE
    assert _conv2d(groups=3, w_shape=(4, 9)) == q8.Q8_ERR_SHAPE   # OC = 4 not divisible by 3
    assert _conv2d(act=b"sigmoid") == q8.Q8_ERR_UNSUPPORTED
    assert _conv2d() == q8.Q8_ERR_WORKSPACE
    assert _conv2d(stride=8, act=b"relu") == q8.Q8_ERR_WORKSPACE
    s = q8.conv2d_shape((2, 96, 10, 12), (64, 9 * 48), 3, 3, 10, 12, 1, 1, 1, 2)
    # relayout: 2 groups of 48 channels padded to 64; packed weight: 2 x 9 x 32 x 64
    assert lib.q8_conv2d_packed_workspace_bytes(ctypes.byref(s)) == 2 * 10 * 12 * 128 * 2
    assert lib.q8_conv2d_packed_weight_bytes(ctypes.byref(s)) == 2 * 9 * 32 * 64 * 2 + 256
    assert lib.q8_conv2d_workspace_bytes(ctypes.byref(s)) == 2 * 10 * 12 * 128 * 2 + 2 * 9 * 32 * 64 * 2
    bad = q8.conv2d_shape((2, 96, 10, 12), (64, 9 * 48), 3, 3, 10, 10, 1, 1, 1, 2)  # W_out % 4
    assert lib.q8_conv2d_workspace_bytes(ctypes.byref(bad)) == 0


def test_packed_acc32_guards():
    """The int32-accumulator forms from packed convolution weights refuse
    bad arguments on the host, before anything is enqueued."""
    st = q8.conv_t_shape((1, 64, 8, 8), (96, 9 * 64), 3, 3, 16, 16, 2, 1, 1)
    sd = q8.conv2d_shape((1, 64, 8, 8), (96, 9 * 64), 3, 3, 8, 8, 1, 1, 1, 1)
    need_t = lib.q8_conv2d_transposed_packed_workspace_bytes(ctypes.byref(st))
    need_d = lib.q8_conv2d_packed_workspace_bytes(ctypes.byref(sd))
    assert need_t > 0 and need_d > 0
    for fn, s, need in ((lib.q8_conv2d_transposed_packed_acc32, st, need_t),
                        (lib.q8_conv2d_packed_acc32, sd, need_d)):
        assert fn(None, ctypes.byref(s), 0, FAKE, FAKE, FAKE, need, None) == q8.Q8_ERR_NULL
        assert fn(FAKE, ctypes.byref(s), 0, None, FAKE, FAKE, need, None) == q8.Q8_ERR_NULL
        assert fn(FAKE, ctypes.byref(s), 0, FAKE, None, FAKE, need, None) == q8.Q8_ERR_NULL
        assert fn(FAKE, None, 0, FAKE, FAKE, FAKE, need, None) == q8.Q8_ERR_NULL
        assert fn(FAKE, ctypes.byref(s), 128, FAKE, FAKE, FAKE, need, None) == q8.Q8_ERR_ARG
        assert fn(FAKE, ctypes.byref(s), 0, FAKE, FAKE, FAKE, need - 1, None) == \
            q8.Q8_ERR_WORKSPACE
        assert fn(FAKE, ctypes.byref(s), 0, FAKE, FAKE, None, need, None) == q8.Q8_ERR_WORKSPACE
        assert fn(FAKE, ctypes.byref(s), 0, FAKE, FAKE, ctypes.c_void_p(0x10010), need,
                  None) == q8.Q8_ERR_ALIGN
    bad = q8.conv_t_shape((1, 64, 8, 8), (96, 9 * 64), 3, 3, 16, 14, 2, 1, 1)   # W_out % 4
    assert lib.q8_conv2d_transposed_packed_acc32(FAKE, ctypes.byref(bad), 0, FAKE, FAKE, FAKE,
                                                 need_t, None) == q8.Q8_ERR_SHAPE


def test_gemv_packed_guards():
    assert lib.q8_linear_gemv_packed_weight_bytes(0, 64) == 0
    assert lib.q8_linear_gemv_packed_weight_bytes(4, 64) == 256
    assert lib.q8_linear_gemv_packed_weight_bytes(1000, 4100) == 4100000 + 96  # up to 256
    pack = lib.q8_linear_gemv_pack_weight
    assert pack(None, 4, 64, FAKE, 256, None) == q8.Q8_ERR_NULL
    assert pack(FAKE, 0, 64, FAKE, 256, None) == q8.Q8_ERR_SHAPE
    assert pack(FAKE, 4, 64, FAKE, 255, None) == q8.Q8_ERR_WORKSPACE
    assert pack(FAKE, 4, 64, ctypes.c_void_p(0x10010), 256, None) == q8.Q8_ERR_ALIGN
    g = lib.q8_linear_gemv_packed
    ok = dict(x=FAKE, K=64, s_in=0.02, izp=0, w=FAKE, N=32, ws=FAKE, s_out=0.05, ozp=0,
              act=b"none", out=FAKE)

    def call(**kw):
        a = dict(ok, **kw)
        return g(a["x"], a["K"], a["s_in"], a["izp"], a["w"], a["N"], a["ws"], None, a["s_out"],
                 a["ozp"], a["act"], a["out"], None)
    assert call(x=None) == q8.Q8_ERR_NULL
    assert call(ws=None) == q8.Q8_ERR_NULL
    assert call(N=30) == q8.Q8_ERR_SHAPE                       # N % 4
    assert call(K=0) == q8.Q8_ERR_SHAPE
    assert call(act=b"gelu") == q8.Q8_ERR_UNSUPPORTED
    assert call(izp=200) == q8.Q8_ERR_ARG
    assert call(w=ctypes.c_void_p(0x10010)) == q8.Q8_ERR_ALIGN  # packed buffers are 256-aligned
