// api_conv.cu -- the extern "C" boundary of the two int8 convolutions:
// q8ta_conv2d_transposed ("Add q8ta_conv2d_transposed op", PR #21205) and the
// direct q8ta_conv2d named in that page's Problem paragraph.
//
// Both run the same three steps on the caller's stream: the channel-blocked
// NHWC bf16 copy of x - input_zero_point (per group, channels padded to a
// multiple of 64), the packed bf16 weight (per group, [taps][IC/64][OC][64]),
// and one tensor-core implicit GEMM per group with the fused epilogue.  The
// *_pack_weight / *_packed forms let a caller pack the weight once.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <cstdint>
#include <mutex>
#include <unordered_map>

#include "api_common.h"
#include "q8ta.h"
#include "q8ta_internal.h"

namespace {

using namespace q8api;
using q8::align_ws;
using q8::kTileK;
using q8::round_up;

// One description of both convolutions.
struct Geom {
  int64_t N, IC, H_in, W_in, OC, Kh, Kw, ldw, H_out, W_out;
  int64_t sh, sw, ph, pw, dh, dw, groups;
  bool direct;
  int64_t ICg() const { return IC / groups; }
  int64_t OCg() const { return OC / groups; }
  int64_t ICgp() const { return round_up(ICg(), kTileK); }
  int64_t taps() const { return Kh * Kw; }
};

Geom geom_t(const q8_conv2d_transposed_shape& s) {
  return Geom{s.N,      s.IC,     s.H_in,  s.W_in,  s.OC,         s.Kh,         s.Kw,
              s.weight_row_stride, s.H_out, s.W_out, s.stride_h, s.stride_w, s.pad_h,
              s.pad_w,  s.dilation_h, s.dilation_w, s.groups, false};
}

Geom geom_d(const q8_conv2d_shape& s) {
  return Geom{s.N,      s.IC,     s.H_in,  s.W_in,  s.OC,         s.Kh,         s.Kw,
              s.weight_row_stride, s.H_out, s.W_out, s.stride_h, s.stride_w, s.pad_h,
              s.pad_w,  s.dilation_h, s.dilation_w, s.groups, true};
}

// Shape guards of both convolutions.  The page's own: stride >= 1,
// W_out % 4 == 0 (one output word = 4 columns), weight row stride >=
// Kh*Kw*IC (per group: Kh*Kw*IC/groups); its fail-loud follow-ups groups > 1
// and dilation != 1 are supported here with groups dividing IC and OC.  The
// direct convolution reads its input through TMA boxes with element strides,
// which the hardware allows up to 8.
q8_status check_geom(const Geom& g) {
  if (g.groups < 1 || g.dh < 1 || g.dw < 1) return Q8_ERR_UNSUPPORTED;
  if (g.sh < 1 || g.sw < 1) return Q8_ERR_SHAPE;
  if (g.direct && (g.sh > 8 || g.sw > 8)) return Q8_ERR_UNSUPPORTED;
  if (g.N < 1 || g.IC < 1 || g.H_in < 1 || g.W_in < 1 || g.OC < 1 || g.Kh < 1 || g.Kw < 1 ||
      g.H_out < 1 || g.W_out < 1)
    return Q8_ERR_SHAPE;
  if (g.IC % g.groups != 0 || g.OC % g.groups != 0) return Q8_ERR_SHAPE;
  if (g.ph < 0 || g.pw < 0) return Q8_ERR_SHAPE;
  if (g.W_out % 4 != 0) return Q8_ERR_SHAPE;
  if (!mul_ok(g.Kh, g.Kw) || !mul_ok(g.Kh * g.Kw, g.ICg())) return Q8_ERR_SHAPE;
  if (g.ldw < g.Kh * g.Kw * g.ICg()) return Q8_ERR_SHAPE;
  // sizes the kernels index with 32-bit tile coordinates
  const int64_t lim = INT32_MAX / 4;
  if (g.N > lim || g.IC > lim || g.H_in > lim || g.W_in > lim || g.OC > lim || g.H_out > lim ||
      g.W_out > lim || g.Kh > 4096 || g.Kw > 4096 || g.sh > 4096 || g.sw > 4096 ||
      g.dh > 4096 || g.dw > 4096 || g.ph > lim || g.pw > lim || g.groups > lim)
    return Q8_ERR_SHAPE;
  if (!mul_ok(g.N * g.H_in, g.W_in) || !mul_ok(g.N * g.H_in * g.W_in, g.groups * g.ICgp()) ||
      !mul_ok(g.N * g.OC, g.H_out * g.W_out))
    return Q8_ERR_SHAPE;
  return Q8_OK;
}

size_t relayout_bytes(const Geom& g) {
  return align_ws(static_cast<size_t>(g.N * g.H_in * g.W_in) * g.groups * g.ICgp() * 2);
}

// The packed weight, then a 256-byte trailer whose first int32 holds the
// largest sum of |w| over one k-block (64 input channels of one tap) of one
// output row, written by the load-time pack.
size_t packed_data_bytes(const Geom& g) {
  return align_ws(static_cast<size_t>(g.groups * g.taps() * g.OCg()) * g.ICgp() * 2);
}

size_t packed_bytes(const Geom& g) { return packed_data_bytes(g) + q8::kWorkspaceAlign; }

int32_t* packed_bound_word(const Geom& g, const void* packed) {
  return reinterpret_cast<int32_t*>(static_cast<char*>(const_cast<void*>(packed)) +
                                    packed_data_bytes(g));
}

// Host copies of the k-block bounds of the weights this library packed, by
// packed buffer and size: with them a launch picks the single-chunk kernel
// without reading the device.  A buffer without an entry (or of another
// size) is taken at the worst case, which never picks that kernel wrongly;
// an entry whose buffer was rewritten behind the library's back is caught
// on the device (the kernel runs nothing and sets the error word).
struct PackedBound {
  size_t bytes;
  int32_t bound;
};
std::mutex& bound_mutex() {
  static std::mutex m;
  return m;
}
std::unordered_map<const void*, PackedBound>& bound_map() {
  static std::unordered_map<const void*, PackedBound> m;
  return m;
}

int host_weight_bound(const Geom& g, const void* packed) {
  std::lock_guard<std::mutex> lock(bound_mutex());
  const auto it = bound_map().find(packed);
  if (it == bound_map().end() || it->second.bytes != packed_data_bytes(g)) return q8::kWorstWBound;
  return it->second.bound;
}

q8_status check_ptr(const void* p, size_t have, size_t need) {
  if (!p || have < need) return Q8_ERR_WORKSPACE;
  if (reinterpret_cast<uintptr_t>(p) % q8::kWorkspaceAlign != 0) return Q8_ERR_ALIGN;
  return Q8_OK;
}

q8_status pack(const Geom& g, const int8_t* weight, void* packed, q8_stream_t stream) {
  return cuda_status(q8::launch_conv_weight_bf16(weight, g.groups, g.OCg(), g.taps(), g.ICg(),
                                                 g.ldw, static_cast<__nv_bfloat16*>(packed),
                                                 g.ICgp(), cs(stream)));
}

// The relayout of x into `relayout`, then one GEMM per group.  w_bound: the
// packed weight's k-block bound word, or null (the worst case); w_bound_host:
// the host's copy, or kWorstWBound.
q8_status run(const Geom& g, const int8_t* x, double input_scale, int32_t izp, const void* packed,
              const int32_t* w_bound, int w_bound_host, const float* ws, const float* bias,
              double output_scale, int32_t ozp, int relu, int8_t* out, int32_t* acc_out,
              void* relayout, q8_stream_t stream) {
  if (reinterpret_cast<uintptr_t>(packed) % q8::kWorkspaceAlign != 0) return Q8_ERR_ALIGN;
  auto* a = static_cast<__nv_bfloat16*>(relayout);
  cudaError_t e = q8::launch_nchw_to_nhwc_bf16(x, g.N, g.groups, g.ICg(), g.H_in, g.W_in, izp, a,
                                                g.ICgp(), cs(stream));
  if (e != cudaSuccess) return Q8_ERR_CUDA;
  const int64_t cbg = g.ICgp() / kTileK;
  const int64_t plane = g.H_out * g.W_out;
  const size_t wgroup = static_cast<size_t>(g.taps() * g.OCg()) * g.ICgp();  // bf16 elements
  for (int64_t j = 0; j < g.groups; ++j) {
    q8::TcConvT C{};
    C.a = a + j * cbg * kTileK * g.H_in * g.W_in;
    C.b = static_cast<const __nv_bfloat16*>(packed) + j * wgroup;
    C.N = g.N;
    C.ICp = g.ICgp();
    C.cb_total = cbg * g.groups;
    C.H_in = g.H_in;
    C.W_in = g.W_in;
    C.OC = g.OCg();
    C.Kh = g.Kh;
    C.Kw = g.Kw;
    C.H_out = g.H_out;
    C.W_out = g.W_out;
    C.stride_h = g.sh;
    C.stride_w = g.sw;
    C.pad_h = g.ph;
    C.pad_w = g.pw;
    C.dil_h = g.dh;
    C.dil_w = g.dw;
    C.out_ch = g.OC;
    C.direct = g.direct;
    C.ws = ws ? ws + j * g.OCg() : nullptr;
    C.bias = bias ? bias + j * g.OCg() : nullptr;
    C.rq = make_rq(input_scale, output_scale, ozp, relu);
    C.out = out ? out + j * g.OCg() * plane : nullptr;
    C.acc_out = acc_out ? acc_out + j * g.OCg() * plane : nullptr;
    C.a_bound = a_bound_of(izp);
    C.w_bound = w_bound;
    C.w_bound_host = w_bound != nullptr ? w_bound_host : q8::kWorstWBound;
    e = q8::launch_tc_conv_t(C, cs(stream));
    if (e != cudaSuccess) return Q8_ERR_CUDA;
  }
  return Q8_OK;
}

q8_status check_epilogue(double input_scale, int32_t izp, const float* ws, double output_scale,
                         int32_t ozp, const char* activation, int* relu) {
  if (!ws || !activation) return Q8_ERR_NULL;
  const int act = parse_activation(activation);
  if (act < 0) return Q8_ERR_UNSUPPORTED;
  *relu = act;
  if (!scale_ok(input_scale) || !scale_ok(output_scale) || !zp_ok(izp) || !zp_ok(ozp))
    return Q8_ERR_ARG;
  return Q8_OK;
}

// The raw-weight forms: workspace = relayout, then the packed weight.
q8_status full(const Geom& g, const int8_t* x, double input_scale, int32_t izp,
               const int8_t* weight, const float* ws, const float* bias, double output_scale,
               int32_t ozp, const char* activation, int8_t* out, int32_t* acc_out,
               void* workspace, size_t workspace_bytes, q8_stream_t stream) {
  if (!x || !weight || (!out && !acc_out)) return Q8_ERR_NULL;
  q8_status st = check_geom(g);
  if (st != Q8_OK) return st;
  int relu = 0;
  if (out) {
    st = check_epilogue(input_scale, izp, ws, output_scale, ozp, activation, &relu);
    if (st != Q8_OK) return st;
  } else if (!zp_ok(izp)) {
    return Q8_ERR_ARG;
  }
  const size_t ra = relayout_bytes(g);
  st = check_ptr(workspace, workspace_bytes, ra + packed_data_bytes(g));
  if (st != Q8_OK) return st;
  void* packed = static_cast<char*>(workspace) + ra;
  st = pack(g, weight, packed, stream);
  if (st != Q8_OK) return st;
  // a per-call weight copy: no bound word (that costs a pass over the weight)
  return run(g, x, input_scale, izp, packed, nullptr, q8::kWorstWBound, ws, bias, output_scale,
             ozp, relu, out, acc_out, workspace, stream);
}

q8_status packed_form(const Geom& g, const int8_t* x, double input_scale, int32_t izp,
                      const void* packed, const float* ws, const float* bias,
                      double output_scale, int32_t ozp, const char* activation, int8_t* out,
                      void* workspace, size_t workspace_bytes, q8_stream_t stream) {
  if (!x || !packed || !out) return Q8_ERR_NULL;
  q8_status st = check_geom(g);
  if (st != Q8_OK) return st;
  int relu = 0;
  st = check_epilogue(input_scale, izp, ws, output_scale, ozp, activation, &relu);
  if (st != Q8_OK) return st;
  st = check_ptr(workspace, workspace_bytes, relayout_bytes(g));
  if (st != Q8_OK) return st;
  return run(g, x, input_scale, izp, packed, packed_bound_word(g, packed),
             host_weight_bound(g, packed), ws, bias, output_scale, ozp, relu, out, nullptr,
             workspace, stream);
}

// The int32 accumulators from a packed weight (exact chunks sized by its
// k-block bound, as in packed_form).
q8_status packed_acc_form(const Geom& g, const int8_t* x, int32_t izp, const void* packed,
                          int32_t* acc, void* workspace, size_t workspace_bytes,
                          q8_stream_t stream) {
  if (!x || !packed || !acc) return Q8_ERR_NULL;
  q8_status st = check_geom(g);
  if (st != Q8_OK) return st;
  if (!zp_ok(izp)) return Q8_ERR_ARG;
  st = check_ptr(workspace, workspace_bytes, relayout_bytes(g));
  if (st != Q8_OK) return st;
  return run(g, x, 1.0, izp, packed, packed_bound_word(g, packed), host_weight_bound(g, packed),
             nullptr, nullptr, 1.0, 0, 0, nullptr, acc, workspace, stream);
}

q8_status pack_form(const Geom& g, const int8_t* weight, void* packed, size_t bytes,
                    q8_stream_t stream) {
  if (!weight) return Q8_ERR_NULL;
  q8_status st = check_geom(g);
  if (st != Q8_OK) return st;
  st = check_ptr(packed, bytes, packed_bytes(g));
  if (st != Q8_OK) return st;
  st = pack(g, weight, packed, stream);
  if (st != Q8_OK) return st;
  int32_t* word = packed_bound_word(g, packed);
  cudaError_t e = q8::launch_weight_block_bound(weight, g.OC, g.ldw, g.taps(), g.ICg(), word,
                                                cs(stream));
  // the host's copy of the bound (load time: the call waits for the pack)
  int32_t host = 0;
  if (e == cudaSuccess)
    e = cudaMemcpyAsync(&host, word, sizeof(host), cudaMemcpyDeviceToHost, cs(stream));
  if (e == cudaSuccess) e = cudaStreamSynchronize(cs(stream));
  if (e != cudaSuccess) return Q8_ERR_CUDA;
  std::lock_guard<std::mutex> lock(bound_mutex());
  bound_map()[packed] = PackedBound{packed_data_bytes(g), host};
  return Q8_OK;
}

size_t sized(const Geom& g, size_t bytes) { return check_geom(g) == Q8_OK ? bytes : 0; }

}  // namespace

extern "C" {

// ------------------------------------------------------------ conv_t
size_t q8_conv2d_transposed_workspace_bytes(const q8_conv2d_transposed_shape* shape) {
  if (!shape) return 0;
  const Geom g = geom_t(*shape);
  return sized(g, relayout_bytes(g) + packed_data_bytes(g));
}

size_t q8_conv2d_transposed_packed_weight_bytes(const q8_conv2d_transposed_shape* shape) {
  if (!shape) return 0;
  const Geom g = geom_t(*shape);
  return sized(g, packed_bytes(g));
}

size_t q8_conv2d_transposed_packed_workspace_bytes(const q8_conv2d_transposed_shape* shape) {
  if (!shape) return 0;
  const Geom g = geom_t(*shape);
  return sized(g, relayout_bytes(g));
}

q8_status q8_conv2d_transposed(const int8_t* x, const q8_conv2d_transposed_shape* shape,
                               double input_scale, int32_t input_zero_point,
                               const int8_t* weight, const int32_t* weight_sums,
                               const float* weight_scales, const float* bias,
                               double output_scale, int32_t output_zero_point,
                               const char* activation, int8_t* out, void* workspace,
                               size_t workspace_bytes, q8_stream_t stream) {
  (void)weight_sums;
  if (!shape || !out) return Q8_ERR_NULL;
  return full(geom_t(*shape), x, input_scale, input_zero_point, weight, weight_scales, bias,
              output_scale, output_zero_point, activation, out, nullptr, workspace,
              workspace_bytes, stream);
}

q8_status q8_conv2d_transposed_acc32(const int8_t* x, const q8_conv2d_transposed_shape* shape,
                                     int32_t input_zero_point, const int8_t* weight, int32_t* acc,
                                     void* workspace, size_t workspace_bytes,
                                     q8_stream_t stream) {
  if (!shape || !acc) return Q8_ERR_NULL;
  return full(geom_t(*shape), x, 1.0, input_zero_point, weight, nullptr, nullptr, 1.0, 0, "none",
              nullptr, acc, workspace, workspace_bytes, stream);
}

q8_status q8_conv2d_transposed_pack_weight(const int8_t* weight,
                                           const q8_conv2d_transposed_shape* shape, void* packed,
                                           size_t packed_bytes_, q8_stream_t stream) {
  if (!shape) return Q8_ERR_NULL;
  return pack_form(geom_t(*shape), weight, packed, packed_bytes_, stream);
}

q8_status q8_conv2d_transposed_packed(const int8_t* x, const q8_conv2d_transposed_shape* shape,
                                      double input_scale, int32_t input_zero_point,
                                      const void* packed_weight, const float* weight_scales,
                                      const float* bias, double output_scale,
                                      int32_t output_zero_point, const char* activation,
                                      int8_t* out, void* workspace, size_t workspace_bytes,
                                      q8_stream_t stream) {
  if (!shape) return Q8_ERR_NULL;
  return packed_form(geom_t(*shape), x, input_scale, input_zero_point, packed_weight,
                     weight_scales, bias, output_scale, output_zero_point, activation, out,
                     workspace, workspace_bytes, stream);
}

q8_status q8_conv2d_transposed_packed_acc32(const int8_t* x,
                                            const q8_conv2d_transposed_shape* shape,
                                            int32_t input_zero_point, const void* packed_weight,
                                            int32_t* acc, void* workspace, size_t workspace_bytes,
                                            q8_stream_t stream) {
  if (!shape) return Q8_ERR_NULL;
  return packed_acc_form(geom_t(*shape), x, input_zero_point, packed_weight, acc, workspace,
                         workspace_bytes, stream);
}

// ------------------------------------------------------------ conv2d
size_t q8_conv2d_workspace_bytes(const q8_conv2d_shape* shape) {
  if (!shape) return 0;
  const Geom g = geom_d(*shape);
  return sized(g, relayout_bytes(g) + packed_data_bytes(g));
}

size_t q8_conv2d_packed_weight_bytes(const q8_conv2d_shape* shape) {
  if (!shape) return 0;
  const Geom g = geom_d(*shape);
  return sized(g, packed_bytes(g));
}

size_t q8_conv2d_packed_workspace_bytes(const q8_conv2d_shape* shape) {
  if (!shape) return 0;
  const Geom g = geom_d(*shape);
  return sized(g, relayout_bytes(g));
}

q8_status q8_conv2d(const int8_t* x, const q8_conv2d_shape* shape, double input_scale,
                    int32_t input_zero_point, const int8_t* weight, const float* weight_scales,
                    const float* bias, double output_scale, int32_t output_zero_point,
                    const char* activation, int8_t* out, void* workspace, size_t workspace_bytes,
                    q8_stream_t stream) {
  if (!shape || !out) return Q8_ERR_NULL;
  return full(geom_d(*shape), x, input_scale, input_zero_point, weight, weight_scales, bias,
              output_scale, output_zero_point, activation, out, nullptr, workspace,
              workspace_bytes, stream);
}

q8_status q8_conv2d_acc32(const int8_t* x, const q8_conv2d_shape* shape, int32_t input_zero_point,
                          const int8_t* weight, int32_t* acc, void* workspace,
                          size_t workspace_bytes, q8_stream_t stream) {
  if (!shape || !acc) return Q8_ERR_NULL;
  return full(geom_d(*shape), x, 1.0, input_zero_point, weight, nullptr, nullptr, 1.0, 0, "none",
              nullptr, acc, workspace, workspace_bytes, stream);
}

q8_status q8_conv2d_pack_weight(const int8_t* weight, const q8_conv2d_shape* shape, void* packed,
                                size_t packed_bytes_, q8_stream_t stream) {
  if (!shape) return Q8_ERR_NULL;
  return pack_form(geom_d(*shape), weight, packed, packed_bytes_, stream);
}

q8_status q8_conv2d_packed(const int8_t* x, const q8_conv2d_shape* shape, double input_scale,
                           int32_t input_zero_point, const void* packed_weight,
                           const float* weight_scales, const float* bias, double output_scale,
                           int32_t output_zero_point, const char* activation, int8_t* out,
                           void* workspace, size_t workspace_bytes, q8_stream_t stream) {
  if (!shape) return Q8_ERR_NULL;
  return packed_form(geom_d(*shape), x, input_scale, input_zero_point, packed_weight,
                     weight_scales, bias, output_scale, output_zero_point, activation, out,
                     workspace, workspace_bytes, stream);
}

q8_status q8_conv2d_packed_acc32(const int8_t* x, const q8_conv2d_shape* shape,
                                 int32_t input_zero_point, const void* packed_weight, int32_t* acc,
                                 void* workspace, size_t workspace_bytes, q8_stream_t stream) {
  if (!shape) return Q8_ERR_NULL;
  return packed_acc_form(geom_d(*shape), x, input_zero_point, packed_weight, acc, workspace,
                         workspace_bytes, stream);
}

}  // extern "C"
