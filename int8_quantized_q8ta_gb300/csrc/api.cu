// api.cu -- the extern "C" boundary declared in include/q8ta.h.
//
// Each entry point validates every argument on the host before anything is
// enqueued (the "fail-loud" guards of the three q8ta pages' Implementation
// paragraphs), forms the f32 reciprocals in double, lays out the caller's
// workspace and enqueues the kernels on the caller's stream.
#include <algorithm>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <cmath>
#include <cstdint>
#include <cstring>

#include "api_common.h"
#include "q8ta.h"
#include "q8ta_internal.h"

namespace {

using namespace q8api;
using q8::align_ws;
using q8::kTileK;
using q8::round_up;

// Guards shared by the q8ta_linear entry points ("Add q8ta_linear op",
// Implementation paragraph): int8 operands (typed), N % 4 == 0,
// (M*K) % 4 == 0, (N*K) % 4 == 0, activation "none" (or the follow-up
// "relu", whose flag goes to *relu).
q8_status check_linear(const int8_t* x, int64_t M, int64_t K, double input_scale,
                       int32_t izp, const void* weight, int64_t N, const float* ws,
                       double output_scale, int32_t ozp, const char* activation,
                       const void* out, int* relu = nullptr) {
  if (!x || !weight || !ws || !out || !activation) return Q8_ERR_NULL;
  if (M < 1 || K < 1 || N < 1) return Q8_ERR_SHAPE;
  if (!mul_ok(M, K) || !mul_ok(N, K) || !mul_ok(M, N)) return Q8_ERR_SHAPE;
  if (N % 4 != 0 || (M * K) % 4 != 0 || (N * K) % 4 != 0) return Q8_ERR_SHAPE;
  if (M > INT32_MAX || N > INT32_MAX || K > INT32_MAX / 2) return Q8_ERR_SHAPE;
  const int act = parse_activation(activation);
  if (act < 0) return Q8_ERR_UNSUPPORTED;
  if (relu) *relu = act;
  if (!scale_ok(input_scale) || !scale_ok(output_scale) || !zp_ok(izp) || !zp_ok(ozp))
    return Q8_ERR_ARG;
  return Q8_OK;
}

size_t bf16_rows_bytes(int64_t rows, int64_t K) {
  return align_ws(static_cast<size_t>(rows) * static_cast<size_t>(round_up(K, kTileK)) * 2);
}

// A prepared operand is the bf16 data followed by one 256-byte trailer whose
// first int32 holds a_bound_of(zp) of the zero point it was prepared with.
// A packed weight likewise: its trailer's first int32 holds the largest sum
// of |w| over one k-block (64 consecutive weights) of one row.
int32_t* operand_bound_word(void* operand, int64_t M, int64_t K) {
  return reinterpret_cast<int32_t*>(static_cast<char*>(operand) + bf16_rows_bytes(M, K));
}

}  // namespace

extern "C" {

const char* q8_status_string(int status) {
  switch (status) {
    case Q8_OK: return "Q8_OK";
    case Q8_ERR_NULL: return "Q8_ERR_NULL: a required pointer is NULL";
    case Q8_ERR_SHAPE: return "Q8_ERR_SHAPE: a size or shape guard failed";
    case Q8_ERR_ALIGN: return "Q8_ERR_ALIGN: a pointer misses a documented alignment";
    case Q8_ERR_UNSUPPORTED:
      return "Q8_ERR_UNSUPPORTED: activation, dilation, groups or stride not supported";
    case Q8_ERR_WORKSPACE: return "Q8_ERR_WORKSPACE: workspace missing or too small";
    case Q8_ERR_CUDA: return "Q8_ERR_CUDA: a CUDA call or kernel launch failed";
    case Q8_ERR_DEVICE: return "Q8_ERR_DEVICE: a kernel raised the device error word";
    case Q8_ERR_ARG: return "Q8_ERR_ARG: a scale or zero point is out of range";
    default: return "unknown q8_status";
  }
}

int q8_version(void) { return 1; }

q8_status q8_device_error(uint32_t* code, int clear) {
  if (!code) return Q8_ERR_NULL;
  return cuda_status(q8::read_device_error(code, clear != 0));
}

// ---------------------------------------------------------------- quantize
q8_status q8_quantize_per_tensor(const float* x, int64_t numel, double scale, int32_t zero_point,
                                 int8_t* out, q8_stream_t stream) {
  if (numel < 0 || numel % 4 != 0) return Q8_ERR_SHAPE;
  if (!scale_ok(scale) || !zp_ok(zero_point)) return Q8_ERR_ARG;
  if (numel == 0) return Q8_OK;  // nothing to read or write
  if (!x || !out) return Q8_ERR_NULL;
  return cuda_status(q8::launch_quantize(x, numel, recip_f32(scale), zero_point, out,
                                         cs(stream)));
}

q8_status q8_dequantize_per_tensor(const int8_t* q, int64_t numel, double scale,
                                   int32_t zero_point, float* out, q8_stream_t stream) {
  if (numel < 0 || numel % 4 != 0) return Q8_ERR_SHAPE;
  if (!scale_ok(scale) || !zp_ok(zero_point)) return Q8_ERR_ARG;
  if (numel == 0) return Q8_OK;  // nothing to read or write
  if (!q || !out) return Q8_ERR_NULL;
  return cuda_status(q8::launch_dequantize(q, numel, static_cast<float>(scale),
                                           static_cast<float>(zero_point), out, cs(stream)));
}

// ---------------------------------------------------------------- linear
size_t q8_linear_workspace_bytes(int64_t M, int64_t K, int64_t N) {
  if (M <= 1 || K < 1 || N < 1) return 0;
  return bf16_rows_bytes(M, K) + bf16_rows_bytes(N, K);
}

size_t q8_linear_packed_weight_bytes(int64_t N, int64_t K) {
  if (N < 1 || K < 1) return 0;
  return bf16_rows_bytes(N, K) + q8::kWorkspaceAlign;
}

size_t q8_linear_operand_bytes(int64_t M, int64_t K) {
  if (M < 1 || K < 1) return 0;
  return bf16_rows_bytes(M, K) + q8::kWorkspaceAlign;
}

q8_status q8_linear_gemv(const int8_t* x, int64_t M, int64_t K, double input_scale,
                         int32_t input_zero_point, const int8_t* weight, int64_t N,
                         const int32_t* weight_sums, const float* weight_scales,
                         const float* bias, double output_scale, int32_t output_zero_point,
                         const char* activation, int8_t* out, void* workspace,
                         size_t workspace_bytes, q8_stream_t stream) {
  (void)weight_sums;
  (void)workspace;
  (void)workspace_bytes;
  int relu = 0;
  q8_status st = check_linear(x, M, K, input_scale, input_zero_point, weight, N, weight_scales,
                              output_scale, output_zero_point, activation, out, &relu);
  if (st != Q8_OK) return st;
  if (M != 1) return Q8_ERR_SHAPE;
  return cuda_status(q8::launch_gemv(x, K, input_zero_point, weight, N, weight_scales, bias,
                                     make_rq(input_scale, output_scale, output_zero_point, relu),
                                     out, cs(stream)));
}

size_t q8_linear_gemv_packed_weight_bytes(int64_t N, int64_t K) {
  if (N < 1 || K < 1 || !mul_ok(N, K)) return 0;
  return align_ws(static_cast<size_t>(N) * static_cast<size_t>(K));
}

q8_status q8_linear_gemv_pack_weight(const int8_t* weight, int64_t N, int64_t K, void* packed,
                                     size_t packed_bytes, q8_stream_t stream) {
  if (!weight || !packed) return Q8_ERR_NULL;
  if (N < 1 || K < 1 || !mul_ok(N, K) || N > INT32_MAX || K > INT32_MAX / 2) return Q8_ERR_SHAPE;
  if (packed_bytes < q8_linear_gemv_packed_weight_bytes(N, K)) return Q8_ERR_WORKSPACE;
  if (reinterpret_cast<uintptr_t>(packed) % q8::kWorkspaceAlign != 0) return Q8_ERR_ALIGN;
  // a copy of the row-major int8 weight, finished before this call returns,
  // so that no kernel launched later ever sees it being written
  cudaError_t e = cudaMemcpyAsync(packed, weight, static_cast<size_t>(N) * static_cast<size_t>(K),
                                  cudaMemcpyDeviceToDevice, cs(stream));
  if (e == cudaSuccess) e = cudaStreamSynchronize(cs(stream));
  return cuda_status(e);
}

q8_status q8_linear_gemv_packed(const int8_t* x, int64_t K, double input_scale,
                                int32_t input_zero_point, const void* packed_weight, int64_t N,
                                const float* weight_scales, const float* bias, double output_scale,
                                int32_t output_zero_point, const char* activation, int8_t* out,
                                q8_stream_t stream) {
  int relu = 0;
  q8_status st = check_linear(x, 1, K, input_scale, input_zero_point, packed_weight, N,
                              weight_scales, output_scale, output_zero_point, activation, out,
                              &relu);
  if (st != Q8_OK) return st;
  if (reinterpret_cast<uintptr_t>(packed_weight) % q8::kWorkspaceAlign != 0) return Q8_ERR_ALIGN;
  return cuda_status(q8::launch_gemv_packed(
      x, K, input_zero_point, static_cast<const int8_t*>(packed_weight), N, weight_scales, bias,
      make_rq(input_scale, output_scale, output_zero_point, relu), out, cs(stream)));
}

q8_status q8_linear(const int8_t* x, int64_t M, int64_t K, double input_scale,
                    int32_t input_zero_point, const int8_t* weight, int64_t N,
                    const int32_t* weight_sums, const float* weight_scales, const float* bias,
                    double output_scale, int32_t output_zero_point, const char* activation,
                    int8_t* out, void* workspace, size_t workspace_bytes, q8_stream_t stream) {
  int relu = 0;
  q8_status st = check_linear(x, M, K, input_scale, input_zero_point, weight, N, weight_scales,
                              output_scale, output_zero_point, activation, out, &relu);
  if (st != Q8_OK) return st;
  if (M == 1)
    return q8_linear_gemv(x, M, K, input_scale, input_zero_point, weight, N, weight_sums,
                          weight_scales, bias, output_scale, output_zero_point, activation, out,
                          nullptr, 0, stream);
  const size_t need = q8_linear_workspace_bytes(M, K, N);
  if (!workspace || workspace_bytes < need) return Q8_ERR_WORKSPACE;
  if (reinterpret_cast<uintptr_t>(workspace) % q8::kWorkspaceAlign != 0) return Q8_ERR_ALIGN;
  const int64_t Kp = round_up(K, kTileK);
  auto* a = static_cast<__nv_bfloat16*>(workspace);
  auto* b = reinterpret_cast<__nv_bfloat16*>(static_cast<char*>(workspace) + bf16_rows_bytes(M, K));
  cudaError_t e = q8::launch_rows_to_bf16(x, M, K, K, input_zero_point, a, Kp, cs(stream));
  if (e == cudaSuccess) e = q8::launch_rows_to_bf16(weight, N, K, K, 0, b, Kp, cs(stream));
  if (e != cudaSuccess) return Q8_ERR_CUDA;
  q8::TcLinear L{};
  L.a = a;
  L.b = b;
  L.M = M;
  L.N = N;
  L.Kp = Kp;
  L.ws = weight_scales;
  L.bias = bias;
  L.rq = make_rq(input_scale, output_scale, output_zero_point, relu);
  L.out = out;
  L.a_bound_host = a_bound_of(input_zero_point);
  return cuda_status(q8::launch_tc_linear(L, cs(stream)));
}

q8_status q8_linear_pack_weight(const int8_t* weight, int64_t N, int64_t K, void* packed,
                                size_t packed_bytes, q8_stream_t stream) {
  if (!weight || !packed) return Q8_ERR_NULL;
  if (N < 1 || K < 1 || !mul_ok(N, K) || N > INT32_MAX || K > INT32_MAX / 2) return Q8_ERR_SHAPE;
  if (packed_bytes < q8_linear_packed_weight_bytes(N, K)) return Q8_ERR_WORKSPACE;
  if (reinterpret_cast<uintptr_t>(packed) % q8::kWorkspaceAlign != 0) return Q8_ERR_ALIGN;
  cudaError_t e = q8::launch_rows_to_bf16(weight, N, K, K, 0, static_cast<__nv_bfloat16*>(packed),
                                          round_up(K, kTileK), cs(stream));
  if (e == cudaSuccess)
    e = q8::launch_weight_block_bound(weight, N, K, 1, K, operand_bound_word(packed, N, K),
                                      cs(stream));
  return cuda_status(e);
}

static q8_status check_operand(const void* operand, size_t operand_bytes, int64_t M, int64_t K) {
  if (!operand) return Q8_ERR_WORKSPACE;
  if (operand_bytes < q8_linear_operand_bytes(M, K)) return Q8_ERR_WORKSPACE;
  if (reinterpret_cast<uintptr_t>(operand) % q8::kWorkspaceAlign != 0) return Q8_ERR_ALIGN;
  return Q8_OK;
}

q8_status q8_linear_prepare_operand(const int8_t* x, int64_t M, int64_t K,
                                    int32_t input_zero_point, void* operand,
                                    size_t operand_bytes, q8_stream_t stream) {
  if (!x) return Q8_ERR_NULL;
  if (M < 1 || K < 1 || !mul_ok(M, K) || (M * K) % 4 != 0) return Q8_ERR_SHAPE;
  if (M > INT32_MAX || K > INT32_MAX / 2) return Q8_ERR_SHAPE;
  if (!zp_ok(input_zero_point)) return Q8_ERR_ARG;
  q8_status st = check_operand(operand, operand_bytes, M, K);
  if (st != Q8_OK) return st;
  return cuda_status(q8::launch_rows_to_bf16(x, M, K, K, input_zero_point,
                                             static_cast<__nv_bfloat16*>(operand),
                                             round_up(K, kTileK), cs(stream),
                                             operand_bound_word(operand, M, K)));
}

q8_status q8_quantize_to_linear_operand(const float* x_f32, int64_t M, int64_t K,
                                        double input_scale, int32_t input_zero_point,
                                        int8_t* x_q, void* operand, size_t operand_bytes,
                                        q8_stream_t stream) {
  if (!x_f32) return Q8_ERR_NULL;
  if (M < 1 || K < 1 || !mul_ok(M, K) || (M * K) % 4 != 0) return Q8_ERR_SHAPE;
  if (M > INT32_MAX || K > INT32_MAX / 2) return Q8_ERR_SHAPE;
  if (!scale_ok(input_scale) || !zp_ok(input_zero_point)) return Q8_ERR_ARG;
  q8_status st = check_operand(operand, operand_bytes, M, K);
  if (st != Q8_OK) return st;
  return cuda_status(q8::launch_quantize_rows_bf16(
      x_f32, M, K, recip_f32(input_scale), input_zero_point, x_q,
      static_cast<__nv_bfloat16*>(operand), round_up(K, kTileK), cs(stream),
      operand_bound_word(operand, M, K)));
}

static q8_status run_operand_packed(const void* operand, int64_t M, int64_t K, double input_scale,
                                    const void* packed, int64_t N, const float* ws,
                                    const float* bias, double output_scale, int32_t ozp,
                                    int relu, int8_t* out, int32_t* acc_out, q8_stream_t stream,
                                    uint64_t wait_ns = 0, int stall_fill = 0) {
  if (reinterpret_cast<uintptr_t>(packed) % q8::kWorkspaceAlign != 0 ||
      reinterpret_cast<uintptr_t>(operand) % q8::kWorkspaceAlign != 0)
    return Q8_ERR_ALIGN;
  q8::TcLinear L{};
  L.a = static_cast<const __nv_bfloat16*>(operand);
  L.b = static_cast<const __nv_bfloat16*>(packed);
  L.M = M;
  L.N = N;
  L.Kp = round_up(K, kTileK);
  L.ws = ws;
  L.bias = bias;
  L.rq = make_rq(input_scale, output_scale, ozp, relu);
  L.out = out;
  L.acc_out = acc_out;
  L.a_bound_dev = operand_bound_word(const_cast<void*>(operand), M, K);
  L.a_bound_host = 255;
  L.w_bound_dev = operand_bound_word(const_cast<void*>(packed), N, K);
  L.wait_ns = wait_ns;
  L.stall_fill = stall_fill;
  return cuda_status(q8::launch_tc_linear(L, cs(stream)));
}

q8_status q8_linear_operand_packed(const void* operand, int64_t M, int64_t K, double input_scale,
                                   const void* packed_weight, int64_t N,
                                   const float* weight_scales, const float* bias,
                                   double output_scale, int32_t output_zero_point,
                                   const char* activation, int8_t* out, q8_stream_t stream) {
  if (!operand) return Q8_ERR_NULL;
  // input_zero_point is already applied inside the operand; 0 passes its guard
  int relu = 0;
  q8_status st = check_linear(static_cast<const int8_t*>(operand), M, K, input_scale, 0,
                              packed_weight, N, weight_scales, output_scale, output_zero_point,
                              activation, out, &relu);
  if (st != Q8_OK) return st;
  return run_operand_packed(operand, M, K, input_scale, packed_weight, N, weight_scales, bias,
                            output_scale, output_zero_point, relu, out, nullptr, stream);
}

q8_status q8_linear_packed(const int8_t* x, int64_t M, int64_t K, double input_scale,
                           int32_t input_zero_point, const void* packed_weight, int64_t N,
                           const float* weight_scales, const float* bias, double output_scale,
                           int32_t output_zero_point, const char* activation, int8_t* out,
                           void* workspace, size_t workspace_bytes, q8_stream_t stream) {
  int relu = 0;
  q8_status st = check_linear(x, M, K, input_scale, input_zero_point, packed_weight, N,
                              weight_scales, output_scale, output_zero_point, activation, out,
                              &relu);
  if (st != Q8_OK) return st;
  st = q8_linear_prepare_operand(x, M, K, input_zero_point, workspace, workspace_bytes, stream);
  if (st != Q8_OK) return st;
  return run_operand_packed(workspace, M, K, input_scale, packed_weight, N, weight_scales, bias,
                            output_scale, output_zero_point, relu, out, nullptr, stream);
}

q8_status q8_quantize_linear_packed(const float* x_f32, int64_t M, int64_t K, double input_scale,
                                    int32_t input_zero_point, const void* packed_weight,
                                    int64_t N, const float* weight_scales, const float* bias,
                                    double output_scale, int32_t output_zero_point,
                                    const char* activation, int8_t* x_q, int8_t* out,
                                    void* workspace, size_t workspace_bytes, q8_stream_t stream) {
  if (!x_f32) return Q8_ERR_NULL;
  // the quantize op's guard (numel % 4) is implied by (M*K) % 4 == 0 below
  int relu = 0;
  q8_status st = check_linear(reinterpret_cast<const int8_t*>(x_f32), M, K, input_scale,
                              input_zero_point, packed_weight, N, weight_scales, output_scale,
                              output_zero_point, activation, out, &relu);
  if (st != Q8_OK) return st;
  st = q8_quantize_to_linear_operand(x_f32, M, K, input_scale, input_zero_point, x_q, workspace,
                                     workspace_bytes, stream);
  if (st != Q8_OK) return st;
  return run_operand_packed(workspace, M, K, input_scale, packed_weight, N, weight_scales, bias,
                            output_scale, output_zero_point, relu, out, nullptr, stream);
}

q8_status q8_linear_operand_init(void* operand, int64_t M, int64_t K, size_t operand_bytes,
                                 q8_stream_t stream) {
  if (M < 1 || K < 1 || !mul_ok(M, K) || M > INT32_MAX || K > INT32_MAX / 2) return Q8_ERR_SHAPE;
  q8_status st = check_operand(operand, operand_bytes, M, K);
  if (st != Q8_OK) return st;
  return cuda_status(q8::launch_fused_trailer_init(
      reinterpret_cast<uint32_t*>(operand_bound_word(operand, M, K)), cs(stream)));
}

q8_status q8_quantize_linear_fused(const float* x_f32, int64_t M, int64_t K, double input_scale,
                                   int32_t input_zero_point, const void* packed_weight, int64_t N,
                                   const float* weight_scales, const float* bias,
                                   double output_scale, int32_t output_zero_point,
                                   const char* activation, int8_t* x_q, int8_t* out,
                                   void* operand, size_t operand_bytes, q8_stream_t stream) {
  if (!x_f32) return Q8_ERR_NULL;
  int relu = 0;
  q8_status st = check_linear(reinterpret_cast<const int8_t*>(x_f32), M, K, input_scale,
                              input_zero_point, packed_weight, N, weight_scales, output_scale,
                              output_zero_point, activation, out, &relu);
  if (st != Q8_OK) return st;
  st = check_operand(operand, operand_bytes, M, K);
  if (st != Q8_OK) return st;
  if (reinterpret_cast<uintptr_t>(packed_weight) % q8::kWorkspaceAlign != 0) return Q8_ERR_ALIGN;
  q8::TcLinear L{};
  L.a = static_cast<const __nv_bfloat16*>(operand);
  L.b = static_cast<const __nv_bfloat16*>(packed_weight);
  L.M = M;
  L.N = N;
  L.Kp = round_up(K, kTileK);
  L.ws = weight_scales;
  L.bias = bias;
  L.rq = make_rq(input_scale, output_scale, output_zero_point, relu);
  L.out = out;
  L.a_bound_host = a_bound_of(input_zero_point);
  L.w_bound_dev = operand_bound_word(const_cast<void*>(packed_weight), N, K);
  L.qx = x_f32;
  L.qxq = x_q;
  L.qinv = recip_f32(input_scale);
  L.qzp = input_zero_point;
  L.qK = K;
  L.qsync = reinterpret_cast<uint32_t*>(operand_bound_word(operand, M, K));
  return cuda_status(q8::launch_tc_linear(L, cs(stream)));
}

q8_status q8_linear_packed_acc32(const int8_t* x, int64_t M, int64_t K, int32_t input_zero_point,
                                 const void* packed_weight, int64_t N, int32_t* acc,
                                 void* workspace, size_t workspace_bytes, q8_stream_t stream) {
  static const float kOne = 1.0f;
  q8_status st = check_linear(x, M, K, 1.0, input_zero_point, packed_weight, N, &kOne, 1.0, 0,
                              "none", acc);
  if (st != Q8_OK) return st;
  st = q8_linear_prepare_operand(x, M, K, input_zero_point, workspace, workspace_bytes, stream);
  if (st != Q8_OK) return st;
  return run_operand_packed(workspace, M, K, 1.0, packed_weight, N, nullptr, nullptr, 1.0, 0, 0,
                            nullptr, acc, stream);
}

// Failure-detection test: q8_linear_packed_acc32 with a short barrier-wait
// limit and one TMA ring fill left out, so the kernel's bounded wait runs out.
q8_status q8_debug_linear_packed_stall(const int8_t* x, int64_t M, int64_t K,
                                       int32_t input_zero_point, const void* packed_weight,
                                       int64_t N, int32_t* acc, void* workspace,
                                       size_t workspace_bytes, uint64_t wait_limit_ns,
                                       int64_t skip_fill, q8_stream_t stream) {
  static const float kOne = 1.0f;
  q8_status st = check_linear(x, M, K, 1.0, input_zero_point, packed_weight, N, &kOne, 1.0, 0,
                              "none", acc);
  if (st != Q8_OK) return st;
  if (wait_limit_ns < 1000000ull || wait_limit_ns > 1000000000ull) return Q8_ERR_ARG;
  if (skip_fill < 0 || skip_fill >= (int64_t{1} << 30)) return Q8_ERR_ARG;
  st = q8_linear_prepare_operand(x, M, K, input_zero_point, workspace, workspace_bytes, stream);
  if (st != Q8_OK) return st;
  return run_operand_packed(workspace, M, K, 1.0, packed_weight, N, nullptr, nullptr, 1.0, 0, 0,
                            nullptr, acc, stream, wait_limit_ns, static_cast<int>(skip_fill) + 1);
}

}  // extern "C"
