// noalloc.cu -- q8_linear_noalloc: q8_linear with its scratch in a fixed,
// library-owned device array instead of a caller-provided workspace.
//
// Why it exists: some callers cannot allocate device memory at the point
// where they run a linear layer.  A plugin inside a host runtime that owns
// the whole device memory pool may be forbidden to call cudaMalloc; a
// latency-critical serving loop cannot afford cudaMalloc/cudaFree, which may
// synchronize the device or stall; an embedded deployment may fix its
// memory budget once, at start-up.  Such callers still own their inputs and
// outputs and pass them in; only the scratch moves here.
//
// The scratch is the file-scope array below: Q8_LINEAR_NOALLOC_SCRATCH_BYTES
// (16 MiB), held on every GPU that loads this library until the process
// exits.  It holds the two bf16 operand copies q8_linear's tensor-core path
// needs (x - input_zero_point and the weight, K rounded up to 64).
#include <algorithm>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <cstdint>
#include <mutex>

#include "api_common.h"
#include "q8ta.h"
#include "q8ta_internal.h"

namespace {

static __device__ __align__(256) uint8_t g_linear_noalloc_scratch[Q8_LINEAR_NOALLOC_SCRATCH_BYTES];

constexpr int kMaxDevices = 64;
std::mutex g_setup_mutex;
void* g_scratch_ptr[kMaxDevices] = {nullptr};

// Set-up, once per device, with that device current: the device address of
// the array.  (In host code the array's name is only a host-side stand-in,
// never a device address.)
cudaError_t scratch_for_current_device(void** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lock(g_setup_mutex);
  if (g_scratch_ptr[dev] == nullptr) {
    void* ptr = nullptr;
    e = cudaGetSymbolAddress(&ptr, g_linear_noalloc_scratch);
    if (e != cudaSuccess) return e;
    g_scratch_ptr[dev] = ptr;
  }
  *out = g_scratch_ptr[dev];
  return cudaSuccess;
}

size_t rows_bytes(int64_t rows, int64_t Kp) {
  return q8::align_ws(static_cast<size_t>(rows) * static_cast<size_t>(Kp) * 2);
}

}  // namespace

extern "C" q8_status q8_linear_noalloc(const int8_t* x, int64_t M, int64_t K, double input_scale,
                                       int32_t input_zero_point, const int8_t* weight, int64_t N,
                                       const int32_t* weight_sums, const float* weight_scales,
                                       const float* bias, double output_scale,
                                       int32_t output_zero_point, const char* activation,
                                       int8_t* out, q8_stream_t stream) {
  if (M == 1) {
    // q8_linear's M == 1 path (the gemv kernel) uses no scratch at all.
    return q8_linear(x, M, K, input_scale, input_zero_point, weight, N, weight_sums,
                     weight_scales, bias, output_scale, output_zero_point, activation, out,
                     nullptr, 0, stream);
  }
  // q8_linear's own guards first (it launches nothing while a guard fails)
  q8_status st = q8_linear(x, M, K, input_scale, input_zero_point, weight, N, weight_sums,
                           weight_scales, bias, output_scale, output_zero_point, activation, out,
                           nullptr, 0, stream);
  if (st != Q8_ERR_WORKSPACE) return st;
  const int64_t Kp = q8::round_up(K, q8::kTileK);
  const size_t a_bytes = rows_bytes(M, Kp);
  const size_t need = a_bytes + rows_bytes(N, Kp);
  if (need > Q8_LINEAR_NOALLOC_SCRATCH_BYTES) return Q8_ERR_WORKSPACE;
  void* scratch = nullptr;
  if (scratch_for_current_device(&scratch) != cudaSuccess) return Q8_ERR_CUDA;
  // Nothing in the scratch needs to start at zero: the two conversions write
  // every byte the GEMM then reads (padding columns included), in stream
  // order, so the previous call's contents are never observed.
  auto* a = static_cast<__nv_bfloat16*>(scratch);
  auto* b = reinterpret_cast<__nv_bfloat16*>(static_cast<uint8_t*>(scratch) + a_bytes);
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  cudaError_t e = q8::launch_rows_to_bf16(x, M, K, K, input_zero_point, a, Kp, s);
  if (e == cudaSuccess) e = q8::launch_rows_to_bf16(weight, N, K, K, 0, b, Kp, s);
  if (e != cudaSuccess) return Q8_ERR_CUDA;
  q8::TcLinear L{};
  L.a = a;
  L.b = b;
  L.M = M;
  L.N = N;
  L.Kp = Kp;
  L.ws = weight_scales;
  L.bias = bias;
  // the guards above passed, so the activation is "none" or "relu"
  L.rq = q8api::make_rq(input_scale, output_scale, output_zero_point,
                        q8api::parse_activation(activation) == 1 ? 1 : 0);
  // largest |x - input_zero_point| over int8 x: sets the exact f32 chunk length
  L.a_bound_host = q8api::a_bound_of(input_zero_point);
  L.out = out;
  return q8::launch_tc_linear(L, s) == cudaSuccess ? Q8_OK : Q8_ERR_CUDA;
}
