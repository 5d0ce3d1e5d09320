// tc_gemm_host.cu -- host-side pieces shared by the tensor-core GEMM launchers:
// the device error word, and TMA tensor-map encoding (driver entry point
// obtained through the runtime, so the library needs no -lcuda).
#include <cuda.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include <cstdint>
#include <mutex>

#include "q8ta_internal.h"

namespace q8 {

// Kernels whose bounded waits expire write a code here (first one wins).
__device__ uint32_t g_q8_error = 0;

uint32_t* device_error_word() {
  static std::mutex mu;
  static uint32_t* cache[64] = {nullptr};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return nullptr;
  std::lock_guard<std::mutex> lock(mu);
  if (cache[dev] == nullptr) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_q8_error) != cudaSuccess) return nullptr;
    cache[dev] = static_cast<uint32_t*>(p);
  }
  return cache[dev];
}

cudaError_t read_device_error(uint32_t* code, bool clear) {
  cudaError_t e = cudaDeviceSynchronize();
  if (e != cudaSuccess) return e;
  e = cudaMemcpyFromSymbol(code, g_q8_error, sizeof(uint32_t));
  if (e != cudaSuccess) return e;
  if (clear) {
    const uint32_t zero = 0;
    e = cudaMemcpyToSymbol(g_q8_error, &zero, sizeof(uint32_t));
  }
  return e;
}

static PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* ptr = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(ptr);
  });
  return fn;
}

bool encode_bf16_tmap(CUtensorMap* map, const void* base, int rank, const uint64_t* dims,
                        const uint64_t* strides_bytes, const uint32_t* box,
                        const uint32_t* element_strides) {
  auto enc = tensor_map_encoder();
  if (!enc) return false;
  uint32_t estr[5] = {1, 1, 1, 1, 1};
  if (rank < 1 || rank > 5) return false;
  if (element_strides != nullptr)
    for (int i = 0; i < rank; ++i) estr[i] = element_strides[i];
  CUresult r = enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, rank, const_cast<void*>(base), dims,
                   strides_bytes, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                   CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                   CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

}  // namespace q8
