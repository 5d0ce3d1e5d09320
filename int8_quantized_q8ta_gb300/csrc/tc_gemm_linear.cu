// tc_gemm_linear.cu -- q8ta_linear on the tensor-core GEMM (tc_gemm_kernel.cuh):
// K-blocked bf16 operands [K/64][rows][64], 128 x BN tiles, one k-block per
// TMA box and ring stage.
#include <cuda.h>
#include <cuda_runtime.h>

#include "q8ta_internal.h"
#include "tc_gemm_kernel.cuh"

namespace q8 {

cudaError_t launch_tc_linear(const TcLinear& L, cudaStream_t s) {
  const int bn = pick_bn(L.N);
  const uint64_t kblocks = static_cast<uint64_t>(L.Kp / kBK);
  // one k-block per TMA box: 128x256 tiles keep 4 ring stages in flight
  const int kd = 1;
  CUtensorMap ma, mb;
  {
    // K-blocked operand: [Kp/64][M][64] bf16
    const uint64_t dims[3] = {kBK, static_cast<uint64_t>(L.M), kblocks};
    const uint64_t str[2] = {kBK * 2, static_cast<uint64_t>(L.M) * kBK * 2};
    const uint32_t box[3] = {kBK, kBM, static_cast<uint32_t>(kd)};
    if (!encode_bf16_tmap(&ma, L.a, 3, dims, str, box)) return cudaErrorInvalidValue;
  }
  {
    const uint64_t dims[3] = {kBK, static_cast<uint64_t>(L.N), kblocks};
    const uint64_t str[2] = {kBK * 2, static_cast<uint64_t>(L.N) * kBK * 2};
    const uint32_t box[3] = {kBK, static_cast<uint32_t>(bn), static_cast<uint32_t>(kd)};
    if (!encode_bf16_tmap(&mb, L.b, 3, dims, str, box)) return cudaErrorInvalidValue;
  }
  TcParams p{};
  p.mode = 0;
  p.kd = kd;
  (void)kd;
  p.M = static_cast<int>(L.M);
  p.N = static_cast<int>(L.N);
  p.kb_total = static_cast<int>(L.Kp / kBK);
  p.tiles_m = static_cast<int>((L.M + kBM - 1) / kBM);
  const int tiles_n = static_cast<int>((L.N + bn - 1) / bn);
  p.total_units = p.tiles_m * tiles_n;
  p.subtiles = 1;
  p.ws = L.ws;
  p.bias = L.bias;
  p.rq = L.rq;
  p.out = L.out;
  p.acc_out = L.acc_out;
  const uintptr_t oa = reinterpret_cast<uintptr_t>(L.out);
  p.store_mode = (L.N % 16 == 0 && oa % 16 == 0) ? 2 : (oa % 4 == 0 ? 1 : 0);
  if (p.total_units == 0) return cudaSuccess;
  // 16 epilogue warps where their register share fits the column slice
  switch (bn) {
    case 64: return launch_tc_kernel<64, 16, 0, 1>(ma, mb, p, 0, s);
    case 128: return launch_tc_kernel<128, 16, 0, 1>(ma, mb, p, 0, s);
    default: return launch_tc_kernel<256, 8, 0, 1>(ma, mb, p, 0, s);
  }
}

}  // namespace q8
