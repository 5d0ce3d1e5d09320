// tc_gemm_linear.cu -- q8ta_linear on the tensor-core GEMM (tc_gemm_kernel.cuh):
// K-blocked bf16 operands [K/64][rows][64].
//
// Tiles: wide problems (M > 128, N > 128) run on CTA pairs, 256 x BN tiles
// through the 2-SM MMA with two k-blocks per TMA box; BN is picked from
// {256, 240, 224, 192} to fill the last wave of the persistent grid best
// (N = 11008: 46 column tiles of 240 make 368 pair tiles = 4.84 waves on 76
// SM pairs, against 4.53 waves of 256-wide tiles, which cost 5 full waves).
// Smaller problems use one CTA per 128 x BN tile.
#include <cuda.h>
#include <cuda_runtime.h>

#include <cstdint>

#include "q8ta_internal.h"
#include "tc_gemm_kernel.cuh"

namespace q8 {

namespace {

// Column-tile width for the pair path: the fewest tile-columns of work in
// the slowest SM pair, i.e. ceil(tiles / pairs) * BN, ties to the wider tile.
int pick_pair_bn(int64_t M, int64_t N, int pairs) {
  static const int kCands[] = {256, 240, 224, 192};
  const int64_t tiles_m = (M + 2 * kBM - 1) / (2 * kBM);
  int best = 256;
  int64_t best_cost = INT64_MAX;
  for (int bn : kCands) {
    const int64_t units = tiles_m * ((N + bn - 1) / bn);
    const int64_t cost = (units + pairs - 1) / pairs * bn;
    if (cost < best_cost) {
      best_cost = cost;
      best = bn;
    }
  }
  return best;
}

// The instantiation for a tile width (MODE 0: prepared operand; MODE 7:
// the same with the fused quantize prologue).
template <int MODE>
cudaError_t launch_linear_bn(bool pair, int bn, const CUtensorMap& ma, const CUtensorMap& mb,
                             const TcParams& p, cudaStream_t s) {
  if (pair) {
    switch (bn) {
      case 256: return launch_tc_kernel<256, 8, MODE, 2, 2>(ma, mb, p, s);
      case 240: return launch_tc_kernel<240, 12, MODE, 2, 2>(ma, mb, p, s);
      case 224: return launch_tc_kernel<224, 8, MODE, 2, 2>(ma, mb, p, s);
      default: return launch_tc_kernel<192, 8, MODE, 2, 2>(ma, mb, p, s);
    }
  }
  // 16 epilogue warps where their register share fits the column slice
  switch (bn) {
    case 64: return launch_tc_kernel<64, 16, MODE, 1, 1>(ma, mb, p, s);
    case 128: return launch_tc_kernel<128, 16, MODE, 1, 1>(ma, mb, p, s);
    default: return launch_tc_kernel<256, 8, MODE, 1, 1>(ma, mb, p, s);
  }
}

}  // namespace

cudaError_t launch_tc_linear(const TcLinear& L, cudaStream_t s) {
  const bool pair = L.M > kBM && L.N > 128;
  const int cg = pair ? 2 : 1;
  // two k-blocks per TMA box on pairs: one k-block per box measured slower
  // (the per-box cost of the TMA unit, not bytes, sets the feed rate)
  const int kd = pair ? 2 : 1;
  const int bn = pair ? pick_pair_bn(L.M, L.N, device_sm_count() / 2) : pick_bn(L.N);
  const uint64_t kblocks = static_cast<uint64_t>(L.Kp / kBK);
  CUtensorMap ma, mb;
  {
    // K-blocked operand: [Kp/64][M][64] bf16; a box is one CTA's 128 rows
    const uint64_t dims[3] = {kBK, static_cast<uint64_t>(L.M), kblocks};
    const uint64_t str[2] = {kBK * 2, static_cast<uint64_t>(L.M) * kBK * 2};
    const uint32_t box[3] = {kBK, kBM, static_cast<uint32_t>(kd)};
    if (!encode_bf16_tmap(&ma, L.a, 3, dims, str, box)) return cudaErrorInvalidValue;
  }
  {
    // packed weight [Kp/64][N][64] bf16; a box is one CTA's bn / cg rows
    const uint64_t dims[3] = {kBK, static_cast<uint64_t>(L.N), kblocks};
    const uint64_t str[2] = {kBK * 2, static_cast<uint64_t>(L.N) * kBK * 2};
    const uint32_t box[3] = {kBK, static_cast<uint32_t>(bn / cg), static_cast<uint32_t>(kd)};
    if (!encode_bf16_tmap(&mb, L.b, 3, dims, str, box)) return cudaErrorInvalidValue;
  }
  TcParams p{};
  p.mode = 0;
  p.kd = kd;
  p.M = static_cast<int>(L.M);
  p.N = static_cast<int>(L.N);
  p.kb_total = static_cast<int>(L.Kp / kBK);
  // row tiles of 128, counted in groups of cg (a CTA pair takes 256 rows)
  p.tiles_m = static_cast<int>(((L.M + kBM - 1) / kBM + cg - 1) / cg);
  const int tiles_n = static_cast<int>((L.N + bn - 1) / bn);
  p.total_units = p.tiles_m * tiles_n;
  p.subtiles = 1;
  p.ws = L.ws;
  p.bias = L.bias;
  p.rq = L.rq;
  p.out = L.out;
  p.acc_out = L.acc_out;
  p.a_bound_dev = L.a_bound_dev;
  p.a_bound_host = L.a_bound_host;
  p.w_bound_dev = L.w_bound_dev;
  p.wait_ns = L.wait_ns;
  p.stall_fill = L.stall_fill;
  if (L.qx != nullptr) {
    const int kb = static_cast<int>(L.Kp / kBK);
    p.qckb = fused_chunk_kb(kb);
    p.qseg_log2 = 0;
    while ((1 << p.qseg_log2) < p.qckb * 8) ++p.qseg_log2;
    p.qnch = (kb + p.qckb - 1) / p.qckb;
    if (L.qsync == nullptr || p.qnch > kFusedMaxChunks) return cudaErrorInvalidValue;
    p.qx = L.qx;
    p.qxq = L.qxq;
    p.qdst = reinterpret_cast<uint4*>(const_cast<__nv_bfloat16*>(L.a));
    p.qsync = L.qsync;
    p.qinv = L.qinv;
    p.qzp = L.qzp;
    p.qK = static_cast<int>(L.qK);
    const uintptr_t xa = reinterpret_cast<uintptr_t>(L.qx), qa = reinterpret_cast<uintptr_t>(L.qxq);
    p.qvec = (L.qK % 8 == 0) && (xa % 16 == 0) && (L.qxq == nullptr || qa % 8 == 0) ? 1 : 0;
  }
  const uintptr_t oa = reinterpret_cast<uintptr_t>(L.out);
  p.store_mode = (L.N % 16 == 0 && oa % 16 == 0) ? 2 : (oa % 4 == 0 ? 1 : 0);
  if (p.total_units == 0) return cudaSuccess;
  return L.qx != nullptr ? launch_linear_bn<7>(pair, bn, ma, mb, p, s)
                        : launch_linear_bn<0>(pair, bn, ma, mb, p, s);
}

__global__ void fused_trailer_init_kernel(uint32_t* t) {
  pdl_wait();  // a launch before this one may still use the trailer
  pdl_launch_dependents();
  // [0] the worst-case |x - zp| bound until a launch writes the real one
  if (threadIdx.x == 0) t[0] = 255u;
  if (threadIdx.x == 1) t[kFusedWordDone] = 0u;
  if (threadIdx.x == 2) *reinterpret_cast<uint64_t*>(t + kFusedWordMagic) = kFusedMagic;
  if (threadIdx.x >= kFusedWordChunk0 && threadIdx.x < kFusedWordChunk0 + kFusedMaxChunks)
    t[threadIdx.x] = 0u;
}

cudaError_t launch_fused_trailer_init(uint32_t* trailer, cudaStream_t s) {
  return launch_pdl(fused_trailer_init_kernel, 1, 64, 0, s, trailer);
}

}  // namespace q8
