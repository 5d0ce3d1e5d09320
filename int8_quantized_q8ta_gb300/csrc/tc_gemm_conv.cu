// tc_gemm_conv.cu -- q8ta_conv2d_transposed on the tensor-core GEMM
// (tc_gemm_kernel.cuh): per-stride-phase implicit GEMM over the
// channel-blocked NHWC copy of x - input_zero_point, read through 5-D TMA
// boxes whose zero fill implements the skipped taps.
#include <cuda.h>
#include <cuda_runtime.h>

#include <algorithm>

#include "q8ta_internal.h"
#include "tc_gemm_kernel.cuh"

namespace q8 {

cudaError_t launch_tc_conv_t(const TcConvT& C, cudaStream_t s) {
  const int bn = pick_bn(C.OC);
  const int64_t Hq = (C.H_out + C.stride_h - 1) / C.stride_h;
  const int64_t Wq = (C.W_out + C.stride_w - 1) / C.stride_w;
  int bw = 1;
  while (bw < Wq && bw < kBM) bw *= 2;
  const int bh = kBM / bw;
  CUtensorMap ma, mb;
  const uint64_t icb = static_cast<uint64_t>(C.ICp / kBK);
  // two k-blocks (channel blocks) per TMA box when they split evenly: the
  // 128-wide tiles need bigger boxes to keep enough bytes in flight per SM
  const int kd = (icb % 2 == 0) ? 2 : 1;
  {
    // channel-blocked NHWC input: [N][ICp/64][H_in][W_in][64] bf16
    const uint64_t dims[5] = {kBK, static_cast<uint64_t>(C.W_in), static_cast<uint64_t>(C.H_in),
                              icb, static_cast<uint64_t>(C.N)};
    const uint64_t row = kBK * 2;
    const uint64_t str[4] = {row, row * C.W_in, row * C.W_in * C.H_in,
                             row * C.W_in * C.H_in * icb};
    const uint32_t box[5] = {kBK, static_cast<uint32_t>(bw), static_cast<uint32_t>(bh),
                             static_cast<uint32_t>(kd), 1};
    if (!encode_bf16_tmap(&ma, C.a, 5, dims, str, box)) return cudaErrorInvalidValue;
  }
  {
    // weight [taps][ICp/64][OC][64] bf16
    const uint64_t dims[3] = {kBK, static_cast<uint64_t>(C.OC),
                              static_cast<uint64_t>(C.Kh * C.Kw) * icb};
    const uint64_t str[2] = {kBK * 2, static_cast<uint64_t>(C.OC) * kBK * 2};
    const uint32_t box[3] = {kBK, static_cast<uint32_t>(bn), static_cast<uint32_t>(kd)};
    if (!encode_bf16_tmap(&mb, C.b, 3, dims, str, box)) return cudaErrorInvalidValue;
  }
  TcParams p{};
  p.mode = 1;
  p.kd = kd;
  p.Nimg = static_cast<int>(C.N);
  p.OC = static_cast<int>(C.OC);
  p.Kh = static_cast<int>(C.Kh);
  p.Kw = static_cast<int>(C.Kw);
  p.H_out = static_cast<int>(C.H_out);
  p.W_out = static_cast<int>(C.W_out);
  p.sh = static_cast<int>(C.stride_h);
  p.sw = static_cast<int>(C.stride_w);
  p.pad_h = static_cast<int>(C.pad_h);
  p.pad_w = static_cast<int>(C.pad_w);
  p.ICp = static_cast<int>(C.ICp);
  p.icb = static_cast<int>(C.ICp / kBK);
  p.BW = bw;
  p.BH = bh;
  p.tiles_w = static_cast<int>((Wq + bw - 1) / bw);
  p.tiles_h = static_cast<int>((Hq + bh - 1) / bh);
  p.tiles_oc = static_cast<int>((C.OC + bn - 1) / bn);
  const int64_t units = C.stride_h * C.N * p.tiles_h * p.tiles_w * p.tiles_oc;
  if (units > (1ll << 30)) return cudaErrorInvalidValue;
  p.total_units = static_cast<int>(units);
  p.subtiles = static_cast<int>(C.stride_w);
  if (C.stride_h <= kMaxPhases) {
    // row phases with more taps first, so the heaviest units start earliest
    int order[kMaxPhases], taps[kMaxPhases];
    for (int ph = 0; ph < C.stride_h; ++ph) {
      const int64_t rh = (ph + C.pad_h) % C.stride_h;
      taps[ph] = rh < C.Kh ? static_cast<int>((C.Kh - rh + C.stride_h - 1) / C.stride_h) : 0;
      order[ph] = ph;
    }
    std::stable_sort(order, order + C.stride_h, [&](int x, int y) { return taps[x] > taps[y]; });
    for (int i = 0; i < C.stride_h; ++i) p.ph_order[i] = static_cast<int8_t>(order[i]);
  }
  p.ws = C.ws;
  p.bias = C.bias;
  p.rq = C.rq;
  p.out = C.out;
  p.acc_out = C.acc_out;
  p.a_bound_dev = nullptr;
  p.a_bound_host = C.a_bound;
  p.store_mode = 0;
  // Whole output rows go through shared memory when a unit's rows fit the
  // stage and split into aligned 16-byte pieces.
  const int64_t wt = static_cast<int64_t>(bw) * C.stride_w;
  const size_t stage_bytes = 2 * static_cast<size_t>(bn) * kBM * C.stride_w;  // two alternating
  const bool staged = C.out != nullptr && C.acc_out == nullptr && bn <= 128 &&
                      C.stride_w <= 2 && wt % 16 == 0 && C.W_out % 16 == 0 &&
                      reinterpret_cast<uintptr_t>(C.out) % 16 == 0;
  p.staged = staged ? 1 : 0;
  if (p.total_units == 0) return cudaSuccess;
  const size_t ostage = staged ? stage_bytes : 0;
  // one CTA per 128-row tile: on this workload the 2-SM MMA measured no
  // faster (its stages fit, but the conv's k-blocks are short and many)
  switch (bn * 4 + kd) {
    case 64 * 4 + 1: return launch_tc_kernel<64, 16, 1, 1, 1>(ma, mb, p, ostage, s);
    case 64 * 4 + 2: return launch_tc_kernel<64, 16, 1, 2, 1>(ma, mb, p, ostage, s);
    case 128 * 4 + 1: return launch_tc_kernel<128, 16, 1, 1, 1>(ma, mb, p, ostage, s);
    case 128 * 4 + 2: return launch_tc_kernel<128, 16, 1, 2, 1>(ma, mb, p, ostage, s);
    case 256 * 4 + 1: return launch_tc_kernel<256, 8, 1, 1, 1>(ma, mb, p, ostage, s);
    default: return launch_tc_kernel<256, 8, 1, 2, 1>(ma, mb, p, ostage, s);
  }
}

}  // namespace q8
