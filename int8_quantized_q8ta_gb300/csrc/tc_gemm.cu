// tc_gemm.cu -- exact int8 contraction on the sm_103a tcgen05 tensor cores.
//
// What it computes: the int32 accumulator of "Add q8ta_linear op" (Solution
// paragraph), acc[m,n] = sum_k (x[m,k] - input_zero_point) * w[n,k], and of
// "Add q8ta_conv2d_transposed op" (Solution paragraph, the gather over valid
// taps), followed by the fused dequantize -> requantize -> int8 epilogue.
//
// How, on GB300: tcgen05 has no integer MMA on sm_103a, so the operands are
// bf16 copies of the integers: x - input_zero_point lies in [-255, 255] and
// w in [-128, 127], both exact in bf16, and every product (|p| <= 32640) is
// exact in the f32 accumulator.  The K loop is cut into chunks of 512 so the
// f32 partial sum of a chunk stays below 2^24 in magnitude (512 * 32640 <
// 2^24) and is therefore an exact integer; each chunk's TMEM accumulator is
// drained by the epilogue warps into int32 registers (exact conversion) while
// the MMA warp already fills the other TMEM buffer.  Integer addition of the
// chunk sums is exact (modulo 2^32, like the pages' i32 accumulator).
//
// Transposed convolution is an implicit GEMM per stride phase: outputs with
// oh % stride_h == ph and ow % stride_w == pw all use the same taps
// kh = (ph + pad_h) mod stride_h + i*stride_h (likewise kw), and tap (kh, kw)
// reads the input at (oh' + dh, ow' + dw) with dh = (ph + pad_h - kh) /
// stride_h, an integer by construction.  A 4-D TMA box over the NHWC bf16
// input fetches that shifted window; coordinates outside the input are
// filled with zeros by the TMA unit, which is exactly "taps outside the input
// contribute nothing" because the stored values are x - input_zero_point.
//
// Warp roles (320 threads, one CTA per SM, persistent over output tiles):
//   warp 0      TMA producer (one thread)
//   warp 1      TMEM allocator and MMA issuer (one thread)
//   warps 2..9  epilogue: warp w reads TMEM lanes 32*(w%4)..+31, half of the
//               tile's columns each, keeps the int32 running sums in registers
// Every mbarrier wait has a time limit (about 1 s); on expiry the CTA records
// a code in g_q8_error, stops issuing work, waits (again bounded) for its own
// copies and MMAs in flight, frees TMEM and returns.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include <algorithm>
#include <cstdint>
#include <mutex>

#include "device_common.cuh"
#include "q8ta_internal.h"

namespace q8 {

__device__ uint32_t g_q8_error = 0;

enum : uint32_t {
  kErrWaitFull = 0x101,
  kErrWaitEmpty = 0x102,
  kErrWaitAccFull = 0x103,
  kErrWaitAccEmpty = 0x104,
  kErrWaitDrain = 0x105,
  kErrWaitEpi = 0x106,
};

constexpr uint64_t kWaitLimitNs = 1000ull * 1000ull * 1000ull;
constexpr int kBM = 128;
constexpr int kBK = 64;             // bf16 per 128-byte row
constexpr int kChunkKb = 8;         // 8 x 64 = 512 products per exact f32 chunk
constexpr int kMaxStages = 8;
constexpr int kMaxPhases = 16;

// Threads of a CTA with E epilogue warps: the TMA warp, the MMA warp, E more.
__host__ __device__ constexpr int cta_threads(int epi_warps) { return 64 + 32 * epi_warps; }
constexpr int kMaxBN = 256;

struct TcParams {
  int mode;          // 0 = linear, 1 = transposed convolution
  int stages;        // smem ring depth
  int total_units;   // work units; a unit is `subtiles` consecutive tiles
  int subtiles;      // 1 (linear) or stride_w (transposed convolution)
  // linear
  int M, N, kb_total, tiles_m;
  // transposed convolution
  int Nimg, OC, Kh, Kw, H_out, W_out, sh, sw, pad_h, pad_w, icb, ICp;
  int BW, BH, tiles_w, tiles_h, tiles_oc;
  int staged;        // conv output goes through the shared-memory stage
  int8_t ph_order[kMaxPhases];  // row phases, most taps first (stride_h <= kMaxPhases)
  uint32_t stage_off;  // byte offset of that stage from the aligned smem base
  // epilogue
  const float* ws;
  const float* bias;
  Requant rq;
  int8_t* out;
  int32_t* acc_out;
  int store_mode;    // linear int8 stores: 2 = 16 B, 1 = 4 B, 0 = bytes
};

struct TileInfo {
  int num_kb;
  // linear
  int mb, nb;
  // conv
  int n, hb, wb, ocb, ph, pw, rh, rw, ntw;
};

// Unit u, sub-tile j -> tile coordinates.  Transposed convolution units are
// (row phase ph, image n, row block hb, column block wb, channel block ocb);
// their sub-tiles are the stride_w column phases pw, so one CTA produces
// every output column of its rows and can write whole rows.
__device__ __forceinline__ TileInfo decode_tile(const TcParams& p, int u, int j) {
  TileInfo ti{};
  if (p.mode == 0) {
    ti.mb = u % p.tiles_m;
    ti.nb = u / p.tiles_m;
    ti.num_kb = p.kb_total;
  } else {
    ti.ocb = u % p.tiles_oc;
    u /= p.tiles_oc;
    ti.wb = u % p.tiles_w;
    u /= p.tiles_w;
    ti.hb = u % p.tiles_h;
    u /= p.tiles_h;
    ti.n = u % p.Nimg;
    const int phx = u / p.Nimg;
    ti.ph = (p.sh <= kMaxPhases) ? p.ph_order[phx] : phx;
    ti.pw = j;
    ti.rh = (ti.ph + p.pad_h) % p.sh;
    ti.rw = (ti.pw + p.pad_w) % p.sw;
    const int nth = ti.rh < p.Kh ? (p.Kh - ti.rh + p.sh - 1) / p.sh : 0;
    ti.ntw = ti.rw < p.Kw ? (p.Kw - ti.rw + p.sw - 1) / p.sw : 0;
    ti.num_kb = nth * ti.ntw * p.icb;
  }
  return ti;
}

struct Ctl {
  uint64_t full[kMaxStages];
  uint64_t empty[kMaxStages];
  uint64_t acc_full[2];
  uint64_t acc_empty[2];
  uint64_t drain;
  uint64_t epi_bar;            // epilogue-warps rendezvous (one arrival per epilogue warp)
  uint32_t tmem_base;
  uint32_t abort_flag;
  alignas(16) float ep_ws[2][kMaxBN];  // per-tile column scales / biases, by tile parity
  alignas(16) float ep_b[2][kMaxBN];
};

// Bounded wait.  Returns false when this CTA is aborting (this wait timed
// out, or another role's did).
__device__ __forceinline__ bool wait_bar(uint32_t bar, uint32_t parity, volatile uint32_t* abort_flag,
                                         uint32_t code) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = global_timer_ns();
  while (true) {
    if (mbar_try_wait(bar, parity)) return true;
    if (*abort_flag) return false;
    if (global_timer_ns() - t0 > kWaitLimitNs) {
      *abort_flag = 1u;
      atomicCAS(&g_q8_error, 0u, code);
      return false;
    }
  }
}

// Bounded wait used while shutting down: ignores the abort flag.
__device__ __forceinline__ void wait_bar_final(uint32_t bar, uint32_t parity) {
  if (mbar_try_wait(bar, parity)) return;
  const uint64_t t0 = global_timer_ns();
  while (!mbar_try_wait(bar, parity)) {
    if (global_timer_ns() - t0 > kWaitLimitNs) {
      atomicCAS(&g_q8_error, 0u, kErrWaitDrain);
      return;
    }
  }
}

// Rendezvous of the epilogue warps on an mbarrier (bounded, unlike
// bar.sync, so one aborted warp cannot strand the others).  Shared-memory
// writes made before the call are visible to every epilogue thread after it.
__device__ __forceinline__ bool epi_sync(Ctl* ctl, uint32_t& phase, volatile uint32_t* abort_flag) {
  // every epilogue warp arrives once per rendezvous
  __syncwarp();
  bool ok = true;
  if ((threadIdx.x & 31) == 0) {
    mbar_arrive(smem_u32(&ctl->epi_bar));
    ok = wait_bar(smem_u32(&ctl->epi_bar), phase, abort_flag, kErrWaitEpi);
  }
  phase ^= 1u;
  ok = __shfl_sync(0xffffffffu, ok ? 1 : 0, 0) != 0;
  __syncwarp();
  return ok;
}

template <int BN, int EPI>
__global__ void __launch_bounds__(cta_threads(EPI), 1)
    tc_gemm_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                   const TcParams p) {
  constexpr int kEpiWarps = EPI;
  constexpr int kEpiThreads = EPI * 32;
  constexpr int kColGroups = EPI / 4;     // epilogue warps sharing one TMEM lane quarter
  constexpr uint32_t kABytes = kBM * kBK * 2;
  constexpr uint32_t kBBytes = BN * kBK * 2;
  constexpr uint32_t kStageBytes = kABytes + kBBytes;
  constexpr uint32_t kTmemCols = 2 * BN;  // two f32 accumulator buffers
  constexpr int kColsPerWarp = BN / kColGroups;
  // columns loaded from TMEM per wait: 32 where registers allow
  constexpr int kDrainCols = kColsPerWarp >= 128 ? 16 : (kColsPerWarp < 32 ? kColsPerWarp : 32);
  static_assert(kColsPerWarp % 16 == 0, "epilogue column slice must be a multiple of 16");
  constexpr uint32_t kIdesc = idesc_bf16_f32(kBM, BN);
  const int S = p.stages;

  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw_base = smem_u32(smem_raw);
  const uint32_t base = (raw_base + 1023u) & ~1023u;
  uint8_t* smem = smem_raw + (base - raw_base);
  Ctl* ctl = reinterpret_cast<Ctl*>(smem + S * kStageBytes);
  uint8_t* ostage = smem + p.stage_off;
  volatile uint32_t* abort_flag = &ctl->abort_flag;

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    for (int s = 0; s < S; ++s) {
      mbar_init(smem_u32(&ctl->full[s]), 1);
      mbar_init(smem_u32(&ctl->empty[s]), 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(smem_u32(&ctl->acc_full[b]), 1);
      mbar_init(smem_u32(&ctl->acc_empty[b]), kEpiWarps);
    }
    mbar_init(smem_u32(&ctl->drain), 1);
    mbar_init(smem_u32(&ctl->epi_bar), kEpiWarps);
    ctl->abort_flag = 0u;
    fence_mbar_init();
    tma_prefetch_desc(&tmA);
    tma_prefetch_desc(&tmB);
  }
  if (warp == 1) {
    tmem_alloc(smem_u32(&ctl->tmem_base), kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = ctl->tmem_base;

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      uint32_t stage = 0, phase = 0;
      uint32_t fills = 0;
      bool ok = true;
      for (int u = blockIdx.x; u < p.total_units && ok; u += gridDim.x) {
        for (int j = 0; j < p.subtiles && ok; ++j) {
          const TileInfo ti = decode_tile(p, u, j);
          for (int kb = 0; kb < ti.num_kb; ++kb) {
            if (!wait_bar(smem_u32(&ctl->empty[stage]), phase ^ 1u, abort_flag, kErrWaitEmpty)) {
              ok = false;
              break;
            }
            const uint32_t full = smem_u32(&ctl->full[stage]);
            const uint32_t sa = base + stage * kStageBytes;
            const uint32_t sb = sa + kABytes;
            mbar_arrive_expect_tx(full, kStageBytes);
            if (p.mode == 0) {
              tma_load_3d(sa, &tmA, full, 0, ti.mb * kBM, kb);
              tma_load_3d(sb, &tmB, full, 0, ti.nb * BN, kb);
            } else {
              const int icx = kb % p.icb;
              const int rest = kb / p.icb;
              const int tw = rest % ti.ntw, th = rest / ti.ntw;
              const int kh = ti.rh + th * p.sh, kw = ti.rw + tw * p.sw;
              const int dh = (ti.ph + p.pad_h - kh) / p.sh;
              const int dw = (ti.pw + p.pad_w - kw) / p.sw;
              tma_load_5d(sa, &tmA, full, 0, ti.wb * p.BW + dw, ti.hb * p.BH + dh, icx, ti.n);
              tma_load_3d(sb, &tmB, full, 0, ti.ocb * BN, (kh * p.Kw + kw) * p.icb + icx);
            }
            ++fills;
            if (++stage == static_cast<uint32_t>(S)) {
              stage = 0;
              phase ^= 1u;
            }
          }
        }
      }
      // Let every copy this thread issued land before the CTA can exit.
      for (int s = 0; s < S; ++s) {
        const uint32_t f = (fills > static_cast<uint32_t>(s)) ? (fills - s + S - 1) / S : 0;
        if (f > 0) wait_bar_final(smem_u32(&ctl->full[s]), (f - 1) & 1u);
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      uint32_t stage = 0, phase = 0, acc_it = 0;
      bool ok = true;
      for (int u = blockIdx.x; u < p.total_units && ok; u += gridDim.x) {
        for (int j = 0; j < p.subtiles && ok; ++j) {
          const TileInfo ti = decode_tile(p, u, j);
          for (int kb0 = 0; kb0 < ti.num_kb && ok; kb0 += kChunkKb) {
            const uint32_t buf = acc_it & 1u, use = acc_it >> 1;
            if (!wait_bar(smem_u32(&ctl->acc_empty[buf]), (use & 1u) ^ 1u, abort_flag,
                          kErrWaitAccEmpty)) {
              ok = false;
              break;
            }
            tc_fence_after();
            const uint32_t d = tmem_base + buf * BN;
            const int kend = min(kb0 + kChunkKb, ti.num_kb);
            for (int kb = kb0; kb < kend; ++kb) {
              if (!wait_bar(smem_u32(&ctl->full[stage]), phase, abort_flag, kErrWaitFull)) {
                ok = false;
                break;
              }
              tc_fence_after();
              const uint32_t sa = base + stage * kStageBytes;
              const uint64_t da = sw128_kmajor_desc(sa);
              const uint64_t db = sw128_kmajor_desc(sa + kABytes);
#pragma unroll
              for (int k = 0; k < kBK / 16; ++k) {
                // +32 bytes along K inside the 128-byte swizzled row
                umma_bf16(d, da + 2u * k, db + 2u * k, kIdesc, (kb > kb0 || k > 0) ? 1u : 0u);
              }
              umma_commit(smem_u32(&ctl->empty[stage]));
              if (++stage == static_cast<uint32_t>(S)) {
                stage = 0;
                phase ^= 1u;
              }
            }
            if (!ok) break;
            umma_commit(smem_u32(&ctl->acc_full[buf]));
            ++acc_it;
          }
        }
      }
      // Every MMA issued so far must finish before TMEM is freed.
      umma_commit(smem_u32(&ctl->drain));
      wait_bar_final(smem_u32(&ctl->drain), 0u);
    }
  } else {
    // ------------------------------------------------------------ epilogue
    const int quarter = warp & 3;           // TMEM lanes this warp may read
    const int group = (warp - 2) >> 2;      // which column slice
    const int row = quarter * 32 + lane;
    const int col0 = group * kColsPerWarp;
    const int et = threadIdx.x - 64;  // 0 .. kEpiThreads-1
    const uint32_t lane_addr = static_cast<uint32_t>(quarter * 32) << 16;
    uint32_t acc_it = 0, epi_phase = 0, tile_par = 0;
    bool ok = true;
    for (int u = blockIdx.x; u < p.total_units && ok; u += gridDim.x) {
      for (int j = 0; j < p.subtiles && ok; ++j) {
        const TileInfo ti = decode_tile(p, u, j);
        int32_t sum[kColsPerWarp];
#pragma unroll
        for (int c = 0; c < kColsPerWarp; ++c) sum[c] = 0;
        for (int kb0 = 0; kb0 < ti.num_kb; kb0 += kChunkKb) {
          const uint32_t buf = acc_it & 1u, use = acc_it >> 1;
          bool got = true;
          if (lane == 0)
            got = wait_bar(smem_u32(&ctl->acc_full[buf]), use & 1u, abort_flag, kErrWaitAccFull);
          got = __shfl_sync(0xffffffffu, got ? 1 : 0, 0) != 0;
          if (!got) {
            ok = false;
            break;
          }
          tc_fence_after();
          // Each chunk sum is an integer below 2^24 in magnitude, so the f32 ->
          // int32 conversion is exact; the int32 adds wrap like the pages' i32.
#pragma unroll
          for (int c = 0; c < kColsPerWarp / kDrainCols; ++c) {
            uint32_t r[kDrainCols];
#pragma unroll
            for (int h = 0; h < kDrainCols / 16; ++h)
              tmem_ld_16cols(tmem_base + lane_addr + buf * BN + col0 + kDrainCols * c + 16 * h,
                             *reinterpret_cast<uint32_t(*)[16]>(&r[16 * h]));
            tmem_ld_wait();
#pragma unroll
            for (int i = 0; i < kDrainCols; ++i)
              sum[kDrainCols * c + i] = static_cast<int32_t>(
                  static_cast<uint32_t>(sum[kDrainCols * c + i]) +
                  static_cast<uint32_t>(__float2int_rn(__uint_as_float(r[i]))));
          }
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(smem_u32(&ctl->acc_empty[buf]));
          ++acc_it;
        }
        if (!ok) break;

        // ---- fused epilogue
        const int gcolbase = (p.mode == 0) ? ti.nb * BN : ti.ocb * BN;
        const int ncols = (p.mode == 0) ? p.N : p.OC;
        if (p.acc_out == nullptr) {
          // this tile's column scales and biases, once, into shared memory
          if (et < BN) {
            const int gc = gcolbase + et;
            ctl->ep_ws[tile_par][et] = (gc < ncols) ? __ldg(p.ws + gc) : 0.0f;
            ctl->ep_b[tile_par][et] = (gc < ncols && p.bias) ? __ldg(p.bias + gc) : 0.0f;
          }
          if (!epi_sync(ctl, epi_phase, abort_flag)) {
            ok = false;
            break;
          }
        }
        const float* sws = ctl->ep_ws[tile_par] + col0;
        const float* sbs = ctl->ep_b[tile_par] + col0;
        tile_par ^= 1u;

        if (p.mode == 0) {
          const int grow = ti.mb * kBM + row;
          const int gcol0 = gcolbase + col0;
          if (grow < p.M) {
            if (p.acc_out) {
              int32_t* dst = p.acc_out + static_cast<int64_t>(grow) * p.N;
#pragma unroll
              for (int c = 0; c < kColsPerWarp; ++c)
                if (gcol0 + c < p.N) dst[gcol0 + c] = sum[c];
            } else {
              int8_t* dst = p.out + static_cast<int64_t>(grow) * p.N;
#pragma unroll
              for (int g = 0; g < kColsPerWarp / 16; ++g) {
                const int c = gcol0 + 16 * g;
                if (c >= p.N) break;
                uint32_t wds[4];
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                  const float4 w4 = *reinterpret_cast<const float4*>(sws + 16 * g + 4 * q);
                  const float4 b4 = *reinterpret_cast<const float4*>(sbs + 16 * g + 4 * q);
                  const int s0 = 16 * g + 4 * q;
                  wds[q] = pack4(requant_one(sum[s0 + 0], w4.x, b4.x, p.rq),
                                 requant_one(sum[s0 + 1], w4.y, b4.y, p.rq),
                                 requant_one(sum[s0 + 2], w4.z, b4.z, p.rq),
                                 requant_one(sum[s0 + 3], w4.w, b4.w, p.rq));
                }
                if (p.store_mode == 2 && c + 16 <= p.N) {
                  *reinterpret_cast<uint4*>(dst + c) = make_uint4(wds[0], wds[1], wds[2], wds[3]);
                } else if (p.store_mode >= 1) {
#pragma unroll
                  for (int q = 0; q < 4; ++q)
                    if (c + 4 * q < p.N) *reinterpret_cast<uint32_t*>(dst + c + 4 * q) = wds[q];
                } else {
                  for (int e = 0; e < 16 && c + e < p.N; ++e)
                    dst[c + e] = static_cast<int8_t>((wds[e >> 2] >> (8 * (e & 3))) & 0xff);
                }
              }
            }
          }
        } else {
          const int hh = row / p.BW, ww = row % p.BW;
          const int oh = (ti.hb * p.BH + hh) * p.sh + ti.ph;
          const int ow = (ti.wb * p.BW + ww) * p.sw + ti.pw;
          const int oc0 = gcolbase + col0;
          const bool inside = (oh < p.H_out && ow < p.W_out);
          if (p.staged && p.acc_out == nullptr) {
            // stage[oc][hh][wl], wl = ww * sw + pw: one unit's rows, all columns
            const int wt = p.BW * p.sw;
            uint8_t* st = ostage + hh * wt + ww * p.sw + ti.pw;
#pragma unroll
            for (int g = 0; g < kColsPerWarp / 16; ++g) {
#pragma unroll
              for (int q = 0; q < 4; ++q) {
                const float4 w4 = *reinterpret_cast<const float4*>(sws + 16 * g + 4 * q);
                const float4 b4 = *reinterpret_cast<const float4*>(sbs + 16 * g + 4 * q);
                const int s0 = 16 * g + 4 * q;
                const int8_t v0 = requant_one(sum[s0 + 0], w4.x, b4.x, p.rq);
                const int8_t v1 = requant_one(sum[s0 + 1], w4.y, b4.y, p.rq);
                const int8_t v2 = requant_one(sum[s0 + 2], w4.z, b4.z, p.rq);
                const int8_t v3 = requant_one(sum[s0 + 3], w4.w, b4.w, p.rq);
                const int ocl = col0 + s0;
                st[(ocl + 0) * p.BH * wt] = static_cast<uint8_t>(v0);
                st[(ocl + 1) * p.BH * wt] = static_cast<uint8_t>(v1);
                st[(ocl + 2) * p.BH * wt] = static_cast<uint8_t>(v2);
                st[(ocl + 3) * p.BH * wt] = static_cast<uint8_t>(v3);
              }
            }
            if (ti.pw == p.sw - 1) {
              // every column phase of this unit is staged: write whole rows
              if (!epi_sync(ctl, epi_phase, abort_flag)) {
                ok = false;
                break;
              }
              const int chunks_per_row = wt / 16;
              const int rows_total = BN * p.BH;
              const int64_t plane = static_cast<int64_t>(p.H_out) * p.W_out;
              const int ow0 = ti.wb * wt;
              for (int it = et; it < rows_total * chunks_per_row; it += kEpiThreads) {
                const int r = it / chunks_per_row, ch = it - r * chunks_per_row;
                const int ocl = r / p.BH, rh = r - ocl * p.BH;
                const int oc = ti.ocb * BN + ocl;
                const int ohh = (ti.hb * p.BH + rh) * p.sh + ti.ph;
                const int oww = ow0 + 16 * ch;
                if (oc < p.OC && ohh < p.H_out && oww < p.W_out) {
                  const uint4 v = *reinterpret_cast<const uint4*>(ostage + r * wt + 16 * ch);
                  int8_t* dst = p.out + (static_cast<int64_t>(ti.n) * p.OC + oc) * plane +
                                static_cast<int64_t>(ohh) * p.W_out + oww;
                  *reinterpret_cast<uint4*>(dst) = v;   // W_out % 16 == 0 when staged
                }
              }
              if (!epi_sync(ctl, epi_phase, abort_flag)) {
                ok = false;
                break;
              }
            }
          } else if (inside) {
            const int64_t plane = static_cast<int64_t>(p.H_out) * p.W_out;
            int8_t* dst = p.out ? p.out + (static_cast<int64_t>(ti.n) * p.OC + oc0) * plane +
                                      static_cast<int64_t>(oh) * p.W_out + ow
                                : nullptr;
            int32_t* adst = p.acc_out ? p.acc_out + (static_cast<int64_t>(ti.n) * p.OC + oc0) * plane +
                                            static_cast<int64_t>(oh) * p.W_out + ow
                                      : nullptr;
#pragma unroll
            for (int g = 0; g < kColsPerWarp / 16; ++g) {
#pragma unroll
              for (int q = 0; q < 4; ++q) {
                const int s0 = 16 * g + 4 * q;
                if (adst) {
#pragma unroll
                  for (int e = 0; e < 4; ++e)
                    if (oc0 + s0 + e < p.OC) adst[(s0 + e) * plane] = sum[s0 + e];
                } else {
                  const float4 w4 = *reinterpret_cast<const float4*>(sws + s0);
                  const float4 b4 = *reinterpret_cast<const float4*>(sbs + s0);
                  const int8_t v[4] = {requant_one(sum[s0 + 0], w4.x, b4.x, p.rq),
                                       requant_one(sum[s0 + 1], w4.y, b4.y, p.rq),
                                       requant_one(sum[s0 + 2], w4.z, b4.z, p.rq),
                                       requant_one(sum[s0 + 3], w4.w, b4.w, p.rq)};
#pragma unroll
                  for (int e = 0; e < 4; ++e)
                    if (oc0 + s0 + e < p.OC) dst[(s0 + e) * plane] = v[e];
                }
              }
            }
          }
        }
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem_base, kTmemCols);
  }
}

// ---------------------------------------------------------------------------
// Host side
// ---------------------------------------------------------------------------
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

static bool encode_bf16(CUtensorMap* map, const void* base, int rank, const uint64_t* dims,
                        const uint64_t* strides_bytes, const uint32_t* box) {
  auto enc = tensor_map_encoder();
  if (!enc) return false;
  uint32_t estr[5] = {1, 1, 1, 1, 1};
  if (rank < 1 || rank > 5) return false;
  CUresult r = enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, rank, const_cast<void*>(base), dims,
                   strides_bytes, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                   CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                   CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

constexpr size_t kSmemBudget = 225 * 1024;   // of the 227 KB a CTA may use

template <int BN, int EPI>
static cudaError_t launch_bn(const CUtensorMap& a, const CUtensorMap& b, TcParams p,
                             size_t out_stage_bytes, cudaStream_t s) {
  constexpr size_t kStage = static_cast<size_t>(kBM) * kBK * 2 + static_cast<size_t>(BN) * kBK * 2;
  const size_t fixed = sizeof(Ctl) + 1024 + out_stage_bytes;
  const int stages = static_cast<int>(std::min<size_t>(kMaxStages, (kSmemBudget - fixed) / kStage));
  if (stages < 2) return cudaErrorInvalidValue;
  p.stages = stages;
  const size_t ctl_end = static_cast<size_t>(stages) * kStage + sizeof(Ctl);
  p.stage_off = static_cast<uint32_t>((ctl_end + 127) / 128 * 128);
  const size_t smem = p.stage_off + out_stage_bytes + 1024;
  static std::once_flag attr_once[64];
  int dev = 0;
  cudaGetDevice(&dev);
  cudaError_t attr_err = cudaSuccess;
  std::call_once(attr_once[dev & 63], [&] {
    attr_err = cudaFuncSetAttribute(tc_gemm_kernel<BN, EPI>,
                                    cudaFuncAttributeMaxDynamicSharedMemorySize,
                                    static_cast<int>(kSmemBudget + 1024));
  });
  if (attr_err != cudaSuccess) return attr_err;
  const int grid = std::max(1, std::min(p.total_units, device_sm_count()));
  tc_gemm_kernel<BN, EPI><<<grid, cta_threads(EPI), smem, s>>>(a, b, p);
  return cudaGetLastError();
}

static int pick_bn(int64_t n) { return n <= 64 ? 64 : (n <= 128 ? 128 : 256); }

static cudaError_t dispatch(int bn, const CUtensorMap& a, const CUtensorMap& b, const TcParams& p,
                            size_t out_stage_bytes, cudaStream_t s) {
  if (p.total_units == 0) return cudaSuccess;
  switch (bn) {
    // 16 epilogue warps where their register share fits the column slice
    case 64: return launch_bn<64, 16>(a, b, p, out_stage_bytes, s);
    case 128: return launch_bn<128, 16>(a, b, p, out_stage_bytes, s);
    default: return launch_bn<256, 8>(a, b, p, out_stage_bytes, s);
  }
}

cudaError_t launch_tc_linear(const TcLinear& L, cudaStream_t s) {
  const int bn = pick_bn(L.N);
  const uint64_t kblocks = static_cast<uint64_t>(L.Kp / kBK);
  CUtensorMap ma, mb;
  {
    // K-blocked operand: [Kp/64][M][64] bf16
    const uint64_t dims[3] = {kBK, static_cast<uint64_t>(L.M), kblocks};
    const uint64_t str[2] = {kBK * 2, static_cast<uint64_t>(L.M) * kBK * 2};
    const uint32_t box[3] = {kBK, kBM, 1};
    if (!encode_bf16(&ma, L.a, 3, dims, str, box)) return cudaErrorInvalidValue;
  }
  {
    const uint64_t dims[3] = {kBK, static_cast<uint64_t>(L.N), kblocks};
    const uint64_t str[2] = {kBK * 2, static_cast<uint64_t>(L.N) * kBK * 2};
    const uint32_t box[3] = {kBK, static_cast<uint32_t>(bn), 1};
    if (!encode_bf16(&mb, L.b, 3, dims, str, box)) return cudaErrorInvalidValue;
  }
  TcParams p{};
  p.mode = 0;
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
  return dispatch(bn, ma, mb, p, 0, s);
}

cudaError_t launch_tc_conv_t(const TcConvT& C, cudaStream_t s) {
  const int bn = pick_bn(C.OC);
  const int64_t Hq = (C.H_out + C.stride_h - 1) / C.stride_h;
  const int64_t Wq = (C.W_out + C.stride_w - 1) / C.stride_w;
  int bw = 1;
  while (bw < Wq && bw < kBM) bw *= 2;
  const int bh = kBM / bw;
  CUtensorMap ma, mb;
  const uint64_t icb = static_cast<uint64_t>(C.ICp / kBK);
  {
    // channel-blocked NHWC input: [N][ICp/64][H_in][W_in][64] bf16
    const uint64_t dims[5] = {kBK, static_cast<uint64_t>(C.W_in), static_cast<uint64_t>(C.H_in),
                              icb, static_cast<uint64_t>(C.N)};
    const uint64_t row = kBK * 2;
    const uint64_t str[4] = {row, row * C.W_in, row * C.W_in * C.H_in,
                             row * C.W_in * C.H_in * icb};
    const uint32_t box[5] = {kBK, static_cast<uint32_t>(bw), static_cast<uint32_t>(bh), 1, 1};
    if (!encode_bf16(&ma, C.a, 5, dims, str, box)) return cudaErrorInvalidValue;
  }
  {
    // weight [taps][ICp/64][OC][64] bf16
    const uint64_t dims[3] = {kBK, static_cast<uint64_t>(C.OC),
                              static_cast<uint64_t>(C.Kh * C.Kw) * icb};
    const uint64_t str[2] = {kBK * 2, static_cast<uint64_t>(C.OC) * kBK * 2};
    const uint32_t box[3] = {kBK, static_cast<uint32_t>(bn), 1};
    if (!encode_bf16(&mb, C.b, 3, dims, str, box)) return cudaErrorInvalidValue;
  }
  TcParams p{};
  p.mode = 1;
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
  p.store_mode = 0;
  // Whole output rows go through shared memory when a unit's rows fit the
  // stage and split into aligned 16-byte pieces.
  const int64_t wt = static_cast<int64_t>(bw) * C.stride_w;
  const size_t stage_bytes = static_cast<size_t>(bn) * kBM * C.stride_w;
  const bool staged = C.out != nullptr && C.acc_out == nullptr && bn <= 128 &&
                      C.stride_w <= 2 && wt % 16 == 0 && C.W_out % 16 == 0 &&
                      reinterpret_cast<uintptr_t>(C.out) % 16 == 0;
  p.staged = staged ? 1 : 0;
  return dispatch(bn, ma, mb, p, staged ? stage_bytes : 0, s);
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

}  // namespace q8
