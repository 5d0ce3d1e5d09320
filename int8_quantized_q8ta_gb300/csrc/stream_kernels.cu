// stream_kernels.cu -- the HBM-bandwidth-bound q8ta kernels for sm_103a:
// quantize_per_tensor, dequantize_per_tensor, the M == 1 q8ta_linear_gemv,
// and the int8 -> bf16 operand preparation for the tensor-core GEMM.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <cstdint>
#include <mutex>

#include "device_common.cuh"
#include "q8ta_internal.h"

namespace q8 {

int device_sm_count() {
  static int cache[64] = {0};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 148;
  if (cache[dev] == 0) {
    int n = 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0)
      n = 148;
    cache[dev] = n;
  }
  return cache[dev];
}

static int stream_grid(int64_t work_items, int threads, int blocks_per_sm) {
  int64_t want = (work_items + threads - 1) / threads;
  int64_t cap = static_cast<int64_t>(device_sm_count()) * blocks_per_sm;
  return static_cast<int>(std::max<int64_t>(1, std::min(want, cap)));
}

// Grid of a grid-stride kernel: no more blocks than fit on the GPU at once
// (its occupancy at `threads`), so every block starts in the first wave and
// no late partial wave stretches the tail.  The occupancy query is made once
// per kernel and device (`cache` is the call site's own table).
template <typename Kernel>
static int resident_grid(Kernel kernel, int (&cache)[64], int64_t work_items, int threads) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) dev = 0;
  if (cache[dev] == 0) {
    int per_sm = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kernel, threads, 0) != cudaSuccess ||
        per_sm < 1) {
      cudaGetLastError();
      per_sm = 4;
    }
    cache[dev] = per_sm;
  }
  return stream_grid(work_items, threads, cache[dev]);
}

// ---------------------------------------------------------------------------
// quantize_per_tensor ("Add quantize_per_tensor op", Solution paragraph):
// q = clamp(rint(x * inv_scale) + zp, -128, 127).
// Vector path: one float4 in, one packed 32-bit word out per item; U items
// per thread per round are loaded before any is converted.
// ---------------------------------------------------------------------------
// (quantize_one: device_common.cuh)
template <int U>
__global__ void __launch_bounds__(256) quantize_vec_kernel(const float4* __restrict__ x, int64_t n4,
                                                           float inv, int32_t zp,
                                                           uint32_t* __restrict__ out) {
  pdl_wait();
  pdl_launch_dependents();
  const int64_t step = static_cast<int64_t>(gridDim.x) * blockDim.x * U;
  for (int64_t base = static_cast<int64_t>(blockIdx.x) * blockDim.x * U + threadIdx.x; base < n4;
       base += step) {
    float4 v[U];
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const int64_t i = base + static_cast<int64_t>(u) * blockDim.x;
      if (i < n4) v[u] = __ldcs(x + i);
    }
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const int64_t i = base + static_cast<int64_t>(u) * blockDim.x;
      if (i < n4)
        __stcs(out + i, pack4(quantize_one(v[u].x, inv, zp), quantize_one(v[u].y, inv, zp),
                              quantize_one(v[u].z, inv, zp), quantize_one(v[u].w, inv, zp)));
    }
  }
}

__global__ void __launch_bounds__(256) quantize_scalar_kernel(const float* __restrict__ x, int64_t n,
                                                              float inv, int32_t zp,
                                                              int8_t* __restrict__ out) {
  pdl_wait();
  pdl_launch_dependents();
  for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < n;
       i += static_cast<int64_t>(gridDim.x) * blockDim.x)
    out[i] = quantize_one(x[i], inv, zp);
}

cudaError_t launch_quantize(const float* x, int64_t numel, float inv, int32_t zp, int8_t* out,
                            cudaStream_t s) {
  if (numel == 0) return cudaSuccess;
  const bool vec = (reinterpret_cast<uintptr_t>(x) % 16 == 0) &&
                   (reinterpret_cast<uintptr_t>(out) % 4 == 0) && (numel % 4 == 0);
  if (vec) {
    constexpr int U = 4;
    const int64_t n4 = numel / 4;
    static int occ[64];
    const int grid = resident_grid(quantize_vec_kernel<U>, occ, (n4 + U - 1) / U, 256);
    return launch_pdl(quantize_vec_kernel<U>, grid, 256, 0, s, reinterpret_cast<const float4*>(x),
                      n4, inv, zp, reinterpret_cast<uint32_t*>(out));
  } else {
    return launch_pdl(quantize_scalar_kernel, stream_grid(numel, 256, 8), 256, 0, s, x, numel, inv,
                      zp, out);
  }
  return cudaGetLastError();
}

// ---------------------------------------------------------------------------
// dequantize_per_tensor: y = ((float)q - (float)zp) * scale.
// ---------------------------------------------------------------------------
__global__ void __launch_bounds__(256) dequantize_kernel(const int8_t* __restrict__ q, int64_t n,
                                                         float scale, float zp,
                                                         float* __restrict__ out) {
  pdl_wait();
  pdl_launch_dependents();
  const bool vec = (reinterpret_cast<uintptr_t>(q) % 4 == 0) &&
                   (reinterpret_cast<uintptr_t>(out) % 16 == 0);
  const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
  if (vec) {
    const int64_t n4 = n / 4;
    const uint32_t* q4 = reinterpret_cast<const uint32_t*>(q);
    float4* o4 = reinterpret_cast<float4*>(out);
    for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < n4;
         i += stride) {
      const uint32_t w = __ldcs(q4 + i);
      float4 r;
      r.x = __fmul_rn(__fsub_rn(static_cast<float>(static_cast<int8_t>(w & 0xff)), zp), scale);
      r.y = __fmul_rn(__fsub_rn(static_cast<float>(static_cast<int8_t>((w >> 8) & 0xff)), zp),
                      scale);
      r.z = __fmul_rn(__fsub_rn(static_cast<float>(static_cast<int8_t>((w >> 16) & 0xff)), zp),
                      scale);
      r.w = __fmul_rn(__fsub_rn(static_cast<float>(static_cast<int8_t>(w >> 24)), zp), scale);
      __stcs(o4 + i, r);
    }
    for (int64_t i = n4 * 4 + static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < n;
         i += stride)
      out[i] = __fmul_rn(__fsub_rn(static_cast<float>(q[i]), zp), scale);
  } else {
    for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < n;
         i += stride)
      out[i] = __fmul_rn(__fsub_rn(static_cast<float>(q[i]), zp), scale);
  }
}

cudaError_t launch_dequantize(const int8_t* q, int64_t numel, float scale, float zp, float* out,
                              cudaStream_t s) {
  if (numel == 0) return cudaSuccess;
  return launch_pdl(dequantize_kernel, stream_grid(numel / 4 + 1, 256, 8), 256, 0, s, q, numel,
                    scale, zp, out);
  return cudaGetLastError();
}

// ---------------------------------------------------------------------------
// q8ta_linear_gemv (M == 1): "Add q8ta_linear op", Solution paragraph, with
// the zero point folded as sum x*w - zp * sum w (Constraints paragraph);
// both sums are exact int32 dp4a dot products, so the fold is exact modulo
// 2^32 like the accumulator itself.
//
// gemv_rows_kernel (K % 16 == 0, 16-byte aligned x and weight): one warp per
// output row, 16 rows per block; each lane keeps 8 16-byte weight loads in
// flight (4 KB of the row per round), and each round's 4 KB of x is brought
// into shared memory once per block instead of every warp reading all of x
// from L2.  The kernel lets the next kernel on the stream launch first
// thing, then, before waiting for the previous one:
//  * the plain form asks for the block's weight slab (16 contiguous rows) to
//    be brought into L2 with one bulk prefetch.  A prefetch into L2 can never
//    hand stale data to the loads that follow the wait, because L2 is where
//    the GPU's memory is coherent (a write by the previous kernel updates the
//    line there);
//  * the packed form (a load-time weight, written only by
//    q8_linear_gemv_pack_weight, which waits for its copy: no kernel that may
//    still run writes it) loads its first round into registers and sums it.
// In a run of gemvs (one per layer of a decode step) each call's weight so
// streams in while the previous call is still running.
// gemv_kernel is the 4-byte and 1-byte fallback: 4 rows per block, x read
// by every warp.
// ---------------------------------------------------------------------------
// FOLD: also sum the weights (the fold term zp * sum w)
template <bool FOLD>
__device__ __forceinline__ void dp4a_acc(uint32_t w, uint32_t x, int& dot, int& wsum) {
  dot = __dp4a(static_cast<int>(w), static_cast<int>(x), dot);
  if constexpr (FOLD) wsum = __dp4a(static_cast<int>(w), 0x01010101, wsum);
}

template <int VEC, bool FOLD>
__global__ void __launch_bounds__(128) gemv_kernel(const int8_t* __restrict__ x, int K, int32_t izp,
                                                   const int8_t* __restrict__ w, int N,
                                                   const float* __restrict__ ws,
                                                   const float* __restrict__ bias, Requant rq,
                                                   int8_t* __restrict__ out) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int n = blockIdx.x * 4 + warp;
  static_assert(VEC == 4 || VEC == 1, "16-byte rows take gemv_rows_kernel");
  if (n < N) {
    const int8_t* wr = w + static_cast<int64_t>(n) * K;
    for (int off = lane * 128; off < K; off += 32 * 128)
      asm volatile("prefetch.global.L2 [%0];" ::"l"(wr + off));
  }
  pdl_launch_dependents();
  pdl_wait();
  // the row's scale and bias are requested now, so their latency hides
  // under the weight stream instead of following the reduction
  float wsn = 0.0f, bn = 0.0f;
  if (n < N && lane == 0) {
    wsn = __ldg(ws + n);
    bn = bias ? __ldg(bias + n) : 0.0f;
  }
  int dot = 0, wsum = 0;
  if (n < N) {
    const int8_t* wr = w + static_cast<int64_t>(n) * K;
    if constexpr (VEC == 4) {
      const uint32_t* w1 = reinterpret_cast<const uint32_t*>(wr);
      const uint32_t* x1 = reinterpret_cast<const uint32_t*>(x);
      for (int j = lane; j < K / 4; j += 32) dp4a_acc<FOLD>(__ldcs(w1 + j), __ldg(x1 + j), dot, wsum);
    } else {
      for (int k = lane; k < K; k += 32) {
        const int wv = wr[k];
        dot = static_cast<int>(static_cast<uint32_t>(dot) +
                               static_cast<uint32_t>(wv * static_cast<int>(x[k])));
        wsum += wv;
      }
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      // modulo-2^32 sums, like the int32 accumulator they form
      dot = static_cast<int>(static_cast<uint32_t>(dot) +
                             static_cast<uint32_t>(__shfl_xor_sync(0xffffffffu, dot, o)));
      wsum = static_cast<int>(static_cast<uint32_t>(wsum) +
                              static_cast<uint32_t>(__shfl_xor_sync(0xffffffffu, wsum, o)));
    }
    if (lane == 0) {
      const int32_t acc = static_cast<int32_t>(static_cast<uint32_t>(dot) -
                                               static_cast<uint32_t>(izp) * static_cast<uint32_t>(wsum));
      out[n] = requant_one(acc, wsn, bn, rq);
    }
  }
}

// Sum over the warp's lanes modulo 2^32 (like the int32 accumulator it forms).
__device__ __forceinline__ int warp_sum_u32(int v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1)
    v = static_cast<int>(static_cast<uint32_t>(v) +
                         static_cast<uint32_t>(__shfl_xor_sync(0xffffffffu, v, o)));
  return v;
}

constexpr int kGemvRows = 16;                   // rows (warps) per block
constexpr int kGemvUnr = 8;                     // 16-byte loads per lane and round
constexpr int kGemvRound = 32 * kGemvUnr;       // 16-byte words of a row per round

// kPacked: the weight is a packed (load-time) one, read before the wait.
template <bool kPacked>
__global__ void __launch_bounds__(32 * kGemvRows, 2)
    gemv_rows_kernel(const int8_t* __restrict__ x, int K, int32_t izp, const int8_t* __restrict__ w,
                     int N, const float* __restrict__ ws, const float* __restrict__ bias,
                     Requant rq, int8_t* __restrict__ out) {
  constexpr int T = 32 * kGemvRows;
  static_assert(kGemvRound <= T, "one round of x is at most one 16-byte word per thread");
  __shared__ int4 xs[kGemvRound];
  pdl_launch_dependents();
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int n = blockIdx.x * kGemvRows + warp;
  const bool row_ok = n < N;
  const int nv = K / 16;
  const bool one_round = nv <= kGemvRound;
  if (threadIdx.x == 0 && (!kPacked || !one_round)) {
    // into L2 now: the block's rows (packed: the rounds after the first),
    // one contiguous, 16-byte aligned run
    const int n0 = blockIdx.x * kGemvRows;
    const uint32_t bytes = static_cast<uint32_t>(min(kGemvRows, N - n0)) * static_cast<uint32_t>(K);
    asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(w + static_cast<int64_t>(n0) * K),
                 "r"(bytes)
                 : "memory");
  }
  const int4* w4 = reinterpret_cast<const int4*>(w + static_cast<int64_t>(row_ok ? n : 0) * K);
  int4 wv[kGemvUnr];
  int dot = 0, wsum = 0;
  if constexpr (kPacked) {
#pragma unroll
    for (int u = 0; u < kGemvUnr; ++u) {
      const int idx = lane + 32 * u;
      wv[u] = (row_ok && idx < nv) ? __ldcs(w4 + idx) : make_int4(0, 0, 0, 0);
    }
#pragma unroll
    for (int u = 0; u < kGemvUnr; ++u) {
      wsum = __dp4a(wv[u].x, 0x01010101, wsum);
      wsum = __dp4a(wv[u].y, 0x01010101, wsum);
      wsum = __dp4a(wv[u].z, 0x01010101, wsum);
      wsum = __dp4a(wv[u].w, 0x01010101, wsum);
    }
    // a row of one round has its whole weight sum now: reduce it before the wait
    if (one_round) wsum = warp_sum_u32(wsum);
  }
  pdl_wait();
  float wsn = 0.0f, bn = 0.0f;
  if (row_ok && lane == 0) {
    wsn = __ldg(ws + n);
    bn = bias ? __ldg(bias + n) : 0.0f;
  }
  const int4* x4 = reinterpret_cast<const int4*>(x);
  for (int base = 0; base < nv; base += kGemvRound) {
    // rounds whose weights are loaded (and summed) after the wait
    const bool late = !kPacked || base > 0;
    if (base > 0) __syncthreads();  // every warp is done with the previous round's x
    if (late) {
#pragma unroll
      for (int u = 0; u < kGemvUnr; ++u) {
        const int idx = base + lane + 32 * u;
        wv[u] = (row_ok && idx < nv) ? __ldcs(w4 + idx) : make_int4(0, 0, 0, 0);
      }
    }
    if (threadIdx.x < kGemvRound) {
      // this round's x, one 16-byte word per thread (zero past K)
      const int i = base + threadIdx.x;
      xs[threadIdx.x] = i < nv ? __ldg(x4 + i) : make_int4(0, 0, 0, 0);
    }
    __syncthreads();
#pragma unroll
    for (int u = 0; u < kGemvUnr; ++u) {
      // past K, both the weight and x words are zero
      const int4 xv = xs[lane + 32 * u];
      dot = __dp4a(wv[u].x, xv.x, dot);
      dot = __dp4a(wv[u].y, xv.y, dot);
      dot = __dp4a(wv[u].z, xv.z, dot);
      dot = __dp4a(wv[u].w, xv.w, dot);
      if (late) {
        wsum = __dp4a(wv[u].x, 0x01010101, wsum);
        wsum = __dp4a(wv[u].y, 0x01010101, wsum);
        wsum = __dp4a(wv[u].z, 0x01010101, wsum);
        wsum = __dp4a(wv[u].w, 0x01010101, wsum);
      }
    }
  }
  if (!row_ok) return;
  dot = warp_sum_u32(dot);
  if (!kPacked || !one_round) wsum = warp_sum_u32(wsum);
  if (lane == 0) {
    const int32_t acc = static_cast<int32_t>(static_cast<uint32_t>(dot) -
                                             static_cast<uint32_t>(izp) * static_cast<uint32_t>(wsum));
    out[n] = requant_one(acc, wsn, bn, rq);
  }
}

// Measured in a chain of 24 calls (1 x 4096 x 4096, packed weight): one warp
// per row in blocks of 4 rows, each warp reading all of x from L2, 3.85 us
// per call; x through shared memory with 8 / 16 / 32 rows per block, 3.49 /
// 3.40 / 3.48 us; 16 rows with the next kernel let in first thing, 3.29 us.
// (A variant staging whole weight slabs in shared memory with bulk copies,
// one block per SM and two calls resident, measured 4.4 us: after the
// dependency wait its work ran behind the next call's copies.)
static cudaError_t launch_gemv_rows(bool packed, const int8_t* x, int64_t K, int32_t izp,
                                    const int8_t* w, int64_t N, const float* ws, const float* bias,
                                    Requant rq, int8_t* out, cudaStream_t s) {
  const int grid = static_cast<int>((N + kGemvRows - 1) / kGemvRows);
  if (packed)
    return launch_pdl(gemv_rows_kernel<true>, grid, 32 * kGemvRows, 0, s, x, (int)K, izp, w, (int)N,
                      ws, bias, rq, out);
  return launch_pdl(gemv_rows_kernel<false>, grid, 32 * kGemvRows, 0, s, x, (int)K, izp, w, (int)N,
                    ws, bias, rq, out);
}

cudaError_t launch_gemv(const int8_t* x, int64_t K, int32_t izp, const int8_t* w, int64_t N,
                        const float* ws, const float* bias, Requant rq, int8_t* out,
                        cudaStream_t s) {
  const int grid = static_cast<int>((N + 3) / 4);
  const uintptr_t xa = reinterpret_cast<uintptr_t>(x), wa = reinterpret_cast<uintptr_t>(w);
  // 16-byte loads need every row start 16-byte aligned, hence K % 16 == 0.
  // (In an earlier 4-row form, skipping the weight sums when the zero point
  // is 0 measured slower in a chain of calls, 4.6 against 4.4 us per call:
  // fewer registers, more blocks resident per SM.)
  if (xa % 16 == 0 && wa % 16 == 0 && K % 16 == 0)
    return launch_gemv_rows(false, x, K, izp, w, N, ws, bias, rq, out, s);
  if (xa % 4 == 0 && wa % 4 == 0 && K % 4 == 0)
    return launch_pdl(gemv_kernel<4, true>, grid, 128, 0, s, x, (int)K, izp, w, (int)N, ws, bias,
                      rq, out);
  return launch_pdl(gemv_kernel<1, true>, grid, 128, 0, s, x, (int)K, izp, w, (int)N, ws, bias, rq,
                    out);
}

// q8ta_linear_gemv from a packed (load-time) weight: the same kernel, its
// first round of weights read before the wait.
cudaError_t launch_gemv_packed(const int8_t* x, int64_t K, int32_t izp, const int8_t* w, int64_t N,
                               const float* ws, const float* bias, Requant rq, int8_t* out,
                               cudaStream_t s) {
  const uintptr_t xa = reinterpret_cast<uintptr_t>(x), wa = reinterpret_cast<uintptr_t>(w);
  if (!(xa % 16 == 0 && wa % 16 == 0 && K % 16 == 0))
    return launch_gemv(x, K, izp, w, N, ws, bias, rq, out, s);
  return launch_gemv_rows(true, x, K, izp, w, N, ws, bias, rq, out, s);
}

// ---------------------------------------------------------------------------
// Operand preparation for the tensor-core GEMM.  int8 values, and the
// differences x - zp in [-255, 255], are exact in bf16 (8 significant bits).
// ---------------------------------------------------------------------------
// (bf16x2_from_ints, kblocked_index16: device_common.cuh)

// One thread converts 8 consecutive elements (16 bytes of output) of a row.
__global__ void __launch_bounds__(256) rows_to_bf16_kernel(const int8_t* __restrict__ src,
                                                           int64_t rows, int64_t K, int64_t ld,
                                                           int32_t zp, uint4* __restrict__ dst,
                                                           int64_t Kp, int32_t* bound_word) {
  pdl_wait();
  pdl_launch_dependents();
  if (bound_word != nullptr && blockIdx.x == 0 && threadIdx.x == 0)
    *bound_word = max(128 + zp, 127 - zp);
  const int64_t per_row = Kp / 8;
  const int64_t total = rows * per_row;
  const bool vec8 = (K % 8 == 0) && (ld % 8 == 0) && (reinterpret_cast<uintptr_t>(src) % 8 == 0);
  for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < total;
       i += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    const int64_t r = i / per_row;
    const int64_t k0 = (i - r * per_row) * 8;
    const int8_t* sp = src + r * ld + k0;
    int v[8];
    if (vec8 && k0 + 8 <= K) {
      const uint2 raw = *reinterpret_cast<const uint2*>(sp);
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        v[j] = static_cast<int8_t>((raw.x >> (8 * j)) & 0xff) - zp;
        v[4 + j] = static_cast<int8_t>((raw.y >> (8 * j)) & 0xff) - zp;
      }
    } else {
#pragma unroll
      for (int j = 0; j < 8; ++j) v[j] = (k0 + j < K) ? static_cast<int>(sp[j]) - zp : 0;
    }
    uint4 o;
    o.x = bf16x2_from_ints(v[0], v[1]);
    o.y = bf16x2_from_ints(v[2], v[3]);
    o.z = bf16x2_from_ints(v[4], v[5]);
    o.w = bf16x2_from_ints(v[6], v[7]);
    dst[kblocked_index16(r, k0, rows)] = o;
  }
}

cudaError_t launch_rows_to_bf16(const int8_t* src, int64_t rows, int64_t K, int64_t ld, int32_t zp,
                                __nv_bfloat16* dst, int64_t Kp, cudaStream_t s,
                                int32_t* bound_word) {
  if (rows == 0) return cudaSuccess;
  const int64_t items = rows * (Kp / 8);
  return launch_pdl(rows_to_bf16_kernel, stream_grid(items, 256, 8), 256, 0, s, src, rows, K, ld,
                    zp, reinterpret_cast<uint4*>(dst), Kp, bound_word);
  return cudaGetLastError();
}

// Fused quantize of fp32 rows into the GEMM operand (and the int8 op output).
// An item is 8 consecutive elements of a row; each thread loads U items
// (U * 32 bytes) before converting any of them.  Idx is the index type:
// 32-bit when the item count allows (integer division is a long sequence of
// instructions, four times longer in 64 bits).
template <int U, typename Idx>
__global__ void __launch_bounds__(256) quantize_rows_bf16_kernel(
    const float* __restrict__ x, Idx rows, Idx K, float inv, int32_t zp,
    int8_t* __restrict__ xq, uint4* __restrict__ dst, Idx Kp, int32_t* bound_word,
    FastDiv fd_row) {
  pdl_wait();
  pdl_launch_dependents();
  if (bound_word != nullptr && blockIdx.x == 0 && threadIdx.x == 0)
    *bound_word = max(128 + zp, 127 - zp);
  const Idx per_row = Kp / 8;
  const Idx total = rows * per_row;
  const int32_t zpf = zp;
  const bool vec = (K % 8 == 0) && (reinterpret_cast<uintptr_t>(x) % 16 == 0) &&
                   (xq == nullptr || reinterpret_cast<uintptr_t>(xq) % 8 == 0);
  const Idx step = static_cast<Idx>(gridDim.x) * blockDim.x * U;
  for (Idx base = static_cast<Idx>(blockIdx.x) * blockDim.x * U + threadIdx.x; base < total;
       base += step) {
    float4 va[U], vb[U];
    Idx rr[U], kk[U];
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const Idx i = base + static_cast<Idx>(u) * blockDim.x;
      // the row of item i: a multiply-shift division in 32 bits (fd_row
      // divides by per_row), a plain one in 64
      if constexpr (sizeof(Idx) == 4)
        rr[u] = static_cast<Idx>(fast_div(static_cast<uint32_t>(i), fd_row));
      else
        rr[u] = i / per_row;
      kk[u] = (i - rr[u] * per_row) * 8;
      if (vec && i < total && kk[u] + 8 <= K) {
        const float4* xp = reinterpret_cast<const float4*>(x + static_cast<int64_t>(rr[u]) * K + kk[u]);
        va[u] = __ldcs(xp);
        vb[u] = __ldcs(xp + 1);
      }
    }
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const Idx i = base + static_cast<Idx>(u) * blockDim.x;
      if (i >= total) break;
      const int64_t r = rr[u];
      const int64_t k0 = kk[u];
      uint4 o;
      if (vec && k0 + 8 <= K) {
        const float xv[8] = {va[u].x, va[u].y, va[u].z, va[u].w, vb[u].x, vb[u].y, vb[u].z, vb[u].w};
        uint2 qw;
        quantize8_operand(xv, inv, zpf, qw, o);
        if (xq) *reinterpret_cast<uint2*>(xq + r * K + k0) = qw;
      } else {
        int v[8];
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          if (k0 + j < K) {
            const int8_t q = quantize_one(x[r * K + k0 + j], inv, zpf);
            if (xq) xq[r * K + k0 + j] = q;
            v[j] = static_cast<int>(q) - zp;
          } else {
            v[j] = 0;
          }
        }
        o.x = bf16x2_from_ints(v[0], v[1]);
        o.y = bf16x2_from_ints(v[2], v[3]);
        o.z = bf16x2_from_ints(v[4], v[5]);
        o.w = bf16x2_from_ints(v[6], v[7]);
      }
      dst[kblocked_index16(r, k0, static_cast<int64_t>(rows))] = o;
    }
  }
}

cudaError_t launch_quantize_rows_bf16(const float* x, int64_t rows, int64_t K, float inv, int32_t zp,
                                      int8_t* xq, __nv_bfloat16* dst, int64_t Kp, cudaStream_t s,
                                      int32_t* bound_word) {
  if (rows == 0) return cudaSuccess;
  const int64_t items = rows * (Kp / 8);
  // one item per thread per round: fewer registers, more threads resident;
  // a sweep of 1 / 2 / 3 / 4 items per thread measured 9.0 / 9.6 / 10.0 /
  // 9.9 us on 2048 x 4096 (medians of nine launches)
  constexpr int U = 1;
  if (items + 256 * U < (int64_t(1) << 31)) {
    static int occ[64];
    const int grid = resident_grid(quantize_rows_bf16_kernel<U, uint32_t>, occ, (items + U - 1) / U, 256);
    return launch_pdl(quantize_rows_bf16_kernel<U, uint32_t>, grid, 256, 0, s, x,
                      static_cast<uint32_t>(rows), static_cast<uint32_t>(K), inv, zp, xq,
                      reinterpret_cast<uint4*>(dst), static_cast<uint32_t>(Kp), bound_word,
                      make_fastdiv(static_cast<uint32_t>(Kp / 8)));
  } else {
    static int occ[64];
    const int grid = resident_grid(quantize_rows_bf16_kernel<U, int64_t>, occ, (items + U - 1) / U, 256);
    return launch_pdl(quantize_rows_bf16_kernel<U, int64_t>, grid, 256, 0, s, x, rows, K, inv, zp,
                      xq, reinterpret_cast<uint4*>(dst), Kp, bound_word, FastDiv{1u, 0u, 0u, 0u});
  }
  return cudaGetLastError();
}

// NCHW int8 -> channel-blocked NHWC bf16 (x - zp), per group:
// dst[n][j*CBg + c/64][h][w][c%64] for channel c of group j (CBg = ICgp/64
// blocks per group); the padding channels ICg <= c < ICgp hold exactly 0, not
// -zp, so the (64 channels x w x h) box of one k-block is contiguous along w.
// One block of 128 threads per (n, channel block, h, 64 columns), the block
// index split by multiply-shift divisions:
//  * load: each thread reads 32 consecutive bytes of one channel's row (two
//    16-byte loads) into shared memory, rows of 16 words (+1 pad);
//  * store: each thread takes 4 columns x 8 channels, i.e. one word of each
//    of 8 channel rows.  Flipping the top bit of every byte gives x + 128 as
//    an unsigned byte; one byte permute puts byte c of a word under the
//    constant high bytes of 1.5 * 2^23, which makes the float 1.5 * 2^23 +
//    x + 128, and one subtraction of 1.5 * 2^23 + 128 + zp leaves exactly
//    x - zp, whose high half is its bf16 (exact: at most 8 significant
//    bits).  The thread stores 4 pieces of 16 bytes (8 channels of one pixel
//    each), and a warp's store covers 4 whole 128-byte pixel rows.
struct RelayoutDiv {
  FastDiv wb, h, cb, cbg;  // by (W + 63) / 64, H, CB (channel blocks), CBg
};

template <bool VEC>
__global__ void __launch_bounds__(128) nchw_to_nhwc_bf16_kernel(const int8_t* __restrict__ x,
                                                                int64_t groups, int64_t ICg,
                                                                int64_t H, int64_t W, int32_t zp,
                                                                uint4* __restrict__ dst,
                                                                int64_t ICgp, RelayoutDiv dv) {
  __shared__ uint32_t tile[64][17];  // [channel][4-column word]
  pdl_wait();
  pdl_launch_dependents();
  const int64_t CBg = ICgp / 64, CB = CBg * groups, C = groups * ICg;
  // the block index in 32 bits (the launch checks it fits)
  uint32_t q, r;
  fast_divmod(blockIdx.x, dv.wb, q, r);
  const int64_t wb = r;
  fast_divmod(q, dv.h, q, r);
  const int64_t h = r;
  fast_divmod(q, dv.cb, q, r);
  const int64_t cb = r, n = q;
  const int64_t g = fast_div(static_cast<uint32_t>(cb), dv.cbg);
  const int64_t cl0 = (cb - g * CBg) * 64;  // first channel of the block, within its group
  const int64_t w0 = wb * 64;
  const int t = threadIdx.x;
  {
    // channel r, columns 32 hq .. 32 hq + 31
    const int r = t >> 1, hq = t & 1;
    uint32_t v[8] = {0u, 0u, 0u, 0u, 0u, 0u, 0u, 0u};
    if (cl0 + r < ICg) {
      const int8_t* src = x + ((n * C + g * ICg + cl0 + r) * H + h) * W + w0 + 32 * hq;
      if (VEC && w0 + 32 * hq + 32 <= W) {
        const uint4 u0 = __ldcs(reinterpret_cast<const uint4*>(src));
        const uint4 u1 = __ldcs(reinterpret_cast<const uint4*>(src) + 1);
        v[0] = u0.x; v[1] = u0.y; v[2] = u0.z; v[3] = u0.w;
        v[4] = u1.x; v[5] = u1.y; v[6] = u1.z; v[7] = u1.w;
      } else {
        for (int e = 0; e < 32; ++e)
          if (w0 + 32 * hq + e < W)
            v[e >> 2] |= static_cast<uint32_t>(static_cast<uint8_t>(src[e])) << (8 * (e & 3));
      }
    }
#pragma unroll
    for (int k = 0; k < 8; ++k) tile[r][8 * hq + k] = v[k];
  }
  __syncthreads();
  const int cq = t >> 3, cs = t & 7;  // columns 4 cq .. 4 cq + 3, channels 8 cs .. 8 cs + 7
  if (w0 + 4 * cq >= W) return;
  uint32_t a[8];
#pragma unroll
  for (int j = 0; j < 8; ++j) a[j] = tile[8 * cs + j][cq] ^ 0x80808080u;  // bytes x + 128
  // channels past the group's last one are padding: exactly 0
  const int64_t left = ICg - (cl0 + 8 * cs);
  const int nvalid = left >= 8 ? 8 : (left <= 0 ? 0 : static_cast<int>(left));
  // 1.5 * 2^23 + 128 + zp: an integer below 2^24, exact in f32
  const float bias = static_cast<float>(12582912 + 128 + zp);
  uint4* out = dst + (((n * CB + cb) * H + h) * W + w0 + 4 * cq) * 8 + cs;
#pragma unroll
  for (int c = 0; c < 4; ++c) {
    if (w0 + 4 * cq + c >= W) break;
    // bytes: [byte c of the word, 0x00, 0x40, 0x4B] = the bits of 1.5 * 2^23 + (x + 128)
    const uint32_t sel = static_cast<uint32_t>(c) | 0x7650u;
    uint32_t f[8];
#pragma unroll
    for (int j = 0; j < 8; ++j)
      f[j] = __float_as_uint(__fsub_rn(__uint_as_float(__byte_perm(a[j], 0x4B400000u, sel)), bias));
    if (nvalid < 8) {
#pragma unroll
      for (int j = 0; j < 8; ++j) f[j] = j < nvalid ? f[j] : 0u;
    }
    uint4 o;
    o.x = __byte_perm(f[0], f[1], 0x7632);
    o.y = __byte_perm(f[2], f[3], 0x7632);
    o.z = __byte_perm(f[4], f[5], 0x7632);
    o.w = __byte_perm(f[6], f[7], 0x7632);
    out[8 * c] = o;
  }
}

cudaError_t launch_nchw_to_nhwc_bf16(const int8_t* x, int64_t N, int64_t groups, int64_t ICg,
                                     int64_t H, int64_t W, int32_t zp, __nv_bfloat16* dst,
                                     int64_t ICgp, cudaStream_t s) {
  if (N * H * W == 0) return cudaSuccess;
  const int64_t WB = (W + 63) / 64, CBg = ICgp / 64, CB = CBg * groups;
  const int64_t blocks = N * CB * H * WB;
  if (blocks > INT32_MAX) return cudaErrorInvalidValue;
  const RelayoutDiv dv{make_fastdiv(static_cast<uint32_t>(WB)), make_fastdiv(static_cast<uint32_t>(H)),
                       make_fastdiv(static_cast<uint32_t>(CB)), make_fastdiv(static_cast<uint32_t>(CBg))};
  const bool vec = (W % 16 == 0) && (reinterpret_cast<uintptr_t>(x) % 16 == 0);
  if (vec)
    return launch_pdl(nchw_to_nhwc_bf16_kernel<true>, static_cast<int>(blocks), 128, 0, s, x,
                      groups, ICg, H, W, zp, reinterpret_cast<uint4*>(dst), ICgp, dv);
  return launch_pdl(nchw_to_nhwc_bf16_kernel<false>, static_cast<int>(blocks), 128, 0, s, x, groups,
                    ICg, H, W, zp, reinterpret_cast<uint4*>(dst), ICgp, dv);
}

// Convolution weight [OC, ldw] (per row: taps x ICg used) -> bf16, per group j:
// dst[j][t][ic/64][ocl][ic%64] for oc = j*OCg + ocl, input channels
// zero-padded to ICgp: the (BN output channels x 64 input channels) tile of
// one k-block is contiguous.
__global__ void __launch_bounds__(256) conv_weight_bf16_kernel(const int8_t* __restrict__ w,
                                                               int64_t groups, int64_t OCg,
                                                               int64_t taps, int64_t ICg,
                                                               int64_t ldw,
                                                               uint32_t* __restrict__ dst,
                                                               int64_t ICgp) {
  pdl_wait();
  pdl_launch_dependents();
  const int64_t icb = ICgp / 64;
  const int64_t total = groups * taps * icb * OCg * 32;  // bf16 pairs
  for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < total;
       i += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    const int64_t jp = i & 31;
    int64_t rest = i >> 5;
    const int64_t ocl = rest % OCg;
    rest /= OCg;
    const int64_t cb = rest % icb;
    rest /= icb;
    const int64_t t = rest % taps;
    const int64_t g = rest / taps;
    const int64_t ic = cb * 64 + 2 * jp;
    const int8_t* row = w + (g * OCg + ocl) * ldw + t * ICg;
    const int a = (ic < ICg) ? row[ic] : 0;
    const int b = (ic + 1 < ICg) ? row[ic + 1] : 0;
    dst[i] = bf16x2_from_ints(a, b);
  }
}

// Largest sum of |w| over one k-block of one output row: rows of
// [taps][ICg] int8 (row stride ldw), a k-block being 64 consecutive input
// channels of one tap (the last one of a tap may be shorter).  One warp per
// k-block; each warp's maximum goes to *bound by atomicMax (the caller zeroes
// it first).  With |x - zp| <= a, the products of one k-block then sum to at
// most a * bound in magnitude, whatever the row.
__global__ void __launch_bounds__(256) weight_block_bound_kernel(const int8_t* __restrict__ w,
                                                                 int64_t rows, int64_t ldw,
                                                                 int64_t taps, int64_t ICg,
                                                                 int32_t* __restrict__ bound) {
  pdl_wait();
  pdl_launch_dependents();
  const int lane = threadIdx.x & 31;
  const int64_t nblk = (ICg + 63) / 64;
  const int64_t items = rows * taps * nblk;
  const int64_t nwarps = (static_cast<int64_t>(gridDim.x) * blockDim.x) >> 5;
  int best = 0;
  for (int64_t it = (static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5; it < items;
       it += nwarps) {
    const int64_t blk = it % nblk;
    const int64_t rt = it / nblk;  // row * taps + tap
    const int8_t* seg = w + (rt / taps) * ldw + (rt % taps) * ICg + blk * 64;
    const int64_t len = ICg - blk * 64;
    int s = 0;
    if (lane < len) s += abs(static_cast<int>(seg[lane]));
    if (lane + 32 < len) s += abs(static_cast<int>(seg[lane + 32]));
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) s += __shfl_xor_sync(0xffffffffu, s, o);
    best = max(best, s);
  }
  if (lane == 0 && best > 0) atomicMax(bound, best);
}

cudaError_t launch_weight_block_bound(const int8_t* w, int64_t rows, int64_t ldw, int64_t taps,
                                      int64_t ICg, int32_t* bound, cudaStream_t s) {
  cudaError_t e = cudaMemsetAsync(bound, 0, sizeof(int32_t), s);
  if (e != cudaSuccess) return e;
  const int64_t items = rows * taps * ((ICg + 63) / 64);
  if (items == 0) return cudaSuccess;
  return launch_pdl(weight_block_bound_kernel, stream_grid(items * 32, 256, 8), 256, 0, s, w, rows,
                    ldw, taps, ICg, bound);
}

cudaError_t launch_conv_weight_bf16(const int8_t* w, int64_t groups, int64_t OCg, int64_t taps,
                                    int64_t ICg, int64_t ldw, __nv_bfloat16* dst, int64_t ICgp,
                                    cudaStream_t s) {
  const int64_t items = groups * OCg * taps * ICgp / 2;
  if (items == 0) return cudaSuccess;
  return launch_pdl(conv_weight_bf16_kernel, stream_grid(items, 256, 8), 256, 0, s, w, groups, OCg,
                    taps, ICg, ldw, reinterpret_cast<uint32_t*>(dst), ICgp);
  return cudaGetLastError();
}

}  // namespace q8
