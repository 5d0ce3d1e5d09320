// tc_gemm_kernel.cuh -- exact int8 contraction on the sm_103a tcgen05 tensor cores.
//
// What it computes: the int32 accumulator of "Add q8ta_linear op" (Solution
// paragraph), acc[m,n] = sum_k (x[m,k] - input_zero_point) * w[n,k], and of
// "Add q8ta_conv2d_transposed op" (Solution paragraph, the gather over valid
// taps), followed by the fused dequantize -> requantize -> int8 epilogue.
//
// How, on GB300: tcgen05 has no integer MMA on sm_103a, so the operands are
// bf16 copies of the integers: x - input_zero_point lies in [-255, 255] and
// w in [-128, 127], both exact in bf16, and every product (|p| <= 32640) is
// exact in the f32 accumulator.  The K loop is cut into chunks whose f32
// partial sums stay within 2^24 in magnitude and are therefore exact
// integers: at most 2^24 / (b * W) k-blocks of 64, b = max(128 + zp,
// 127 - zp) being the largest |x - zp| and W the largest sum of |w| over one
// k-block of one weight row (64 * 128 when the weight's own bound is not
// known: 8 k-blocks for b = 255, 16 for zp = 0).  Each chunk's TMEM
// accumulator is drained by the epilogue warps into int32 registers (exact
// conversion) while the MMA warp already fills the other TMEM buffer.
// Integer addition of the chunk sums is exact (modulo 2^32, like the pages'
// i32 accumulator).
//
// Transposed convolution is an implicit GEMM per stride phase: outputs with
// oh % stride_h == ph and ow % stride_w == pw all use the same taps, those
// kh with kh * dil_h = ph + pad_h (mod stride_h) -- kh0 + i * stride_h / g
// for g = gcd(dil_h, stride_h) (likewise kw) -- and tap (kh, kw) reads the
// input at (oh' + dh, ow' + dw) with dh = (ph + pad_h - kh * dil_h) /
// stride_h, an integer by construction.  A 5-D TMA box over the
// channel-blocked NHWC bf16 input fetches that shifted window; coordinates
// outside the input are filled with zeros by the TMA unit, which is exactly
// "taps outside the input contribute nothing" because the stored values are
// x - input_zero_point.  The direct convolution (mode 2) reads each tap's
// window through a box with element strides (stride_w, stride_h).  Above 64
// output channels per group the convolutions exchange the operands (modes
// 3 to 6, see the kernel): 128 output channels on the MMA's M side, 256
// output pixels on N.
//
// Warp roles (one CTA per SM, persistent over output tiles):
//   warp 0      TMA producer (one thread)
//   warp 1      TMEM allocator and MMA issuer (one thread)
//   warps 2..   E epilogue warps (8, 12 or 16): warp w reads TMEM lanes
//               32*(w%4)..+31 and BN / (E/4) of the tile's columns
// With CTA pairs (CG = 2, a cluster of two CTAs on neighbouring SMs) one
// 256 x BN tile is computed by the 2-SM MMA: each CTA loads its own 128 rows
// of A and half of the BN rows of B, the leader CTA's MMA thread issues the
// MMAs for both, and each CTA's epilogue drains its own TMEM rows.  Per SM
// that is 16 KB of B per k-block instead of 32 KB at BN = 256.
// Every mbarrier wait has a time limit (about 1 s); on expiry the CTA records
// a code in g_q8_error, stops issuing work, waits (again bounded) for its own
// copies and MMAs in flight, frees TMEM and returns.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <cstdint>
#include <mutex>

#include "device_common.cuh"
#include "q8ta_internal.h"

namespace q8 {

enum : uint32_t {
  kErrWaitFull = 0x101,
  kErrWaitEmpty = 0x102,
  kErrWaitAccFull = 0x103,
  kErrWaitAccEmpty = 0x104,
  kErrWaitDrain = 0x105,
  kErrWaitEpi = 0x106,
  kErrChunks = 0x107,  // a single-chunk kernel met a tile of several chunks
  kErrWaitQuant = 0x108,  // a fused-quantize chunk of the operand never became ready
  kErrFusedInit = 0x109,  // fused quantize: the operand's trailer was never initialized
};

// Fused quantize -> linear: the operand's 256-byte trailer holds, as 32-bit
// words, [0] the |x - zp| bound, [1] the count of CTAs that finished the
// launch, [2..3] kFusedMagic (written by the trailer's initialization) and
// [4 + c] the count of CTAs that wrote their share of operand chunk c, a
// chunk being qckb consecutive k-blocks of every row (at most 60 chunks).
constexpr uint64_t kFusedMagic = 0x51a8d7e3c0f1b2a4ull;
constexpr int kFusedWordDone = 1;
constexpr int kFusedWordMagic = 2;
constexpr int kFusedWordChunk0 = 4;
constexpr int kFusedMaxChunks = 60;
// k-blocks per chunk: 2 (one ring stage of the pair GEMM), doubled until
// the chunk count fits kFusedMaxChunks
__host__ __device__ constexpr int fused_chunk_kb(int kb_total) {
  int kb = 2;
  while ((kb_total + kb - 1) / kb > kFusedMaxChunks) kb *= 2;
  return kb;
}

constexpr uint64_t kWaitLimitNs = 1000ull * 1000ull * 1000ull;
constexpr int kBM = 128;
constexpr int kBK = 64;             // bf16 per 128-byte row
// Exact f32 chunks: with |x - zp| <= a_bound and at most w_bound for the sum
// of |w| over the 64 weights of any k-block of any row, every partial sum of
// a chunk of c k-blocks is an integer of magnitude at most c * a_bound *
// w_bound, exact in f32 while that is <= 2^24.  Without a measured weight
// bound, w_bound = 64 * 128: c <= 2048 / a_bound (8 k-blocks for the int8
// worst case a_bound = 255, 16 for a zero point of 0).  kWorstWBound:
// q8ta_internal.h.
constexpr int kMaxChunkKb = 256;
constexpr int kMaxStages = 8;
constexpr int kMaxPhases = 16;
constexpr int kMaxEpiWarps = 16;
constexpr int kMaxColsPerWarp = 128;

// Threads of a CTA with E epilogue warps: the TMA warp, the MMA warp, E more.
__host__ __device__ constexpr int cta_threads(int epi_warps) { return 64 + 32 * epi_warps; }
constexpr int kMaxBN = 256;
constexpr int kEpFloats = 8 * kMaxBN;  // scale/bias staging (see Ctl::ep)

struct TcParams {
  int mode;          // 0 = linear, 1 = transposed convolution, 2 = direct convolution
  int stages;        // smem ring depth
  int kd;            // k-blocks per ring stage (1 or 2): one TMA box holds kd k-blocks
  int total_units;   // work units; a unit is `subtiles` consecutive tiles
  int subtiles;      // 1 (linear) or stride_w (transposed convolution)
  int max_nstages;   // the most ring stages of any sub-tile (convolutions)
  // linear
  int M, N, kb_total, tiles_m;
  // transposed convolution
  // (OC: the GEMM's columns, one group's output channels; out_ch: channels
  // of the output tensor)
  int Nimg, OC, Kh, Kw, H_out, W_out, sh, sw, pad_h, pad_w, icb, ICp, out_ch;
  int dil_h, dil_w;
  // transposed convolution: the row taps of a phase are kh0 + i * tsh and
  // read input rows dh0 - i * dsh, with gh = gcd(dil_h, sh), tsh = sh / gh,
  // dsh = dil_h / gh and kh0 = ((ph + pad_h) mod sh / gh) * invh mod tsh,
  // invh being the inverse of dsh modulo tsh (columns likewise)
  int gh, gw, tsh, tsw, dsh, dsw, invh, invw;
  int osh, osw;      // output pixel step of a tile's rows / columns (conv_t: stride; conv2d: 1)
  int BW, BH, tiles_w, tiles_h, tiles_oc;
  int staged;        // conv output: 2 = column phases held in registers, one
                     // store per channel; 0 = one byte store per output
  int8_t ph_order[kMaxPhases];  // row phases, most taps first (stride_h <= kMaxPhases)
  // tile decomposition without integer division: divisors of the unit index
  FastDiv fd_oc, fd_w, fd_h, fd_n;
  // per stride phase (phase_tab: both strides <= kMaxPhases), the first
  // tap, the tap count and the input offset of the first tap: row phase ph
  // (ph_r, ph_nt, ph_d0) and column phase pw (pw_r, pw_nt, pw_d0), as
  // decode_tile would compute them
  int phase_tab;
  int ph_r[kMaxPhases], ph_nt[kMaxPhases], ph_d0[kMaxPhases];
  int pw_r[kMaxPhases], pw_nt[kMaxPhases], pw_d0[kMaxPhases];
  // epilogue
  const float* ws;
  const float* bias;
  Requant rq;
  int8_t* out;
  int32_t* acc_out;
  int store_mode;    // linear int8 stores: 2 = 16 B, 1 = 4 B, 0 = bytes
  uint32_t* err;     // the library's device error word
  const int32_t* a_bound_dev;  // largest |x - zp| of A, on the device (or null)
  int a_bound_host;            // the same, when a_bound_dev is null
  const int32_t* w_bound_dev;  // largest sum of |w| over one k-block of one row (or null)
  // failure detection: every barrier wait gives up after wait_ns (0: the
  // default kWaitLimitNs); stall_fill = f + 1 makes the TMA producer skip
  // its f-th ring fill (a test of the timeout path; 0: none)
  uint64_t wait_ns;
  int stall_fill;
  // fused quantize -> linear (MODE 0 with qx != null): the epilogue warps of
  // all CTAs first quantize fp32 x into the operand (and x_q), chunk by
  // chunk; a producer loads an operand chunk only once every CTA has
  // signalled it in the trailer (see kFusedMagic)
  const float* qx;     // fp32 activations [M, qK], row-major
  int8_t* qxq;         // int8 quantize output [M, qK], or null
  uint4* qdst;         // the operand the A tensor map reads, K-blocked
  uint32_t* qsync;     // the operand's trailer
  float qinv;          // (float)(1 / input_scale)
  int qzp;             // input zero point
  int qK;              // K (the operand is zero-padded to kb_total * 64)
  int qvec;            // x (and x_q) rows allow 16-byte (8-byte) vector access
  int qckb;            // k-blocks per operand chunk (fused_chunk_kb, a power of two)
  int qseg_log2;       // log2(qckb * 8): 8-element items per row and chunk
  int qnch;            // operand chunks
};

// Ring stages per exact f32 chunk (see kWorstWBound), from A's and W's bounds.
__device__ __forceinline__ int chunk_stages(const TcParams& p, int kd) {
  int bound = p.a_bound_dev != nullptr ? __ldg(p.a_bound_dev) : p.a_bound_host;
  if (bound < 1 || bound > 255) bound = 255;  // anything else: the int8 worst case
  int wb = p.w_bound_dev != nullptr ? __ldg(p.w_bound_dev) : kWorstWBound;
  if (wb > kWorstWBound || wb < 0) wb = kWorstWBound;
  wb = max(wb, 1);  // all-zero weights: any length is exact
  const int kb = min(kMaxChunkKb, (1 << 24) / (bound * wb));
  return max(1, kb / kd);
}

struct TileInfo {
  int num_kb;   // k-blocks of the tile
  int nstages;  // ring stages that carry them (KD k-blocks each; a stage
                // past a tap's last channel block holds zeros of A)
  // linear
  int mb, nb;
  // conv: output phase (ph, pw), first taps (rh, rw), tap counts (nth, ntw),
  // input offsets of the first taps (dh0, dw0)
  int n, hb, wb, ocb, ph, pw, rh, rw, nth, ntw, dh0, dw0;
};

// Unit u, sub-tile j -> tile coordinates.  Transposed convolution units are
// (row phase ph, image n, row block hb, column block wb, channel block ocb);
// their sub-tiles are the stride_w column phases pw, so one CTA produces
// every output column of its rows and can write whole rows.
// With CTA pairs (CG == 2) a unit spans CG row blocks of 128: the CTA of
// rank r takes row block (u % tiles) * CG + r, and p.tiles_m / p.tiles_h
// count pairs of row blocks.
template <int MODE, int CG, int KD>
__device__ __forceinline__ TileInfo decode_tile(const TcParams& p, int u, int j, int rank) {
  TileInfo ti{};
  if constexpr (MODE == 0) {
    ti.mb = (u % p.tiles_m) * CG + rank;
    ti.nb = u / p.tiles_m;
    ti.num_kb = p.kb_total;
    ti.nstages = (p.kb_total + KD - 1) / KD;
  } else if constexpr (MODE == 2) {
    // direct convolution: one output tile of image n, every tap
    uint32_t q, r;
    fast_divmod(static_cast<uint32_t>(u), p.fd_oc, q, r);
    ti.ocb = static_cast<int>(r);
    fast_divmod(q, p.fd_w, q, r);
    ti.wb = static_cast<int>(r);
    fast_divmod(q, p.fd_h, q, r);
    ti.hb = static_cast<int>(r) * CG + rank;
    ti.n = static_cast<int>(q);
    ti.nth = p.Kh;
    ti.ntw = p.Kw;
    ti.num_kb = p.Kh * p.Kw * p.icb;
    ti.nstages = p.Kh * p.Kw * ((p.icb + KD - 1) / KD);
  } else {
    uint32_t q, r;
    fast_divmod(static_cast<uint32_t>(u), p.fd_oc, q, r);
    ti.ocb = static_cast<int>(r);
    fast_divmod(q, p.fd_w, q, r);
    ti.wb = static_cast<int>(r);
    fast_divmod(q, p.fd_h, q, r);
    ti.hb = static_cast<int>(r) * CG + rank;
    fast_divmod(q, p.fd_n, q, r);
    ti.n = static_cast<int>(r);
    const int phx = static_cast<int>(q);
    ti.ph = (p.sh <= kMaxPhases) ? p.ph_order[phx] : phx;
    ti.pw = j;
    if (p.phase_tab) {
      ti.rh = p.ph_r[ti.ph];
      ti.nth = p.ph_nt[ti.ph];
      ti.dh0 = p.ph_d0[ti.ph];
      ti.rw = p.pw_r[j];
      ti.ntw = p.pw_nt[j];
      ti.dw0 = p.pw_d0[j];
      ti.num_kb = ti.nth * ti.ntw * p.icb;
      ti.nstages = ti.nth * ti.ntw * ((p.icb + KD - 1) / KD);
      return ti;
    }
    // first taps: the least kh >= 0 with kh * dil_h = ph + pad_h (mod sh), if any
    const int th0 = (ti.ph + p.pad_h) % p.sh, tw0 = (ti.pw + p.pad_w) % p.sw;
    ti.nth = 0;
    ti.ntw = 0;
    if (th0 % p.gh == 0) {
      ti.rh = (th0 / p.gh) * p.invh % p.tsh;
      ti.nth = ti.rh < p.Kh ? (p.Kh - ti.rh + p.tsh - 1) / p.tsh : 0;
      ti.dh0 = (ti.ph + p.pad_h - ti.rh * p.dil_h) / p.sh;  // exact
    }
    if (tw0 % p.gw == 0) {
      ti.rw = (tw0 / p.gw) * p.invw % p.tsw;
      ti.ntw = ti.rw < p.Kw ? (p.Kw - ti.rw + p.tsw - 1) / p.tsw : 0;
      ti.dw0 = (ti.pw + p.pad_w - ti.rw * p.dil_w) / p.sw;
    }
    ti.num_kb = ti.nth * ti.ntw * p.icb;
    ti.nstages = ti.nth * ti.ntw * ((p.icb + KD - 1) / KD);
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
  uint32_t qwarps[kFusedMaxChunks];  // fused quantize: this CTA's warps done with each chunk
  // column scales and biases of the current tile:
  //   linear: shared by all epilogue warps, two buffers by tile parity, [2][2][BN]
  //   conv:   one slice per epilogue warp, [warp][2][BN / (warps / 4)] = 8 * BN
  alignas(16) float ep[kEpFloats];
};

// Bounded wait.  Returns false when this CTA is aborting (this wait timed
// out, or another role's did).
__device__ __forceinline__ uint64_t wait_limit(const TcParams& p) {
  return p.wait_ns != 0 ? p.wait_ns : kWaitLimitNs;
}

__device__ __forceinline__ bool wait_bar(uint32_t bar, uint32_t parity, volatile uint32_t* abort_flag,
                                         uint32_t code, uint32_t* err, uint64_t limit_ns) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = global_timer_ns();
  while (true) {
    if (mbar_try_wait(bar, parity)) return true;
    if (*abort_flag) return false;
    if (global_timer_ns() - t0 > limit_ns) {
      *abort_flag = 1u;
      atomicCAS(err, 0u, code);
      return false;
    }
  }
}

// Bounded wait used while shutting down: ignores the abort flag.
__device__ __forceinline__ void wait_bar_final(uint32_t bar, uint32_t parity, uint32_t* err,
                                               uint64_t limit_ns) {
  if (mbar_try_wait(bar, parity)) return;
  const uint64_t t0 = global_timer_ns();
  while (!mbar_try_wait(bar, parity)) {
    if (global_timer_ns() - t0 > limit_ns) {
      atomicCAS(err, 0u, kErrWaitDrain);
      return;
    }
  }
}

// Rendezvous of the epilogue warps on an mbarrier (bounded, unlike
// bar.sync, so one aborted warp cannot strand the others).  Shared-memory
// writes made before the call are visible to every epilogue thread after it.
__device__ __forceinline__ bool epi_sync(Ctl* ctl, uint32_t& phase, volatile uint32_t* abort_flag,
                                         uint32_t* err, uint64_t limit_ns) {
  // every epilogue warp arrives once per rendezvous
  __syncwarp();
  bool ok = true;
  if ((threadIdx.x & 31) == 0) {
    mbar_arrive(smem_u32(&ctl->epi_bar));
    ok = wait_bar(smem_u32(&ctl->epi_bar), phase, abort_flag, kErrWaitEpi, err, limit_ns);
  }
  phase ^= 1u;
  ok = __shfl_sync(0xffffffffu, ok ? 1 : 0, 0) != 0;
  __syncwarp();
  return ok;
}

// ---- fused quantize -> linear ---------------------------------------------
__device__ __forceinline__ uint32_t ld_relaxed_gpu(const uint32_t* p) {
  uint32_t v;
  asm volatile("ld.relaxed.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}
__device__ __forceinline__ void fence_acq_rel_gpu() {
  asm volatile("fence.acq_rel.gpu;" ::: "memory");
}
__device__ __forceinline__ void red_relaxed_gpu_add(uint32_t* p, uint32_t v) {
  asm volatile("red.relaxed.gpu.global.add.u32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}
// Generic-proxy stores made before this fence are ordered before later
// async-proxy (TMA) accesses, and the other way round.
__device__ __forceinline__ void fence_proxy_async_global() {
  asm volatile("fence.proxy.async.global;" ::: "memory");
}
__device__ __forceinline__ uint32_t atom_add_acq_rel_cta(uint32_t* p, uint32_t v) {
  uint32_t old;
  asm volatile("atom.acq_rel.cta.shared::cta.add.u32 %0, [%1], %2;"
               : "=r"(old)
               : "r"(smem_u32(p)), "r"(v)
               : "memory");
  return old;
}

// Bounded wait until every CTA of the launch has signalled operand chunk c:
// relaxed polling, then one acquire fence (the counter's increments follow a
// release fence on the writers' side).
static __device__ __noinline__ bool wait_chunk(const TcParams& p, int c, volatile uint32_t* abort_flag) {
  const uint32_t* word = p.qsync + kFusedWordChunk0 + c;
  const uint32_t target = gridDim.x;
  const uint64_t t0 = global_timer_ns();
  while (true) {
    if (ld_relaxed_gpu(word) >= target) {
      fence_acq_rel_gpu();
      return true;
    }
    if (*abort_flag) return false;
    if (global_timer_ns() - t0 > wait_limit(p)) {
      *abort_flag = 1u;
      atomicCAS(p.err, 0u, kErrWaitQuant);
      return false;
    }
    __nanosleep(32);
  }
}

// This CTA's share of quantize_per_tensor fused with the operand
// preparation.  The work is a list of items of 8 consecutive elements of
// one row, chunk after chunk: item I is (chunk c, index i) = (I / P, I % P),
// P = M * segs, segs = qckb * 8 items per row and chunk; index i is row
// i / segs, elements (c * segs + i % segs) * 8 .. + 7.  Thread g of the
// grid's converter threads takes items g, g + GT, g + 2 GT, ... (GT of
// them in the grid), loads IU items before converting any, writes x_q
// (when asked) and the bf16 of q - zp (0 past K), and never waits on a
// barrier: after each batch its warp counts, in shared memory, the chunks
// all its lanes have passed, and the warp that completes a chunk for the
// CTA adds one to the chunk's counter in the trailer (a release at GPU
// scope, after the stores were ordered before the TMA unit's reads).
__device__ __forceinline__ void fused_report(const TcParams& p, uint32_t* qwarps, uint32_t nwarps,
                                             int& done, int upto) {
  bool fenced = false;  // one GPU-scope release fence covers every count that follows
  for (; done < upto; ++done) {
    const uint32_t prev = atom_add_acq_rel_cta(qwarps + done, 1u);
    if (prev == nwarps - 1) {
      if (!fenced) {
        fence_acq_rel_gpu();
        fenced = true;
      }
      red_relaxed_gpu_add(p.qsync + kFusedWordChunk0 + done, 1u);
    }
  }
}

template <int IU>
__device__ __noinline__ void fused_quantize(const TcParams& p, uint32_t* qwarps, int t, int nt) {
  const int lane = t & 31;
  const uint32_t nwarps = static_cast<uint32_t>(nt >> 5);
  const int sh = p.qseg_log2;
  const int64_t M = p.M, K = p.qK, Kp = static_cast<int64_t>(p.kb_total) * 64;
  const int64_t P = M << sh;
  const int64_t GT = static_cast<int64_t>(gridDim.x) * nt;
  const int64_t gc = GT / P, gi = GT - gc * P;
  const int64_t I = static_cast<int64_t>(blockIdx.x) * nt + t;
  int64_t c = I / P, i = I - c * P;
  int done = 0;  // chunks this warp has reported
  while (__shfl_sync(0xffffffffu, (c < p.qnch ? static_cast<int>(c) : p.qnch), 0) < p.qnch) {
    float4 va[IU], vb[IU];
    int cu[IU];
    int64_t iu[IU];
#pragma unroll
    for (int u = 0; u < IU; ++u) {
      cu[u] = (c < p.qnch ? static_cast<int>(c) : p.qnch);
      iu[u] = i;
      if (c < p.qnch) {
        const int64_t row = i >> sh;
        const int64_t k0 = ((c << sh) + (i - (row << sh))) * 8;
        if (p.qvec && k0 + 8 <= K) {
          const float4* xp = reinterpret_cast<const float4*>(p.qx + row * K + k0);
          va[u] = __ldcs(xp);
          vb[u] = __ldcs(xp + 1);
        }
      }
      c += gc;
      i += gi;
      if (i >= P) {
        i -= P;
        ++c;
      }
    }
#pragma unroll
    for (int u = 0; u < IU; ++u) {
      if (cu[u] >= p.qnch) break;
      const int64_t row = iu[u] >> sh;
      const int64_t k0 = ((static_cast<int64_t>(cu[u]) << sh) + (iu[u] - (row << sh))) * 8;
      if (k0 >= Kp) continue;  // the last chunk's k-blocks past the operand
      int v[8];
      if (p.qvec && k0 + 8 <= K) {
        int8_t q[8];
        q[0] = quantize_one(va[u].x, p.qinv, p.qzp); q[1] = quantize_one(va[u].y, p.qinv, p.qzp);
        q[2] = quantize_one(va[u].z, p.qinv, p.qzp); q[3] = quantize_one(va[u].w, p.qinv, p.qzp);
        q[4] = quantize_one(vb[u].x, p.qinv, p.qzp); q[5] = quantize_one(vb[u].y, p.qinv, p.qzp);
        q[6] = quantize_one(vb[u].z, p.qinv, p.qzp); q[7] = quantize_one(vb[u].w, p.qinv, p.qzp);
        if (p.qxq != nullptr)
          *reinterpret_cast<uint2*>(p.qxq + row * K + k0) =
              make_uint2(pack4(q[0], q[1], q[2], q[3]), pack4(q[4], q[5], q[6], q[7]));
#pragma unroll
        for (int j = 0; j < 8; ++j) v[j] = static_cast<int>(q[j]) - p.qzp;
      } else {
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          v[j] = 0;
          if (k0 + j < K) {
            const int8_t q = quantize_one(p.qx[row * K + k0 + j], p.qinv, p.qzp);
            if (p.qxq != nullptr) p.qxq[row * K + k0 + j] = q;
            v[j] = static_cast<int>(q) - p.qzp;
          }
        }
      }
      uint4 o;
      o.x = bf16x2_from_ints(v[0], v[1]);
      o.y = bf16x2_from_ints(v[2], v[3]);
      o.z = bf16x2_from_ints(v[4], v[5]);
      o.w = bf16x2_from_ints(v[6], v[7]);
      p.qdst[kblocked_index16(row, k0, M)] = o;
    }
    // every item of this warp below lane 0's next one is done: the chunks
    // before that item's chunk are complete for the warp
    fence_proxy_async_global();
    __syncwarp();
    const int passed = __shfl_sync(0xffffffffu, (c < p.qnch ? static_cast<int>(c) : p.qnch), 0);
    if (lane == 0) fused_report(p, qwarps, nwarps, done, passed);
    done = passed;
  }
  // chunks past this warp's last item (or all of them, for a warp with none)
  if (lane == 0) fused_report(p, qwarps, nwarps, done, p.qnch);
}

// Exchanged operands (MODE 3 / 4): one epilogue thread holds one output
// channel (its TMEM lane) and a run of kCols pixels of the tile (TMEM
// columns col0 ..), row-major in the tile, BW (a power of two) per row.
struct PixRun {
  int64_t chan;  // offset of the output channel's plane
  int8_t* dst;   // one-row runs: the output byte of the first pixel, phase 0
  int oh, ow0;   // one-row runs: its output row and column (phase 0)
  bool row;      // the run is one tile row (BW a multiple of kCols)
  bool vec;      // ... inside the output row and 32-byte aligned: sector stores
};

template <int kCols>
__device__ __forceinline__ PixRun pix_run(const TcParams& p, const TileInfo& ti, int oc, int col0) {
  PixRun r;
  r.chan = (static_cast<int64_t>(ti.n) * p.out_ch + oc) * (static_cast<int64_t>(p.H_out) * p.W_out);
  r.row = (p.BW % kCols) == 0;
  const int bw_log = __ffs(p.BW) - 1;
  r.oh = (ti.hb * p.BH + (col0 >> bw_log)) * p.osh + ti.ph;
  r.ow0 = (ti.wb * p.BW + (col0 & (p.BW - 1))) * p.osw;
  r.dst = p.out != nullptr ? p.out + r.chan + static_cast<int64_t>(r.oh) * p.W_out + r.ow0 : nullptr;
  r.vec = r.row && r.dst != nullptr && (p.osw == 1 || p.osw == 2) && r.oh < p.H_out &&
          r.ow0 + kCols * p.osw <= p.W_out && (reinterpret_cast<uintptr_t>(r.dst) & 31u) == 0;
  return r;
}

// Four f32 accumulators of one output channel -> one word of four
// requantized bytes: the epilogue's arithmetic in the order of requant_f,
// the floor on the float and the upper clamp in the saturating pack.
__device__ __forceinline__ int32_t rq_unclamped(float a, float ws, float b, const Requant& rq) {
  const float u = __fmul_rn(__fadd_rn(__fmul_rn(__fmul_rn(a, rq.s_in), ws), b), rq.inv_out);
  return round_floor_first(u, rq.ozp_i, rq.lo_f);
}
__device__ __forceinline__ uint32_t rq_pack4(float a0, float a1, float a2, float a3, float ws,
                                             float b, const Requant& rq) {
  return pack4_sat(rq_unclamped(a0, ws, b, rq), rq_unclamped(a1, ws, b, rq),
                   rq_unclamped(a2, ws, b, rq), rq_unclamped(a3, ws, b, rq));
}

// Output pixel of run column c (generic placement).
__device__ __forceinline__ bool pix_at(const TcParams& p, const TileInfo& ti, int c, int& oh,
                                       int& ow) {
  const int bw_log = __ffs(p.BW) - 1;
  oh = (ti.hb * p.BH + (c >> bw_log)) * p.osh + ti.ph;
  ow = (ti.wb * p.BW + (c & (p.BW - 1))) * p.osw + ti.pw;
  return oh < p.H_out && ow < p.W_out;
}

// One whole 32-byte sector per thread and instruction (256-bit accesses):
// the lanes of a warp hold different output channels, so narrower stores
// would leave partial sectors in L2.
__device__ __forceinline__ void st_global_v8(void* ptr, const uint32_t (&w)[8]) {
  asm volatile("st.global.v8.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8};" ::"l"(ptr), "r"(w[0]),
               "r"(w[1]), "r"(w[2]), "r"(w[3]), "r"(w[4]), "r"(w[5]), "r"(w[6]), "r"(w[7])
               : "memory");
}
__device__ __forceinline__ void ld_global_v8(const void* ptr, uint32_t (&w)[8]) {
  asm volatile("ld.global.v8.b32 {%0, %1, %2, %3, %4, %5, %6, %7}, [%8];"
               : "=r"(w[0]), "=r"(w[1]), "=r"(w[2]), "=r"(w[3]), "=r"(w[4]), "=r"(w[5]),
                 "=r"(w[6]), "=r"(w[7])
               : "l"(ptr)
               : "memory");
}

// Requantize and store the run's columns 16g .. 16g + 15 (f: the exact f32
// accumulators), whole sectors where the run allows:
//   stride 1: 16 bytes; even groups wait in hold[], odd ones store both;
//   stride 2: one sector of the output row per group.  The two column
//     phases of a unit meet in the output: phase 0 writes its bytes to the
//     even positions (odd ones zero), phase 1 (the same thread, later) merges
//     its bytes into the sector phase 0 wrote, read back into e[] before.
template <int kCols>
__device__ __forceinline__ void pix_store16(const TcParams& p, const TileInfo& ti, const PixRun& r,
                                            int col0, int g, const float (&f)[16], float ws,
                                            float b, uint32_t (&hold)[4], const uint32_t (&e)[8]) {
  if (r.vec) {
    uint32_t q[4];
#pragma unroll
    for (int k = 0; k < 4; ++k)
      q[k] = rq_pack4(f[4 * k], f[4 * k + 1], f[4 * k + 2], f[4 * k + 3], ws, b, p.rq);
    uint32_t w[8];
    if (p.osw == 1) {
      if ((g & 1) == 0) {
#pragma unroll
        for (int k = 0; k < 4; ++k) hold[k] = q[k];
        return;
      }
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        w[k] = hold[k];
        w[4 + k] = q[k];
      }
      st_global_v8(r.dst + 16 * (g - 1), w);
    } else if (ti.pw == 0) {
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        w[2 * k] = __byte_perm(q[k], 0u, 0x4140);
        w[2 * k + 1] = __byte_perm(q[k], 0u, 0x4342);
      }
      st_global_v8(r.dst + 32 * g, w);
    } else {
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        w[2 * k] = __byte_perm(e[2 * k], q[k], 0x5240);
        w[2 * k + 1] = __byte_perm(e[2 * k + 1], q[k], 0x7260);
      }
      st_global_v8(r.dst + 32 * g, w);
    }
  } else if (r.row) {
    if (r.oh >= p.H_out) return;
#pragma unroll
    for (int i = 0; i < 16; ++i) {
      const int k = p.osw * (16 * g + i) + ti.pw;
      if (r.ow0 + k < p.W_out) r.dst[k] = static_cast<int8_t>(requant_f(f[i], ws, b, p.rq));
    }
  } else {
#pragma unroll
    for (int i = 0; i < 16; ++i) {
      int oh, ow;
      if (pix_at(p, ti, col0 + 16 * g + i, oh, ow))
        p.out[r.chan + static_cast<int64_t>(oh) * p.W_out + ow] =
            static_cast<int8_t>(requant_f(f[i], ws, b, p.rq));
    }
  }
}

// The single-chunk kernels' form of pix_store16: with stride 2 the two
// column phases of a unit meet in registers instead of in the output.
// Phase 0 keeps its four packed words of group G in ph0[4G .. 4G + 3] and
// stores nothing; phase 1 (the same thread, next sub-tile) interleaves them
// with its own bytes and writes whole sectors once.  (G is a compile-time
// index, so ph0 stays in registers.)
template <int kCols, int G>
__device__ __forceinline__ void pix_store16_reg(const TcParams& p, const TileInfo& ti,
                                                const PixRun& r, int col0, const float (&f)[16],
                                                float ws, float b, uint32_t (&hold)[4],
                                                uint32_t (&ph0)[kCols / 4]) {
  if (r.vec && p.osw == 2) {
    uint32_t q[4];
#pragma unroll
    for (int k = 0; k < 4; ++k)
      q[k] = rq_pack4(f[4 * k], f[4 * k + 1], f[4 * k + 2], f[4 * k + 3], ws, b, p.rq);
    if (ti.pw == 0) {
#pragma unroll
      for (int k = 0; k < 4; ++k) ph0[4 * G + k] = q[k];
      return;
    }
    uint32_t w[8];
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      w[2 * k] = __byte_perm(ph0[4 * G + k], q[k], 0x5140);
      w[2 * k + 1] = __byte_perm(ph0[4 * G + k], q[k], 0x7362);
    }
    st_global_v8(r.dst + 32 * G, w);
    return;
  }
  const uint32_t e[8] = {0u, 0u, 0u, 0u, 0u, 0u, 0u, 0u};  // (no stride-2 sector merge here)
  pix_store16<kCols>(p, ti, r, col0, G, f, ws, b, hold, e);
}

// The sector that phase 0 of a stride-2 unit wrote for group g (read before
// the group's accumulators, so the load overlaps them).
__device__ __forceinline__ void pix_phase0(const TcParams& p, const TileInfo& ti, const PixRun& r,
                                           int g, uint32_t (&e)[8]) {
  if (r.vec && p.osw == 2 && ti.pw == 1) ld_global_v8(r.dst + 32 * g, e);
}

// The int32 accumulators of the run's columns 16g .. 16g + 15 (debug output).
__device__ __forceinline__ void pix_store16_acc(const TcParams& p, const TileInfo& ti,
                                                const PixRun& r, int col0, int g,
                                                const int32_t (&a)[16]) {
#pragma unroll
  for (int i = 0; i < 16; ++i) {
    int oh, ow;
    if (pix_at(p, ti, col0 + 16 * g + i, oh, ow))
      p.acc_out[r.chan + static_cast<int64_t>(oh) * p.W_out + ow] = a[i];
  }
}

// Exchanged operands, a tile of several exact chunks (a long k-loop with
// wide input and weight bounds): the chunks' int32 sums, then the same
// stores.  Out of line, so that its 64 live sums do not crowd the registers
// of the single-chunk path.
struct PixChunks {
  uint32_t acc_it;
  bool ok;
};

template <int kCols, uint32_t kAccStride>
__device__ __noinline__ PixChunks pix_chunks(const TcParams& p, TileInfo ti, PixRun run, Ctl* ctl,
                                             uint32_t tmem_row, int col0, bool mine, float ws,
                                             float b, uint32_t acc_it, int chunk_st) {
  const int lane = threadIdx.x & 31;
  volatile uint32_t* abort_flag = &ctl->abort_flag;
  int32_t sum[kCols];
#pragma unroll
  for (int c = 0; c < kCols; ++c) sum[c] = 0;
  for (int st0 = 0; st0 < ti.nstages; st0 += chunk_st) {
    const uint32_t buf = acc_it & 1u, use = acc_it >> 1;
    bool got = true;
    if (lane == 0)
      got = wait_bar(smem_u32(&ctl->acc_full[buf]), use & 1u, abort_flag, kErrWaitAccFull, p.err,
                     wait_limit(p));
    got = __shfl_sync(0xffffffffu, got ? 1 : 0, 0) != 0;
    if (!got) return {acc_it, false};
    tc_fence_after();
#pragma unroll
    for (int g = 0; g < kCols / 16; ++g) {
      uint32_t r[16];
      tmem_ld_16cols(tmem_row + buf * kAccStride + col0 + 16 * g, r);
      tmem_ld_wait();
#pragma unroll
      for (int i = 0; i < 16; ++i)
        sum[16 * g + i] = static_cast<int32_t>(static_cast<uint32_t>(sum[16 * g + i]) +
                                               static_cast<uint32_t>(__float2int_rn(__uint_as_float(r[i]))));
    }
    tc_fence_before();
    __syncwarp();
    if (lane == 0) mbar_arrive(smem_u32(&ctl->acc_empty[buf]));
    ++acc_it;
  }
  if (mine) {
    uint32_t hold[4] = {0u, 0u, 0u, 0u};
#pragma unroll
    for (int g = 0; g < kCols / 16; ++g) {
      if (p.acc_out != nullptr) {
        int32_t a[16];
#pragma unroll
        for (int i = 0; i < 16; ++i) a[i] = sum[16 * g + i];
        pix_store16_acc(p, ti, run, col0, g, a);
      } else {
        uint32_t e[8];
        pix_phase0(p, ti, run, g, e);
        float fv[16];
#pragma unroll
        for (int i = 0; i < 16; ++i) fv[i] = __int2float_rn(sum[16 * g + i]);
        pix_store16<kCols>(p, ti, run, col0, g, fv, ws, b, hold, e);
      }
    }
  }
  return {acc_it, true};
}

// MODE 0: q8ta_linear tiles; MODE 1: transposed-convolution units; MODE 2:
// direct-convolution tiles.  MODE 3 / 4 (5 / 6): the same convolutions with the
// roles of the operands exchanged: A is 128 output channels of the packed
// weight and B is a tile of BN output pixels, so the accumulator holds one
// output channel per TMEM lane and a run of pixels per lane (each epilogue
// thread writes contiguous output bytes of one channel plane), and a k-block
// moves 16 + 32 KB for a 128 x 256 product instead of 32 KB for 128 x 128.
// MODE 5 / 6 hold only the single-chunk path (no register pressure from the
// multi-chunk ones); the host picks them when every sub-tile fits one chunk.
// KD: k-blocks per ring stage (one TMA box spans KD k-blocks).
// CG: 1 = one CTA per 128-row tile (cta_group::1); 2 = a cluster of two CTAs
// shares one 256-row tile through the 2-SM MMA (cta_group::2): each CTA
// loads its 128 rows of A and half of B's BN rows, the leader CTA issues
// the MMAs, and each CTA's TMEM holds the accumulators of its own rows.
template <int BN, int EPI, int MODE_IN, int KD, int CG>
__global__ void __launch_bounds__(cta_threads(EPI), 1)
    tc_gemm_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                   const __grid_constant__ TcParams p) {
  // MODE_IN 7: the linear (MODE 0) with the fused quantize prologue
  constexpr int MODE = MODE_IN == 7 ? 0 : MODE_IN;
  constexpr bool kFusedQ = (MODE_IN == 7);
  constexpr int kEpiWarps = EPI;
  constexpr int kColGroups = EPI / 4;     // epilogue warps sharing one TMEM lane quarter
  constexpr uint32_t kABytes = kBM * kBK * 2;   // one k-block of A
  constexpr uint32_t kBBytes = (BN / CG) * kBK * 2;  // this CTA's part of one k-block of B
  // two f32 accumulator buffers, 32-column aligned; the allocation is a power of two
  constexpr uint32_t kAccStride = (BN + 31) / 32 * 32;
  constexpr uint32_t kTmemCols = 2 * kAccStride <= 64 ? 64 : (2 * kAccStride <= 128 ? 128
                                 : (2 * kAccStride <= 256 ? 256 : 512));
  static_assert(2 * kAccStride <= 512, "two accumulator buffers fit TMEM");
  constexpr int kColsPerWarp = BN / kColGroups;
  // columns loaded from TMEM per wait: 32 where registers allow
  constexpr int kDrainCols = (kColsPerWarp >= 128 || kColsPerWarp % 32 != 0) ? 16 : 32;
  static_assert(kColsPerWarp % 16 == 0, "epilogue column slice must be a multiple of 16");
  static_assert(BN % 16 == 0 && BN >= 16 * CG && BN <= 256, "MMA N: a multiple of 16 up to 256");
  static_assert((BN / CG) % 8 == 0, "B tiles keep the 1024-byte swizzle-atom alignment");
  static_assert(EPI <= kMaxEpiWarps && kColsPerWarp <= kMaxColsPerWarp, "epilogue smem slices");
  static_assert(MODE != 0 || 4 * BN <= kEpFloats, "linear scale/bias buffers exceed Ctl::ep");
  static_assert(MODE == 0 || EPI * 2 * kColsPerWarp <= kEpFloats,
                "per-warp scale/bias slices exceed Ctl::ep");
  constexpr uint32_t kIdesc = idesc_bf16_f32(kBM * CG, BN);
  constexpr bool kPair = (CG == 2);
  constexpr bool kPixN = (MODE >= 3);                  // output channels on M, pixels on N
  constexpr bool kSingleOnly = (MODE >= 5);            // every sub-tile one exact chunk
  constexpr int CM = kPixN ? (MODE - 3) % 2 + 1 : MODE;  // the tile geometry: 0, 1 or 2
  static_assert(!kPixN || CG == 1, "exchanged operands: one CTA per tile");
  static_assert(8 % KD == 0, "the worst-case chunk holds whole stages");
  constexpr uint32_t kStageBytes = static_cast<uint32_t>(KD) * (kABytes + kBBytes);
  const int S = p.stages;

  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw_base = smem_u32(smem_raw);
  const uint32_t base = (raw_base + 1023u) & ~1023u;
  uint8_t* smem = smem_raw + (base - raw_base);
  Ctl* ctl = reinterpret_cast<Ctl*>(smem + S * kStageBytes);
  volatile uint32_t* abort_flag = &ctl->abort_flag;

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int rank = kPair ? static_cast<int>(cluster_ctarank()) : 0;
  const bool leader = (rank == 0);
  // persistent loop over units: a CTA pair walks the units together
  const int unit0 = static_cast<int>(blockIdx.x) / CG;
  const int unit_step = static_cast<int>(gridDim.x) / CG;

  if (threadIdx.x == 0) {
    for (int s = 0; s < S; ++s) {
      mbar_init(smem_u32(&ctl->full[s]), 1);
      mbar_init(smem_u32(&ctl->empty[s]), 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(smem_u32(&ctl->acc_full[b]), 1);
      // the leader's MMA reuses a buffer once both CTAs' epilogues drained it
      mbar_init(smem_u32(&ctl->acc_empty[b]), kEpiWarps * CG);
    }
    mbar_init(smem_u32(&ctl->drain), 1);
    mbar_init(smem_u32(&ctl->epi_bar), kEpiWarps);
    ctl->abort_flag = 0u;
    for (int c = 0; c < kFusedMaxChunks; ++c) ctl->qwarps[c] = 0u;
    fence_mbar_init();
    tma_prefetch_desc(&tmA);
    tma_prefetch_desc(&tmB);
  }
  if (warp == 1) {
    if constexpr (kPair) {
      tmem_alloc_pair(smem_u32(&ctl->tmem_base), kTmemCols);
      tmem_relinquish_pair();
    } else {
      tmem_alloc(smem_u32(&ctl->tmem_base), kTmemCols);
      tmem_relinquish();
    }
  }
  tc_fence_before();
  __syncthreads();
  if constexpr (kPair) cluster_sync_all();  // the peer's barriers exist before any remote use
  tc_fence_after();
  const uint32_t tmem_base = ctl->tmem_base;
  // set-up done: from here on global memory is read and written
  pdl_wait();
  pdl_launch_dependents();
  // exact-f32 chunk length in ring stages (MMA issuer and epilogue agree),
  // from bound words that the previous kernel may have written
  const int chunk_st = chunk_stages(p, KD);
  // The single-chunk instantiation runs only where the host's choice holds
  // on the device too; otherwise (a packed weight changed after packing)
  // nothing runs and the error word says why.
  bool run = true;
  if constexpr (kSingleOnly) {
    if (p.max_nstages > chunk_st) {
      run = false;
      if (threadIdx.x == 0 && blockIdx.x == 0) atomicCAS(p.err, 0u, kErrChunks);
    }
  }
  // Fused quantize: the chunk counters must start at zero, which the
  // trailer's initialization (kFusedMagic) and every launch's last CTA
  // guarantee; a trailer without the magic runs nothing (every CTA reads the
  // same word, written before this launch).
  constexpr bool fused = kFusedQ;
  if constexpr (fused) {
    const uint64_t magic = *reinterpret_cast<const volatile uint64_t*>(p.qsync + kFusedWordMagic);
    if (magic != kFusedMagic) {
      run = false;
      if (threadIdx.x == 0 && blockIdx.x == 0) atomicCAS(p.err, 0u, kErrFusedInit);
    } else if (threadIdx.x == 0 && blockIdx.x == 0) {
      p.qsync[0] = static_cast<uint32_t>(p.a_bound_host);  // the operand's |x - zp| bound
    }
  }

  if (!run) {
    // nothing to do (see above)
  } else if (warp == 0) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      uint32_t stage = 0, phase = 0;
      uint32_t fills = 0;
      int chunks_ready = 0;  // fused quantize: operand chunks known complete
      bool ok = true;
      for (int u = unit0; u < p.total_units && ok; u += unit_step) {
        for (int j = 0; j < p.subtiles && ok; ++j) {
          const TileInfo ti = decode_tile<CM, CG, KD>(p, u, j, rank);
          // k-blocks in (row tap, column tap, channel block) order, with the
          // input offsets stepped incrementally: no division in this loop.
          // Linear tiles are one "tap" of kb_total channel blocks.
          const int ntaps_h = (MODE == 0) ? 1 : ti.nth;
          const int ntaps_w = (MODE == 0) ? 1 : ti.ntw;
          // channel blocks per tap, KD per stage (a last stage may run past them)
          const int nblk = (MODE == 0) ? ti.num_kb : p.icb;
          // input coordinates of the tile's first tap: conv_t phases read
          // (oh' + dh0 - th*dsh); the direct convolution reads
          // (oh*sh - pad_h + th*dil_h) through a box with element stride sh
          const int a_w = (CM == 2) ? ti.wb * p.BW * p.sw - p.pad_w : ti.wb * p.BW + ti.dw0;
          const int a_h = (CM == 2) ? ti.hb * p.BH * p.sh - p.pad_h : ti.hb * p.BH + ti.dh0;
          const int step_w = (CM == 2) ? p.dil_w : -p.dsw;
          const int step_h = (CM == 2) ? p.dil_h : -p.dsh;
          for (int th = 0; th < ntaps_h && ok; ++th) {
            for (int tw = 0; tw < ntaps_w && ok; ++tw) {
              // tap (kh, kw): conv_t (rh + th*tsh, rw + tw*tsw); conv2d (th, tw)
              const int b_blk = (CM == 2)
                                    ? (th * p.Kw + tw) * p.icb
                                    : ((ti.rh + th * p.tsh) * p.Kw + ti.rw + tw * p.tsw) * p.icb;
              const int c_w = a_w + tw * step_w, c_h = a_h + th * step_h;
              for (int blk = 0; blk < nblk; blk += KD) {
                if (!wait_bar(smem_u32(&ctl->empty[stage]), phase ^ 1u, abort_flag,
                              kErrWaitEmpty, p.err, wait_limit(p))) {
                  ok = false;
                  break;
                }
                const uint32_t sa = base + stage * kStageBytes;
                const uint32_t sb = sa + KD * kABytes;
                const int b_row = (MODE == 0 ? ti.nb : ti.ocb) * BN + rank * (BN / CG);
                if constexpr (fused) {
                  // the stage's k-blocks blk .. blk + KD - 1 must be converted
                  // by every CTA before the TMA unit reads them
                  const int need = (min(blk + KD, p.kb_total) - 1) / p.qckb;
                  while (ok && chunks_ready <= need) {
                    ok = wait_chunk(p, chunks_ready, abort_flag);
                    if (ok) ++chunks_ready;
                  }
                  if (!ok) break;
                  fence_proxy_async_global();
                }
                if (p.stall_fill != 0 && fills + 1u == static_cast<uint32_t>(p.stall_fill)) {
                  // failure-detection test: this fill is never issued, so the
                  // MMA's wait on its full barrier runs out (bounded)
                } else if constexpr (kPair) {
                  // both CTAs' copies complete on the leader's full barrier
                  const uint32_t full = map_to_cta(smem_u32(&ctl->full[stage]), 0);
                  if (leader) mbar_arrive_expect_tx(smem_u32(&ctl->full[stage]), CG * kStageBytes);
                  if constexpr (MODE == 0) {
                    tma_load_3d_pair(sa, &tmA, full, 0, ti.mb * kBM, blk);
                    tma_load_3d_pair(sb, &tmB, full, 0, b_row, blk);
                  } else {
                    tma_load_5d_pair(sa, &tmA, full, 0, c_w, c_h, blk, ti.n);
                    tma_load_3d_pair(sb, &tmB, full, 0, b_row, b_blk + blk);
                  }
                } else {
                  const uint32_t full = smem_u32(&ctl->full[stage]);
                  mbar_arrive_expect_tx(full, kStageBytes);
                  if constexpr (MODE == 0) {
                    tma_load_3d(sa, &tmA, full, 0, ti.mb * kBM, blk);
                    tma_load_3d(sb, &tmB, full, 0, b_row, blk);
                  } else if constexpr (kPixN) {
                    // the weight's 128 output-channel rows are the M operand,
                    // the pixel box the N operand
                    tma_load_3d(sa, &tmB, full, 0, ti.ocb * kBM, b_blk + blk);
                    tma_load_5d(sb, &tmA, full, 0, c_w, c_h, blk, ti.n);
                  } else {
                    tma_load_5d(sa, &tmA, full, 0, c_w, c_h, blk, ti.n);
                    tma_load_3d(sb, &tmB, full, 0, b_row, b_blk + blk);
                  }
                }
                ++fills;
                if (++stage == static_cast<uint32_t>(S)) {
                  stage = 0;
                  phase ^= 1u;
                }
              }
            }
          }
        }
      }
      // Let every copy this thread issued land before the CTA can exit (a
      // peer's copies complete on the leader's barriers; the leader waits
      // for both, and the closing cluster barrier holds the peer until then).
      for (int s = 0; s < S && leader; ++s) {
        const uint32_t f = (fills > static_cast<uint32_t>(s)) ? (fills - s + S - 1) / S : 0;
        if (f > 0) wait_bar_final(smem_u32(&ctl->full[s]), (f - 1) & 1u, p.err, wait_limit(p));
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0 && leader) {
      uint32_t stage = 0, phase = 0, acc_it = 0;
      bool ok = true;
      for (int u = unit0; u < p.total_units && ok; u += unit_step) {
        for (int j = 0; j < p.subtiles && ok; ++j) {
          const TileInfo ti = decode_tile<CM, CG, KD>(p, u, j, rank);
          // chunks of chunk_st stages (at most 2048 / a_bound k-blocks each)
          for (int st0 = 0; st0 < ti.nstages && ok; st0 += chunk_st) {
            const uint32_t buf = acc_it & 1u, use = acc_it >> 1;
            if (!wait_bar(smem_u32(&ctl->acc_empty[buf]), (use & 1u) ^ 1u, abort_flag,
                          kErrWaitAccEmpty, p.err, wait_limit(p))) {
              ok = false;
              break;
            }
            tc_fence_after();
            const uint32_t d = tmem_base + buf * kAccStride;
            const int st_end = min(st0 + chunk_st, ti.nstages);
            for (int st = st0; st < st_end; ++st) {
              if (!wait_bar(smem_u32(&ctl->full[stage]), phase, abort_flag, kErrWaitFull, p.err,
                            wait_limit(p))) {
                ok = false;
                break;
              }
              tc_fence_after();
              const uint32_t sa = base + stage * kStageBytes;
              const uint32_t sb = sa + KD * kABytes;
#pragma unroll
              for (int k2 = 0; k2 < KD; ++k2) {
                const uint64_t da = sw128_kmajor_desc(sa + k2 * kABytes);
                const uint64_t db = sw128_kmajor_desc(sb + k2 * kBBytes);
#pragma unroll
                for (int k = 0; k < kBK / 16; ++k) {
                  // +32 bytes along K inside the 128-byte swizzled row
                  const uint32_t acc = (st > st0 || k2 > 0 || k > 0) ? 1u : 0u;
                  if constexpr (kPair)
                    umma_bf16_pair(d, da + 2u * k, db + 2u * k, kIdesc, acc);
                  else
                    umma_bf16(d, da + 2u * k, db + 2u * k, kIdesc, acc);
                }
              }
              // the stage is free in every CTA that supplied it
              if constexpr (kPair)
                umma_commit_pair(smem_u32(&ctl->empty[stage]), 0x3);
              else
                umma_commit(smem_u32(&ctl->empty[stage]));
              if (++stage == static_cast<uint32_t>(S)) {
                stage = 0;
                phase ^= 1u;
              }
            }
            if (!ok) break;
            if constexpr (kPair)
              umma_commit_pair(smem_u32(&ctl->acc_full[buf]), 0x3);
            else
              umma_commit(smem_u32(&ctl->acc_full[buf]));
            ++acc_it;
          }
        }
      }
      // Every MMA issued so far must finish before TMEM is freed.
      if constexpr (kPair)
        umma_commit_pair(smem_u32(&ctl->drain), 0x1);
      else
        umma_commit(smem_u32(&ctl->drain));
      wait_bar_final(smem_u32(&ctl->drain), 0u, p.err, wait_limit(p));
    }
  } else {
    // ------------------------------------------------------------ epilogue
    const int quarter = warp & 3;           // TMEM lanes this warp may read
    const int group = (warp - 2) >> 2;      // which column slice
    const int row = quarter * 32 + lane;
    const int col0 = group * kColsPerWarp;
    const int et = threadIdx.x - 64;  // 0 .. 32 * EPI - 1
    const uint32_t lane_addr = static_cast<uint32_t>(quarter * 32) << 16;
    uint32_t acc_it = 0, epi_phase = 0, tile_par = 0;
    int cur_ocb = -1;
    float px_ws = 0.0f, px_b = 0.0f;  // exchanged operands: this lane's channel
    const int ew = warp - 2;  // epilogue warp index
    bool ok = true;
    if constexpr (fused) {
      // fused quantize: this CTA's share of the operand, before any tile
      // 8 items in flight per thread where the registers allow (<= 448 threads)
      fused_quantize<(cta_threads(EPI) <= 448 ? 8 : 4)>(p, ctl->qwarps, et, 32 * kEpiWarps);
    }
    for (int u = unit0; u < p.total_units && ok; u += unit_step) {
      // register staging: this thread's bytes of the unit's earlier column
      // phases, four output channels per word
      constexpr int kHeld = (MODE != 0 && !kPixN && kColsPerWarp <= 64) ? kColsPerWarp / 4 : 1;
      uint32_t held[kHeld];
      // single-chunk exchanged kernels: phase 0's packed bytes (see pix_store16_reg)
      constexpr int kPh0 = (kPixN && kSingleOnly) ? kColsPerWarp / 4 : 4;
      uint32_t ph0[kPh0];
      for (int j = 0; j < p.subtiles && ok; ++j) {
        const TileInfo ti = decode_tile<CM, CG, KD>(p, u, j, rank);
        if constexpr (kPixN) {
          // ---- exchanged operands: lane = output channel, columns = pixels
          const int oc = ti.ocb * kBM + row;
          if (p.acc_out == nullptr && ti.ocb != cur_ocb) {
            px_ws = (oc < p.OC) ? __ldg(p.ws + oc) : 0.0f;
            px_b = (oc < p.OC && p.bias) ? __ldg(p.bias + oc) : 0.0f;
            cur_ocb = ti.ocb;
          }
          const PixRun run = pix_run<kColsPerWarp>(p, ti, oc, col0);
          const bool mine = oc < p.OC;
          const int nchunks = (ti.nstages + chunk_st - 1) / chunk_st;
          if (nchunks <= 1) {
            // one exact chunk (or none: no tap reaches these pixels): the f32
            // accumulators stream from TMEM through the requantization, 16
            // columns at a time
            const uint32_t buf = acc_it & 1u, use = acc_it >> 1;
            if (nchunks == 1) {
              bool got = true;
              if (lane == 0)
                got = wait_bar(smem_u32(&ctl->acc_full[buf]), use & 1u, abort_flag, kErrWaitAccFull,
                               p.err, wait_limit(p));
              got = __shfl_sync(0xffffffffu, got ? 1 : 0, 0) != 0;
              if (!got) {
                ok = false;
                break;
              }
              tc_fence_after();
            }
            uint32_t hold[4] = {0u, 0u, 0u, 0u};
            if constexpr (kSingleOnly) {
              // groups unrolled, so ph0 stays in registers
              static_assert(!kSingleOnly || kColsPerWarp == 64, "four 16-column groups per thread");
              uint32_t r[1][16];
              const uint32_t taddr = tmem_base + lane_addr + buf * kAccStride + col0;
#pragma unroll
              for (int g = 0; g < 4; ++g) {
                if (nchunks == 1) {
                  tmem_ld_16cols(taddr + 16 * g, r[0]);
                  tmem_ld_wait();
                } else {
#pragma unroll
                  for (int i = 0; i < 16; ++i) r[0][i] = 0u;
                }
                if (mine) {
                  if (p.acc_out != nullptr) {
                    int32_t a[16];
#pragma unroll
                    for (int i = 0; i < 16; ++i) a[i] = __float2int_rn(__uint_as_float(r[0][i]));
                    pix_store16_acc(p, ti, run, col0, g, a);
                  } else {
                    float fv[16];
#pragma unroll
                    for (int i = 0; i < 16; ++i) fv[i] = __uint_as_float(r[0][i]);
                    if (g == 0) pix_store16_reg<kColsPerWarp, 0>(p, ti, run, col0, fv, px_ws, px_b, hold, ph0);
                    if (g == 1) pix_store16_reg<kColsPerWarp, 1>(p, ti, run, col0, fv, px_ws, px_b, hold, ph0);
                    if (g == 2) pix_store16_reg<kColsPerWarp, 2>(p, ti, run, col0, fv, px_ws, px_b, hold, ph0);
                    if (g == 3) pix_store16_reg<kColsPerWarp, 3>(p, ti, run, col0, fv, px_ws, px_b, hold, ph0);
                  }
                }
              }
            } else
#pragma unroll 1
            for (int g = 0; g < kColsPerWarp / 16; ++g) {
              uint32_t e[8];
              if (mine && p.acc_out == nullptr) pix_phase0(p, ti, run, g, e);
              uint32_t r[16];
              if (nchunks == 1) {
                tmem_ld_16cols(tmem_base + lane_addr + buf * kAccStride + col0 + 16 * g, r);
                tmem_ld_wait();
              } else {
#pragma unroll
                for (int i = 0; i < 16; ++i) r[i] = 0u;
              }
              if (mine) {
                if (p.acc_out != nullptr) {
                  int32_t a[16];
#pragma unroll
                  for (int i = 0; i < 16; ++i) a[i] = __float2int_rn(__uint_as_float(r[i]));
                  pix_store16_acc(p, ti, run, col0, g, a);
                } else {
                  float fv[16];
#pragma unroll
                  for (int i = 0; i < 16; ++i) fv[i] = __uint_as_float(r[i]);
                  pix_store16<kColsPerWarp>(p, ti, run, col0, g, fv, px_ws, px_b, hold, e);
                }
              }
            }
            if (nchunks == 1) {
              tc_fence_before();
              __syncwarp();
              if (lane == 0) mbar_arrive(smem_u32(&ctl->acc_empty[buf]));
              ++acc_it;
            }
          } else if constexpr (kSingleOnly) {
            ok = false;  // excluded on entry (max_nstages <= chunk_st)
            break;
          } else if (nchunks == 2) {
            // two exact chunks in the two TMEM buffers: held together and
            // streamed as one.  Each chunk sum is an integer below 2^24 in
            // magnitude, so one f32 add rounds their exact sum once, to
            // float(acc) (what the requantization starts from); the int32
            // output adds the two exact conversions.  The MMA waits for both
            // buffers meanwhile.
            const uint32_t b0 = acc_it & 1u, b1 = (acc_it + 1u) & 1u;
            bool got = true;
            if (lane == 0) {
              got = wait_bar(smem_u32(&ctl->acc_full[b0]), (acc_it >> 1) & 1u, abort_flag,
                             kErrWaitAccFull, p.err, wait_limit(p)) &&
                    wait_bar(smem_u32(&ctl->acc_full[b1]), ((acc_it + 1u) >> 1) & 1u, abort_flag,
                             kErrWaitAccFull, p.err, wait_limit(p));
            }
            got = __shfl_sync(0xffffffffu, got ? 1 : 0, 0) != 0;
            if (!got) {
              ok = false;
              break;
            }
            tc_fence_after();
            uint32_t hold[4] = {0u, 0u, 0u, 0u};
#pragma unroll 1
            for (int g = 0; g < kColsPerWarp / 16; ++g) {
              uint32_t e[8];
              if (mine && p.acc_out == nullptr) pix_phase0(p, ti, run, g, e);
              uint32_t r0[16], r1[16];
              const uint32_t ta = tmem_base + lane_addr + col0 + 16 * g;
              tmem_ld_16cols(ta + b0 * kAccStride, r0);
              tmem_ld_16cols(ta + b1 * kAccStride, r1);
              tmem_ld_wait();
              if (mine) {
                if (p.acc_out != nullptr) {
                  int32_t a[16];
#pragma unroll
                  for (int i = 0; i < 16; ++i)
                    a[i] = static_cast<int32_t>(
                        static_cast<uint32_t>(__float2int_rn(__uint_as_float(r0[i]))) +
                        static_cast<uint32_t>(__float2int_rn(__uint_as_float(r1[i]))));
                  pix_store16_acc(p, ti, run, col0, g, a);
                } else {
                  float fv[16];
#pragma unroll
                  for (int i = 0; i < 16; ++i)
                    fv[i] = __fadd_rn(__uint_as_float(r0[i]), __uint_as_float(r1[i]));
                  pix_store16<kColsPerWarp>(p, ti, run, col0, g, fv, px_ws, px_b, hold, e);
                }
              }
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) {
              mbar_arrive(smem_u32(&ctl->acc_empty[b0]));
              mbar_arrive(smem_u32(&ctl->acc_empty[b1]));
            }
            acc_it += 2u;
          } else {
            // three chunks or more (each chunk's f32 sum is an exact integer)
            const PixChunks c = pix_chunks<kColsPerWarp, kAccStride>(
                p, ti, run, ctl, tmem_base + lane_addr, col0, mine, px_ws, px_b, acc_it, chunk_st);
            acc_it = c.acc_it;
            if (!c.ok) {
              ok = false;
              break;
            }
          }
          continue;
        }
        const int gcolbase = (MODE == 0) ? ti.nb * BN : ti.ocb * BN;
        const int ncols = (MODE == 0) ? p.N : p.OC;
        // The tile's column scales and biases into shared memory, loaded
        // before the accumulator waits so their latency hides there.
        //   linear: one copy per tile for all warps (et < BN loads it), two
        //     buffers by tile parity, published by the rendezvous below;
        //   conv: each warp keeps its own columns, reloaded only when the
        //     output-channel block changes (for OC <= BN: once per CTA).
        const float* sws;
        const float* sbs;
        // linear: this thread's column scale and bias, loaded now and
        // written to shared memory after the accumulator drains, so the
        // load latency is spent there
        float ld_ws = 0.0f, ld_b = 0.0f;
        float* ws_buf = ctl->ep + tile_par * (2 * kMaxBN);
        if constexpr (MODE == 0) {
          if (p.acc_out == nullptr && et < BN) {
            const int gc = gcolbase + et;
            ld_ws = (gc < ncols) ? __ldg(p.ws + gc) : 0.0f;
            ld_b = (gc < ncols && p.bias) ? __ldg(p.bias + gc) : 0.0f;
          }
          sws = ws_buf + col0;
          sbs = ws_buf + kMaxBN + col0;
        } else {
          float* slice = ctl->ep + ew * (2 * kColsPerWarp);
          if (p.acc_out == nullptr && ti.ocb != cur_ocb) {
            __syncwarp();
#pragma unroll
            for (int c0 = 0; c0 < kColsPerWarp; c0 += 32) {
              const int c = c0 + lane;
              if (c < kColsPerWarp) {
                const int gc = gcolbase + col0 + c;
                slice[c] = (gc < ncols) ? __ldg(p.ws + gc) : 0.0f;
                slice[kColsPerWarp + c] = (gc < ncols && p.bias) ? __ldg(p.bias + gc) : 0.0f;
              }
            }
            cur_ocb = ti.ocb;
          }
          sws = slice;
          sbs = slice + kColsPerWarp;
        }
        // A convolution tile of a single exact chunk keeps the f32
        // accumulator as it is (an exact integer: converting it to int32 and
        // back would return the same value); longer tiles add the chunks as
        // int32.  (Only where the column slice is small: the extra path
        // costs registers that the wide linear slices do not have.)
        constexpr bool kSingleChunkPath = (MODE != 0) && (kColsPerWarp <= 64);
        const bool single = kSingleChunkPath && ti.nstages <= chunk_st;
        int32_t sum[kColsPerWarp];
#pragma unroll
        for (int c = 0; c < kColsPerWarp; ++c) sum[c] = 0;
        for (int st0 = 0; st0 < ti.nstages; st0 += chunk_st) {
          const uint32_t buf = acc_it & 1u, use = acc_it >> 1;
          bool got = true;
          if (lane == 0)
            got = wait_bar(smem_u32(&ctl->acc_full[buf]), use & 1u, abort_flag, kErrWaitAccFull, p.err,
                           wait_limit(p));
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
              tmem_ld_16cols(tmem_base + lane_addr + buf * kAccStride + col0 + kDrainCols * c + 16 * h,
                             *reinterpret_cast<uint32_t(*)[16]>(&r[16 * h]));
            tmem_ld_wait();
            if (single) {
#pragma unroll
              for (int i = 0; i < kDrainCols; ++i) sum[kDrainCols * c + i] = static_cast<int32_t>(r[i]);
            } else {
#pragma unroll
              for (int i = 0; i < kDrainCols; ++i)
                sum[kDrainCols * c + i] = static_cast<int32_t>(
                    static_cast<uint32_t>(sum[kDrainCols * c + i]) +
                    static_cast<uint32_t>(__float2int_rn(__uint_as_float(r[i]))));
            }
          }
          tc_fence_before();
          __syncwarp();
          if (lane == 0) {
            // the MMA issuer (the leader CTA's) may reuse this buffer
            if (kPair && !leader)
              mbar_arrive_cluster(map_to_cta(smem_u32(&ctl->acc_empty[buf]), 0));
            else
              mbar_arrive(smem_u32(&ctl->acc_empty[buf]));
          }
          ++acc_it;
        }
        if (!ok) break;
        // sum[] in one form for what follows: int32 accumulators for the
        // acc_out debug output, else the f32 value (float(acc), rounded to
        // nearest even when |acc| > 2^24) the requantization starts from
        if (p.acc_out != nullptr) {
          if (single) {
#pragma unroll
            for (int c = 0; c < kColsPerWarp; ++c) sum[c] = __float2int_rn(__int_as_float(sum[c]));
          }
        } else if (!single) {
#pragma unroll
          for (int c = 0; c < kColsPerWarp; ++c) sum[c] = __float_as_int(__int2float_rn(sum[c]));
        }

        // ---- fused epilogue
        if constexpr (MODE == 0) {
          if (p.acc_out == nullptr && et < BN) {
            ws_buf[et] = ld_ws;
            ws_buf[kMaxBN + et] = ld_b;
          }
          if (p.acc_out == nullptr && !epi_sync(ctl, epi_phase, abort_flag, p.err, wait_limit(p))) {
            ok = false;
            break;
          }
          tile_par ^= 1u;
        } else {
          __syncwarp();  // this warp's scale/bias slice is visible to all its lanes
        }
        if constexpr (MODE == 0) {
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
                  wds[q] = pack4_sat(rq_unclamped(__int_as_float(sum[s0 + 0]), w4.x, b4.x, p.rq),
                                     rq_unclamped(__int_as_float(sum[s0 + 1]), w4.y, b4.y, p.rq),
                                     rq_unclamped(__int_as_float(sum[s0 + 2]), w4.z, b4.z, p.rq),
                                     rq_unclamped(__int_as_float(sum[s0 + 3]), w4.w, b4.w, p.rq));
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
          const int oh = (ti.hb * p.BH + hh) * p.osh + ti.ph;
          const int ow = (ti.wb * p.BW + ww) * p.osw + ti.pw;
          const int oc0 = gcolbase + col0;
          const bool inside = (oh < p.H_out && ow < p.W_out);
          bool done = false;
          if constexpr (kHeld > 1) {
            if (p.staged == 2) {
              // Register staging (osw <= 2): the unit's column phases of one
              // output pixel pair are processed by this same thread; earlier
              // phases wait packed in held[], and the last one writes osw
              // consecutive bytes per output channel (a warp covers 32 * osw
              // contiguous bytes of an output row).
              done = true;
              const bool last = (ti.pw == p.osw - 1);
              const int64_t plane = static_cast<int64_t>(p.H_out) * p.W_out;
              int8_t* dst = p.out + (static_cast<int64_t>(ti.n) * p.out_ch + oc0) * plane +
                            static_cast<int64_t>(oh) * p.W_out + (ow - ti.pw);
#pragma unroll
              for (int g = 0; g < kColsPerWarp / 16; ++g) {
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                  const float4 w4 = *reinterpret_cast<const float4*>(sws + 16 * g + 4 * q);
                  const float4 b4 = *reinterpret_cast<const float4*>(sbs + 16 * g + 4 * q);
                  const int s0 = 16 * g + 4 * q;
                  const int32_t v[4] = {requant_f(__int_as_float(sum[s0 + 0]), w4.x, b4.x, p.rq),
                                        requant_f(__int_as_float(sum[s0 + 1]), w4.y, b4.y, p.rq),
                                        requant_f(__int_as_float(sum[s0 + 2]), w4.z, b4.z, p.rq),
                                        requant_f(__int_as_float(sum[s0 + 3]), w4.w, b4.w, p.rq)};
                  if (!last) {
                    held[s0 / 4] = pack4_i(v[0], v[1], v[2], v[3]);
                  } else if (inside) {
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                      if (oc0 + s0 + e >= p.OC) continue;
                      if (p.osw == 2) {
                        const uint32_t lo = (held[s0 / 4] >> (8 * e)) & 0xffu;
                        *reinterpret_cast<uint16_t*>(dst + (s0 + e) * plane) =
                            static_cast<uint16_t>(lo | ((static_cast<uint32_t>(v[e]) & 0xffu) << 8));
                      } else {
                        dst[(s0 + e) * plane] = static_cast<int8_t>(v[e]);
                      }
                    }
                  }
                }
              }
            }
          }
          if (done) {
            // stored above
          } else if (inside) {
            const int64_t plane = static_cast<int64_t>(p.H_out) * p.W_out;
            int8_t* dst = p.out ? p.out + (static_cast<int64_t>(ti.n) * p.out_ch + oc0) * plane +
                                      static_cast<int64_t>(oh) * p.W_out + ow
                                : nullptr;
            int32_t* adst = p.acc_out ? p.acc_out + (static_cast<int64_t>(ti.n) * p.out_ch + oc0) * plane +
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
                  const int32_t v[4] = {requant_f(__int_as_float(sum[s0 + 0]), w4.x, b4.x, p.rq),
                                        requant_f(__int_as_float(sum[s0 + 1]), w4.y, b4.y, p.rq),
                                        requant_f(__int_as_float(sum[s0 + 2]), w4.z, b4.z, p.rq),
                                        requant_f(__int_as_float(sum[s0 + 3]), w4.w, b4.w, p.rq)};
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
  // neither CTA of a pair leaves while the leader's MMAs may still read the
  // peer's shared memory or signal its barriers
  if constexpr (kPair) cluster_sync_all();
  if (warp == 1) {
    tc_fence_after();
    if constexpr (kPair)
      tmem_dealloc_pair(tmem_base, kTmemCols);
    else
      tmem_dealloc(tmem_base, kTmemCols);
  }
  if (fused && run && threadIdx.x == 0) {  // (fused: constexpr)
    // The last CTA to finish (no producer polls the counters any more) puts
    // them back to zero for the next launch on this operand.
    __threadfence();
    const uint32_t done = atomicAdd(p.qsync + kFusedWordDone, 1u);
    if (done == gridDim.x - 1) {
      __threadfence();
      for (int c = 0; c < p.qnch; ++c) p.qsync[kFusedWordChunk0 + c] = 0u;
      p.qsync[kFusedWordDone] = 0u;
      __threadfence();
    }
  }
}


// ---------------------------------------------------------------------------
// Host launch of one instantiation (smem ring sized from the budget)
// ---------------------------------------------------------------------------
constexpr size_t kSmemBudget = 225 * 1024;   // of the 227 KB a CTA may use

inline int pick_bn(int64_t n) { return n <= 64 ? 64 : (n <= 128 ? 128 : 256); }

template <int BN, int EPI, int MODE, int KD, int CG>
inline cudaError_t launch_tc_kernel(const CUtensorMap& a, const CUtensorMap& b, TcParams p,
                                    cudaStream_t s) {
  const size_t kStage = static_cast<size_t>(KD) * (static_cast<size_t>(kBM) * kBK * 2 +
                                                   static_cast<size_t>(BN / CG) * kBK * 2);
  const size_t fixed = sizeof(Ctl) + 1024;
  const int stages = static_cast<int>(std::min<size_t>(kMaxStages, (kSmemBudget - fixed) / kStage));
  if (stages < 2) return cudaErrorInvalidValue;
  p.err = device_error_word();
  if (p.err == nullptr) return cudaErrorInvalidValue;
  p.stages = stages;
  p.kd = KD;
  const size_t smem = static_cast<size_t>(stages) * kStage + sizeof(Ctl) + 1024;
  auto kernel = tc_gemm_kernel<BN, EPI, MODE, KD, CG>;
  static std::once_flag attr_once[64];
  int dev = 0;
  cudaGetDevice(&dev);
  cudaError_t attr_err = cudaSuccess;
  std::call_once(attr_once[dev & 63], [&] {
    attr_err = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                    static_cast<int>(kSmemBudget + 1024));
  });
  if (attr_err != cudaSuccess) return attr_err;
  cudaLaunchConfig_t cfg = {};
  cfg.blockDim = dim3(static_cast<unsigned>(cta_threads(EPI)), 1, 1);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = CG;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  // programmatic dependent launch: the set-up above the kernel's pdl_wait()
  // overlaps the previous kernel on the stream
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 2;
  // persistent: one CTA per SM, or one CTA pair per co-resident SM pair (a
  // pair must share a GPC, so fewer than SMs / 2 pairs may fit at once)
  int resident = device_sm_count() / CG;
  if (CG > 1) {
    static int pairs_cache[64] = {};
    int& cached = pairs_cache[dev & 63];
    if (cached == 0) {
      cfg.gridDim = dim3(static_cast<unsigned>(resident * CG), 1, 1);
      int n = 0;
      if (cudaOccupancyMaxActiveClusters(&n, kernel, &cfg) != cudaSuccess || n <= 0) {
        cudaGetLastError();
        n = resident;
      }
      cached = n;
    }
    resident = std::min(resident, cached);
  }
  const int groups = std::max(1, std::min(p.total_units, resident));
  cfg.gridDim = dim3(static_cast<unsigned>(groups * CG), 1, 1);
  cudaError_t e = cudaLaunchKernelEx(&cfg, kernel, a, b, p);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

}  // namespace q8
