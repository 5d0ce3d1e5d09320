// device_common.cuh -- device helpers shared by the q8ta kernels (sm_103a).
//
// Hand-written inline PTX for the Blackwell pieces the kernels use
// (mbarrier, TMA bulk tensor copies, tcgen05 MMA / TMEM), and the f32
// dequantize -> requantize epilogue of the q8ta ops.
#pragma once

#include <cstdint>
#include <cuda_runtime.h>

#include "fastdiv.h"

namespace q8 {

// ---------------------------------------------------------------------------
// The requantize epilogue ("Add q8ta_linear op" and "Add
// q8ta_conv2d_transposed op", Solution paragraphs): one f32 rounding per
// step, fixed order, no contraction into FMA (explicit _rn intrinsics are
// never fused by the compiler), round half to even.
// ---------------------------------------------------------------------------
struct Requant {
  float s_in;     // (float)input_scale
  float inv_out;  // (float)(1.0 / output_scale), formed on the host in double
  float ozp;      // output zero point, exactly representable
  int32_t ozp_i;  // the same zero point as an integer
  int32_t lo;     // output floor: -128, or ozp_i for activation "relu"
  float lo_f;     // lo - ozp_i and 127 - ozp_i: the clamp bounds of rint(u)
  float hi_f;
};

// clamp(rint(u) + zp, -128, 127) with rint half-to-even, as an int32, on
// plain FP32/INT32 ALU operations (no float<->int conversion instruction):
//  * u is first raised to at least -2^22 (fmaxf maps NaN to -2^22 too);
//  * adding 1.5 * 2^23 rounds to an integer (round-to-nearest-even: for
//    -2^22 <= u < 2^22 the sum lies in [2^23, 2^24), where the spacing of
//    floats is exactly 1), and the integer is the low bits of the sum's
//    encoding: bits(sum) - 0x4B400000.  For larger u the encoding only grows
//    (the sum stays positive), so the clamp saturates at 127 as it should;
//    for u < -2^22, and NaN, it gives -128 (the float form's fmaxf/fminf
//    clamp gives the same).
// Equal to the float form -- r = rint(u); t = r + zp; clamp t to
// [-128, 127]; (int8)t -- for every float u and every zp in [-128, 127]
// when lo = -128.  lo = zp gives the relu form: max(v, 0) before the
// requantization is max(q, zp) after it, v * inv_out being monotone and
// rint(0) = 0.
constexpr float kRoundMagic = 12582912.0f;   // 1.5 * 2^23, encoded 0x4B400000
constexpr float kRoundFloor = -4194304.0f;   // -2^22

__device__ __forceinline__ int32_t magic_to_q(float y, int32_t zp, int32_t lo) {
  const int32_t q = __float_as_int(y) - (0x4B400000 - zp);
  return min(max(q, lo), 127);
}

__device__ __forceinline__ int32_t round_add_clamp_i(float u, int32_t zp, int32_t lo) {
  const float y = __fadd_rn(fmaxf(u, kRoundFloor), kRoundMagic);
  return magic_to_q(y, zp, lo);
}

// The same result with the clamp taken first, on the float: u is clamped to
// [lo - zp, 127 - zp], whose bounds are integers, so that rint(clamp(u)) + zp
// = clamp(rint(u) + zp, lo, 127) for every u (NaN takes the lower bound, as
// fmaxf does above); then 1.5 * 2^23 is added and the integer read off the
// encoding, already in range.  One instruction fewer per output.
__device__ __forceinline__ int32_t round_clamp_first(float u, int32_t zp, float lo_f, float hi_f) {
  const float c = fminf(fmaxf(u, lo_f), hi_f);
  return __float_as_int(__fadd_rn(c, kRoundMagic)) - (0x4B400000 - zp);
}

// The same result with only the floor taken on the float: u is raised to
// at least lo - zp (NaN takes it, as fmaxf does), 1.5 * 2^23 is added and
// the integer read off the encoding; that integer is rint(u) + zp below
// 2^22 and only larger above, so a saturating conversion to int8 (see
// pack4_sat) supplies the upper clamp.  Returns the unsaturated int32.
__device__ __forceinline__ int32_t round_floor_first(float u, int32_t zp, float lo_f) {
  return __float_as_int(__fadd_rn(fmaxf(u, lo_f), kRoundMagic)) - (0x4B400000 - zp);
}

// Four int32 values saturated to [-128, 127] as bytes 0..3 of a word: two
// cvt.pack.sat (each converts two values with saturation into the low 16
// bits and copies the low bits of its third operand above them).
__device__ __forceinline__ uint32_t pack4_sat(int32_t a, int32_t b, int32_t c, int32_t d) {
  uint32_t hi, r;
  asm("cvt.pack.sat.s8.s32.b32 %0, %1, %2, %3;" : "=r"(hi) : "r"(d), "r"(c), "r"(0u));
  asm("cvt.pack.sat.s8.s32.b32 %0, %1, %2, %3;" : "=r"(r) : "r"(b), "r"(a), "r"(hi));
  return r;
}

// The fused epilogue of one accumulator, in the order of "Add q8ta_linear op"
// (Solution paragraph): ((acc * input_scale) * weight_scale + bias) *
// (1 / output_scale), rounded, plus the output zero point, clamped (from
// below at the zero point under the relu activation).  requant_f takes
// a = (float)acc.
__device__ __forceinline__ int32_t requant_f(float a, float ws, float b, const Requant& rq) {
  float t = __fmul_rn(a, rq.s_in);
  t = __fmul_rn(t, ws);
  float v = __fadd_rn(t, b);
  float u = __fmul_rn(v, rq.inv_out);
  return round_clamp_first(u, rq.ozp_i, rq.lo_f, rq.hi_f);
}

// From the int32 accumulator: a = (float)acc, rounded to nearest even.
__device__ __forceinline__ int32_t requant_i(int32_t acc, float ws, float b, const Requant& rq) {
  return requant_f(__int2float_rn(acc), ws, b, rq);
}

__device__ __forceinline__ int8_t requant_one(int32_t acc, float ws, float b, const Requant& rq) {
  return static_cast<int8_t>(requant_i(acc, ws, b, rq));
}

// Four values in [-128, 127] as bytes 0..3 of a word.
__device__ __forceinline__ uint32_t pack4_i(int32_t a, int32_t b, int32_t c, int32_t d) {
  const uint32_t lo = __byte_perm(static_cast<uint32_t>(a), static_cast<uint32_t>(b), 0x0040);
  const uint32_t hi = __byte_perm(static_cast<uint32_t>(c), static_cast<uint32_t>(d), 0x0040);
  return __byte_perm(lo, hi, 0x5410);
}

__device__ __forceinline__ uint32_t pack4(int8_t a, int8_t b, int8_t c, int8_t d) {
  return (uint32_t)(uint8_t)a | ((uint32_t)(uint8_t)b << 8) | ((uint32_t)(uint8_t)c << 16) |
         ((uint32_t)(uint8_t)d << 24);
}

// quantize_per_tensor of one value ("Add quantize_per_tensor op", Solution
// paragraph): clamp(rint(x * inv) + zp, -128, 127) on ALU instructions
// (round_add_clamp_i, equal to the float form for every x; zp in [-128, 127]).
__device__ __forceinline__ int8_t quantize_one(float x, float inv, int32_t zp) {
  return static_cast<int8_t>(round_add_clamp_i(__fmul_rn(x, inv), zp, -128));
}

// Operand preparation for the tensor-core GEMM: int8 values, and the
// differences x - zp in [-255, 255], are exact in bf16 (8 significant bits).
// On integer and FP32 ALU instructions only (no conversion instruction): for
// |v| < 2^22, bits(1.5 * 2^23) + v is the encoding of 1.5 * 2^23 + v, so one
// exact f32 subtraction gives (float)v; with at most 8 significant bits its
// low 16 encoding bits are zero, and the high 16 are its bf16 encoding.
__device__ __forceinline__ uint32_t bf16_bits_hi(int v) {
  return __float_as_uint(__fsub_rn(__int_as_float(0x4B400000 + v), 12582912.0f));
}
__device__ __forceinline__ uint32_t bf16x2_from_ints(int lo, int hi) {
  return __byte_perm(bf16_bits_hi(lo), bf16_bits_hi(hi), 0x7632);
}

// quantize_per_tensor of 8 values and the bf16 of their q - zp, together:
// u = x * inv is clamped first to [-128 - zp, 127 - zp] (integer bounds, so
// rint(clamp(u)) + zp = clamp(rint(u) + zp, -128, 127), NaN taking the lower
// bound as in quantize_one), then y = u + 1.5 * 2^23 rounds it: the low byte
// of bits(y) + zp is q, and y - 1.5 * 2^23 is exactly the float of q - zp,
// whose high half is its bf16.  qw: the 8 int8 q; ow: the 8 bf16.
__device__ __forceinline__ void quantize8_operand(const float (&x)[8], float inv, int32_t zp,
                                                  uint2& qw, uint4& ow) {
  const float lo_f = static_cast<float>(-128 - zp), hi_f = static_cast<float>(127 - zp);
  uint32_t qb[8], d[8];
#pragma unroll
  for (int j = 0; j < 8; ++j) {
    const float c = fminf(fmaxf(__fmul_rn(x[j], inv), lo_f), hi_f);
    const float y = __fadd_rn(c, kRoundMagic);
    qb[j] = __float_as_uint(y) + static_cast<uint32_t>(zp);
    d[j] = __float_as_uint(__fsub_rn(y, kRoundMagic));
  }
  qw.x = __byte_perm(__byte_perm(qb[0], qb[1], 0x0040), __byte_perm(qb[2], qb[3], 0x0040), 0x5410);
  qw.y = __byte_perm(__byte_perm(qb[4], qb[5], 0x0040), __byte_perm(qb[6], qb[7], 0x0040), 0x5410);
  ow.x = __byte_perm(d[0], d[1], 0x7632);
  ow.y = __byte_perm(d[2], d[3], 0x7632);
  ow.z = __byte_perm(d[4], d[5], 0x7632);
  ow.w = __byte_perm(d[6], d[7], 0x7632);
}

// Destination layout of the GEMM operands ("K-blocked"): dst[kb][r][kk] with
// kb = k / 64 and kk = k % 64, so the 128 x 64 (or BN x 64) tile the tensor
// cores read for one k-block is a single contiguous run in memory.
__device__ __forceinline__ int64_t kblocked_index16(int64_t r, int64_t k0, int64_t rows) {
  // index of the 16-byte chunk holding elements k0 .. k0 + 7 of row r
  return (((k0 >> 6) * rows + r) * 64 + (k0 & 63)) / 8;
}

// ---------------------------------------------------------------------------
// Programmatic dependent launch.  Every kernel of the library is launched
// with programmatic stream serialization: it may start while the previous
// kernel on the stream is still finishing.  pdl_wait() returns once that
// kernel has completed and its memory operations are visible, so a kernel
// calls it before its first access to global memory (reads and writes);
// pdl_launch_dependents() lets the next kernel's blocks be scheduled.
// Outside such a launch both are no-ops.
// ---------------------------------------------------------------------------
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_launch_dependents() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// ---------------------------------------------------------------------------
// Shared memory, mbarrier
// ---------------------------------------------------------------------------
__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}

__device__ __forceinline__ void fence_mbar_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes)
               : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}

__device__ __forceinline__ uint64_t global_timer_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

// ---------------------------------------------------------------------------
// TMA (cp.async.bulk.tensor), completion counted on an mbarrier
// ---------------------------------------------------------------------------
__device__ __forceinline__ void tma_prefetch_desc(const void* map) {
  asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(map)) : "memory");
}

__device__ __forceinline__ void tma_load_2d(uint32_t dst, const void* map, uint32_t bar, int32_t c0,
                                            int32_t c1) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%3, %4}], [%2];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(bar), "r"(c0), "r"(c1)
      : "memory");
}

__device__ __forceinline__ void tma_load_3d(uint32_t dst, const void* map, uint32_t bar, int32_t c0,
                                            int32_t c1, int32_t c2) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%3, %4, %5}], [%2];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(bar), "r"(c0), "r"(c1), "r"(c2)
      : "memory");
}

__device__ __forceinline__ void tma_load_5d(uint32_t dst, const void* map, uint32_t bar, int32_t c0,
                                            int32_t c1, int32_t c2, int32_t c3, int32_t c4) {
  asm volatile(
      "cp.async.bulk.tensor.5d.shared::cluster.global.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%3, %4, %5, %6, %7}], [%2];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(bar), "r"(c0), "r"(c1), "r"(c2), "r"(c3), "r"(c4)
      : "memory");
}

__device__ __forceinline__ void tma_load_4d(uint32_t dst, const void* map, uint32_t bar, int32_t c0,
                                            int32_t c1, int32_t c2, int32_t c3) {
  asm volatile(
      "cp.async.bulk.tensor.4d.shared::cluster.global.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%3, %4, %5, %6}], [%2];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(bar), "r"(c0), "r"(c1), "r"(c2), "r"(c3)
      : "memory");
}

// ---------------------------------------------------------------------------
// tcgen05: TMEM allocation, MMA, commit, loads
// ---------------------------------------------------------------------------
__device__ __forceinline__ void tmem_alloc(uint32_t dst_smem, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(dst_smem),
               "r"(ncols)
               : "memory");
}
__device__ __forceinline__ void tmem_relinquish() {
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols)
               : "memory");
}
__device__ __forceinline__ void tc_fence_before() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

// D[tmem] (+)= A[smem] * B[smem]^T, bf16 inputs, f32 accumulate, M=128.
__device__ __forceinline__ void umma_bf16(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc,
                                          uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}

// Arrive once on `bar` when every tcgen05.mma issued so far by this thread
// has completed.
__device__ __forceinline__ void umma_commit(uint32_t bar) {
  asm volatile(
      "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar)
      : "memory");
}

// 32 consecutive 32-bit TMEM columns of this thread's lane.
__device__ __forceinline__ void tmem_ld_32cols(uint32_t taddr, uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
      "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, "
      "%16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}, [%32];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
        "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]),
        "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]),
        "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
      : "r"(taddr)
      : "memory");
}

// 16 consecutive 32-bit TMEM columns of this thread's lane.
__device__ __forceinline__ void tmem_ld_16cols(uint32_t taddr, uint32_t (&r)[16]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 "
      "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15}, [%16];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
        "=r"(r[14]), "=r"(r[15])
      : "r"(taddr)
      : "memory");
}

__device__ __forceinline__ void tmem_ld_wait() {
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}

// ---------------------------------------------------------------------------
// CTA pairs (clusters of 2) for the 2-SM MMA: rank, cluster barrier, peer
// shared-memory addresses, remote mbarrier arrival, and the cta_group::2
// forms of TMA, TMEM allocation, MMA and commit.
// ---------------------------------------------------------------------------
__device__ __forceinline__ uint32_t cluster_ctarank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}
__device__ __forceinline__ void cluster_sync_all() {
  asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::
                   : "memory");
}
// The shared::cluster address of `local_addr` in CTA `rank` of the cluster.
__device__ __forceinline__ uint32_t map_to_cta(uint32_t local_addr, uint32_t rank) {
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(local_addr), "r"(rank));
  return r;
}
// Arrival on a barrier of another CTA of the cluster.  Default semantics
// (release at CTA scope): the arrivals here publish TMEM reads, which
// tcgen05.wait::ld and tcgen05.fence::before_thread_sync already order; a
// cluster-scope release would also hold the warp until its earlier global
// stores were visible cluster-wide.
__device__ __forceinline__ void mbar_arrive_cluster(uint32_t cluster_addr) {
  asm volatile("mbarrier.arrive.shared::cluster.b64 _, [%0];" ::"r"(cluster_addr) : "memory");
}
// TMA loads into this CTA's shared memory whose completion is counted on an
// mbarrier that may live in the peer CTA (cluster address).
__device__ __forceinline__ void tma_load_3d_pair(uint32_t dst, const void* map, uint32_t bar,
                                                 int32_t c0, int32_t c1, int32_t c2) {
  asm volatile(
      "cp.async.bulk.tensor.3d.cta_group::2.shared::cluster.global.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%3, %4, %5}], [%2];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(bar), "r"(c0), "r"(c1), "r"(c2)
      : "memory");
}
__device__ __forceinline__ void tma_load_5d_pair(uint32_t dst, const void* map, uint32_t bar,
                                                 int32_t c0, int32_t c1, int32_t c2, int32_t c3,
                                                 int32_t c4) {
  asm volatile(
      "cp.async.bulk.tensor.5d.cta_group::2.shared::cluster.global.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%3, %4, %5, %6, %7}], [%2];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(bar), "r"(c0), "r"(c1), "r"(c2), "r"(c3), "r"(c4)
      : "memory");
}
// Collective over the CTA pair: one warp of each CTA executes it.
__device__ __forceinline__ void tmem_alloc_pair(uint32_t dst_smem, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(dst_smem),
               "r"(ncols)
               : "memory");
}
__device__ __forceinline__ void tmem_relinquish_pair() {
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc_pair(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols)
               : "memory");
}
// D (+)= A * B^T over the pair: M = 256, each CTA supplies 128 rows of A and
// half of B's N rows from the same shared-memory offsets; the leader CTA
// issues it, and each CTA's TMEM receives the accumulators of its own rows.
__device__ __forceinline__ void umma_bf16_pair(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc,
                                               uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::2.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}
// Arrive once on the mbarrier at `bar`'s offset in every CTA of `mask` when
// this thread's prior cta_group::2 MMAs complete.
__device__ __forceinline__ void umma_commit_pair(uint32_t bar, uint16_t mask) {
  asm volatile(
      "tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64"
      " [%0], %1;" ::"r"(bar),
      "h"(mask)
      : "memory");
}

// Shared-memory matrix descriptor of a K-major operand tile written by TMA
// with 128-byte swizzling: rows of 128 bytes (64 bf16), 8-row core groups
// 1024 bytes apart.  Tile bases are 1024-byte aligned.
__device__ __forceinline__ uint64_t sw128_kmajor_desc(uint32_t saddr) {
  uint64_t d = 0;
  d |= static_cast<uint64_t>((saddr & 0x3FFFFu) >> 4);  // start address
  d |= static_cast<uint64_t>(1) << 16;                    // leading offset (unused here)
  d |= static_cast<uint64_t>(1024 >> 4) << 32;            // stride offset: 8 rows x 128 B
  d |= static_cast<uint64_t>(1) << 46;                    // descriptor version (tcgen05)
  d |= static_cast<uint64_t>(2) << 61;                    // 128-byte swizzle
  return d;
}

// Instruction descriptor: kind::f16 with bf16 A/B, f32 D, both K-major,
// M = 128, N = n.
__host__ __device__ constexpr uint32_t idesc_bf16_f32(uint32_t m, uint32_t n) {
  return (1u << 4) | (1u << 7) | (1u << 10) | ((n >> 3) << 17) | ((m >> 4) << 24);
}

}  // namespace q8
