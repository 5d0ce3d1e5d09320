// q8ta_internal.h -- host-side declarations shared by the library's
// translation units (kernel launchers and the tensor-core GEMM plan).
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <cstddef>
#include <cstdint>

#include "device_common.cuh"

namespace q8 {

constexpr int64_t kTileK = 64;          // bf16 elements per 128-byte swizzled row
constexpr size_t kWorkspaceAlign = 256;

inline int64_t round_up(int64_t v, int64_t m) { return (v + m - 1) / m * m; }
inline size_t align_ws(size_t v) { return (v + kWorkspaceAlign - 1) / kWorkspaceAlign * kWorkspaceAlign; }

// Number of SMs of the current device (cached per device).
int device_sm_count();

// Launch with programmatic stream serialization (the kernel calls
// pdl_wait() before touching global memory, see device_common.cuh).
template <typename... KArgs, typename... Args>
inline cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem,
                              cudaStream_t s, Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  cudaError_t e = cudaLaunchKernelEx(&cfg, kernel, static_cast<KArgs>(args)...);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

// ---- bandwidth-bound kernels (stream_kernels.cu) --------------------------
cudaError_t launch_quantize(const float* x, int64_t numel, float inv_scale, int32_t zp, int8_t* out,
                            cudaStream_t s);
cudaError_t launch_dequantize(const int8_t* q, int64_t numel, float scale, float zp, float* out,
                              cudaStream_t s);
cudaError_t launch_gemv(const int8_t* x, int64_t K, int32_t izp, const int8_t* w, int64_t N,
                        const float* ws, const float* bias, Requant rq, int8_t* out,
                        cudaStream_t s);
// The gemv from a packed weight: reads its first round of weights before
// waiting for the previous kernel (a packed weight is never written by a
// kernel that may still be running); falls back to launch_gemv when the
// 16-byte path does not apply.
cudaError_t launch_gemv_packed(const int8_t* x, int64_t K, int32_t izp, const int8_t* w, int64_t N,
                               const float* ws, const float* bias, Requant rq, int8_t* out,
                               cudaStream_t s);
// dst[r, k] = bf16(src[r*ld + k] - zp) for k < K, 0 for K <= k < Kp.
// When bound_word is non-null, one thread also stores there the largest
// |x - zp| an int8 x can give, max(128 + zp, 127 - zp): the operand's bound
// read by the GEMM (see TcLinear::a_bound).
cudaError_t launch_rows_to_bf16(const int8_t* src, int64_t rows, int64_t K, int64_t ld, int32_t zp,
                                __nv_bfloat16* dst, int64_t Kp, cudaStream_t s,
                                int32_t* bound_word = nullptr);
// Fused quantize of fp32 rows: q = quantize(x) (written to xq when non-null)
// and dst[r, k] = bf16(q - zp), zero-padded to Kp.
cudaError_t launch_quantize_rows_bf16(const float* x, int64_t rows, int64_t K, float inv_scale,
                                      int32_t zp, int8_t* xq, __nv_bfloat16* dst, int64_t Kp,
                                      cudaStream_t s, int32_t* bound_word = nullptr);
// Channel-blocked NHWC copy for the convolutions, per group:
// dst[n][j*ICgp/64 + c/64][h][w][c%64] = bf16(x[n, j*ICg + c, h, w] - zp) for
// c < ICg in group j, 0 for ICg <= c < ICgp (ICgp = ICg rounded up to 64).
cudaError_t launch_nchw_to_nhwc_bf16(const int8_t* x, int64_t N, int64_t groups, int64_t ICg,
                                     int64_t H, int64_t W, int32_t zp, __nv_bfloat16* dst,
                                     int64_t ICgp, cudaStream_t s);
// Packed convolution weight, per group j (rows oc = j*OCg + ocl):
// dst[j][t][ic/64][ocl][ic%64] = bf16(w[oc*ldw + t*ICg + ic]) for ic < ICg, else 0.
// Largest sum of |w| over one k-block (64 input channels of one tap) of
// one output row of a rows x [taps][ICg] int8 weight (row stride ldw), into
// the device word *bound (zeroed here first).
cudaError_t launch_weight_block_bound(const int8_t* w, int64_t rows, int64_t ldw, int64_t taps,
                                      int64_t ICg, int32_t* bound, cudaStream_t s);
cudaError_t launch_conv_weight_bf16(const int8_t* w, int64_t groups, int64_t OCg, int64_t taps,
                                    int64_t ICg, int64_t ldw, __nv_bfloat16* dst, int64_t ICgp,
                                    cudaStream_t s);

// ---- tensor-core GEMM (tc_gemm.cu) -----------------------------------------
// The largest sum of |w| over one k-block (64 weights) of one row for any
// int8 weight: the chunk bound used when a weight's own bound is unknown.
constexpr int kWorstWBound = 64 * 128;

struct TcLinear {
  const __nv_bfloat16* a;  // [M, Kp] bf16, values x - input_zero_point
  const __nv_bfloat16* b;  // [N, Kp] bf16, weight values
  int64_t M, N, Kp;
  const float* ws;
  const float* bias;
  Requant rq;
  int8_t* out;       // [M, N] (or null when acc_out is set)
  int32_t* acc_out;  // [M, N] int32 debug output, or null
  // Largest |x - input_zero_point| of the operand: read on the device from
  // a_bound_dev when that is non-null (an operand prepared by an earlier
  // launch), else a_bound_host.  It sets how many k-blocks one exact f32
  // chunk may hold (255, the int8 worst case, gives 8).
  const int32_t* a_bound_dev;
  int a_bound_host;
  // Largest sum of |w| over one k-block of one weight row (a device word
  // written when the weight was packed), or null for the worst case 64 * 128.
  const int32_t* w_bound_dev;
  // Failure-detection test hooks (see TcParams): the barrier-wait time limit
  // in ns (0: the default) and a ring fill the producer skips (f + 1; 0: none).
  uint64_t wait_ns;
  int stall_fill;
  // Fused quantize -> linear (qx non-null): the kernel itself quantizes fp32
  // x [M, qK] with (qinv, qzp) into the operand `a` (and into qxq when
  // non-null) before multiplying it; qsync is the operand's trailer, which
  // q8_linear_operand_init prepared (see tc_gemm_kernel.cuh, kFusedMagic).
  const float* qx;
  int8_t* qxq;
  float qinv;
  int qzp;
  int64_t qK;
  uint32_t* qsync;
};
cudaError_t launch_tc_linear(const TcLinear& p, cudaStream_t s);
// Writes the synchronization words of a fused-quantize operand trailer.
cudaError_t launch_fused_trailer_init(uint32_t* trailer, cudaStream_t s);

struct TcConvT {
  // One group's implicit GEMM of a transposed (direct == false) or direct
  // (direct == true) convolution.
  // a: the group's first channel block in the channel-blocked NHWC copy of
  //    x - input_zero_point, [N][cb_total][H_in][W_in][64] bf16;
  // b: the group's packed weight [taps][ICp/64][OC][64] bf16.
  const __nv_bfloat16* a;
  const __nv_bfloat16* b;
  int64_t N, ICp, cb_total, H_in, W_in, OC, Kh, Kw, H_out, W_out;
  int64_t stride_h, stride_w, pad_h, pad_w, dil_h, dil_w;
  int64_t out_ch;    // channels of the output tensor (the group's OC columns start at out)
  bool direct;
  const float* ws;
  const float* bias;
  Requant rq;
  int8_t* out;       // the group's first output channel of [N, out_ch, H_out, W_out]
  int32_t* acc_out;  // int32 debug output laid out like out, or null
  int a_bound;       // largest |x - input_zero_point| (see TcLinear)
  const int32_t* w_bound;  // per-k-block weight bound on the device, or null (see TcLinear)
  // The host's copy of that bound (recorded when the weight was packed), or
  // 64 * 128, the worst case, when unknown: with it the host picks the
  // single-chunk kernel, which checks the device bound again.
  int w_bound_host;
};
cudaError_t launch_tc_conv_t(const TcConvT& p, cudaStream_t s);

// Device error word (written by kernels whose pipeline waits time out):
// its device address for the current device, and a synchronizing read.
uint32_t* device_error_word();
cudaError_t read_device_error(uint32_t* code, bool clear);

// TMA tensor map of a bf16 tensor with 128-byte swizzle (tc_gemm_host.cu).
// element_strides (optional, rank entries, 1..8): the box reads every
// element_strides[i]-th element along dimension i, box[i] / element_strides[i]
// of them, packed densely in shared memory.
bool encode_bf16_tmap(CUtensorMap* map, const void* base, int rank, const uint64_t* dims,
                      const uint64_t* strides_bytes, const uint32_t* box,
                      const uint32_t* element_strides = nullptr);

}  // namespace q8
