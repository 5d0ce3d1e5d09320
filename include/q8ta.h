/*
 * q8ta.h -- C ABI of the GB300 (sm_103a) q8ta int8 quantized contraction.
 *
 * The operations follow three ExecuTorch WebGPU pull-request pages:
 *   [quantize] "Add quantize_per_tensor op (int8 buffer path)", PR #21187,
 *              Solution and Implementation paragraphs;
 *   [linear]   "Add q8ta_linear op", PR #21197, Solution, Implementation
 *              and Constraints paragraphs;
 *   [conv_t]   "Add q8ta_conv2d_transposed op (int8 transposed conv)",
 *              PR #21205, Solution, Implementation and Constraints paragraphs.
 *
 * Conventions shared by every entry point
 * ---------------------------------------
 * - Every tensor pointer is caller-owned DEVICE memory (cudaMalloc, a torch
 *   CUDA tensor, ...), unless a parameter says "host".  The library keeps
 *   no pointer after a call returns and allocates no device memory: scratch
 *   space is passed in as `workspace` (size from the matching
 *   *_workspace_bytes query).
 * - All work is enqueued on `stream` (a cudaStream_t; NULL is the legacy
 *   default stream) and is asynchronous: inputs, outputs and workspace must
 *   stay valid until the stream has passed the call.  Calls that share a
 *   workspace must be ordered on one stream.
 * - Tensors are dense, row-major (C order) unless stated.  int8 outputs are
 *   plain bytes; the pages' "4 int8 packed per 32-bit word" layout is the
 *   same memory read as little-endian words (byte j of word i is element
 *   4*i + j).
 * - Every argument check runs on the host BEFORE anything is enqueued; a
 *   failing check returns its status and launches nothing ("fail-loud" on
 *   the pages).  Q8_ERR_CUDA reports a failed launch or runtime call.
 * - Rounding is round-half-to-even everywhere.  Scales arrive as double
 *   (the schema's float); reciprocals are taken in double and cast to f32:
 *   inv_scale = (float)(1.0 / scale)                                [quantize]
 *   inv_output_scale = (float)(1.0 / output_scale)   (same convention)
 *   The dequantize/requantize epilogue is evaluated in f32, one rounding per
 *   step, in this order and without fused multiply-add:
 *     a = (float)acc; t = a * (float)input_scale; t = t * weight_scales[n];
 *     v = t + bias[n]; u = v * inv_output_scale;
 *     q = clamp(rint(u) + output_zero_point, -128, 127)        [linear]
 * - Scales must be finite and > 0; zero points must lie in [-128, 127]
 *   (they are zero points of int8 tensors); otherwise Q8_ERR_ARG.  These
 *   scalar checks are this library's own, not the pages': the pages state
 *   no range for scales or zero points.  Below, each guard list says which
 *   guards the pages state ("page") and which are this library's ("lib").
 * - Per-device state: the device error word and the scratch array of
 *   q8_linear_noalloc live in this library's device globals, whose device
 *   addresses are looked up once per device and kept for the life of the
 *   process.  Do not call the library across a cudaDeviceReset (or any
 *   other destruction of the device's primary context): the kept addresses
 *   would then be stale.
 */
#ifndef Q8TA_H_
#define Q8TA_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Same object as cudaStream_t / CUstream. */
typedef struct CUstream_st* q8_stream_t;

typedef enum q8_status {
  Q8_OK = 0,
  Q8_ERR_NULL = 1,        /* a required pointer is NULL */
  Q8_ERR_SHAPE = 2,       /* a size or shape guard failed */
  Q8_ERR_ALIGN = 3,       /* a pointer misses a documented alignment */
  Q8_ERR_UNSUPPORTED = 4, /* activation other than "none"/"relu", dilation or
                             groups < 1, conv2d stride > 8 */
  Q8_ERR_WORKSPACE = 5,   /* workspace NULL or smaller than required */
  Q8_ERR_CUDA = 6,        /* a CUDA runtime call or kernel launch failed */
  Q8_ERR_DEVICE = 7,      /* a kernel raised the library's device error word */
  Q8_ERR_ARG = 8          /* a scalar argument is out of range */
} q8_status;

/* Static, human-readable name of a status code (never NULL). */
const char* q8_status_string(int status);

/* Library ABI version, currently 1. */
int q8_version(void);

/*
 * Device error word.  Kernels that wait on pipeline barriers give every wait
 * a time limit (about one second); on expiry they record a code here, stop
 * issuing work and return, leaving the CUDA context usable (codes 0x101 ..
 * 0x106: which wait ran out).  Code 0x107: a convolution launched from a
 * packed weight whose buffer was rewritten after packing (the host's copy of
 * its k-block bound no longer held); that launch wrote nothing.  Codes
 * 0x108 / 0x109: q8_quantize_linear_fused waited too long for an operand
 * chunk / met an operand trailer that q8_linear_operand_init never prepared.  This call
 * synchronizes the current device, copies the word to *code (host pointer)
 * and, if clear != 0, resets it to 0.  Q8_OK is returned when the copy
 * succeeded, whatever the word holds.
 */
q8_status q8_device_error(uint32_t* code, int clear);

/* ------------------------------------------------------------------------ */
/* quantize_per_tensor: fp32 -> int8                               [quantize] */
/* ------------------------------------------------------------------------ */
/*
 * out[i] = clamp(rint(x[i] * inv_scale) + zero_point, -128, 127).
 * x: float32[numel]; out: int8[numel].
 * Guards: page -- x, out non-NULL; numel % 4 == 0 (the page's packed-word
 * binding; [quantize] Implementation).  lib -- numel >= 0 (0 is a no-op,
 * and then the pointers may be NULL); the scale and zero-point ranges.
 */
q8_status q8_quantize_per_tensor(const float* x, int64_t numel, double scale,
                                 int32_t zero_point, int8_t* out, q8_stream_t stream);

/*
 * dequantize_per_tensor: int8 -> fp32, the op that closes the
 * quantize -> q8ta_* -> dequantize subgraph named in the Problem paragraphs
 * of [linear] and [conv_t].  out[i] = ((float)q[i] - (float)zero_point) *
 * (float)scale, one f32 rounding per step.  Same guards as quantize (the
 * pages print no guard for this op; numel % 4 mirrors quantize's).
 */
q8_status q8_dequantize_per_tensor(const int8_t* q, int64_t numel, double scale,
                                   int32_t zero_point, float* out, q8_stream_t stream);

/* ------------------------------------------------------------------------ */
/* q8ta_linear / q8ta_linear_gemv                                   [linear] */
/* ------------------------------------------------------------------------ */
/*
 * acc[m,n] = sum_k (x[m,k] - input_zero_point) * weight[n,k]   (exact int32,
 * wrapping modulo 2^32), then the epilogue above with weight_scales[n] and
 * bias[n]; out[m,n] int8.
 *   x             int8 [M, K] row-major
 *   weight        int8 [N, K] row-major (per-output-channel symmetric)
 *   weight_sums   accepted and ignored (the pages fold the zero point per
 *                 element instead of using precomputed sums); may be NULL
 *   weight_scales float [>= N]; only [0, N) is read
 *   bias          float [>= N] or NULL (= zero bias)
 *   activation    host C string: "none", or "relu" (the page's follow-up:
 *                 the dequantized value is raised to 0 before the
 *                 requantization, i.e. out = max(out, output_zero_point));
 *                 anything else gives Q8_ERR_UNSUPPORTED
 *   out           int8 [M, N] row-major
 * Guards: page ([linear] Implementation) -- N % 4 == 0, (M*K) % 4 == 0,
 * (N*K) % 4 == 0, activation "none" (the page's fail-loud follow-up "relu"
 * is supported here instead of refused), and for q8_linear_gemv M == 1.
 * lib -- M, N, K >= 1; M, N <= INT32_MAX and K <= INT32_MAX / 2 (32-bit
 * tile coordinates); no product of two sizes overflows int64; the scale
 * and zero-point ranges.
 *
 * The contraction runs on the tcgen05 tensor cores with bf16 operands that
 * hold the int8 values exactly; workspace holds the bf16 operand copies:
 * q8_linear_workspace_bytes(M, K, N) bytes, 256-byte aligned.  When
 * M == 1 the bandwidth-bound gemv kernel runs instead and workspace may be
 * NULL (the query returns 0).
 */
size_t q8_linear_workspace_bytes(int64_t M, int64_t K, int64_t N);
q8_status q8_linear(const int8_t* x, int64_t M, int64_t K, double input_scale,
                    int32_t input_zero_point, const int8_t* weight, int64_t N,
                    const int32_t* weight_sums, const float* weight_scales, const float* bias,
                    double output_scale, int32_t output_zero_point, const char* activation,
                    int8_t* out, void* workspace, size_t workspace_bytes, q8_stream_t stream);

/*
 * q8_linear without any allocation or workspace: the pages have no
 * counterpart; this entry point exists for callers that cannot allocate
 * device memory where they run the layer (a plugin whose host runtime owns
 * the device memory pool and forbids cudaMalloc, a latency-critical loop
 * that cannot afford cudaMalloc/cudaFree, a deployment whose memory budget
 * is fixed at start-up).  Same arguments, guards and results as q8_linear,
 * minus the workspace.  The scratch is a library-owned device array of
 * Q8_LINEAR_NOALLOC_SCRATCH_BYTES (16 MiB) that every GPU loading this
 * library holds until the process exits; no call allocates or frees memory.
 *   - Limit: 2*(M + N)*ceil64(K) bytes (each half rounded up to 256) must fit
 *     the array, else Q8_ERR_WORKSPACE and nothing is launched.  M == 1 uses
 *     no scratch (the gemv kernel) and has no such limit.
 *   - The first call on each device looks up the array's device address
 *     (once per device, with that device current); make that first call
 *     before any stream capture.
 *   - All calls on a device share the one array, which keeps the last
 *     call's contents (nothing in it needs to start at zero).  Calls whose
 *     work overlaps on the GPU (other streams, other host threads) race on
 *     it: order them on one stream.
 */
#define Q8_LINEAR_NOALLOC_SCRATCH_BYTES (16u * 1024u * 1024u)
q8_status q8_linear_noalloc(const int8_t* x, int64_t M, int64_t K, double input_scale,
                            int32_t input_zero_point, const int8_t* weight, int64_t N,
                            const int32_t* weight_sums, const float* weight_scales,
                            const float* bias, double output_scale, int32_t output_zero_point,
                            const char* activation, int8_t* out, q8_stream_t stream);

/* The M == 1 case with the identical schema; returns Q8_ERR_SHAPE unless
 * M == 1.  Needs no workspace (pass NULL, 0). */
q8_status q8_linear_gemv(const int8_t* x, int64_t M, int64_t K, double input_scale,
                         int32_t input_zero_point, const int8_t* weight, int64_t N,
                         const int32_t* weight_sums, const float* weight_scales,
                         const float* bias, double output_scale, int32_t output_zero_point,
                         const char* activation, int8_t* out, void* workspace,
                         size_t workspace_bytes, q8_stream_t stream);

/*
 * The gemv from a packed weight (decode-shaped layers, whose weights are
 * constants): q8_linear_gemv_pack_weight copies the int8 [N, K] weight into
 * `packed` (q8_linear_gemv_packed_weight_bytes(N, K) bytes, 256-byte
 * aligned, owned by the caller) and waits for the copy (load time).  A packed
 * buffer is rewritten only by packing into it again.  q8_linear_gemv_packed
 * then computes exactly what q8_linear_gemv computes, but reads its first
 * 4 KB of each weight row before waiting for the previous kernel on the
 * stream (which never writes a packed weight), so that in a run of layers
 * each layer's weight streams in while the previous layer runs.  x is int8
 * [1, K].  Guards: those of q8_linear_gemv.
 */
size_t q8_linear_gemv_packed_weight_bytes(int64_t N, int64_t K);
q8_status q8_linear_gemv_pack_weight(const int8_t* weight, int64_t N, int64_t K, void* packed,
                                     size_t packed_bytes, q8_stream_t stream);
q8_status q8_linear_gemv_packed(const int8_t* x, int64_t K, double input_scale,
                                int32_t input_zero_point, const void* packed_weight, int64_t N,
                                const float* weight_scales, const float* bias, double output_scale,
                                int32_t output_zero_point, const char* activation, int8_t* out,
                                q8_stream_t stream);

/*
 * Load-time weight packing.  A linear layer's weight is a constant, so the
 * bf16 copy the tensor cores read can be made once:
 *   q8_linear_pack_weight writes q8_linear_packed_weight_bytes(N, K) bytes
 *   (256-byte aligned buffer) from the int8 [N, K] weight: the bf16 rows,
 *   then a 256-byte trailer whose first int32 is the largest sum of |w| over
 *   64 consecutive weights of one row (the kernels size their exact f32
 *   partial sums from it; results never depend on it).
 * Results of every *_packed call are identical to q8_linear.
 */
size_t q8_linear_packed_weight_bytes(int64_t N, int64_t K);
q8_status q8_linear_pack_weight(const int8_t* weight, int64_t N, int64_t K, void* packed,
                                size_t packed_bytes, q8_stream_t stream);

/*
 * The activation operand: the bf16 copy of x - input_zero_point that the
 * tensor cores read, q8_linear_operand_bytes(M, K) bytes (256-byte aligned).
 *   q8_linear_prepare_operand      from int8 x [M, K];
 *   q8_quantize_to_linear_operand  from fp32 x [M, K]: quantize_per_tensor
 *       with (input_scale, input_zero_point) exactly as
 *       q8_quantize_per_tensor does, fused with the operand preparation
 *       (the pages' quantize -> q8ta_linear subgraph); x_q (int8 [M, K],
 *       may be NULL) receives the quantized activations.
 *   q8_linear_operand_packed       runs the contraction and the epilogue
 *       from a prepared operand and a packed weight (one kernel).
 * Guards: those of q8_linear (and of quantize for the fp32 form).
 */
size_t q8_linear_operand_bytes(int64_t M, int64_t K);
q8_status q8_linear_prepare_operand(const int8_t* x, int64_t M, int64_t K,
                                    int32_t input_zero_point, void* operand,
                                    size_t operand_bytes, q8_stream_t stream);
q8_status q8_quantize_to_linear_operand(const float* x_f32, int64_t M, int64_t K,
                                        double input_scale, int32_t input_zero_point,
                                        int8_t* x_q, void* operand, size_t operand_bytes,
                                        q8_stream_t stream);
q8_status q8_linear_operand_packed(const void* operand, int64_t M, int64_t K, double input_scale,
                                   const void* packed_weight, int64_t N,
                                   const float* weight_scales, const float* bias,
                                   double output_scale, int32_t output_zero_point,
                                   const char* activation, int8_t* out, q8_stream_t stream);

/* Convenience forms: prepare the operand into `workspace`
 * (q8_linear_operand_bytes(M, K) bytes), then q8_linear_operand_packed. */
q8_status q8_linear_packed(const int8_t* x, int64_t M, int64_t K, double input_scale,
                           int32_t input_zero_point, const void* packed_weight, int64_t N,
                           const float* weight_scales, const float* bias, double output_scale,
                           int32_t output_zero_point, const char* activation, int8_t* out,
                           void* workspace, size_t workspace_bytes, q8_stream_t stream);
q8_status q8_quantize_linear_packed(const float* x_f32, int64_t M, int64_t K, double input_scale,
                                    int32_t input_zero_point, const void* packed_weight,
                                    int64_t N, const float* weight_scales, const float* bias,
                                    double output_scale, int32_t output_zero_point,
                                    const char* activation, int8_t* x_q, int8_t* out,
                                    void* workspace, size_t workspace_bytes, q8_stream_t stream);

/*
 * Fused quantize -> q8ta_linear in ONE kernel (the pages' delegated
 * quantize_per_tensor -> q8ta_linear subgraph, [linear] Problem paragraph):
 * the GEMM's own warps quantize fp32 x [M, K] exactly as
 * q8_quantize_per_tensor does (input_scale, input_zero_point), write x_q
 * (int8 [M, K], may be NULL) and the bf16 operand into `operand`, chunk by
 * chunk along K, and the tensor cores start on each chunk as soon as every
 * CTA has written its share of it.  Results equal q8_quantize_linear_packed.
 *   operand: q8_linear_operand_bytes(M, K) bytes, 256-byte aligned, whose
 *     trailer q8_linear_operand_init prepared once (before the first fused
 *     call on it; each call leaves it ready for the next).  A buffer that
 *     was never initialized runs nothing and sets device error 0x109.
 *   Calls sharing an operand buffer must be ordered on one stream.
 * The kernel's CTAs wait on one another (bounded, device error 0x108 on
 * expiry): its persistent grid is sized to fit the GPU at once, so do not
 * run other long-lived kernels concurrently on the same GPU.
 * Guards: those of q8_quantize_linear_packed.
 */
q8_status q8_linear_operand_init(void* operand, int64_t M, int64_t K, size_t operand_bytes,
                                 q8_stream_t stream);
q8_status q8_quantize_linear_fused(const float* x_f32, int64_t M, int64_t K, double input_scale,
                                   int32_t input_zero_point, const void* packed_weight, int64_t N,
                                   const float* weight_scales, const float* bias,
                                   double output_scale, int32_t output_zero_point,
                                   const char* activation, int8_t* x_q, int8_t* out,
                                   void* operand, size_t operand_bytes, q8_stream_t stream);

/* Test and debugging form of q8_linear_packed: writes the exact int32
 * accumulators acc[m,n] (int32 [M, N]) instead of the int8 output. */
q8_status q8_linear_packed_acc32(const int8_t* x, int64_t M, int64_t K, int32_t input_zero_point,
                                 const void* packed_weight, int64_t N, int32_t* acc,
                                 void* workspace, size_t workspace_bytes, q8_stream_t stream);

/*
 * Failure-detection test hook (no counterpart on the pages).  Runs
 * q8_linear_packed_acc32 with every pipeline-barrier wait limited to
 * wait_limit_ns (1 ms .. 1 s; else Q8_ERR_ARG) and with the kernel's TMA
 * producer leaving out its skip_fill-th ring fill (0-based), so that the
 * matching wait runs out.  The kernel then records a code in the device
 * error word (0x101 .. 0x106, q8_device_error), stops, waits (bounded) for
 * its own copies and tensor-core work in flight, frees its tensor memory
 * and returns: nothing hangs and the CUDA context stays usable.  acc is
 * left partly written.  For tests only.
 */
q8_status q8_debug_linear_packed_stall(const int8_t* x, int64_t M, int64_t K,
                                       int32_t input_zero_point, const void* packed_weight,
                                       int64_t N, int32_t* acc, void* workspace,
                                       size_t workspace_bytes, uint64_t wait_limit_ns,
                                       int64_t skip_fill, q8_stream_t stream);

/* ------------------------------------------------------------------------ */
/* q8ta_conv2d_transposed                                            [conv_t] */
/* ------------------------------------------------------------------------ */
typedef struct q8_conv2d_transposed_shape {
  int64_t N, IC, H_in, W_in;          /* x      int8 [N, IC, H_in, W_in] (NCHW) */
  int64_t OC, Kh, Kw;                 /* weight int8 [OC, weight_row_stride]    */
  int64_t weight_row_stride;          /* >= Kh*Kw*IC/groups (tolerates padding) */
  int64_t H_out, W_out;               /* out    int8 [N, OC, H_out, W_out]      */
  int64_t stride_h, stride_w;         /* >= 1                                   */
  int64_t pad_h, pad_w;               /* >= 0                                   */
  int64_t output_padding_h, output_padding_w; /* accepted, unused: the output
                                         size is H_out/W_out as given           */
  int64_t dilation_h, dilation_w;     /* >= 1                                   */
  int64_t groups;                     /* >= 1, divides IC and OC                */
} q8_conv2d_transposed_shape;

/*
 * For every output (n, oc, oh, ow), with group j = oc / (OC/groups) and
 * ICg = IC/groups:
 *   acc = sum over icl < ICg, kh, kw of
 *         (x[n, j*ICg + icl, ih, iw] - input_zero_point) *
 *         weight[oc, (kh*Kw + kw)*ICg + icl]
 * where ih = (oh + pad_h - kh*dilation_h) / stride_h is used only when the
 * numerator is >= 0, divisible by stride_h and ih < H_in (iw likewise); taps
 * that fail contribute nothing.  Then the epilogue above with
 * weight_scales[oc] and bias[oc] (arrays of length >= OC; only [0, OC) is
 * read).  For groups == 1 the weight layout is the page's reshape
 * weight[oc, (kh*Kw+kw)*IC + ic] = original[ic, oc, kh, kw]; group j of a
 * grouped weight holds original[j*ICg + icl, oc - j*OC/groups, kh, kw].
 * Guards: page ([conv_t] Implementation) -- stride >= 1, W_out % 4 == 0,
 * weight_row_stride >= Kh*Kw*IC/groups, activation "none"; the page's
 * fail-loud follow-ups (activation "relu", groups != 1, dilation != 1) are
 * supported here: activation "none" or "relu", groups dividing IC and OC,
 * dilation >= 1.  lib -- every size >= 1, pad >= 0, the scale and
 * zero-point ranges.  weight_sums is accepted and ignored.
 * workspace: q8_conv2d_transposed_workspace_bytes(shape) bytes, 256-byte
 * aligned (an NHWC bf16 copy of x - input_zero_point, channels padded per
 * group to a multiple of 64, then the packed weight); the size functions
 * return 0 when a shape guard fails.
 */
size_t q8_conv2d_transposed_workspace_bytes(const q8_conv2d_transposed_shape* shape);
q8_status q8_conv2d_transposed(const int8_t* x, const q8_conv2d_transposed_shape* shape,
                               double input_scale, int32_t input_zero_point,
                               const int8_t* weight, const int32_t* weight_sums,
                               const float* weight_scales, const float* bias,
                               double output_scale, int32_t output_zero_point,
                               const char* activation, int8_t* out, void* workspace,
                               size_t workspace_bytes, q8_stream_t stream);

/* Test and debugging form: writes the exact int32 accumulators
 * acc int32 [N, OC, H_out, W_out] instead of the int8 output. */
q8_status q8_conv2d_transposed_acc32(const int8_t* x, const q8_conv2d_transposed_shape* shape,
                                     int32_t input_zero_point, const int8_t* weight,
                                     int32_t* acc, void* workspace, size_t workspace_bytes,
                                     q8_stream_t stream);

/* Packed-weight form, for weights that are fixed across calls (the page's
 * weight arrives ahead of time, reshaped):
 *   q8_conv2d_transposed_pack_weight writes the weight's tensor-core layout
 *     (bf16, per group [taps][IC/64][OC/groups][64]) into `packed`
 *     (q8_conv2d_transposed_packed_weight_bytes(shape) bytes, 256-byte
 *     aligned, owned by the caller), followed by a 256-byte trailer whose
 *     first int32 is the largest sum of |w| over 64 input channels of one
 *     tap of one output channel: the kernels size their exact f32 partial
 *     sums from it (with |x - input_zero_point|), so results never depend
 *     on it.  The call waits for the packing to finish (load time) and keeps
 *     a host copy of that bound for the buffer, from which launches pick the
 *     kernel; rewrite a packed buffer only by packing into it again;
 *   q8_conv2d_transposed_packed runs the op from it; its workspace holds only
 *     the input copy (q8_conv2d_transposed_packed_workspace_bytes(shape));
 *   q8_conv2d_transposed_packed_acc32 writes the exact int32 accumulators
 *     (as q8_conv2d_transposed_acc32) from it, same workspace.
 * Guards: those of q8_conv2d_transposed. */
size_t q8_conv2d_transposed_packed_weight_bytes(const q8_conv2d_transposed_shape* shape);
size_t q8_conv2d_transposed_packed_workspace_bytes(const q8_conv2d_transposed_shape* shape);
q8_status q8_conv2d_transposed_pack_weight(const int8_t* weight,
                                           const q8_conv2d_transposed_shape* shape, void* packed,
                                           size_t packed_bytes, q8_stream_t stream);
q8_status q8_conv2d_transposed_packed(const int8_t* x, const q8_conv2d_transposed_shape* shape,
                                      double input_scale, int32_t input_zero_point,
                                      const void* packed_weight, const float* weight_scales,
                                      const float* bias, double output_scale,
                                      int32_t output_zero_point, const char* activation,
                                      int8_t* out, void* workspace, size_t workspace_bytes,
                                      q8_stream_t stream);
q8_status q8_conv2d_transposed_packed_acc32(const int8_t* x,
                                            const q8_conv2d_transposed_shape* shape,
                                            int32_t input_zero_point, const void* packed_weight,
                                            int32_t* acc, void* workspace, size_t workspace_bytes,
                                            q8_stream_t stream);

/* ------------------------------------------------------------------------ */
/* q8ta_conv2d (direct convolution)                                   [conv] */
/* ------------------------------------------------------------------------ */
/* The general int8 convolution whose scaffold and [OC, Kh*Kw*IC] weight
 * layout the transposed convolution reuses ("Add q8ta_conv2d_transposed op",
 * Problem and Solution paragraphs). */
typedef struct q8_conv2d_shape {
  int64_t N, IC, H_in, W_in;          /* x      int8 [N, IC, H_in, W_in] (NCHW) */
  int64_t OC, Kh, Kw;                 /* weight int8 [OC, weight_row_stride]    */
  int64_t weight_row_stride;          /* >= Kh*Kw*IC/groups                     */
  int64_t H_out, W_out;               /* out    int8 [N, OC, H_out, W_out]      */
  int64_t stride_h, stride_w;         /* 1 .. 8                                 */
  int64_t pad_h, pad_w;               /* >= 0                                   */
  int64_t dilation_h, dilation_w;     /* >= 1                                   */
  int64_t groups;                     /* >= 1, divides IC and OC                */
} q8_conv2d_shape;

/*
 * For every output (n, oc, oh, ow), with group j = oc / (OC/groups) and
 * ICg = IC/groups:
 *   acc = sum over icl < ICg, kh, kw of
 *         (x[n, j*ICg + icl, ih, iw] - input_zero_point) *
 *         weight[oc, (kh*Kw + kw)*ICg + icl]
 * with ih = oh*stride_h - pad_h + kh*dilation_h, the tap used only when
 * 0 <= ih < H_in (iw likewise); weight[oc, (kh*Kw+kw)*ICg + icl] =
 * original[oc, icl, kh, kw].  Then the shared epilogue with per-oc scales.
 * H_out and W_out are the caller's (normally (H_in + 2*pad_h -
 * dilation_h*(Kh-1) - 1) / stride_h + 1); outputs whose window lies wholly
 * in the padding hold the requantized bias.
 * Guards: as q8_conv2d_transposed (the pages name this op but print no
 * guard of its own), plus lib -- stride_h, stride_w <= 8
 * (Q8_ERR_UNSUPPORTED above: the input is read through TMA boxes with
 * element strides).  Workspace and packed forms as for the transposed op.
 */
size_t q8_conv2d_workspace_bytes(const q8_conv2d_shape* shape);
q8_status q8_conv2d(const int8_t* x, const q8_conv2d_shape* shape, double input_scale,
                    int32_t input_zero_point, const int8_t* weight, const float* weight_scales,
                    const float* bias, double output_scale, int32_t output_zero_point,
                    const char* activation, int8_t* out, void* workspace, size_t workspace_bytes,
                    q8_stream_t stream);
q8_status q8_conv2d_acc32(const int8_t* x, const q8_conv2d_shape* shape, int32_t input_zero_point,
                          const int8_t* weight, int32_t* acc, void* workspace,
                          size_t workspace_bytes, q8_stream_t stream);
size_t q8_conv2d_packed_weight_bytes(const q8_conv2d_shape* shape);
size_t q8_conv2d_packed_workspace_bytes(const q8_conv2d_shape* shape);
q8_status q8_conv2d_pack_weight(const int8_t* weight, const q8_conv2d_shape* shape, void* packed,
                                size_t packed_bytes, q8_stream_t stream);
q8_status q8_conv2d_packed(const int8_t* x, const q8_conv2d_shape* shape, double input_scale,
                           int32_t input_zero_point, const void* packed_weight,
                           const float* weight_scales, const float* bias, double output_scale,
                           int32_t output_zero_point, const char* activation, int8_t* out,
                           void* workspace, size_t workspace_bytes, q8_stream_t stream);
q8_status q8_conv2d_packed_acc32(const int8_t* x, const q8_conv2d_shape* shape,
                                 int32_t input_zero_point, const void* packed_weight, int32_t* acc,
                                 void* workspace, size_t workspace_bytes, q8_stream_t stream);

#ifdef __cplusplus
}
#endif
#endif /* Q8TA_H_ */
