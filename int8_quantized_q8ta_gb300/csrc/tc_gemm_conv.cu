// tc_gemm_conv.cu -- q8ta_conv2d_transposed on the tensor-core GEMM
// (tc_gemm_kernel.cuh): per-stride-phase implicit GEMM over the
// channel-blocked NHWC copy of x - input_zero_point, read through 5-D TMA
// boxes whose zero fill implements the skipped taps.  One launch per group.
// More than 64 output channels per group: 128 channels x 256 pixels per tile
// (exchanged operands, MODE 3); otherwise 128 pixels x 64..256 channels.
#include <cuda.h>
#include <cuda_runtime.h>

#include "q8ta_internal.h"
#include "tc_gemm_conv_setup.cuh"

namespace q8 {

cudaError_t launch_tc_conv2d(const TcConvT& C, cudaStream_t s);  // tc_gemm_conv2d.cu

cudaError_t launch_tc_conv_t(const TcConvT& C, cudaStream_t s) {
  if (C.direct) return launch_tc_conv2d(C, s);
  ConvSetup S;
  if (!conv_setup(C, S)) return cudaErrorInvalidValue;
  if (S.p.total_units == 0) return cudaSuccess;
  // one CTA per tile: on the transposed-convolution workload the 2-SM MMA
  // measured no faster (its k-blocks are short and many)
  if (S.pixn) {
    if (S.kd != 1) return cudaErrorInvalidValue;
    return S.single ? launch_tc_kernel<kPixTile, 16, 5, 1, 1>(S.ma, S.mb, S.p, s)
                    : launch_tc_kernel<kPixTile, 16, 3, 1, 1>(S.ma, S.mb, S.p, s);
  }
  switch (S.bn * 4 + S.kd) {
    case 64 * 4 + 1: return launch_tc_kernel<64, 16, 1, 1, 1>(S.ma, S.mb, S.p, s);
    case 64 * 4 + 2: return launch_tc_kernel<64, 16, 1, 2, 1>(S.ma, S.mb, S.p, s);
    case 128 * 4 + 1: return launch_tc_kernel<128, 16, 1, 1, 1>(S.ma, S.mb, S.p, s);
    case 128 * 4 + 2: return launch_tc_kernel<128, 16, 1, 2, 1>(S.ma, S.mb, S.p, s);
    case 256 * 4 + 1: return launch_tc_kernel<256, 8, 1, 1, 1>(S.ma, S.mb, S.p, s);
    default: return launch_tc_kernel<256, 8, 1, 2, 1>(S.ma, S.mb, S.p, s);
  }
}

}  // namespace q8
