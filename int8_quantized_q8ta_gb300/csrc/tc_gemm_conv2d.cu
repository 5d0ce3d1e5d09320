// tc_gemm_conv2d.cu -- q8ta_conv2d (the direct convolution) on the
// tensor-core GEMM (tc_gemm_kernel.cuh): an implicit GEMM over 128-pixel
// output tiles whose input taps are 5-D TMA boxes with element strides
// (stride_w, stride_h), starting at (ow*stride_w - pad_w + kw*dil_w, ...);
// the boxes' zero fill covers the padding.  One launch per group.  More
// than 64 output channels per group: 128 channels x 256 pixels per tile
// (exchanged operands, MODE 4).
#include <cuda.h>
#include <cuda_runtime.h>

#include "q8ta_internal.h"
#include "tc_gemm_conv_setup.cuh"

namespace q8 {

cudaError_t launch_tc_conv2d(const TcConvT& C, cudaStream_t s) {
  ConvSetup S;
  if (!conv_setup(C, S)) return cudaErrorInvalidValue;
  if (S.p.total_units == 0) return cudaSuccess;
  if (S.pixn) {
    if (S.kd != 1) return cudaErrorInvalidValue;
    return S.single ? launch_tc_kernel<kPixTile, 16, 6, 1, 1>(S.ma, S.mb, S.p, s)
                    : launch_tc_kernel<kPixTile, 16, 4, 1, 1>(S.ma, S.mb, S.p, s);
  }
  switch (S.bn * 4 + S.kd) {
    case 64 * 4 + 1: return launch_tc_kernel<64, 16, 2, 1, 1>(S.ma, S.mb, S.p, s);
    case 64 * 4 + 2: return launch_tc_kernel<64, 16, 2, 2, 1>(S.ma, S.mb, S.p, s);
    case 128 * 4 + 1: return launch_tc_kernel<128, 16, 2, 1, 1>(S.ma, S.mb, S.p, s);
    case 128 * 4 + 2: return launch_tc_kernel<128, 16, 2, 2, 1>(S.ma, S.mb, S.p, s);
    case 256 * 4 + 1: return launch_tc_kernel<256, 8, 2, 1, 1>(S.ma, S.mb, S.p, s);
    default: return launch_tc_kernel<256, 8, 2, 2, 1>(S.ma, S.mb, S.p, s);
  }
}

}  // namespace q8
