// api_common.h -- host-side helpers shared by the extern "C" entry points
// (api.cu, api_conv.cu, noalloc.cu): argument checks, the f32 reciprocal,
// the activation string, the epilogue constants.
#pragma once

#include <cuda_runtime.h>

#include <algorithm>
#include <cmath>
#include <cstdint>
#include <cstring>

#include "q8ta.h"
#include "q8ta_internal.h"

namespace q8api {

inline cudaStream_t cs(q8_stream_t s) { return reinterpret_cast<cudaStream_t>(s); }

inline q8_status cuda_status(cudaError_t e) { return e == cudaSuccess ? Q8_OK : Q8_ERR_CUDA; }

inline bool scale_ok(double s) { return std::isfinite(s) && s > 0.0; }
inline bool zp_ok(int32_t z) { return z >= -128 && z <= 127; }
inline bool mul_ok(int64_t a, int64_t b) { return a == 0 || b <= INT64_MAX / a; }

// (float)(1.0 / scale): the reciprocal in double, then one rounding to f32
// ("Add quantize_per_tensor op", Solution paragraph).
inline float recip_f32(double scale) { return static_cast<float>(1.0 / scale); }

// The activation string: "none" -> 0, "relu" -> 1, anything else -> -1.
// ("Add q8ta_linear op", Implementation paragraph, reads it as a string and
// names the relu-fused form as its follow-up.)
inline int parse_activation(const char* a) {
  if (a == nullptr) return -1;
  if (std::strcmp(a, "none") == 0) return 0;
  if (std::strcmp(a, "relu") == 0) return 1;
  return -1;
}

// Epilogue constants.  relu: the dequantized value is raised to 0 before the
// requantization, which is the output floor max(q, ozp).
inline q8::Requant make_rq(double input_scale, double output_scale, int32_t ozp, int relu) {
  q8::Requant r;
  r.s_in = static_cast<float>(input_scale);
  r.inv_out = recip_f32(output_scale);
  r.ozp = static_cast<float>(ozp);
  r.ozp_i = ozp;
  r.lo = relu ? ozp : -128;
  r.lo_f = static_cast<float>(r.lo - ozp);
  r.hi_f = static_cast<float>(127 - ozp);
  return r;
}

// Largest |x - zp| over int8 x.
inline int a_bound_of(int32_t zp) { return std::max(128 + zp, 127 - zp); }

}  // namespace q8api
