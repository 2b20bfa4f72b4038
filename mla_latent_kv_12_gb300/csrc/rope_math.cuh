// One rotary pair of the partial interleaved RoPE ("glm52-mla.ts",
// partialInterleavedRopeMlx), shared by the RoPE kernel and the fused
// RoPE + absorb kernel.  The angle is f32(p * invf_j), formed exactly in double
// and rounded once (the page forms it in f64 and rounds with fround); sin/cos
// are CUDA's accurate sincosf of that f32 angle.
#pragma once

#include <stdint.h>

namespace mla {

__device__ __forceinline__ void rope_rotate_pair(float a, float b, int64_t pos, float inv_freq, float& re,
                                                 float& im) {
  const float ang = __double2float_rn((double)pos * (double)inv_freq);
  float s, c;
  sincosf(ang, &s, &c);
  re = a * c - b * s;
  im = b * c + a * s;
}

}  // namespace mla
