// One rotary pair of the partial interleaved RoPE ("glm52-mla.ts",
// partialInterleavedRopeMlx), shared by the RoPE kernel and the fused
// RoPE + absorb kernel.  The angle is f32(p * invf_j), the exact product
// rounded once (the page forms it in f64 and rounds with fround); sin/cos are
// CUDA's accurate sincosf of that f32 angle.
#pragma once

#include <stdint.h>

namespace mla {

// f32(pos * inv_freq), the exact product rounded once.  While |pos| <= 2^24
// the position is an exact f32 and the f32 product is already that rounding
// (the exact product of two f32 values fits a double, so both routes round the
// same real number); beyond, the product is formed in double.
__device__ __forceinline__ float rope_angle(int64_t pos, float inv_freq) {
  if (pos >= -(1LL << 24) && pos <= (1LL << 24)) return __fmul_rn((float)pos, inv_freq);
  return __double2float_rn((double)pos * (double)inv_freq);
}

__device__ __forceinline__ void rope_rotate_pair(float a, float b, int64_t pos, float inv_freq, float& re,
                                                 float& im) {
  const float ang = rope_angle(pos, inv_freq);
  float s, c;
  sincosf(ang, &s, &c);
  re = a * c - b * s;
  im = b * c + a * s;
}

}  // namespace mla
