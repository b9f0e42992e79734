// Device helpers shared by the kernel files.
#pragma once

#include <cuda_bf16.h>
#include <stdint.h>

namespace yr {

// cos and sin of the angle m * theta for an integer position m < 2^24, with
// theta given as f = theta / (2 pi) turns per position split into f.x + f.y.
// The fractional turn is formed from the rounded product, its exact
// residual (fmaf), and the low part, so the reduction is exact up to two
// roundings of a value below one turn.
//   precise: sincospif of the reduced turn (float32 outputs)
//   fast   : __sincosf on the reduced angle in [-pi, pi] (bfloat16 outputs)
template <bool PRECISE>
__device__ __forceinline__ void turn_cos_sin(float m, float2 f, float& c, float& s) {
  const float p = m * f.x;
  const float e = fmaf(m, f.x, -p);
  float r = p - rintf(p);
  r += fmaf(m, f.y, e);
  if (PRECISE) {
    sincospif(2.0f * r, &s, &c);
  } else {
    __sincosf(r * 6.28318530717958647692f, &s, &c);
  }
}

__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xffff0000u); }

__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi) {
  __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&v);
}

}  // namespace yr
