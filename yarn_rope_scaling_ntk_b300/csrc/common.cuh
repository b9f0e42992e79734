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

// Two float32 lanes at once (sm_100 family packed arithmetic); each lane is
// an ordinary round-to-nearest float32 fma / multiply.
__device__ __forceinline__ void fma2(float& d0, float& d1, float a0, float a1, float b0, float b1, float c0,
                                     float c1) {
  asm("{\n .reg .b64 a, b, c, d;\n mov.b64 a, {%2, %3};\n mov.b64 b, {%4, %5};\n mov.b64 c, {%6, %7};\n"
      " fma.rn.f32x2 d, a, b, c;\n mov.b64 {%0, %1}, d;\n}\n"
      : "=f"(d0), "=f"(d1)
      : "f"(a0), "f"(a1), "f"(b0), "f"(b1), "f"(c0), "f"(c1));
}
__device__ __forceinline__ void mul2(float& d0, float& d1, float a0, float a1, float b0, float b1) {
  asm("{\n .reg .b64 a, b, d;\n mov.b64 a, {%2, %3};\n mov.b64 b, {%4, %5};\n"
      " mul.rn.f32x2 d, a, b;\n mov.b64 {%0, %1}, d;\n}\n"
      : "=f"(d0), "=f"(d1)
      : "f"(a0), "f"(a1), "f"(b0), "f"(b1));
}

__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xffff0000u); }

__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi) {
  __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&v);
}

}  // namespace yr
