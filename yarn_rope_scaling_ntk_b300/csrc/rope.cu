// rope_apply: rotate every pair (x_i, x_{i+d/2}) of a [B, H, S, d] tensor by
// m * theta'_i ("Context Window Scaling ...", Section 2, Formal RoPE
// Mechanics; rotate-half pairing as in that section's listing).  The same
// kernel, with a bfloat16 output, prepares the rotated operands of the
// attention entry point.
//
// Memory-bound: each thread owns VEC pairs of one row -- one 16-byte vector
// from the first half and one from the second half -- and keeps its VEC
// frequencies in registers while it strides over rows.
#include <algorithm>

#include "common.cuh"
#include "internal.h"

namespace yr {
namespace {

template <typename T> struct Vec;
template <> struct Vec<float> { static constexpr int N = 4; };
template <> struct Vec<__nv_bfloat16> { static constexpr int N = 8; };

template <typename T, int N>
__device__ __forceinline__ void load_vec(const T* p, float (&v)[N]);

template <>
__device__ __forceinline__ void load_vec<float, 4>(const float* p, float (&v)[4]) {
  const float4 t = *reinterpret_cast<const float4*>(p);
  v[0] = t.x; v[1] = t.y; v[2] = t.z; v[3] = t.w;
}
template <>
__device__ __forceinline__ void load_vec<float, 8>(const float* p, float (&v)[8]) {
  const float4 a = reinterpret_cast<const float4*>(p)[0];
  const float4 b = reinterpret_cast<const float4*>(p)[1];
  v[0] = a.x; v[1] = a.y; v[2] = a.z; v[3] = a.w; v[4] = b.x; v[5] = b.y; v[6] = b.z; v[7] = b.w;
}
template <>
__device__ __forceinline__ void load_vec<__nv_bfloat16, 8>(const __nv_bfloat16* p, float (&v)[8]) {
  const uint4 t = *reinterpret_cast<const uint4*>(p);
  v[0] = bf16_lo(t.x); v[1] = bf16_hi(t.x); v[2] = bf16_lo(t.y); v[3] = bf16_hi(t.y);
  v[4] = bf16_lo(t.z); v[5] = bf16_hi(t.z); v[6] = bf16_lo(t.w); v[7] = bf16_hi(t.w);
}

template <typename T, int N>
__device__ __forceinline__ void store_vec(T* p, const float (&v)[N]);

template <>
__device__ __forceinline__ void store_vec<float, 4>(float* p, const float (&v)[4]) {
  *reinterpret_cast<float4*>(p) = make_float4(v[0], v[1], v[2], v[3]);
}
template <>
__device__ __forceinline__ void store_vec<__nv_bfloat16, 8>(__nv_bfloat16* p, const float (&v)[8]) {
  *reinterpret_cast<uint4*>(p) =
      make_uint4(pack_bf16(v[0], v[1]), pack_bf16(v[2], v[3]), pack_bf16(v[4], v[5]), pack_bf16(v[6], v[7]));
}

// Plain (coherent) loads: y may alias x, each element read then written by
// the same thread.
//
// One thread: pairs [c*VEC, c*VEC + VEC) of rows r, r + rows_per_pass, ...
// VEC is the output vector width (8 for bf16 out, 4 for f32 out); float32
// inputs converted to bf16 read two float4 per half.
template <typename Tin, typename Tout, bool PRECISE>
__global__ void __launch_bounds__(256) rope_kernel(RopeLaunch a, RopeFreqs f) {
  constexpr int VEC = Vec<Tout>::N;
  const int half = a.d >> 1;
  const int tpr = half / VEC;  // threads per row (power of two)
  const int c = threadIdx.x & (tpr - 1);
  const int64_t rows = (int64_t)a.B * a.H * a.S;
  const int rows_per_pass = blockDim.x / tpr;
  const bool identity = f.identity != 0;
  const float scale = a.apply_mscale ? f.mscale : 1.0f;

  float2 fr[VEC];
#pragma unroll
  for (int k = 0; k < VEC; ++k) fr[k] = f.f[c * VEC + k];

  const Tin* x = static_cast<const Tin*>(a.x);
  Tout* y = static_cast<Tout*>(a.y);
  for (int64_t r = (int64_t)blockIdx.x * rows_per_pass + threadIdx.x / tpr; r < rows;
       r += (int64_t)gridDim.x * rows_per_pass) {
    const int s = (int)(r % a.S);
    const int64_t bh = r / a.S;
    const int h = (int)(bh % a.H);
    const int b = (int)(bh / a.H);
    const Tin* xr = x + b * a.xs[0] + h * a.xs[1] + (int64_t)s * a.xs[2] + c * VEC;
    Tout* yr_ = y + b * a.ys[0] + h * a.ys[1] + (int64_t)s * a.ys[2] + c * VEC;
    float x1[VEC], x2[VEC];
    load_vec<Tin, VEC>(xr, x1);
    load_vec<Tin, VEC>(xr + half, x2);
    float y1[VEC], y2[VEC];
    if (identity) {
#pragma unroll
      for (int k = 0; k < VEC; ++k) { y1[k] = x1[k] * scale; y2[k] = x2[k] * scale; }
    } else {
      const float m = (float)(a.positions ? __ldg(a.positions + s) : a.pos0 + s);
#pragma unroll
      for (int k = 0; k < VEC; ++k) {
        float cs, sn;
        turn_cos_sin<PRECISE>(m, fr[k], cs, sn);
        y1[k] = (x1[k] * cs - x2[k] * sn) * scale;
        y2[k] = (x1[k] * sn + x2[k] * cs) * scale;
      }
    }
    store_vec<Tout, VEC>(yr_, y1);
    store_vec<Tout, VEC>(yr_ + half, y2);
  }
}

}  // namespace

cudaError_t launch_rope(const RopeLaunch& a, const RopeFreqs& f, cudaStream_t st) {
  const int vec = a.out_bf16 ? 8 : 4;
  const int tpr = a.d / 2 / vec;
  const int rows_per_block = 256 / tpr;
  const int64_t rows = (int64_t)a.B * a.H * a.S;
  const int64_t need = (rows + rows_per_block - 1) / rows_per_block;
  const int blocks = (int)std::min<int64_t>(need, (int64_t)sm_count() * 8);
  if (blocks <= 0) return cudaSuccess;
  if (a.in_bf16 && a.out_bf16)
    rope_kernel<__nv_bfloat16, __nv_bfloat16, false><<<blocks, 256, 0, st>>>(a, f);
  else if (!a.in_bf16 && a.out_bf16)
    rope_kernel<float, __nv_bfloat16, false><<<blocks, 256, 0, st>>>(a, f);
  else if (!a.in_bf16 && !a.out_bf16)
    rope_kernel<float, float, true><<<blocks, 256, 0, st>>>(a, f);
  else
    return cudaErrorInvalidValue;
  return launched(1);
}

}  // namespace yr
