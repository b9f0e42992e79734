// attn_merge_partial: exact merge of two attention partials over disjoint key
// sets, each given as (O, LSE) with O normalised over its own keys.  With
// L = ln(e^La + e^Lb), the merged row is O = e^(La - L) Oa + e^(Lb - L) Ob:
// the combination of per-block results by their softmax denominators that
// ring attention uses for the blocks a device receives ("Context Length
// Extension", Ring Attention: partial results combined with online
// softmax; "Context Window Scaling ...", Section 5).
//
// Memory-bound: one warp per row; each lane owns 4 consecutive float32
// elements of each 128-element chunk (16-byte loads and stores).
#include "common.cuh"
#include "internal.h"

namespace yr {
namespace {

// CH = chunks of 128 floats per row (d <= 128 CH).
template <int CH>
__global__ void __launch_bounds__(256) merge_kernel(MergeLaunch a) {
  const int lane = threadIdx.x & 31;
  const int64_t rows = (int64_t)a.B * a.H * a.S;
  const int64_t row = (int64_t)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
  if (row >= rows) return;
  const int s = (int)(row % a.S);
  const int64_t bh = row / a.S;
  const int h = (int)(bh % a.H), b = (int)(bh / a.H);
  float* oa = a.o_acc + b * a.as[0] + h * a.as[1] + (int64_t)s * a.as[2];
  const float* op = a.o_part + b * a.ps[0] + h * a.ps[1] + (int64_t)s * a.ps[2];
  // Both rows are loaded together with the lse values (no dependent second
  // round trip); a side with weight 0 (an empty partial, lse = -inf) is
  // dropped by a select, never multiplied, so an accumulator that holds
  // nothing yet may contain anything.
  constexpr int kMaxChunks = CH;
  float4 xa[kMaxChunks], xp[kMaxChunks];
#pragma unroll
  for (int i = 0; i < kMaxChunks; ++i) {
    const int c = lane * 4 + i * 128;
    if (c < a.d) {
      xa[i] = *reinterpret_cast<const float4*>(oa + c);
      xp[i] = *reinterpret_cast<const float4*>(op + c);
    }
  }
  const float la = a.lse_acc[row], lp = a.lse_part[row];
  const float mx = fmaxf(la, lp);
  float wa = 0.f, wp = 0.f, lnew = -INFINITY;
  if (mx != -INFINITY) {
    const float ea = expf(la - mx), ep = expf(lp - mx);
    const float tot = ea + ep;
    wa = ea / tot;
    wp = ep / tot;
    lnew = mx + logf(tot);
  }
#pragma unroll
  for (int i = 0; i < kMaxChunks; ++i) {
    const int c = lane * 4 + i * 128;
    if (c >= a.d) continue;
    const float4 x = xa[i], y = xp[i];
    float4 z;
    z.x = (wa != 0.f ? wa * x.x : 0.f) + (wp != 0.f ? wp * y.x : 0.f);
    z.y = (wa != 0.f ? wa * x.y : 0.f) + (wp != 0.f ? wp * y.y : 0.f);
    z.z = (wa != 0.f ? wa * x.z : 0.f) + (wp != 0.f ? wp * y.z : 0.f);
    z.w = (wa != 0.f ? wa * x.w : 0.f) + (wp != 0.f ? wp * y.w : 0.f);
    *reinterpret_cast<float4*>(oa + c) = z;
    if (a.o_final) {
      const int64_t off = b * a.fs[0] + h * a.fs[1] + (int64_t)s * a.fs[2] + c;
      if (a.final_bf16)
        *reinterpret_cast<uint2*>(static_cast<__nv_bfloat16*>(a.o_final) + off) =
            make_uint2(pack_bf16(z.x, z.y), pack_bf16(z.z, z.w));
      else
        *reinterpret_cast<float4*>(static_cast<float*>(a.o_final) + off) = z;
    }
  }
  if (lane == 0) a.lse_acc[row] = lnew;
}

// Rows with no key at all: o = 0 and lse = -inf (the empty softmax).
__global__ void __launch_bounds__(256) fill_empty_kernel(void* o, int out_bf16, float* lse, int B, int H, int S,
                                                         int d, int64_t s0, int64_t s1, int64_t s2) {
  const int64_t rows = (int64_t)B * H * S;
  const int lane = threadIdx.x & 31;
  const int64_t row = (int64_t)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
  if (row >= rows) return;
  const int s = (int)(row % S);
  const int64_t bh = row / S;
  const int h = (int)(bh % H), b = (int)(bh / H);
  const int64_t base = b * s0 + h * s1 + (int64_t)s * s2;
  for (int c = lane; c < d; c += 32) {
    if (out_bf16) static_cast<__nv_bfloat16*>(o)[base + c] = __float2bfloat16_rn(0.f);
    else static_cast<float*>(o)[base + c] = 0.f;
  }
  if (lse && lane == 0) lse[row] = -INFINITY;
}

}  // namespace

cudaError_t launch_fill_empty(void* o, int out_bf16, float* lse, int B, int H, int S, int d, const int64_t os[3],
                              cudaStream_t st) {
  const int64_t rows = (int64_t)B * H * S;
  if (rows == 0) return cudaSuccess;
  const int64_t blocks = (rows + 7) / 8;
  if (blocks > 0x7fffffff) return cudaErrorInvalidValue;
  fill_empty_kernel<<<(unsigned)blocks, 256, 0, st>>>(o, out_bf16, lse, B, H, S, d, os[0], os[1], os[2]);
  return launched(1);
}

cudaError_t launch_merge(const MergeLaunch& a, cudaStream_t st) {
  const int64_t rows = (int64_t)a.B * a.H * a.S;
  if (rows == 0) return cudaSuccess;
  const int64_t blocks = (rows + 7) / 8;  // 8 warps (rows) per CTA
  if (blocks > 0x7fffffff) return cudaErrorInvalidValue;
  const int ch = (a.d + 127) / 128;
  if (ch <= 1) merge_kernel<1><<<(unsigned)blocks, 256, 0, st>>>(a);
  else if (ch <= 2) merge_kernel<2><<<(unsigned)blocks, 256, 0, st>>>(a);
  else if (ch <= 4) merge_kernel<4><<<(unsigned)blocks, 256, 0, st>>>(a);
  else if (ch <= 8) merge_kernel<8><<<(unsigned)blocks, 256, 0, st>>>(a);
  else return cudaErrorInvalidValue;
  return launched(1);
}

}  // namespace yr
