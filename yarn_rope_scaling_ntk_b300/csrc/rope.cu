// rope_apply and the rotation pass of the attention entry points: rotate every
// pair (x_i, x_{i+d/2}) of [B, H, S, d] tensors by m * theta'_i ("Context
// Window Scaling ...", Section 2, Formal RoPE Mechanics; rotate-half pairing
// as in that section's listing).  One launch may cover several tensors
// (segments): the attention entry points rotate Q and K (and convert V for
// float32 inputs) in a single pass.
//
// Memory-bound: one read and one write of every element.  The reads do not
// depend on registers for their depth: a producer warp streams tiles of
// consecutive rows of one (batch, head) into a four-stage shared-memory ring
// with bulk asynchronous copies (one copy per tile when the rows are
// contiguous, one per row otherwise), so each CTA keeps up to four 24 KB
// tiles in flight.  Eight compute warps rotate each landed tile -- a thread
// owns VEC pairs of a few consecutive rows, one vector from each half of a
// row -- and store the result with 16-byte writes.  Persistent CTAs, two per
// SM, walk the tiles with a grid stride.  Every wait is bounded.
#include <algorithm>

#include "common.cuh"
#include "internal.h"
#include "tc_ptx.cuh"

namespace yr {
namespace {

using tc::mbar_arrive;
using tc::mbar_arrive_expect_tx;
using tc::mbar_init;
using tc::mbar_wait;
using tc::mbar_wait_drain;

constexpr int kComputeWarps = 8;
constexpr int kThreads = (kComputeWarps + 1) * 32;  // + one producer warp
// Four 24 KB stages (96 rows of bf16 at d = 128, three rows per thread):
// timed against 3 x 32, 2 x 48, 4 x 16, 6 x 16 and 8 x 12 KB.
constexpr int kStages = 4;
constexpr int kStageBytes = 24576;  // input bytes of one tile
constexpr int kMaxTileRows = 256;

template <typename T> struct Vec;
template <> struct Vec<float> { static constexpr int N = 4; };
template <> struct Vec<__nv_bfloat16> { static constexpr int N = 8; };

// VEC consecutive input elements (from shared memory) as float.
template <typename T, int N>
__device__ __forceinline__ void load_vec(const uint8_t* p, float (&v)[N]);

template <>
__device__ __forceinline__ void load_vec<float, 4>(const uint8_t* p, float (&v)[4]) {
  const float4 t = *reinterpret_cast<const float4*>(p);
  v[0] = t.x; v[1] = t.y; v[2] = t.z; v[3] = t.w;
}
template <>
__device__ __forceinline__ void load_vec<float, 8>(const uint8_t* p, float (&v)[8]) {
  const float4 a = reinterpret_cast<const float4*>(p)[0];
  const float4 b = reinterpret_cast<const float4*>(p)[1];
  v[0] = a.x; v[1] = a.y; v[2] = a.z; v[3] = a.w; v[4] = b.x; v[5] = b.y; v[6] = b.z; v[7] = b.w;
}
template <>
__device__ __forceinline__ void load_vec<__nv_bfloat16, 8>(const uint8_t* p, float (&v)[8]) {
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

// Tile t of the launch -> segment, (batch, head) and first row.  Tiles are
// numbered segment by segment, (batch, head) by (batch, head), rows
// ascending; a tile never crosses a (batch, head).
struct TileRef {
  int seg, b, h, s0, rows;
};
// (32-bit arithmetic: the launcher keeps the tile count below 2^31)
__device__ __forceinline__ TileRef tile_ref(const RopeLaunch& a, int rows_per_tile, int t) {
  TileRef r;
  int g = 0;
  while (g + 1 < a.n_seg && t >= (int)a.seg[g + 1].tile0) ++g;
  const RopeSegment& sg = a.seg[g];
  const unsigned local = (unsigned)(t - (int)sg.tile0);
  const unsigned tph = (unsigned)((sg.S + rows_per_tile - 1) / rows_per_tile);  // tiles per (batch, head)
  const unsigned bh = local / tph;
  r.seg = g;
  r.h = (int)(bh % (unsigned)sg.H);
  r.b = (int)(bh / (unsigned)sg.H);
  r.s0 = (int)(local - bh * tph) * rows_per_tile;
  r.rows = min(rows_per_tile, sg.S - r.s0);
  return r;
}

template <typename Tin, typename Tout, bool PRECISE>
__global__ void __launch_bounds__(kThreads, 2)
    rope_kernel(const __grid_constant__ RopeLaunch a, const __grid_constant__ RopeFreqs f) {
  constexpr int VEC = Vec<Tout>::N;
  constexpr int EIN = (int)sizeof(Tin);
  extern __shared__ __align__(128) uint8_t smem[];
  __shared__ uint64_t full[kStages], empty[kStages];
  __shared__ volatile int abort_flag;

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int half = a.d >> 1;
  const int row_bytes = a.d * EIN;
  const int rpt = a.rows_per_tile;
  const int stage_bytes = rpt * row_bytes;

  if (tid == 0) {
    abort_flag = 0;
    for (int s = 0; s < kStages; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], kComputeWarps);
    }
    tc::fence_mbar_init();
  }
  __syncthreads();

  if (warp == kComputeWarps) {
    // ---------------- producer ----------------
    if (lane == 0) {
      int issued[kStages] = {0};
      int i = 0;
      for (int t = blockIdx.x; t < (int)a.n_tiles; t += gridDim.x, ++i) {
        const int s = i % kStages;
        if (!mbar_wait(&empty[s], ((i / kStages) & 1) ^ 1, &abort_flag, a.status, 51)) break;
        const TileRef r = tile_ref(a, rpt, t);
        const RopeSegment& sg = a.seg[r.seg];
        const uint8_t* src = static_cast<const uint8_t*>(sg.x) +
                             (r.b * sg.xs[0] + r.h * sg.xs[1] + (int64_t)r.s0 * sg.xs[2]) * EIN;
        uint8_t* dst = smem + s * stage_bytes;
        mbar_arrive_expect_tx(&full[s], (uint32_t)(r.rows * row_bytes));
        if (sg.xs[2] == a.d) {
          tc::bulk_g2s(dst, src, (uint32_t)(r.rows * row_bytes), &full[s]);
        } else {
          for (int k = 0; k < r.rows; ++k)
            tc::bulk_g2s(dst + k * row_bytes, src + (int64_t)k * sg.xs[2] * EIN, (uint32_t)row_bytes, &full[s]);
        }
        ++issued[s];
      }
      // every copy issued lands before the CTA exits, also when the compute
      // warps gave up on an earlier tile
      for (int s = 0; s < kStages; ++s)
        if (issued[s]) mbar_wait_drain(&full[s], (issued[s] - 1) & 1, 200000000ll);
    }
    __syncwarp();
    __syncthreads();
    return;
  }

  // ---------------- compute warps ----------------
  // Thread (slot, c): chunk c of rows slot * rpt_thr ... of each tile, i.e.
  // consecutive rows, so that after an exact angle at the first row the
  // rotation of the next row follows by one complex multiply by the step
  // e^(i theta) (positions pos0 + s, bfloat16 outputs; explicit positions and
  // float32 outputs take the exact angle on every row).  Each 8-lane phase of
  // a shared-memory read is one row's 128 contiguous bytes.
  const int tpr = half / VEC;               // threads per row (power of two)
  const int c = tid & (tpr - 1);            // this thread's chunk of the half row
  const int slot = tid / tpr;
  const int rows_thr = (rpt + kComputeWarps * 32 / tpr - 1) / (kComputeWarps * 32 / tpr);
  const float scale = a.apply_mscale ? f.mscale : 1.0f;
  const bool recur = !PRECISE && a.positions == nullptr;
  float stc[VEC], sts[VEC];  // cos / sin of one position step
#pragma unroll
  for (int e = 0; e < VEC; ++e) turn_cos_sin<false>(1.0f, f.f[c * VEC + e], stc[e], sts[e]);

  int i = 0;
  for (int t = blockIdx.x; t < (int)a.n_tiles; t += gridDim.x, ++i) {
    const int s = i % kStages;
    if (!__all_sync(0xffffffffu, mbar_wait(&full[s], (i / kStages) & 1, &abort_flag, a.status, 52))) break;
    const TileRef r = tile_ref(a, rpt, t);
    const RopeSegment& sg = a.seg[r.seg];
    const bool identity = f.identity != 0 || sg.identity != 0;
    const uint8_t* st = smem + s * stage_bytes;
    Tout* ybase = static_cast<Tout*>(sg.y) + r.b * sg.ys[0] + r.h * sg.ys[1];
    const int k0 = slot * rows_thr, k1 = min(r.rows, k0 + rows_thr);
    float cs[VEC], sn[VEC];  // rotation of the current row, times scale
    for (int k = k0; k < k1; ++k) {
      const int srow = r.s0 + k;
      const uint8_t* xr = st + k * row_bytes + c * VEC * EIN;
      float x1[VEC], x2[VEC], y1[VEC], y2[VEC];
      load_vec<Tin, VEC>(xr, x1);
      load_vec<Tin, VEC>(xr + half * EIN, x2);
      if (identity) {
#pragma unroll
        for (int e = 0; e < VEC; ++e) { y1[e] = x1[e] * scale; y2[e] = x2[e] * scale; }
      } else {
        if (k == k0 || !recur) {
          const float m = (float)(a.positions ? __ldg(a.positions + srow) : sg.pos0 + srow);
#pragma unroll
          for (int e = 0; e < VEC; ++e) {
            turn_cos_sin<PRECISE>(m, f.f[c * VEC + e], cs[e], sn[e]);
            cs[e] *= scale;
            sn[e] *= scale;
          }
        } else {
#pragma unroll
          for (int e = 0; e < VEC; ++e) {  // next position: multiply by e^(i theta)
            const float c0 = cs[e], s0 = sn[e];
            cs[e] = c0 * stc[e] - s0 * sts[e];
            sn[e] = s0 * stc[e] + c0 * sts[e];
          }
        }
#pragma unroll
        for (int e = 0; e < VEC; ++e) {
          y1[e] = x1[e] * cs[e] - x2[e] * sn[e];
          y2[e] = x1[e] * sn[e] + x2[e] * cs[e];
        }
      }
      Tout* yr_ = ybase + (int64_t)srow * sg.ys[2] + c * VEC;
      store_vec<Tout, VEC>(yr_, y1);
      store_vec<Tout, VEC>(yr_ + half, y2);
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(&empty[s]);
  }
  __syncthreads();
}

template <typename Tin, typename Tout, bool PRECISE>
cudaError_t launch_t(const RopeLaunch& a, const RopeFreqs& f, int smem, cudaStream_t st) {
  auto kern = rope_kernel<Tin, Tout, PRECISE>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  const int64_t grid = std::min<int64_t>(a.n_tiles, 2 * (int64_t)sm_count());
  kern<<<(unsigned)grid, kThreads, smem, st>>>(a, f);
  return launched(1);
}

}  // namespace

cudaError_t launch_rope(const RopeLaunch& a_in, const RopeFreqs& f, cudaStream_t st) {
  RopeLaunch a = a_in;
  if (a.n_seg < 1 || a.n_seg > kMaxRopeSegments) return cudaErrorInvalidValue;
  if (a.in_bf16 && !a.out_bf16) return cudaErrorInvalidValue;
  const int row_bytes = a.d * (a.in_bf16 ? 2 : 4);
  a.rows_per_tile = std::max(1, std::min(kMaxTileRows, kStageBytes / row_bytes));
  int64_t tiles = 0;
  for (int g = 0; g < a.n_seg; ++g) {
    RopeSegment& sg = a.seg[g];
    sg.tile0 = tiles;
    tiles += (int64_t)a.B * sg.H * ((sg.S + a.rows_per_tile - 1) / a.rows_per_tile);
  }
  a.n_tiles = tiles;
  if (tiles == 0) return cudaSuccess;
  if (tiles >= (int64_t(1) << 31)) return cudaErrorInvalidValue;
  a.status = device_status_word();
  if (!a.status) return cudaErrorInvalidValue;
  const int smem = kStages * a.rows_per_tile * row_bytes;
  if (a.in_bf16) return launch_t<__nv_bfloat16, __nv_bfloat16, false>(a, f, smem, st);
  if (a.out_bf16) return launch_t<float, __nv_bfloat16, false>(a, f, smem, st);
  return launch_t<float, float, true>(a, f, smem, st);
}

}  // namespace yr
