// attn_fwd_prefill, warp-level tensor-core path (mma.sync m16n8k16, bf16 in,
// fp32 accumulate): exact softmax attention over pre-rotated bfloat16 Q/K,
// key/value tiles folded with an online-softmax merge in ring order.
//
// Sources: softmax(QK^T / sqrt(d)) V ("Context Window Scaling ...", Section
// 1); attention as a sum over key blocks merged with online softmax
// ("Context Length Extension", Ring Attention); ring order and the causal
// skip of future blocks ("Context Window Scaling ...", Section 5 and FAQ 2);
// the sink + window mask ("Context Length Extension", Sliding Window +
// Attention Sinks).
//
// CTA = 128 query rows (8 warps x 16 rows); key/value tiles of 64 rows are
// double-buffered in shared memory with cp.async; 16-byte chunks are XOR-
// swizzled by row so ldmatrix reads are bank-conflict free.
#include <math.h>

#include "common.cuh"
#include "internal.h"

namespace yr {
namespace {

constexpr int BM = 128;
constexpr int BN = 64;
constexpr int kThreads = 256;

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

template <int D>
__device__ __forceinline__ int swz(int row, int col) {
  // element offset of (row, col) in a [rows][D] bf16 tile
  return row * D + ((((col >> 3) ^ (row & 7))) << 3) + (col & 7);
}

__device__ __forceinline__ void cp_async16(uint32_t dst, const void* src, bool valid) {
  const int n = valid ? 16 : 0;
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;\n" ::"r"(dst), "l"(src), "r"(n));
}
__device__ __forceinline__ void cp_commit() { asm volatile("cp.async.commit_group;\n" ::); }
template <int N>
__device__ __forceinline__ void cp_wait() { asm volatile("cp.async.wait_group %0;\n" ::"n"(N)); }

__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2, uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];\n"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3) : "r"(addr));
}
__device__ __forceinline__ void ldsm_x4_t(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2, uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];\n"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3) : "r"(addr));
}
__device__ __forceinline__ void mma16816(float (&c)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%0,%1,%2,%3};\n"
      : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

// Order of key tiles for one query tile: ring blocks I, I-1, ..., 0 (then
// N-1, ..., I+1 when no mask hides the future), tiles ascending inside a
// block.  I is the ring block of the tile's last row.
struct TileOrder {
  int n_tiles, tiles_per_block, N, I;
  __device__ int tile(int u) const {
    const int blk = u / tiles_per_block;
    const int rb = ((I - blk) % N + N) % N;
    return rb * tiles_per_block + (u % tiles_per_block);
  }
};

__device__ __forceinline__ bool tile_visible(int n0, int m0, int m1, int S, int mask, int sink, int window) {
  if (n0 >= S) return false;
  if (mask == YR_MASK_NONE) return true;
  if (n0 > m1) return false;                                   // future keys
  if (mask == YR_MASK_SINK_WINDOW && n0 >= sink && n0 + BN - 1 <= m0 - window) return false;
  return true;
}

template <int D, bool OUT_BF16>
__global__ void __launch_bounds__(kThreads, 1) prefill_mma_kernel(PrefillLaunch a) {
  extern __shared__ __align__(128) uint8_t smem_raw[];
  __nv_bfloat16* sQ = reinterpret_cast<__nv_bfloat16*>(smem_raw);
  __nv_bfloat16* sK = sQ + BM * D;
  __nv_bfloat16* sV = sK + 2 * BN * D;

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int n_qt = (a.S + BM - 1) / BM;
  const int qt = n_qt - 1 - (int)blockIdx.x;  // heaviest tiles first
  const int bhq = blockIdx.y;
  const int b = bhq / a.Hq, hq = bhq % a.Hq;
  const int hkv = hq / (a.Hq / a.Hkv);
  const int m0 = qt * BM, m1 = min(a.S, m0 + BM) - 1;

  const __nv_bfloat16* Qg = static_cast<const __nv_bfloat16*>(a.q) + b * a.qs[0] + hq * a.qs[1];
  const __nv_bfloat16* Kg = static_cast<const __nv_bfloat16*>(a.k) + b * a.ks[0] + hkv * a.ks[1];
  const __nv_bfloat16* Vg = static_cast<const __nv_bfloat16*>(a.v) + b * a.vs[0] + hkv * a.vs[1];

  constexpr int CPR = D / 8;  // 16-byte chunks per row
  // Q tile
  for (int i = tid; i < BM * CPR; i += kThreads) {
    const int r = i / CPR, ch = i % CPR;
    const bool ok = m0 + r < a.S;
    cp_async16(smem_u32(sQ + swz<D>(r, ch * 8)), Qg + (int64_t)(ok ? m0 + r : 0) * a.qs[2] + ch * 8, ok);
  }
  cp_commit();

  TileOrder ord;
  ord.n_tiles = (a.S + BN - 1) / BN;
  ord.N = a.ring_blocks;
  ord.tiles_per_block = a.ring_blocks > 1 ? (a.S / a.ring_blocks) / BN : ord.n_tiles;
  ord.I = a.ring_blocks > 1 ? m1 / (a.S / a.ring_blocks) : 0;

  auto next_visible = [&](int u) {
    while (u < ord.n_tiles && !tile_visible(ord.tile(u) * BN, m0, m1, a.S, a.mask, a.sink, a.window)) ++u;
    return u;
  };
  auto load_kv = [&](int t, int buf) {
    const int n0 = t * BN;
    __nv_bfloat16* dK = sK + buf * BN * D;
    __nv_bfloat16* dV = sV + buf * BN * D;
    for (int i = tid; i < BN * CPR; i += kThreads) {
      const int r = i / CPR, ch = i % CPR;
      const bool ok = n0 + r < a.S;
      const int64_t row = ok ? n0 + r : 0;
      cp_async16(smem_u32(dK + swz<D>(r, ch * 8)), Kg + row * a.ks[2] + ch * 8, ok);
      cp_async16(smem_u32(dV + swz<D>(r, ch * 8)), Vg + row * a.vs[2] + ch * 8, ok);
    }
  };

  int u = next_visible(0);
  if (u < ord.n_tiles) load_kv(ord.tile(u), 0);
  cp_commit();

  // Q fragments of this warp's 16 rows
  cp_wait<1>();
  __syncthreads();
  uint32_t qf[D / 16][4];
#pragma unroll
  for (int kk = 0; kk < D / 16; ++kk) {
    const int r = warp * 16 + (lane & 15), c = kk * 16 + (lane >> 4) * 8;
    ldsm_x4(smem_u32(sQ + swz<D>(r, c)), qf[kk][0], qf[kk][1], qf[kk][2], qf[kk][3]);
  }

  float o_acc[D / 8][4];
#pragma unroll
  for (int i = 0; i < D / 8; ++i) o_acc[i][0] = o_acc[i][1] = o_acc[i][2] = o_acc[i][3] = 0.f;
  float row_m[2] = {-INFINITY, -INFINITY}, row_l[2] = {0.f, 0.f};
  const int g = lane >> 2, t4 = lane & 3;
  const int mrow0 = m0 + warp * 16 + g;  // and mrow0 + 8

  int buf = 0;
  while (u < ord.n_tiles) {
    const int t = ord.tile(u);
    const int n0 = t * BN;
    const int un = next_visible(u + 1);
    if (un < ord.n_tiles) load_kv(ord.tile(un), buf ^ 1);
    cp_commit();
    cp_wait<1>();
    __syncthreads();

    const __nv_bfloat16* cK = sK + buf * BN * D;
    const __nv_bfloat16* cV = sV + buf * BN * D;
    float s[BN / 8][4];
#pragma unroll
    for (int i = 0; i < BN / 8; ++i) s[i][0] = s[i][1] = s[i][2] = s[i][3] = 0.f;
#pragma unroll
    for (int kk = 0; kk < D / 16; ++kk) {
#pragma unroll
      for (int p = 0; p < BN / 16; ++p) {
        const int r = p * 16 + (lane & 7) + (lane >> 4) * 8, c = kk * 16 + ((lane >> 3) & 1) * 8;
        uint32_t b0, b1, b2, b3;
        ldsm_x4(smem_u32(cK + swz<D>(r, c)), b0, b1, b2, b3);
        mma16816(s[2 * p], qf[kk], b0, b1);
        mma16816(s[2 * p + 1], qf[kk], b2, b3);
      }
    }

    // scale to base-2 logits and mask
    const bool need_mask = (n0 + BN - 1 > m0) || (n0 + BN > a.S) ||
                           (a.mask == YR_MASK_SINK_WINDOW && n0 <= m1 - a.window);
#pragma unroll
    for (int i = 0; i < BN / 8; ++i) {
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        float x = s[i][e] * a.scale_log2;
        if (need_mask) {
          const int m = mrow0 + (e >> 1) * 8;
          const int n = n0 + i * 8 + t4 * 2 + (e & 1);
          bool vis = n < a.S;
          if (a.mask != YR_MASK_NONE) {
            vis = vis && n <= m;
            if (a.mask == YR_MASK_SINK_WINDOW) vis = vis && (n < a.sink || m - n < a.window);
          }
          if (!vis) x = -INFINITY;
        }
        s[i][e] = x;
      }
    }

    // online softmax, two rows per thread (g and g + 8)
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      float mx = -INFINITY;
#pragma unroll
      for (int i = 0; i < BN / 8; ++i) mx = fmaxf(mx, fmaxf(s[i][2 * h], s[i][2 * h + 1]));
      mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 1));
      mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 2));
      const float mn = fmaxf(row_m[h], mx);
      const float ref = mn == -INFINITY ? 0.f : mn;
      const float corr = row_m[h] == -INFINITY ? 0.f : exp2f(row_m[h] - ref);
      float sum = 0.f;
#pragma unroll
      for (int i = 0; i < BN / 8; ++i) {
        s[i][2 * h] = exp2f(s[i][2 * h] - ref);
        s[i][2 * h + 1] = exp2f(s[i][2 * h + 1] - ref);
        sum += s[i][2 * h] + s[i][2 * h + 1];
      }
      row_l[h] = row_l[h] * corr + sum;
      row_m[h] = mn;
#pragma unroll
      for (int i = 0; i < D / 8; ++i) { o_acc[i][2 * h] *= corr; o_acc[i][2 * h + 1] *= corr; }
    }

    // O += P V
#pragma unroll
    for (int kk = 0; kk < BN / 16; ++kk) {
      uint32_t pa[4];
      pa[0] = pack_bf16(s[2 * kk][0], s[2 * kk][1]);
      pa[1] = pack_bf16(s[2 * kk][2], s[2 * kk][3]);
      pa[2] = pack_bf16(s[2 * kk + 1][0], s[2 * kk + 1][1]);
      pa[3] = pack_bf16(s[2 * kk + 1][2], s[2 * kk + 1][3]);
#pragma unroll
      for (int p = 0; p < D / 16; ++p) {
        const int r = kk * 16 + (lane & 7) + ((lane >> 3) & 1) * 8, c = p * 16 + (lane >> 4) * 8;
        uint32_t b0, b1, b2, b3;
        ldsm_x4_t(smem_u32(cV + swz<D>(r, c)), b0, b1, b2, b3);
        mma16816(o_acc[2 * p], pa, b0, b1);
        mma16816(o_acc[2 * p + 1], pa, b2, b3);
      }
    }
    __syncthreads();
    buf ^= 1;
    u = un;
  }
  cp_wait<0>();

  // epilogue: normalise and store
#pragma unroll
  for (int h = 0; h < 2; ++h) {
    float l = row_l[h];
    l += __shfl_xor_sync(0xffffffffu, l, 1);
    l += __shfl_xor_sync(0xffffffffu, l, 2);
    const int m = mrow0 + h * 8;
    if (m >= a.S) continue;
    const float inv = l > 0.f ? 1.f / l : 0.f;
    if (OUT_BF16) {
      __nv_bfloat16* Og = static_cast<__nv_bfloat16*>(a.o) + b * a.os[0] + hq * a.os[1] + (int64_t)m * a.os[2];
#pragma unroll
      for (int i = 0; i < D / 8; ++i)
        *reinterpret_cast<uint32_t*>(Og + i * 8 + t4 * 2) = pack_bf16(o_acc[i][2 * h] * inv, o_acc[i][2 * h + 1] * inv);
    } else {
      float* Og = static_cast<float*>(a.o) + b * a.os[0] + hq * a.os[1] + (int64_t)m * a.os[2];
#pragma unroll
      for (int i = 0; i < D / 8; ++i)
        *reinterpret_cast<float2*>(Og + i * 8 + t4 * 2) = make_float2(o_acc[i][2 * h] * inv, o_acc[i][2 * h + 1] * inv);
    }
    if (a.lse && t4 == 0)
      a.lse[((int64_t)b * a.Hq + hq) * a.S + m] =
          l > 0.f ? (row_m[h] + log2f(l)) * 0.69314718055994530942f : -INFINITY;
  }
}

template <int D, bool OB>
cudaError_t launch_dt(const PrefillLaunch& a, cudaStream_t st) {
  const int smem = (BM + 4 * BN) * D * 2;
  cudaError_t e = cudaFuncSetAttribute(prefill_mma_kernel<D, OB>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  dim3 grid((unsigned)((a.S + BM - 1) / BM), (unsigned)(a.B * a.Hq));
  prefill_mma_kernel<D, OB><<<grid, kThreads, smem, st>>>(a);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_prefill(const PrefillLaunch& a, cudaStream_t st) {
  if (a.ring_blocks > 1 && (a.S / a.ring_blocks) % BN != 0) return cudaErrorInvalidValue;
  if (a.d == 128) return a.out_bf16 ? launch_dt<128, true>(a, st) : launch_dt<128, false>(a, st);
  return a.out_bf16 ? launch_dt<64, true>(a, st) : launch_dt<64, false>(a, st);
}

}  // namespace yr
