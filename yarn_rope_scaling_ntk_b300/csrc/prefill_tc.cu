// attn_fwd_prefill, tcgen05 path for sm_103a: exact softmax attention over
// rotated bfloat16 Q/K with key/value tiles folded by an online-softmax merge
// in ring order.
//
// Sources: softmax(QK^T / sqrt(d)) V ("Context Window Scaling ...", Section
// 1); attention as a sum over key blocks combined with online softmax
// ("Context Length Extension", Ring Attention); ring rotation and the skip
// of future blocks ("Context Window Scaling ...", Section 5 and FAQ 2); the
// sink + window mask ("Context Length Extension", Sliding Window + Attention
// Sinks).
//
// One CTA = one 128-row query tile of one (batch, head).  Roles:
//   warp 4  TMA producer: Q once, then K and V tiles of 128 keys into a
//           two-stage ring of 128-byte-swizzled shared-memory buffers.
//   warp 5  TMEM owner and MMA issuer (one thread): S = Q K^T into one of two
//           128-column TMEM buffers, then O += P V with P read from TMEM.
//   warps 0-3  softmax: thread r owns query row r (TMEM lane r); it reads its
//           row of S, masks, updates the running max / sum, writes P as
//           bf16 pairs over the first 64 columns of the same buffer, and
//           rescales O in TMEM only when the max grew by more than 2^8.
// The MMA of S for tile i+1 overlaps the softmax of tile i.  Every mbarrier
// wait is bounded; a wait that gives up records a code in the status word and
// makes every role leave its loop, drain its asynchronous work and free TMEM.
#include <cudaTypedefs.h>
#include <math.h>
#include <string.h>

#include "common.cuh"
#include "internal.h"
#include "tc_ptx.cuh"

namespace yr {
namespace {

using namespace tc;

constexpr int BM = 128;   // query rows per CTA
constexpr int BN = 128;   // keys per tile
constexpr int NS = 2;     // K / V pipeline stages
constexpr int kThreads = 192;
constexpr uint32_t kTmemCols = 512;
constexpr float kRescaleThreshold = 8.0f;  // log2 units

struct TcParams {
  int B, Hq, Hkv, S, group;
  int mask, sink, window, ring_blocks, cs;
  float scale_log2;
  void* o;
  int64_t os[3];
  float* lse;
  int out_bf16;
  int* status;
};

// Key chunks in ring order for one query tile: ring blocks I, I-1, ... (then
// the rest of the ring when nothing is masked), chunks ascending in a block.
// A chunk holds cs <= 128 keys (cs = 64 when a ring block is an odd multiple
// of 64 keys); the MMA tile always spans 128 keys and masks the excess.
struct Walk {
  int u, n_chunks, cpb, N, I, cs, S, m0, m1, mask, sink, window;
  __device__ void init(const TcParams& p, int qt) {
    u = 0;
    cs = p.cs;
    S = p.S;
    n_chunks = (p.S + cs - 1) / cs;
    N = p.ring_blocks;
    const int bs = N > 1 ? p.S / N : 0;
    cpb = N > 1 ? bs / cs : n_chunks;
    m0 = qt * BM;
    m1 = min(p.S, m0 + BM) - 1;
    I = N > 1 ? m1 / bs : 0;
    mask = p.mask;
    sink = p.sink;
    window = p.window;
  }
  __device__ bool visible(int n0) const {
    if (n0 >= S) return false;
    if (mask == YR_MASK_NONE) return true;
    if (n0 > m1) return false;
    if (mask == YR_MASK_SINK_WINDOW && n0 >= sink && n0 + cs - 1 <= m0 - window) return false;
    return true;
  }
  // next visible chunk start, or -1
  __device__ int next() {
    while (u < n_chunks) {
      const int blk = u / cpb;
      const int rb = ((I - blk) % N + N) % N;
      const int n0 = (rb * cpb + (u % cpb)) * cs;
      ++u;
      if (visible(n0)) return n0;
    }
    return -1;
  }
};

__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

template <int D>
struct Smem {
  static constexpr int kTile = BM * D * 2;  // bytes of one 128-row bf16 tile
  static constexpr int kQ = 0;
  static constexpr int kK = kTile;
  static constexpr int kV = kK + NS * kTile;
  static constexpr int kBytes = kV + NS * kTile;
};

template <int D>
__global__ void __launch_bounds__(kThreads, 1)
    prefill_tc_kernel(const __grid_constant__ CUtensorMap tq, const __grid_constant__ CUtensorMap tk,
                      const __grid_constant__ CUtensorMap tv, const TcParams p) {
  constexpr int ATOMS = D / 64;              // 64-column swizzle atoms per row
  constexpr int ATOM_BYTES = BM * 128;       // one atom column of a 128-row tile
  constexpr uint32_t S_COLS = 128;
  constexpr uint32_t O_COL = 2 * S_COLS;
  constexpr uint32_t ID_QK = idesc_bf16_f32(BM, BN, false);
  constexpr uint32_t ID_PV = idesc_bf16_f32(BM, D, true);

  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* sQ = smem + Smem<D>::kQ;
  uint8_t* sK = smem + Smem<D>::kK;
  uint8_t* sV = smem + Smem<D>::kV;

  __shared__ uint64_t q_full, k_full[NS], k_empty[NS], v_full[NS], v_empty[NS];
  __shared__ uint64_t s_full[2], p_full[2], o_done, drain;
  __shared__ uint32_t tmem_slot;
  __shared__ volatile int abort_flag;

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int n_qt = (p.S + BM - 1) / BM;
  const int qt = n_qt - 1 - (int)blockIdx.x;
  const int bh = blockIdx.y;
  const int b = bh / p.Hq, hq = bh % p.Hq;
  const int hkv = hq / p.group;

  if (tid == 0) {
    abort_flag = 0;
    mbar_init(&q_full, 1);
    for (int s = 0; s < NS; ++s) {
      mbar_init(&k_full[s], 1);
      mbar_init(&k_empty[s], 1);
      mbar_init(&v_full[s], 1);
      mbar_init(&v_empty[s], 1);
    }
    for (int s = 0; s < 2; ++s) {
      mbar_init(&s_full[s], 1);
      mbar_init(&p_full[s], 128);
    }
    mbar_init(&o_done, 1);
    mbar_init(&drain, 1);
    fence_mbar_init();
  }
  if (warp == 5) tmem_alloc(&tmem_slot, kTmemCols);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = tmem_slot;

  Walk walk;
  walk.init(p, qt);

  if (warp == 4) {
    // ---------------- TMA producer ----------------
    if (lane == 0) {
      tma_prefetch_desc(&tq);
      tma_prefetch_desc(&tk);
      tma_prefetch_desc(&tv);
      mbar_arrive_expect_tx(&q_full, Smem<D>::kTile);
      for (int a = 0; a < ATOMS; ++a) tma_load_4d(sQ + a * ATOM_BYTES, &tq, &q_full, a * 64, walk.m0, hq, b);
      int i = 0;
      int k_uses[NS] = {0}, v_uses[NS] = {0};
      for (int n0 = walk.next(); n0 >= 0; n0 = walk.next(), ++i) {
        const int s = i % NS;
        const uint32_t par = ((i / NS) & 1) ^ 1;
        if (!mbar_wait(&k_empty[s], par, &abort_flag, p.status, 11)) break;
        mbar_arrive_expect_tx(&k_full[s], Smem<D>::kTile);
        for (int a = 0; a < ATOMS; ++a)
          tma_load_4d(sK + s * Smem<D>::kTile + a * ATOM_BYTES, &tk, &k_full[s], a * 64, n0, hkv, b);
        ++k_uses[s];
        if (!mbar_wait(&v_empty[s], par, &abort_flag, p.status, 12)) break;
        mbar_arrive_expect_tx(&v_full[s], Smem<D>::kTile);
        for (int a = 0; a < ATOMS; ++a)
          tma_load_4d(sV + s * Smem<D>::kTile + a * ATOM_BYTES, &tv, &v_full[s], a * 64, n0, hkv, b);
        ++v_uses[s];
      }
      if (abort_flag) {
        // let the copies already issued land before the CTA exits
        mbar_wait_drain(&q_full, 0, 100000000ull);
        for (int s = 0; s < NS; ++s) {
          if (k_uses[s]) mbar_wait_drain(&k_full[s], (k_uses[s] - 1) & 1, 100000000ull);
          if (v_uses[s]) mbar_wait_drain(&v_full[s], (v_uses[s] - 1) & 1, 100000000ull);
        }
      }
    }
    __syncwarp();
  } else if (warp == 5) {
    // ---------------- MMA issuer ----------------
    if (lane == 0) {
      bool ok = mbar_wait(&q_full, 0, &abort_flag, p.status, 21);
      const uint32_t q_base = smem_u32(sQ);
      int i = 0;
      for (int n0 = ok ? walk.next() : -1; n0 >= 0; n0 = walk.next(), ++i) {
        const int s = i % NS, sb = i & 1;
        if (!mbar_wait(&k_full[s], (i / NS) & 1, &abort_flag, p.status, 22)) { ok = false; break; }
        tc_fence_after();
        const uint32_t k_base = smem_u32(sK + s * Smem<D>::kTile);
        const uint32_t d_s = tmem + sb * S_COLS;
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint32_t off = (kk >> 2) * ATOM_BYTES + (kk & 3) * 32;
          mma_ss(d_s, sdesc_sw128(q_base + off, 16, 1024), sdesc_sw128(k_base + off, 16, 1024), ID_QK, kk > 0);
        }
        mma_commit(&s_full[sb]);
        mma_commit(&k_empty[s]);
        if (i > 0) {
          const int j = i - 1, sj = j % NS, pb = j & 1;
          if (!mbar_wait(&p_full[pb], (j >> 1) & 1, &abort_flag, p.status, 23)) { ok = false; break; }
          if (!mbar_wait(&v_full[sj], (j / NS) & 1, &abort_flag, p.status, 24)) { ok = false; break; }
          tc_fence_after();
          const uint32_t v_base = smem_u32(sV + sj * Smem<D>::kTile);
#pragma unroll
          for (int kk = 0; kk < BN / 16; ++kk)
            mma_ts(tmem + O_COL, tmem + pb * S_COLS + kk * 8, sdesc_sw128(v_base + kk * 2048, ATOM_BYTES, 1024),
                   ID_PV, (j > 0 || kk > 0) ? 1u : 0u);
          mma_commit(&v_empty[sj]);
          mma_commit(&o_done);
        }
      }
      if (ok && i > 0) {
        const int j = i - 1, sj = j % NS, pb = j & 1;
        if (mbar_wait(&p_full[pb], (j >> 1) & 1, &abort_flag, p.status, 25) &&
            mbar_wait(&v_full[sj], (j / NS) & 1, &abort_flag, p.status, 26)) {
          tc_fence_after();
          const uint32_t v_base = smem_u32(sV + sj * Smem<D>::kTile);
#pragma unroll
          for (int kk = 0; kk < BN / 16; ++kk)
            mma_ts(tmem + O_COL, tmem + pb * S_COLS + kk * 8, sdesc_sw128(v_base + kk * 2048, ATOM_BYTES, 1024),
                   ID_PV, (j > 0 || kk > 0) ? 1u : 0u);
          mma_commit(&v_empty[sj]);
          mma_commit(&o_done);
        }
      }
      // all issued MMAs complete before TMEM is released
      mma_commit(&drain);
      mbar_wait_drain(&drain, 0, 100000000ull);
    }
    __syncwarp();
  } else {
    // ---------------- softmax (warps 0-3) ----------------
    const int r = tid;  // query row within the tile == TMEM lane
    const int m = walk.m0 + r;
    const uint32_t lane_addr = tmem + ((uint32_t)(warp * 32) << 16);
    float m_used = -INFINITY, l = 0.f;
    int i = 0;
    bool ok = true;
    for (int n0 = walk.next(); n0 >= 0; n0 = walk.next(), ++i) {
      const int sb = i & 1;
      // warp-uniform decisions: tcgen05.ld / st are warp-collective
      ok = __all_sync(0xffffffffu, mbar_wait(&s_full[sb], (i >> 1) & 1, &abort_flag, p.status, 31));
      if (!ok) break;
      tc_fence_after();
      float x[BN];
#pragma unroll
      for (int c = 0; c < BN / 32; ++c) {
        uint32_t rr[32];
        tmem_ld32(lane_addr + sb * S_COLS + c * 32, rr);
        tmem_ld_wait();
#pragma unroll
        for (int e = 0; e < 32; ++e) x[c * 32 + e] = __uint_as_float(rr[e]) * p.scale_log2;
      }
      const bool need_mask = walk.cs < BN || n0 + BN > p.S || (p.mask != YR_MASK_NONE && n0 + BN - 1 > walk.m0) ||
                             (p.mask == YR_MASK_SINK_WINDOW && n0 <= walk.m1 - p.window);
      if (need_mask) {
#pragma unroll
        for (int e = 0; e < BN; ++e) {
          const int n = n0 + e;
          bool vis = e < walk.cs && n < p.S;
          if (p.mask != YR_MASK_NONE) {
            vis = vis && n <= m;
            if (p.mask == YR_MASK_SINK_WINDOW) vis = vis && (n < p.sink || m - n < p.window);
          }
          if (!vis) x[e] = -INFINITY;
        }
      }
      float mx = x[0];
#pragma unroll
      for (int e = 1; e < BN; ++e) mx = fmaxf(mx, x[e]);
      // Lazy rescale: the reference max moves only when the row max exceeds it
      // by more than 2^8; the whole warp rescales its O rows when any lane must.
      const bool grow = mx > m_used + kRescaleThreshold;
      const bool rescale = grow && m_used != -INFINITY && i > 0;
      const float corr = rescale ? ex2(m_used - mx) : 1.0f;
      if (grow) m_used = mx;
      if (__any_sync(0xffffffffu, rescale)) {
        l *= corr;
        ok = __all_sync(0xffffffffu, mbar_wait(&o_done, (i - 1) & 1, &abort_flag, p.status, 32));
        if (!ok) break;
        tc_fence_after();
#pragma unroll
        for (int c = 0; c < D / 32; ++c) {
          uint32_t rr[32];
          tmem_ld32(lane_addr + O_COL + c * 32, rr);
          tmem_ld_wait();
#pragma unroll
          for (int e = 0; e < 32; ++e) rr[e] = __float_as_uint(__uint_as_float(rr[e]) * corr);
          tmem_st32(lane_addr + O_COL + c * 32, rr);
        }
      }
      const float ref = m_used == -INFINITY ? 0.f : m_used;
      float sum = 0.f;
#pragma unroll
      for (int c = 0; c < BN / 64; ++c) {
        uint32_t pk[32];
#pragma unroll
        for (int e = 0; e < 32; ++e) {
          const float a0 = ex2(x[c * 64 + 2 * e] - ref);
          const float a1 = ex2(x[c * 64 + 2 * e + 1] - ref);
          sum += a0 + a1;
          pk[e] = pack_bf16(a0, a1);
        }
        tmem_st32(lane_addr + sb * S_COLS + c * 32, pk);
      }
      l += sum;
      tmem_st_wait();
      tc_fence_before();
      mbar_arrive(&p_full[sb]);
    }
    // epilogue: O / l -> global, lse
    if (__all_sync(0xffffffffu, ok && !abort_flag)) {
      bool have = true;
      if (i > 0) have = __all_sync(0xffffffffu, mbar_wait(&o_done, (i - 1) & 1, &abort_flag, p.status, 33));
      tc_fence_after();
      if (have) {
        const float inv = l > 0.f ? 1.f / l : 0.f;
        const bool row_ok = m < p.S;
        char* orow = static_cast<char*>(p.o) +
                     (b * p.os[0] + hq * p.os[1] + (int64_t)m * p.os[2]) * (p.out_bf16 ? 2 : 4);
#pragma unroll
        for (int c = 0; c < D / 32; ++c) {
          uint32_t rr[32];
          if (i > 0) {
            tmem_ld32(lane_addr + O_COL + c * 32, rr);
            tmem_ld_wait();
          } else {
#pragma unroll
            for (int e = 0; e < 32; ++e) rr[e] = 0u;
          }
          if (!row_ok) continue;
          if (p.out_bf16) {
            uint4* dst = reinterpret_cast<uint4*>(orow + c * 64);
#pragma unroll
            for (int q4 = 0; q4 < 4; ++q4) {
              uint32_t w4[4];
#pragma unroll
              for (int e = 0; e < 4; ++e)
                w4[e] = pack_bf16(__uint_as_float(rr[q4 * 8 + 2 * e]) * inv, __uint_as_float(rr[q4 * 8 + 2 * e + 1]) * inv);
              dst[q4] = make_uint4(w4[0], w4[1], w4[2], w4[3]);
            }
          } else {
            float4* dst = reinterpret_cast<float4*>(orow + c * 128);
#pragma unroll
            for (int q4 = 0; q4 < 8; ++q4)
              dst[q4] = make_float4(__uint_as_float(rr[q4 * 4]) * inv, __uint_as_float(rr[q4 * 4 + 1]) * inv,
                                    __uint_as_float(rr[q4 * 4 + 2]) * inv, __uint_as_float(rr[q4 * 4 + 3]) * inv);
          }
        }
        if (p.lse && row_ok)
          p.lse[((int64_t)b * p.Hq + hq) * p.S + m] =
              l > 0.f ? (m_used + log2f(l)) * 0.69314718055994530942f : -INFINITY;
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 5) tmem_dealloc(tmem, kTmemCols);
}

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  if (!fn) {
    void* ptr = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(ptr);
  }
  return fn;
}

// [B, H, S, D] bf16 with element strides (b, h, s) -> 4-D map, 64 x 128 boxes,
// 128-byte swizzle, zero fill outside the tensor.
bool make_map(CUtensorMap* map, const void* base, int B, int H, int S, int D, const int64_t st[3]) {
  auto fn = encode_fn();
  if (!fn) return false;
  cuuint64_t dims[4] = {(cuuint64_t)D, (cuuint64_t)S, (cuuint64_t)H, (cuuint64_t)B};
  cuuint64_t strides[3] = {(cuuint64_t)st[2] * 2, (cuuint64_t)st[1] * 2, (cuuint64_t)st[0] * 2};
  // broadcast-free strides must be non-zero for TMA; a single head or batch
  // can take any stride
  if (H == 1) strides[1] = strides[0] * (cuuint64_t)S;
  if (B == 1) strides[2] = strides[1] * (cuuint64_t)H;
  cuuint32_t box[4] = {64, 128, 1, 1};
  cuuint32_t es[4] = {1, 1, 1, 1};
  CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void*>(base), dims, strides, box, es,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

template <int D>
cudaError_t launch_d(const PrefillLaunch& a, cudaStream_t st) {
  CUtensorMap mq, mk, mv;
  if (!make_map(&mq, a.q, a.B, a.Hq, a.S, D, a.qs) || !make_map(&mk, a.k, a.B, a.Hkv, a.S, D, a.ks) ||
      !make_map(&mv, a.v, a.B, a.Hkv, a.S, D, a.vs))
    return cudaErrorInvalidValue;
  TcParams p;
  memset(&p, 0, sizeof(p));
  p.B = a.B; p.Hq = a.Hq; p.Hkv = a.Hkv; p.S = a.S; p.group = a.Hq / a.Hkv;
  p.mask = a.mask; p.sink = a.sink; p.window = a.window; p.ring_blocks = a.ring_blocks;
  p.cs = (a.ring_blocks > 1 && (a.S / a.ring_blocks) % BN != 0) ? 64 : BN;
  p.scale_log2 = a.scale_log2;
  p.o = a.o;
  for (int i = 0; i < 3; ++i) p.os[i] = a.os[i];
  p.lse = a.lse;
  p.out_bf16 = a.out_bf16;
  p.status = device_status_word();
  if (!p.status) return cudaErrorInvalidValue;
  const int smem = Smem<D>::kBytes + 1024;
  cudaError_t e = cudaFuncSetAttribute(prefill_tc_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  dim3 grid((unsigned)((a.S + BM - 1) / BM), (unsigned)(a.B * a.Hq));
  prefill_tc_kernel<D><<<grid, kThreads, smem, st>>>(mq, mk, mv, p);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_prefill(const PrefillLaunch& a, cudaStream_t st) {
  if (a.ring_blocks > 1 && (a.S / a.ring_blocks) % 64 != 0) return cudaErrorInvalidValue;
  return a.d == 128 ? launch_d<128>(a, st) : launch_d<64>(a, st);
}

}  // namespace yr
