// attn_bwd: gradients of the exact softmax attention with the rotation applied
// to Q and K, on the tcgen05 tensor cores of sm_103a.
//
// For O = softmax(scale * Qr Kr^T) V (Qr, Kr the rotated q and k; "Context
// Window Scaling ...", Section 1 for the attention and Section 2 for the
// rotation), with dO the gradient of the output, LSE the forward's row
// log-sum-exp and D = rowsum(dO * O):
//   P = exp(scale S - LSE),  dP = dO V^T,  dS = P * (dP - D)
//   dV = P^T dO,  dKr = scale dS^T Qr,  dQr = scale dS Kr
//   dk = R_n^T dKr,  dq = R_m^T dQr  (the rotation is orthogonal).
// Two kernels, each one CTA per 128-row tile:
//   bwd_kv_kernel: a 128-key tile of one (batch, KV head) walks the query
//     tiles (of every query head of its group) that see it.  TMEM: S^T | dP^T
//     | dV | dK.  Each query tile is taken as two 64-query halves with their
//     own barriers: P^T and dS^T of a half are written as bf16 over its first
//     32 columns of S^T and dP^T and feed its dV and dK products from TMEM,
//     after which that half's S^T and dP^T of the next query tile are
//     computed, while the other half's rows run.
//   bwd_q_kernel: a 128-query tile walks its key tiles.  TMEM: S | S | dP |
//     dQ; dS overwrites S and feeds the dQ product.
// Roles (384 threads): warps 0-3 and 4-7 are two row groups on the same TMEM
// lanes (thread r owns tile row r), group 0 taking columns 0-63 and group 1
// columns 64-127 of each S / dP tile, so two warps per SM sub-partition hide
// each other's latency; warp 8 MMA (converged, one elected lane issues),
// warp 9 TMA producer, warps 10-11 only lend registers (setmaxnreg).  Each
// group writes its bf16 P / dS over its own, already read, columns (group 0
// at 0-31, group 1 at 64-95).  The epilogues apply the softmax scale and the
// inverse rotation.  Every wait is bounded.
#include <math.h>
#include <string.h>

#include <algorithm>
#include <type_traits>

#include "common.cuh"
#include "internal.h"
#include "tc_ptx.cuh"

namespace yr {
namespace {

using namespace tc;

constexpr int BT = 128;        // rows per tile
constexpr int kThreads = 384;  // warps 0-7 rows, 8 MMA, 9 TMA, 10-11 idle
constexpr int kMmaWarp = 8;
constexpr int kLoadWarp = 9;
constexpr uint32_t kRegsRows = 216;   // 2 x 128 x 216 + 128 x 72 = 384 x 168
constexpr uint32_t kRegsControl = 72;
static_assert(2 * 128 * kRegsRows + 128 * kRegsControl <= kThreads * 168, "register split");
constexpr int NS = 2;          // pipeline stages
constexpr uint32_t kTmemCols = 512;
constexpr float kLog2e = 1.4426950408889634f;
constexpr int kPrefetch = 4;   // iterations whose tiles the producer prefetches into L2

struct BwdParams {
  int B, Hq, Hkv, S, group, n_tiles;
  int hgroup;        // heads per scheduling group
  int mask, sink, window;
  float scale_log2;  // scale * log2(e)
  float scale;       // softmax scale (applied to dQ and dK)
  const float* lse2; // [B, Hq, S], -LSE * log2(e)
  const float* dsum; // [B, Hq, S], rowsum(dO * O)
  void* out_a;       // dK (kv kernel) or dQ (q kernel)
  int64_t oas[3];
  void* out_b;       // dV (kv kernel)
  int64_t obs[3];
  int out_bf16;
  int* status;
  RopeFreqs f;       // frequencies of the inverse rotation
};

__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

__device__ __forceinline__ float4 lds_f4(uint32_t addr) {
  float4 v;
  asm volatile("ld.shared.v4.f32 {%0, %1, %2, %3}, [%4];" : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w) : "r"(addr));
  return v;
}

// CTA i of a grid of U units (batch x head) x n_tiles tiles, taken in groups
// of hg units: every tile of a group before the next group, tile-major inside
// a group, so the CTAs resident at once share a few heads and the tiles they
// all re-read (Q and dO, or K and V) stay in L2.
__device__ __forceinline__ void sched_unit(int i, int U, int n_tiles, int hg, int& tile, int& unit) {
  const int per_group = hg * n_tiles;
  const int full = U / hg;
  int g, r, hc;
  if (i < full * per_group) {
    g = i / per_group;
    r = i - g * per_group;
    hc = hg;
  } else {
    g = full;
    r = i - full * per_group;
    hc = U - full * hg;
  }
  tile = r / hc;
  unit = g * hg + r % hc;
}

// Does a (query tile, key tile) pair need the element mask?
__device__ __forceinline__ bool tile_needs_mask(const BwdParams& p, int m0, int n0) {
  if (p.mask == YR_MASK_NONE) return false;
  const int m1 = m0 + BT - 1, n1 = n0 + BT - 1;
  if (n1 > m0) return true;  // some key is after some query
  // some non-sink key farther than the window from some query
  return p.mask == YR_MASK_SINK_WINDOW && n1 >= p.sink && m1 - max(n0, p.sink) >= p.window;
}

// Query tiles that see key tile kt: [lo, hi] (hi < lo when none).
__device__ __forceinline__ void query_tiles(const BwdParams& p, int kt, int& lo, int& hi) {
  lo = p.mask == YR_MASK_NONE ? 0 : kt;
  hi = p.n_tiles - 1;
  const int n0 = kt * BT, n1 = n0 + BT - 1;
  if (p.mask == YR_MASK_SINK_WINDOW && n0 >= p.sink) hi = min(hi, (n1 + p.window - 1) / BT);
}

// Key tiles that query tile qt sees: sink tiles [0, sink_hi] and the window
// tiles [w_lo, hi]; returns the key tile of step u, or -1 past the end.
struct KeyWalk {
  int hi, sink_hi, w_lo;
  __device__ void init(const BwdParams& p, int qt) {
    const int m0 = qt * BT, m1 = m0 + BT - 1;
    hi = p.mask == YR_MASK_NONE ? p.n_tiles - 1 : qt;
    sink_hi = -1;
    w_lo = 0;
    if (p.mask == YR_MASK_SINK_WINDOW) {
      sink_hi = p.sink > 0 ? min(hi, (p.sink - 1) / BT) : -1;
      const int first = m0 - p.window + 1;  // the first key row m0 sees
      w_lo = first <= 0 ? 0 : first / BT;
      if (w_lo <= sink_hi + 1) { w_lo = 0; sink_hi = -1; }
    }
    (void)m1;
  }
  __device__ int count() const { return (sink_hi + 1) + (hi - w_lo + 1); }
  __device__ int tile(int u) const { return u <= sink_hi ? u : w_lo + (u - sink_hi - 1); }
};

template <int D>
struct Cfg {
  static constexpr int kTile = BT * D * 2;  // bytes of a 128-row bf16 tile
  static constexpr int kVec = BT * 4;       // 128 floats
  // kv kernel: K, V once; per stage Q, dO, LSE, D
  static constexpr int kvK = 0, kvV = kTile, kvStage0 = 2 * kTile;
  static constexpr int kvStage = 2 * kTile + 2 * 1024;  // Q | dO | LSE | D (vectors padded to 1 KB)
  static constexpr int kvBytes = kvStage0 + NS * kvStage;
  // q kernel: Q, dO once; K in three slots, V in two
  static constexpr int qKSlots = 3, qVSlots = 2;
  static constexpr int qQ = 0, qDO = kTile, qK0 = 2 * kTile, qV0 = qK0 + qKSlots * kTile;
  static constexpr int qBytes = qV0 + qVSlots * kTile;
};

// Row `row` of a 128 x D fp32 TMEM block -> global, scaled by `mult` and,
// when `unrotate`, rotated back by -row * theta (pairs (i, i + D/2)).
// Columns [32c, 32c + 32) and their partners [D/2 + 32c, ...) are handled
// together, 64 values at a time.
template <int D>
__device__ __forceinline__ void store_rows(const BwdParams& p, uint32_t taddr, void* out, const int64_t st[3],
                                           int b, int h, int row, float mult, bool unrotate, bool have, int c_begin,
                                           int c_end) {
  char* dst = static_cast<char*>(out) + (b * st[0] + h * st[1] + (int64_t)row * st[2]) * (p.out_bf16 ? 2 : 4);
#pragma unroll
  for (int c = 0; c < D / 64; ++c) {
    if (c < c_begin || c >= c_end) continue;
    uint32_t lo[32], hi[32];
    if (have) {
      tmem_ld32(taddr + c * 32, lo);
      tmem_ld32(taddr + D / 2 + c * 32, hi);
      tmem_ld_wait();
      reg_fence32(lo);
      reg_fence32(hi);
    }
    float a[32], bb[32];
#pragma unroll
    for (int e = 0; e < 32; ++e) {
      a[e] = have ? __uint_as_float(lo[e]) * mult : 0.f;
      bb[e] = have ? __uint_as_float(hi[e]) * mult : 0.f;
    }
    if (unrotate && !p.f.identity) {
#pragma unroll
      for (int e = 0; e < 32; ++e) {
        float cs, sn;
        turn_cos_sin<true>((float)row, p.f.f[c * 32 + e], cs, sn);
        const float x = a[e], y = bb[e];
        a[e] = x * cs + y * sn;
        bb[e] = y * cs - x * sn;
      }
    }
#pragma unroll
    for (int part = 0; part < 2; ++part) {
      const float* v = part ? bb : a;
      const int col = part * (D / 2) + c * 32;
      if (p.out_bf16) {
        uint4* d4 = reinterpret_cast<uint4*>(dst + col * 2);
#pragma unroll
        for (int q = 0; q < 4; ++q)
          d4[q] = make_uint4(pack_bf16(v[8 * q], v[8 * q + 1]), pack_bf16(v[8 * q + 2], v[8 * q + 3]),
                             pack_bf16(v[8 * q + 4], v[8 * q + 5]), pack_bf16(v[8 * q + 6], v[8 * q + 7]));
      } else {
        float4* d4 = reinterpret_cast<float4*>(dst + col * 4);
#pragma unroll
        for (int q = 0; q < 8; ++q) d4[q] = make_float4(v[4 * q], v[4 * q + 1], v[4 * q + 2], v[4 * q + 3]);
      }
    }
  }
}

// ---------------------------------------------------------------------------
// dK, dV: one CTA per (key tile, batch, KV head); in each scheduling group key
// tiles ascending (the causal tiles with the most query tiles first).
template <int D>
__global__ void __launch_bounds__(kThreads, 1)
    bwd_kv_kernel(const __grid_constant__ CUtensorMap tq, const __grid_constant__ CUtensorMap tk,
                  const __grid_constant__ CUtensorMap tv, const __grid_constant__ CUtensorMap tdo,
                  const __grid_constant__ BwdParams p) {
  using C = Cfg<D>;
  constexpr int ATOMS = D / 64;
  constexpr int ATOM_BYTES = BT * 128;
  constexpr uint32_t ID_SSH = idesc_bf16_f32(BT, BT / 2, false);  // [128 x D] x [64 x D]^T
  constexpr uint32_t ID_TS = idesc_bf16_f32(BT, D, true);         // TMEM [128 x 16] x smem [16 x D]
  constexpr uint32_t C_S = 0, C_DP = 128, C_DV = 256, C_DK = 256 + D;

  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  __shared__ uint64_t kv_full, full[NS], empty[NS], s_full[2], p_full[2], o_done, drain;
  __shared__ uint32_t tmem_slot;
  __shared__ volatile int abort_flag;

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  int kt, bkv;
  sched_unit((int)blockIdx.x, p.B * p.Hkv, p.n_tiles, p.hgroup, kt, bkv);
  const int b = bkv / p.Hkv, hkv = bkv % p.Hkv;
  const int n0 = kt * BT;
  int qlo, qhi;
  query_tiles(p, kt, qlo, qhi);
  const int per_head = max(0, qhi - qlo + 1);
  const int iters = per_head * p.group;  // (query head of the group, query tile)

  if (tid == 0) {
    abort_flag = 0;
    mbar_init(&kv_full, 1);
    for (int s = 0; s < NS; ++s) { mbar_init(&full[s], 1); mbar_init(&empty[s], 1); }
    for (int h = 0; h < 2; ++h) {
      mbar_init(&s_full[h], 1);
      mbar_init(&p_full[h], 4);  // one arrival per warp of the half's row group
    }
    mbar_init(&o_done, 1);
    mbar_init(&drain, 1);
    fence_mbar_init();
  }
  if (warp == kMmaWarp) tmem_alloc(&tmem_slot, kTmemCols);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = tmem_slot;

  if (warp >= 8) {
   reg_dealloc<kRegsControl>();
   if (warp == kLoadWarp) {
    if (lane == 0) {
      tma_prefetch_desc(&tq); tma_prefetch_desc(&tk); tma_prefetch_desc(&tv); tma_prefetch_desc(&tdo);
      // with no query tile to visit nothing is loaded (nobody would wait)
      if (iters > 0) {
        mbar_arrive_expect_tx(&kv_full, 2 * C::kTile);
        for (int a = 0; a < ATOMS; ++a) {
          tma_load_4d(smem + C::kvK + a * ATOM_BYTES, &tk, &kv_full, a * 64, n0, hkv, b);
          tma_load_4d(smem + C::kvV + a * ATOM_BYTES, &tv, &kv_full, a * 64, n0, hkv, b);
        }
      }
      int uses[NS] = {0, 0};
      // the tiles of the first iterations go to L2 ahead of their loads
      auto prefetch = [&](int i) {
        if (i >= iters) return;
        const int hq = hkv * p.group + i / per_head;
        const int m0 = (qlo + i % per_head) * BT;
        for (int a = 0; a < ATOMS; ++a) {
          tma_prefetch_l2_4d(&tq, a * 64, m0, hq, b);
          tma_prefetch_l2_4d(&tdo, a * 64, m0, hq, b);
        }
        const int64_t row0 = ((int64_t)b * p.Hq + hq) * p.S + m0;
        bulk_prefetch_l2(p.lse2 + row0, C::kVec);
        bulk_prefetch_l2(p.dsum + row0, C::kVec);
      };
      for (int i = 0; i < kPrefetch; ++i) prefetch(i);
      for (int i = 0; i < iters; ++i) {
        const int s = i % NS;
        const int hq = hkv * p.group + i / per_head;
        const int m0 = (qlo + i % per_head) * BT;
        prefetch(i + kPrefetch);
        if (!mbar_wait(&empty[s], ((i / NS) & 1) ^ 1, &abort_flag, p.status, 51)) break;
        uint8_t* st = smem + C::kvStage0 + s * C::kvStage;
        mbar_arrive_expect_tx(&full[s], 2 * C::kTile + 2 * C::kVec);
        for (int a = 0; a < ATOMS; ++a) {
          tma_load_4d(st + a * ATOM_BYTES, &tq, &full[s], a * 64, m0, hq, b);
          tma_load_4d(st + C::kTile + a * ATOM_BYTES, &tdo, &full[s], a * 64, m0, hq, b);
        }
        const int64_t row0 = ((int64_t)b * p.Hq + hq) * p.S + m0;
        bulk_g2s(st + 2 * C::kTile, p.lse2 + row0, C::kVec, &full[s]);
        bulk_g2s(st + 2 * C::kTile + 1024, p.dsum + row0, C::kVec, &full[s]);
        ++uses[s];
      }
      if (abort_flag) {
        if (iters > 0) mbar_wait_drain(&kv_full, 0, 200000000ll);
        for (int s = 0; s < NS; ++s)
          if (uses[s]) mbar_wait_drain(&full[s], (uses[s] - 1) & 1, 200000000ll);
      }
    }
    __syncwarp();
   } else if (warp == kMmaWarp) {
    const bool leader = elect_one();
    const uint64_t dK = sdesc_sw128(smem_u32(smem + C::kvK), 16, 1024);
    const uint64_t dV = sdesc_sw128(smem_u32(smem + C::kvV), 16, 1024);
    auto wait = [&](uint64_t* bar, uint32_t par, int code) -> bool {
      return __all_sync(0xffffffffu, mbar_wait(bar, par, &abort_flag, p.status, code));
    };
    // S^T and dP^T of query half h (64 queries) of iteration i: N = 64
    auto issue_sdp = [&](int i, int h) {
      const uint32_t st = smem_u32(smem + C::kvStage0 + (i % NS) * C::kvStage) + h * (BT / 2) * 128;
      const uint64_t dQk = sdesc_sw128(st, 16, 1024), dDOk = sdesc_sw128(st + C::kTile, 16, 1024);
#pragma unroll
      for (int kk = 0; kk < D / 16; ++kk) {
        const uint64_t off = (uint64_t)(((kk >> 2) * ATOM_BYTES + (kk & 3) * 32) >> 4);
        mma_ss(tmem + C_S + 64 * h, dK + off, dQk + off, ID_SSH, kk > 0);     // S^T = K Q^T
        mma_ss(tmem + C_DP + 64 * h, dV + off, dDOk + off, ID_SSH, kk > 0);   // dP^T = V dO^T
      }
      mma_commit(&s_full[h]);
    };
    // dV += P^T dO and dK += dS^T Q over the 64 queries of half h
    auto issue_dvdk = [&](int i, int h) {
      const uint32_t st = smem_u32(smem + C::kvStage0 + (i % NS) * C::kvStage);
      const uint64_t dQn = sdesc_sw128(st, ATOM_BYTES, 1024), dDOn = sdesc_sw128(st + C::kTile, ATOM_BYTES, 1024);
#pragma unroll
      for (int kq = 0; kq < 4; ++kq) {
        const int kk = 4 * h + kq;  // 16-query step within the tile
        const uint64_t off = (uint64_t)(kk * 2048 >> 4);
        const uint32_t a_off = 64 * h + kq * 8;  // the half's packed bf16 columns
        mma_ts(tmem + C_DV, tmem + C_S + a_off, dDOn + off, ID_TS, (i > 0 || kk > 0) ? 1u : 0u);
        mma_ts(tmem + C_DK, tmem + C_DP + a_off, dQn + off, ID_TS, (i > 0 || kk > 0) ? 1u : 0u);
      }
    };
    bool ok = iters == 0 || wait(&kv_full, 0, 61);
    if (ok && iters > 0) {
      ok = wait(&full[0], 0, 62);
      tc_fence_after();
      if (ok && leader) { issue_sdp(0, 0); issue_sdp(0, 1); }
      __syncwarp();
    }
    // per half: its dV/dK products of iteration i, then its S^T/dP^T of
    // iteration i + 1 (into the columns those products have just read; the
    // tensor pipe runs a CTA's MMAs in issue order), so one row group's
    // softmax overlaps the other half's products
    for (int i = 0; ok && i < iters; ++i) {
      const int s = i % NS;
      for (int h = 0; h < 2; ++h) {
        if (!wait(&p_full[h], i & 1, 63 + h)) { ok = false; break; }
        tc_fence_after();
        if (leader) {
          issue_dvdk(i, h);
          if (h == 1) mma_commit(&empty[s]);
        }
        __syncwarp();
        if (i + 1 < iters) {
          if (h == 0 && !wait(&full[(i + 1) % NS], ((i + 1) / NS) & 1, 62)) { ok = false; break; }
          tc_fence_after();
          if (leader) issue_sdp(i + 1, h);
          __syncwarp();
        }
      }
    }
    if (leader) {
      mma_commit(&o_done);
      mma_commit(&drain);
      mbar_wait_drain(&drain, 0, 200000000ll);
    }
    __syncwarp();
   }
  } else {
    reg_alloc<kRegsRows>();
    // ---------------- rows: thread r = key row n0 + r; group wg takes query
    // half wg (columns 64 wg .. 64 wg + 63) of each S^T / dP^T tile ---------
    const int wg = warp >> 2;
    const int r = (warp & 3) * 32 + lane;
    const int n = n0 + r;
    const uint32_t lane_addr = tmem + ((uint32_t)((warp & 3) * 32) << 16);
    const int col0 = wg * 64;
    const float sl2 = p.scale_log2;
    bool ok = true;
    for (int i = 0; i < iters; ++i) {
      const int s = i % NS;
      const int m0 = (qlo + i % per_head) * BT;
      const uint32_t vec = smem_u32(smem + C::kvStage0 + s * C::kvStage + 2 * C::kTile);  // -LSE*log2e | D
      ok = __all_sync(0xffffffffu, mbar_wait(&s_full[wg], i & 1, &abort_flag, p.status, 71));
      // the LSE / D vectors of this stage landed with full[s] (already
      // complete: the MMA waited for it before the products of s_full); the
      // stage is refilled only after both halves' products have run
      if (ok) ok = __all_sync(0xffffffffu, mbar_wait(&full[s], (i / NS) & 1, &abort_flag, p.status, 73));
      if (!ok) break;
      tc_fence_after();
      const bool need_mask = tile_needs_mask(p, m0, n0);
      uint32_t sr[2][32], dr[2][32];
      tmem_ld32(lane_addr + C_S + col0, sr[0]);
      tmem_ld32(lane_addr + C_S + col0 + 32, sr[1]);
      tmem_ld32(lane_addr + C_DP + col0, dr[0]);
      tmem_ld32(lane_addr + C_DP + col0 + 32, dr[1]);
      tmem_ld_wait();
      reg_fence32(sr[0]); reg_fence32(sr[1]); reg_fence32(dr[0]); reg_fence32(dr[1]);
      // Visible columns of key row n: e >= e_lo (causal: query m0 + col0 + e
      // >= n) and, for a non-sink key under the window, e < e_hi.  The
      // masked and unmasked loops are separate copies: a per-element test
      // on the tile flag costs more than the whole unmasked pass.
      const int e_lo = n - (m0 + col0);
      const int e_hi = (p.mask == YR_MASK_SINK_WINDOW && n >= p.sink) ? n + p.window - (m0 + col0) : BT;
      uint32_t pk[32], dk[32];
      auto softmax = [&](auto masked) {
#pragma unroll
        for (int q4 = 0; q4 < 16; ++q4) {  // 4 query columns per step
          const float4 l4 = lds_f4(vec + (col0 + 4 * q4) * 4);
          const float4 d4 = lds_f4(vec + 1024 + (col0 + 4 * q4) * 4);
          const float nl[4] = {l4.x, l4.y, l4.z, l4.w}, dvv[4] = {d4.x, d4.y, d4.z, d4.w};
          float pp[4], dd[4];
          // two columns per packed op: P = 2^(S scale log2e - LSE log2e),
          // dS = P (dP - D)
#pragma unroll
          for (int t = 0; t < 4; t += 2) {
            const int e = 4 * q4 + t;  // column within the group's 64
            const float sv0 = __uint_as_float(sr[e >> 5][e & 31]), sv1 = __uint_as_float(sr[(e + 1) >> 5][(e + 1) & 31]);
            const float dv0 = __uint_as_float(dr[e >> 5][e & 31]), dv1 = __uint_as_float(dr[(e + 1) >> 5][(e + 1) & 31]);
            float a0, a1, g0, g1;
            fma2(a0, a1, sv0, sv1, sl2, sl2, nl[t], nl[t + 1]);
            float p0 = ex2(a0), p1 = ex2(a1);
            if (decltype(masked)::value) {
              if (e < e_lo || e >= e_hi) p0 = 0.f;
              if (e + 1 < e_lo || e + 1 >= e_hi) p1 = 0.f;
            }
            fma2(g0, g1, dvv[t], dvv[t + 1], -1.f, -1.f, dv0, dv1);
            mul2(dd[t], dd[t + 1], p0, p1, g0, g1);
            pp[t] = p0;
            pp[t + 1] = p1;
          }
          pk[2 * q4] = pack_bf16(pp[0], pp[1]);
          pk[2 * q4 + 1] = pack_bf16(pp[2], pp[3]);
          dk[2 * q4] = pack_bf16(dd[0], dd[1]);
          dk[2 * q4 + 1] = pack_bf16(dd[2], dd[3]);
        }
      };
      if (need_mask) softmax(std::true_type{});
      else softmax(std::false_type{});
      tmem_st32(lane_addr + C_S + col0, pk);
      tmem_st32(lane_addr + C_DP + col0, dk);
      tmem_st_wait();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&p_full[wg]);
    }
    if (__all_sync(0xffffffffu, ok && !abort_flag)) {
      bool have = iters > 0;
      if (have) have = __all_sync(0xffffffffu, mbar_wait(&o_done, 0, &abort_flag, p.status, 72));
      tc_fence_after();
      if (!abort_flag) {
        // each group stores half of the column pairs (i, i + D/2)
        store_rows<D>(p, lane_addr + C_DV, p.out_b, p.obs, b, hkv, n, 1.f, false, have, wg, wg + 1);
        store_rows<D>(p, lane_addr + C_DK, p.out_a, p.oas, b, hkv, n, p.scale, true, have, wg, wg + 1);
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == kMmaWarp) tmem_dealloc(tmem, kTmemCols);
}

// ---------------------------------------------------------------------------
// dQ: one CTA per (query tile, batch, query head); in each scheduling group the
// heaviest query tiles first.
// TMEM: S[0] | S[1] | dP | dQ.  S is double-buffered, so S(i + 1) is computed
// while the rows work on iteration i; dP(i + 1) waits only until the rows have
// read dP(i) into registers.  K has three shared-memory slots (read by S and
// dQ) and V two (read by dP alone), so the load of a later tile never waits
// for the products of the current one.
template <int D>
__global__ void __launch_bounds__(kThreads, 1)
    bwd_q_kernel(const __grid_constant__ CUtensorMap tq, const __grid_constant__ CUtensorMap tk,
                 const __grid_constant__ CUtensorMap tv, const __grid_constant__ CUtensorMap tdo,
                 const __grid_constant__ BwdParams p) {
  using C = Cfg<D>;
  constexpr int ATOMS = D / 64;
  constexpr int ATOM_BYTES = BT * 128;
  constexpr uint32_t ID_SS = idesc_bf16_f32(BT, BT, false);
  constexpr uint32_t ID_TS = idesc_bf16_f32(BT, D, true);
  constexpr uint32_t C_S0 = 0, C_DP = 256, C_DQ = 384;

  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  __shared__ uint64_t q_full, k_full[C::qKSlots], k_empty[C::qKSlots], v_full[C::qVSlots], v_empty[C::qVSlots];
  __shared__ uint64_t s_full[2], dp_free, p_full[2], o_done, drain;
  __shared__ uint32_t tmem_slot;
  __shared__ volatile int abort_flag;

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  int t, bh;
  sched_unit((int)blockIdx.x, p.B * p.Hq, p.n_tiles, p.hgroup, t, bh);
  const int qt = p.n_tiles - 1 - t;
  const int b = bh / p.Hq, hq = bh % p.Hq;
  const int hkv = hq / p.group;
  const int m0 = qt * BT;
  KeyWalk walk;
  walk.init(p, qt);
  const int iters = walk.count();

  if (tid == 0) {
    abort_flag = 0;
    mbar_init(&q_full, 1);
    for (int s = 0; s < C::qKSlots; ++s) { mbar_init(&k_full[s], 1); mbar_init(&k_empty[s], 1); }
    for (int s = 0; s < C::qVSlots; ++s) { mbar_init(&v_full[s], 1); mbar_init(&v_empty[s], 1); }
    mbar_init(&s_full[0], 1);
    mbar_init(&s_full[1], 1);
    mbar_init(&dp_free, 8);  // one arrival per row warp
    // p_full alternates with the S buffer: the rows may finish iteration i + 1
    // before the MMA warp has seen iteration i complete
    mbar_init(&p_full[0], 8);
    mbar_init(&p_full[1], 8);
    mbar_init(&o_done, 1);
    mbar_init(&drain, 1);
    fence_mbar_init();
  }
  if (warp == kMmaWarp) tmem_alloc(&tmem_slot, kTmemCols);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = tmem_slot;

  if (warp >= 8) {
   reg_dealloc<kRegsControl>();
   if (warp == kLoadWarp) {
    if (lane == 0) {
      tma_prefetch_desc(&tq); tma_prefetch_desc(&tk); tma_prefetch_desc(&tv); tma_prefetch_desc(&tdo);
      if (iters > 0) {
        mbar_arrive_expect_tx(&q_full, 2 * C::kTile);
        for (int a = 0; a < ATOMS; ++a) {
          tma_load_4d(smem + C::qQ + a * ATOM_BYTES, &tq, &q_full, a * 64, m0, hq, b);
          tma_load_4d(smem + C::qDO + a * ATOM_BYTES, &tdo, &q_full, a * 64, m0, hq, b);
        }
      }
      int kuses[C::qKSlots] = {}, vuses[C::qVSlots] = {};
      auto prefetch = [&](int i) {
        if (i >= iters) return;
        const int nk = walk.tile(i) * BT;
        for (int a = 0; a < ATOMS; ++a) {
          tma_prefetch_l2_4d(&tk, a * 64, nk, hkv, b);
          tma_prefetch_l2_4d(&tv, a * 64, nk, hkv, b);
        }
      };
      for (int i = 0; i < kPrefetch; ++i) prefetch(i);
      for (int i = 0; i < iters; ++i) {
        const int ks = i % C::qKSlots, vs = i % C::qVSlots;
        const int nk0 = walk.tile(i) * BT;
        prefetch(i + kPrefetch);
        if (!mbar_wait(&k_empty[ks], ((i / C::qKSlots) & 1) ^ 1, &abort_flag, p.status, 81)) break;
        uint8_t* kd = smem + C::qK0 + ks * C::kTile;
        mbar_arrive_expect_tx(&k_full[ks], C::kTile);
        for (int a = 0; a < ATOMS; ++a) tma_load_4d(kd + a * ATOM_BYTES, &tk, &k_full[ks], a * 64, nk0, hkv, b);
        ++kuses[ks];
        if (!mbar_wait(&v_empty[vs], ((i / C::qVSlots) & 1) ^ 1, &abort_flag, p.status, 82)) break;
        uint8_t* vd = smem + C::qV0 + vs * C::kTile;
        mbar_arrive_expect_tx(&v_full[vs], C::kTile);
        for (int a = 0; a < ATOMS; ++a) tma_load_4d(vd + a * ATOM_BYTES, &tv, &v_full[vs], a * 64, nk0, hkv, b);
        ++vuses[vs];
      }
      if (abort_flag) {
        if (iters > 0) mbar_wait_drain(&q_full, 0, 200000000ll);
        for (int s = 0; s < C::qKSlots; ++s)
          if (kuses[s]) mbar_wait_drain(&k_full[s], (kuses[s] - 1) & 1, 200000000ll);
        for (int s = 0; s < C::qVSlots; ++s)
          if (vuses[s]) mbar_wait_drain(&v_full[s], (vuses[s] - 1) & 1, 200000000ll);
      }
    }
    __syncwarp();
   } else if (warp == kMmaWarp) {
    const bool leader = elect_one();
    const uint64_t dQk = sdesc_sw128(smem_u32(smem + C::qQ), 16, 1024);
    const uint64_t dDOk = sdesc_sw128(smem_u32(smem + C::qDO), 16, 1024);
    auto wait = [&](uint64_t* bar, uint32_t par, int code) -> bool {
      return __all_sync(0xffffffffu, mbar_wait(bar, par, &abort_flag, p.status, code));
    };
    auto k_addr = [&](int i) { return smem_u32(smem + C::qK0 + (i % C::qKSlots) * C::kTile); };
    auto v_addr = [&](int i) { return smem_u32(smem + C::qV0 + (i % C::qVSlots) * C::kTile); };
    auto issue_s = [&](int i) {  // S(i) = Q K(i)^T into S[i & 1]
      const uint64_t dKk = sdesc_sw128(k_addr(i), 16, 1024);
#pragma unroll
      for (int kk = 0; kk < D / 16; ++kk) {
        const uint64_t off = (uint64_t)(((kk >> 2) * ATOM_BYTES + (kk & 3) * 32) >> 4);
        mma_ss(tmem + C_S0 + 128 * (i & 1), dQk + off, dKk + off, ID_SS, kk > 0);
      }
    };
    auto issue_dp = [&](int i) {  // dP(i) = dO V(i)^T
      const uint64_t dVk = sdesc_sw128(v_addr(i), 16, 1024);
#pragma unroll
      for (int kk = 0; kk < D / 16; ++kk) {
        const uint64_t off = (uint64_t)(((kk >> 2) * ATOM_BYTES + (kk & 3) * 32) >> 4);
        mma_ss(tmem + C_DP, dDOk + off, dVk + off, ID_SS, kk > 0);
      }
      mma_commit(&v_empty[i % C::qVSlots]);
      mma_commit(&s_full[i & 1]);
    };
    bool ok = iters == 0 || wait(&q_full, 0, 91);
    if (ok && iters > 0) {
      ok = wait(&k_full[0], 0, 92) && wait(&v_full[0], 0, 94);
      tc_fence_after();
      if (ok && leader) { issue_s(0); issue_dp(0); }
      __syncwarp();
    }
    for (int i = 0; ok && i < iters; ++i) {
      if (i + 1 < iters) {
        const int j = i + 1;
        if (!wait(&k_full[j % C::qKSlots], (j / C::qKSlots) & 1, 92)) { ok = false; break; }
        tc_fence_after();
        if (leader) issue_s(j);  // the other S buffer: dQ(i - 1) read it and was issued before
        __syncwarp();
        if (!wait(&v_full[j % C::qVSlots], (j / C::qVSlots) & 1, 94) || !wait(&dp_free, i & 1, 95)) {
          ok = false;
          break;
        }
        tc_fence_after();
        if (leader) issue_dp(j);
        __syncwarp();
      }
      if (!wait(&p_full[i & 1], (i >> 1) & 1, 93)) { ok = false; break; }
      tc_fence_after();
      if (leader) {
        const uint64_t dKn = sdesc_sw128(k_addr(i), ATOM_BYTES, 1024);
        const uint32_t a0 = tmem + C_S0 + 128 * (i & 1);
#pragma unroll
        for (int kk = 0; kk < BT / 16; ++kk)
          mma_ts(tmem + C_DQ, a0 + (kk >> 2) * 64 + (kk & 3) * 8, dKn + (uint64_t)(kk * 2048 >> 4), ID_TS,
                 (i > 0 || kk > 0) ? 1u : 0u);  // dQ += dS K
        mma_commit(&k_empty[i % C::qKSlots]);
      }
      __syncwarp();
    }
    if (leader) {
      mma_commit(&o_done);
      mma_commit(&drain);
      mbar_wait_drain(&drain, 0, 200000000ll);
    }
    __syncwarp();
   }
  } else {
    reg_alloc<kRegsRows>();
    // ---------------- rows: thread r = query row m0 + r; group wg takes the
    // key columns 64 wg .. 64 wg + 63 of each S / dP tile --------------------
    const int wg = warp >> 2;
    const int r = (warp & 3) * 32 + lane;
    const int m = m0 + r;
    const uint32_t lane_addr = tmem + ((uint32_t)((warp & 3) * 32) << 16);
    const int col0 = wg * 64;
    const int64_t row = ((int64_t)b * p.Hq + hq) * p.S + m;
    const float nlse_l2 = p.lse2[row];  // -LSE * log2(e)
    const float dsum = p.dsum[row];
    const float sl2 = p.scale_log2;
    bool ok = true;
    for (int i = 0; i < iters; ++i) {
      const int nk0 = walk.tile(i) * BT;
      const uint32_t c_s = C_S0 + 128 * (i & 1);
      ok = __all_sync(0xffffffffu, mbar_wait(&s_full[i & 1], (i >> 1) & 1, &abort_flag, p.status, 101));
      if (!ok) break;
      tc_fence_after();
      const bool need_mask = tile_needs_mask(p, m0, nk0);
      uint32_t sr[2][32], dr[2][32];
      tmem_ld32(lane_addr + c_s + col0, sr[0]);
      tmem_ld32(lane_addr + c_s + col0 + 32, sr[1]);
      tmem_ld32(lane_addr + C_DP + col0, dr[0]);
      tmem_ld32(lane_addr + C_DP + col0 + 32, dr[1]);
      tmem_ld_wait();
      reg_fence32(sr[0]); reg_fence32(sr[1]); reg_fence32(dr[0]); reg_fence32(dr[1]);
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&dp_free);  // dP(i) is in registers: dP(i + 1) may overwrite it
      // Visible columns of query row m (key nk0 + col0 + e): e <= e_max
      // (causal) and, under the window, a sink key (e < e_sink) or one
      // inside the window (e > e_win).  Masked and unmasked loops are
      // separate copies, as in the dK/dV kernel.
      const int base = nk0 + col0;
      const bool sw = p.mask == YR_MASK_SINK_WINDOW;
      const int e_max = m - base;
      const int e_sink = sw ? p.sink - base : BT;
      const int e_win = sw ? m - p.window - base : -1;
      uint32_t dk[32];
      auto softmax = [&](auto masked) {
#pragma unroll
        for (int e2 = 0; e2 < 32; ++e2) {
          // two columns per packed op: P = 2^(S scale log2e - LSE log2e),
          // dS = P (dP - D)
          const int e = 2 * e2;
          const float sv0 = __uint_as_float(sr[e >> 5][e & 31]), sv1 = __uint_as_float(sr[(e + 1) >> 5][(e + 1) & 31]);
          const float dv0 = __uint_as_float(dr[e >> 5][e & 31]), dv1 = __uint_as_float(dr[(e + 1) >> 5][(e + 1) & 31]);
          float a0, a1, g0, g1, d0, d1;
          fma2(a0, a1, sv0, sv1, sl2, sl2, nlse_l2, nlse_l2);
          float p0 = ex2(a0), p1 = ex2(a1);
          if (decltype(masked)::value) {
            if (e > e_max || (e >= e_sink && e <= e_win)) p0 = 0.f;
            if (e + 1 > e_max || (e + 1 >= e_sink && e + 1 <= e_win)) p1 = 0.f;
          }
          fma2(g0, g1, dsum, dsum, -1.f, -1.f, dv0, dv1);
          mul2(d0, d1, p0, p1, g0, g1);
          dk[e2] = pack_bf16(d0, d1);
        }
      };
      if (need_mask) softmax(std::true_type{});
      else softmax(std::false_type{});
      tmem_st32(lane_addr + c_s + col0, dk);
      tmem_st_wait();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&p_full[i & 1]);
    }
    if (__all_sync(0xffffffffu, ok && !abort_flag)) {
      bool have = iters > 0;
      if (have) have = __all_sync(0xffffffffu, mbar_wait(&o_done, 0, &abort_flag, p.status, 102));
      tc_fence_after();
      if (!abort_flag) store_rows<D>(p, lane_addr + C_DQ, p.out_a, p.oas, b, hq, m, p.scale, true, have, wg, wg + 1);
    }
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == kMmaWarp) tmem_dealloc(tmem, kTmemCols);
}

// D = rowsum(dO * O) of [B, H, S, d] and lse2 = -LSE * log2(e) per row.  Each
// lane takes 16 contiguous bytes of a row of both tensors (8 bf16 or 4
// float32 elements), d / that many lanes share a row, so one warp covers
// 32 / (lanes per row) rows with one 16-byte load of each tensor per lane.
template <typename T>
__global__ void __launch_bounds__(256) dsum_kernel(const T* dout, const T* o, float* dsum, const float* lse,
                                                   float* lse2, int B, int H, int S, int d, int64_t ds0, int64_t ds1,
                                                   int64_t ds2, int64_t os0, int64_t os1, int64_t os2) {
  constexpr int EPL = 16 / (int)sizeof(T);  // elements per lane
  const int64_t rows = (int64_t)B * H * S;
  const int lane = threadIdx.x & 31;
  const int lpr = d / EPL;  // lanes per row: 8, 16 or 32 (d = 64 or 128)
  const int64_t row = ((int64_t)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5)) * (32 / lpr) + lane / lpr;
  const int sub = lane % lpr;
  float acc = 0.f;
  if (row < rows) {
    const int s = (int)(row % S);
    const int64_t bh = row / S;
    const int h = (int)(bh % H), b = (int)(bh / H);
    const uint4 x = *reinterpret_cast<const uint4*>(dout + b * ds0 + h * ds1 + (int64_t)s * ds2 + sub * EPL);
    const uint4 y = *reinterpret_cast<const uint4*>(o + b * os0 + h * os1 + (int64_t)s * os2 + sub * EPL);
    const uint32_t xw[4] = {x.x, x.y, x.z, x.w}, yw[4] = {y.x, y.y, y.z, y.w};
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      if constexpr (sizeof(T) == 2) {  // bf16 pairs: the low half is the even element
        acc = fmaf(__uint_as_float(xw[j] << 16), __uint_as_float(yw[j] << 16), acc);
        acc = fmaf(__uint_as_float(xw[j] & 0xffff0000u), __uint_as_float(yw[j] & 0xffff0000u), acc);
      } else {
        acc = fmaf(__uint_as_float(xw[j]), __uint_as_float(yw[j]), acc);
      }
    }
  }
  for (int off = lpr >> 1; off > 0; off >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, off);
  if (row < rows && sub == 0) {
    dsum[row] = acc;
    lse2[row] = -lse[row] * kLog2e;
  }
}

template <int D>
cudaError_t launch_bwd_d(const BwdLaunch& a, cudaStream_t st) {
  CUtensorMap mq, mk, mv, mdo;
  if (!make_map(&mq, a.q, a.B, a.Hq, a.S, D, a.qs) || !make_map(&mk, a.k, a.B, a.Hkv, a.S, D, a.ks) ||
      !make_map(&mv, a.v, a.B, a.Hkv, a.S, D, a.vs) || !make_map(&mdo, a.dout, a.B, a.Hq, a.S, D, a.dos))
    return cudaErrorInvalidValue;
  BwdParams p;
  memset(&p, 0, sizeof(p));
  p.B = a.B; p.Hq = a.Hq; p.Hkv = a.Hkv; p.S = a.S; p.group = a.Hq / a.Hkv; p.n_tiles = a.S / BT;
  p.mask = a.mask; p.sink = a.sink; p.window = a.window;
  p.scale = a.scale; p.scale_log2 = a.scale * kLog2e;
  p.lse2 = a.lse2; p.dsum = a.dsum;
  p.out_bf16 = a.out_bf16;
  p.f = a.f;
  p.status = device_status_word();
  if (!p.status) return cudaErrorInvalidValue;
  using C = Cfg<D>;
  // about four waves of CTAs per scheduling group
  auto heads_per_group = [&](int units) { return std::max(1, std::min(units, (4 * sm_count() + p.n_tiles - 1) / p.n_tiles)); };
  // dK, dV
  p.hgroup = heads_per_group(a.B * a.Hkv);
  p.out_a = a.dk; p.out_b = a.dv;
  for (int i = 0; i < 3; ++i) { p.oas[i] = a.dks[i]; p.obs[i] = a.dvs[i]; }
  int smem = C::kvBytes + 1024;
  cudaError_t e = cudaFuncSetAttribute(bwd_kv_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  bwd_kv_kernel<D><<<(unsigned)(p.n_tiles * a.B * a.Hkv), kThreads, smem, st>>>(mq, mk, mv, mdo, p);
  if ((e = launched(1)) != cudaSuccess) return e;
  // dQ
  p.hgroup = heads_per_group(a.B * a.Hq);
  p.out_a = a.dq; p.out_b = nullptr;
  for (int i = 0; i < 3; ++i) p.oas[i] = a.dqs[i];
  smem = C::qBytes + 1024;
  e = cudaFuncSetAttribute(bwd_q_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  bwd_q_kernel<D><<<(unsigned)(p.n_tiles * a.B * a.Hq), kThreads, smem, st>>>(mq, mk, mv, mdo, p);
  return launched(1);
}

}  // namespace

cudaError_t launch_dsum(const void* dout, const void* o, int bf16, float* dsum, const float* lse, float* lse2, int B,
                        int H, int S, int d, const int64_t ds[3], const int64_t os[3], cudaStream_t st) {
  const int64_t rows = (int64_t)B * H * S;
  if (rows == 0) return cudaSuccess;
  if (d != 64 && d != 128) return cudaErrorInvalidValue;
  const int lpr = d / (bf16 ? 8 : 4);
  const int64_t warps = (rows + 32 / lpr - 1) / (32 / lpr);
  const int64_t blocks = (warps + 7) / 8;
  if (blocks > 0x7fffffff) return cudaErrorInvalidValue;
  if (bf16)
    dsum_kernel<__nv_bfloat16><<<(unsigned)blocks, 256, 0, st>>>(
        static_cast<const __nv_bfloat16*>(dout), static_cast<const __nv_bfloat16*>(o), dsum, lse, lse2, B, H, S, d,
        ds[0], ds[1], ds[2], os[0], os[1], os[2]);
  else
    dsum_kernel<float><<<(unsigned)blocks, 256, 0, st>>>(static_cast<const float*>(dout), static_cast<const float*>(o),
                                                         dsum, lse, lse2, B, H, S, d, ds[0], ds[1], ds[2], os[0], os[1],
                                                         os[2]);
  return launched(1);
}

cudaError_t launch_bwd(const BwdLaunch& a, cudaStream_t st) {
  if (a.S % BT != 0) return cudaErrorInvalidValue;
  return a.d == 128 ? launch_bwd_d<128>(a, st) : launch_bwd_d<64>(a, st);
}

}  // namespace yr
