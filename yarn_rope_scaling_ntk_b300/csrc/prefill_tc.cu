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
// One CTA = two 128-row query tiles (256 consecutive rows) of one (batch,
// head); both tiles share every key/value tile the CTA loads.  Roles:
//   warp 9     TMA producer: Q0 and Q1 once, then K and V tiles of 128 keys
//              into two-stage rings of 128-byte-swizzled shared memory.
//   warp 8     TMEM owner and MMA issuer: the warp runs the loop converged
//              and one elected lane issues the MMAs.  For key tile j it
//              issues, in this order, O0 += P0(j) V(j), S0(j+1) = Q0 K(j+1)^T,
//              O1 += P1(j) V(j), S1(j+1) = Q1 K(j+1)^T, so that while one
//              softmax group works on its S the tensor pipe runs the other
//              group's products (ping-pong).
//   warps 10-11 idle: their registers go to the softmax groups.
//   warps 0-3  softmax group 0 (query tile 0), warps 4-7 group 1 (tile 1):
//              thread r owns query row r (TMEM lane r).  It reads its row of
//              S, masks, updates the running max / sum, writes P as bf16
//              pairs over the first 64 columns of the same TMEM buffer, and
//              rescales its O rows in TMEM only when the max grew by more
//              than 2^8 (lazy rescale).  Each group then writes its O / l and
//              the log-sum-exp.
// TMEM (512 columns): S0 | S1 | O0 | O1.  Every mbarrier wait is bounded; a
// wait that gives up records a code in the status word and makes every role
// leave its loop, drain its asynchronous work and free TMEM.
#include <math.h>
#include <string.h>

#include "common.cuh"
#include "internal.h"
#include "tc_ptx.cuh"

namespace yr {
namespace {

using namespace tc;

constexpr int BM = 128;   // query rows per tile (two tiles per CTA)
constexpr int BN = 128;   // keys per tile
constexpr int kThreads = 384;              // 3 warpgroups
constexpr int kMmaWarp = 8;
constexpr int kLoadWarp = 9;               // warps 10 and 11 only lend registers
// Register budgets (launch: 384 threads x 168).  The softmax groups hold a
// full 128-column row of S in registers; the control warpgroup keeps the
// MMA issue loop in registers: 2 x 128 x 216 + 128 x 72 = 64512 = 384 x 168.
constexpr uint32_t kRegsSoftmax = 216;
constexpr uint32_t kRegsControl = 72;
static_assert(2 * 128 * kRegsSoftmax + 128 * kRegsControl <= kThreads * 168, "register split");
constexpr uint32_t kTmemCols = 512;
constexpr float kRescaleThreshold = 8.0f;  // log2 units
// Waves of CTAs per scheduling group of KV heads (see the CTA order below):
// the K/V of a group's heads stays in L2 while its CTAs stream it.
#ifndef YR_PREFILL_SCHED_WAVES
#define YR_PREFILL_SCHED_WAVES 3
#endif
constexpr int kSchedWaves = YR_PREFILL_SCHED_WAVES;

struct TcParams {
  int B, Hq, Hkv, group, n_pairs;
  int Sq, Skv, qp0, kp0;  // query rows, keys, position of query row 0 / key 0
  int kv_per_sched;  // KV heads per scheduling group (see the CTA order below)
  int mask, sink, window, ring_blocks, cs;
  float scale_log2;
  void* o;
  int64_t os[3];
  float* lse;
  int out_bf16;
  int* status;
  long long wait_limit;  // first-level wait bound in cycles
  int skip_unit;         // fault injection: load unit never issued (-1: none)
};

// Key chunks in ring order for one CTA (two query tiles a and b): ring
// blocks I, I-1, ... (I = block of the CTA's last row), chunks ascending in a
// block.  A chunk holds cs <= 128 keys (cs = 64 when a ring block is an odd
// multiple of 64 keys); the MMA tile always spans 128 keys and masks the
// excess.  A chunk is walked when either tile sees part of it; v0 / v1 say
// which tiles do.  Under a mask the chunks any row of the CTA can see form the
// range [0, last] minus at most one gap [gap_lo, gap_hi) (chunks between the
// sinks and the start of the window), so the walk is a few compares per chunk.
struct Walk {
  int N, cpb, cs, mask, sink, window, qp0, kp0;
  int r0a, r1a, r0b, r1b;  // local query rows of tiles a and b
  bool hasa, hasb;
  int last, gap_lo, gap_hi, I;
  int t, c, c_end, rb;  // ring step, chunk, end of the block's visible chunks, block
  __device__ void init(const TcParams& p, int pair) {
    cs = p.cs;
    N = p.ring_blocks;
    const int n_chunks = (p.Skv + cs - 1) / cs;
    const int bs = N > 1 ? p.Skv / N : 0;  // ring blocks only when Sq == Skv and both start at 0
    cpb = N > 1 ? bs / cs : n_chunks;
    r0a = pair * 2 * BM;
    r0b = r0a + BM;
    hasa = r0a < p.Sq;
    hasb = r0b < p.Sq;
    r1a = min(p.Sq, r0a + BM) - 1;
    r1b = min(p.Sq, r0b + BM) - 1;
    qp0 = p.qp0;
    kp0 = p.kp0;
    const int lim = hasb ? r1b : r1a;
    mask = p.mask;
    sink = p.sink;
    window = p.window;
    // positions: query row r sits at qp0 + r, key n at kp0 + n
    if (mask == YR_MASK_NONE) {
      last = n_chunks - 1;
    } else {
      const int reach = qp0 + lim - kp0;  // the last key index any row sees
      last = reach < 0 ? -1 : min(n_chunks - 1, reach / cs);
    }
    gap_lo = gap_hi = 0;
    if (mask == YR_MASK_SINK_WINDOW) {
      // chunks with a sink: kp0 + c * cs < sink; chunks that reach the window
      // of row r0a: kp0 + c * cs + cs - 1 > qp0 + r0a - window
      const int sink_chunks = sink > kp0 ? (sink - kp0 + cs - 1) / cs : 0;
      const int x = qp0 + r0a - window - cs + 1 - kp0;
      const int w_lo = x < 0 ? 0 : x / cs + 1;
      if (sink_chunks < w_lo) { gap_lo = sink_chunks; gap_hi = w_lo; }
    }
    I = N > 1 ? lim / bs : 0;
    t = -1;
    c = c_end = 0;
    rb = 0;
  }
  __device__ __forceinline__ bool visible(bool has, int r0, int r1, int n0) const {
    const int ng = kp0 + n0, r0g = qp0 + r0, r1g = qp0 + r1;
    const bool in_window = (mask != YR_MASK_SINK_WINDOW) | (ng < sink) | (ng + cs - 1 > r0g - window);
    return has & ((mask == YR_MASK_NONE) | ((ng <= r1g) & in_window));
  }
  // next chunk start seen by either tile (or -1), with per-tile visibility
  __device__ __forceinline__ int next(bool& v0, bool& v1) {
    while (true) {
      if (c >= c_end) {
        if (++t >= N) return -1;
        rb = t == 0 ? I : (rb == 0 ? N - 1 : rb - 1);
        c = rb * cpb;
        c_end = min(c + cpb, last + 1);
        continue;
      }
      if (c >= gap_lo && c < gap_hi) {
        c = gap_hi;
        continue;
      }
      const int n0 = c * cs;
      ++c;
      v0 = visible(hasa, r0a, r1a, n0);
      v1 = visible(hasb, r0b, r1b, n0);
      if (v0 | v1) return n0;
    }
  }
};

// does a tile with rows [r0, r1] need the per-element mask on chunk n0?
__device__ __forceinline__ bool needs_mask(const TcParams& p, int r0, int r1, int n0) {
  const int ng = p.kp0 + n0, r0g = p.qp0 + r0, r1g = p.qp0 + r1;
  return p.cs < BN || n0 + BN > p.Skv || (p.mask != YR_MASK_NONE && ng + BN - 1 > r0g) ||
         (p.mask == YR_MASK_SINK_WINDOW && ng <= r1g - p.window);
}

__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

__device__ __forceinline__ float max3(float a, float b, float c) {
  float d;
  asm("max.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
  return d;
}

template <int D>
struct Cfg {
  static constexpr int NS = D == 128 ? 2 : 4;  // K / V pipeline stages
  static constexpr int kTile = BM * D * 2;     // bytes of one 128-row bf16 tile
  static constexpr int kQ = 0;                 // Q0, Q1
  static constexpr int kK = 2 * kTile;
  static constexpr int kV = kK + NS * kTile;
  static constexpr int kBytes = kV + NS * kTile;
};

template <int D>
__global__ void __launch_bounds__(kThreads, 1)
    prefill_tc_kernel(const __grid_constant__ CUtensorMap tq, const __grid_constant__ CUtensorMap tk,
                      const __grid_constant__ CUtensorMap tv, const TcParams p) {
  using C = Cfg<D>;
  constexpr int NS = C::NS;
  constexpr int ATOMS = D / 64;         // 64-column swizzle atoms per row
  constexpr int ATOM_BYTES = BM * 128;  // one atom column of a 128-row tile
  constexpr uint32_t S_COLS = 128;
  constexpr uint32_t O_COL = 2 * S_COLS;
  constexpr uint32_t ID_QK = idesc_bf16_f32(BM, BN, false);
  constexpr uint32_t ID_PV = idesc_bf16_f32(BM, D, true);

  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* sQ = smem + C::kQ;
  uint8_t* sK = smem + C::kK;
  uint8_t* sV = smem + C::kV;

  __shared__ uint64_t q_full, kv_full[NS], kv_empty[NS];
  __shared__ uint64_t s_full[2], p_full[2], o_done[2], drain;
  __shared__ uint32_t tmem_slot;
  __shared__ volatile int abort_flag;

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  // Launch order: the (batch, KV head) pairs are taken in scheduling groups
  // of kv_per_sched; inside a group, every query head that reads one of its
  // KV heads runs its heaviest query-tile pairs first (longest-first keeps
  // the tail short).  CTAs that run together then stream the same K/V tiles,
  // which stay in L2.
  const int n_kv = p.B * p.Hkv;
  const int per_kv = p.n_pairs * p.group;  // CTAs per (batch, KV head)
  const int g0 = (int)(blockIdx.x / ((unsigned)per_kv * p.kv_per_sched)) * p.kv_per_sched;
  const int gsz = min(p.kv_per_sched, n_kv - g0);
  const int r = (int)(blockIdx.x - (unsigned)g0 * per_kv);
  const int heads = gsz * p.group;  // query heads in this group
  const int pair = p.n_pairs - 1 - r / heads;
  const int hg = r % heads;
  const int bkv = g0 + hg / p.group;  // batch * Hkv + KV head
  const int b = bkv / p.Hkv, hkv = bkv % p.Hkv;
  const int hq = hkv * p.group + hg % p.group;

  if (tid == 0) {
    abort_flag = 0;
    mbar_init(&q_full, 1);
    for (int s = 0; s < NS; ++s) {
      mbar_init(&kv_full[s], 1);
      mbar_init(&kv_empty[s], 1);
    }
    for (int w = 0; w < 2; ++w) {
      mbar_init(&s_full[w], 1);
      mbar_init(&p_full[w], 4);  // one arrival per softmax warp
      mbar_init(&o_done[w], 1);
    }
    mbar_init(&drain, 1);
    fence_mbar_init();
  }
  if (warp == kMmaWarp) tmem_alloc(&tmem_slot, kTmemCols);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = tmem_slot;

  Walk walk;
  walk.init(p, pair);
  int uses[NS] = {0};  // producer: load units issued per stage

  if (warp >= 8) {
    reg_dealloc<kRegsControl>();
    if (warp == kLoadWarp) {
      // ---------------- TMA producer ----------------
      if (lane == 0) {
        tma_prefetch_desc(&tq);
        tma_prefetch_desc(&tk);
        tma_prefetch_desc(&tv);
        const int nq = walk.hasb ? 2 : 1;
        mbar_arrive_expect_tx(&q_full, nq * C::kTile);
        for (int w = 0; w < nq; ++w)
          for (int a = 0; a < ATOMS; ++a)
            tma_load_4d(sQ + w * C::kTile + a * ATOM_BYTES, &tq, &q_full, a * 64, w ? walk.r0b : walk.r0a, hq, b);
        // Load unit u: K(0) for u = 0; V(u-1) and (when chunk u exists) K(u)
        // otherwise, on barrier u % NS.  K(c) lives in K buffer c % NS and
        // V(c) in V buffer c % NS, so unit u reuses exactly the buffers of
        // unit u - NS and waits for that unit's release.
        bool v0, v1;
        int prev = -1;
        int cur = walk.next(v0, v1);
        for (int u = 0; cur >= 0 || prev >= 0; ++u) {
          const int s = u % NS;
          if (!mbar_wait(&kv_empty[s], ((u / NS) & 1) ^ 1, &abort_flag, p.status, 11, p.wait_limit)) break;
          if (u != p.skip_unit) {  // (fault injection: a skipped unit is never loaded)
            mbar_arrive_expect_tx(&kv_full[s], (prev >= 0 ? C::kTile : 0) + (cur >= 0 ? C::kTile : 0));
            if (prev >= 0)
              for (int a = 0; a < ATOMS; ++a)
                tma_load_4d(sV + ((u - 1) % NS) * C::kTile + a * ATOM_BYTES, &tv, &kv_full[s], a * 64, prev, hkv, b);
            if (cur >= 0)
              for (int a = 0; a < ATOMS; ++a)
                tma_load_4d(sK + s * C::kTile + a * ATOM_BYTES, &tk, &kv_full[s], a * 64, cur, hkv, b);
            ++uses[s];
          }
          prev = cur;
          cur = cur >= 0 ? walk.next(v0, v1) : -1;
        }
      }
      __syncwarp();
    } else if (warp == kMmaWarp) {
      // ---------------- MMA issuer ----------------
      // The whole warp runs the loop (waits, walk, descriptors: warp-uniform
      // values) and one elected lane issues each group of MMAs and commits.
      {
        const bool leader = elect_one();
        // Shared-memory descriptors of every operand buffer, built once; a
        // K step adds its (compile-time) byte offset / 16 to the start
        // address field, which cannot carry out (shared addresses < 256 KB).
        const uint64_t dq = sdesc_sw128(smem_u32(sQ), 16, 1024);
        const uint64_t dk = sdesc_sw128(smem_u32(sK), 16, 1024);
        const uint64_t dv = sdesc_sw128(smem_u32(sV), ATOM_BYTES, 1024);
        constexpr uint64_t kTile16 = C::kTile >> 4;
        auto issue_s = [&](int w, int s) {
          const uint64_t a0 = dq + (w ? kTile16 : 0), b0 = dk + (uint64_t)s * kTile16;
          const uint32_t d_s = tmem + w * S_COLS;
          if (leader) {
#pragma unroll
            for (int kk = 0; kk < D / 16; ++kk) {
              const uint64_t off = (uint64_t)(((kk >> 2) * ATOM_BYTES + (kk & 3) * 32) >> 4);
              mma_ss(d_s, a0 + off, b0 + off, ID_QK, kk > 0);
            }
            mma_commit(&s_full[w]);
          }
          __syncwarp();
        };
        auto issue_pv = [&](int w, int s, bool acc) {
          const uint64_t b0 = dv + (uint64_t)s * kTile16;
          const uint32_t d_o = tmem + O_COL + w * D, a_p = tmem + w * S_COLS;
          if (leader) {
#pragma unroll
            for (int kk = 0; kk < BN / 16; ++kk)
              mma_ts(d_o, a_p + kk * 8, b0 + (uint64_t)(kk * 2048 >> 4), ID_PV, (acc || kk > 0) ? 1u : 0u);
          }
          __syncwarp();
        };
        auto commit = [&](uint64_t* bar) {
          if (leader) mma_commit(bar);
          __syncwarp();
        };
        auto wait = [&](uint64_t* bar, uint32_t par, int code) -> bool {
          return __all_sync(0xffffffffu, mbar_wait(bar, par, &abort_flag, p.status, code, p.wait_limit));
        };
        bool ok = wait(&q_full, 0, 21);
        int pv_count[2] = {0, 0};
        bool cv0 = false, cv1 = false, nv0 = false, nv1 = false;
        int cur = ok ? walk.next(cv0, cv1) : -1;
        int nxt = -1;
        if (cur >= 0) {
          ok = wait(&kv_full[0], 0, 22);
          if (ok) {
            tc_fence_after();
            if (cv0) issue_s(0, 0);
            if (cv1) issue_s(1, 0);
            commit(&kv_empty[0]);
            nxt = walk.next(nv0, nv1);
            ok = wait(&kv_full[1 % NS], (1 / NS) & 1, 23);
          }
        }
        // Step i (load unit i + 1 = V(i), K(i + 1) has landed; nxt, nv0, nv1
        // describe chunk i + 1).  The walk and the wait for the next unit come
        // after S1(i + 1) is queued, while the tensor pipe still has work.
        for (int i = 0; ok && cur >= 0; ++i) {
          const int s = i % NS, sn = (i + 1) % NS;
          tc_fence_after();
          if (cv0) {
            if (!wait(&p_full[0], pv_count[0] & 1, 25)) { ok = false; break; }
            tc_fence_after();
            issue_pv(0, s, pv_count[0] > 0);
            ++pv_count[0];
          }
          if (nxt >= 0 && nv0) issue_s(0, sn);
          if (cv1) {
            if (!wait(&p_full[1], pv_count[1] & 1, 26)) { ok = false; break; }
            tc_fence_after();
            issue_pv(1, s, pv_count[1] > 0);
            ++pv_count[1];
          }
          if (nxt >= 0 && nv1) issue_s(1, sn);
          commit(&kv_empty[sn]);
          cur = nxt;
          cv0 = nv0;
          cv1 = nv1;
          if (cur >= 0) {
            nv0 = nv1 = false;
            nxt = walk.next(nv0, nv1);
            const int un = i + 2;
            if (!wait(&kv_full[un % NS], (un / NS) & 1, 24)) { ok = false; break; }
          }
        }
        // the epilogues read O once every product is done
        commit(&o_done[0]);
        commit(&o_done[1]);
        // all issued MMAs complete before TMEM is released
        commit(&drain);
        if (leader) mbar_wait_drain(&drain, 0, 200000000ll);
        __syncwarp();
      }
    }
  } else {
    reg_alloc<kRegsSoftmax>();
    // ---------------- softmax (warps 0-3: tile 0, warps 4-7: tile 1) --------
    const int wg = warp >> 2;
    const int r = (warp & 3) * 32 + lane;  // query row within the tile == TMEM lane
    const int my_r0 = wg ? walk.r0b : walk.r0a, my_r1 = wg ? walk.r1b : walk.r1a;
    const int m = my_r0 + r;
    const uint32_t lane_addr = tmem + ((uint32_t)((warp & 3) * 32) << 16);
    const uint32_t s_addr = lane_addr + wg * S_COLS;
    const uint32_t o_addr = lane_addr + O_COL + wg * D;
    const float sc = p.scale_log2;
    float m_used = -INFINITY, l = 0.f;
    int i = 0;
    bool ok = true;
    bool v0, v1;
    for (int n0 = walk.next(v0, v1); n0 >= 0; n0 = walk.next(v0, v1)) {
      if (!(wg ? v1 : v0)) continue;
      // warp-uniform decisions: tcgen05.ld / st are warp-collective
      ok = __all_sync(0xffffffffu, mbar_wait(&s_full[wg], i & 1, &abort_flag, p.status, 31, p.wait_limit));
      if (!ok) break;
      tc_fence_after();
      uint32_t raw[4][32];
#pragma unroll
      for (int c = 0; c < 4; ++c) tmem_ld32(s_addr + c * 32, raw[c]);
      tmem_ld_wait();
#pragma unroll
      for (int c = 0; c < 4; ++c) reg_fence32(raw[c]);
      float x[BN];
#pragma unroll
      for (int c = 0; c < 4; ++c)
#pragma unroll
        for (int e = 0; e < 32; ++e) x[c * 32 + e] = __uint_as_float(raw[c][e]);
      if (needs_mask(p, my_r0, my_r1, n0)) {
        // Visible columns of row m, as bounds on the column e (key position
        // kp0 + n0 + e, query position qp0 + m): e <= hi (inside the chunk,
        // inside the keys, not after the query) and, under the sink-window
        // mask, a sink (e < s_end) or inside the window (e > w_lo).
        const int ng0 = p.kp0 + n0, mg = p.qp0 + m;
        int hi = min(p.cs, p.Skv - n0) - 1;
        if (p.mask != YR_MASK_NONE) hi = min(hi, mg - ng0);
        const bool sw = p.mask == YR_MASK_SINK_WINDOW;
        const int s_end = sw ? p.sink - ng0 : BN;
        const int w_lo = sw ? mg - p.window - ng0 : -1;
#pragma unroll
        for (int e = 0; e < BN; ++e)
          if (e > hi || (e >= s_end && e <= w_lo)) x[e] = -INFINITY;
      }
      // row max of the raw logits: eight independent 3-input chains
      float mx8[8];
#pragma unroll
      for (int t = 0; t < 8; ++t) mx8[t] = x[t];
#pragma unroll
      for (int e = 8; e + 16 <= BN; e += 16)
#pragma unroll
        for (int t = 0; t < 8; ++t) mx8[t] = max3(mx8[t], x[e + 2 * t], x[e + 2 * t + 1]);
      // the loop above covers x[8, 120); fold the last 8 in
#pragma unroll
      for (int t = 0; t < 8; ++t) mx8[t] = fmaxf(mx8[t], x[BN - 8 + t]);
      const float mx_raw = max3(max3(mx8[0], mx8[1], mx8[2]), max3(mx8[3], mx8[4], mx8[5]), fmaxf(mx8[6], mx8[7]));
      const float mx = mx_raw * sc;  // -inf stays -inf (sc > 0)
      // Lazy rescale: the reference max moves only when the row max exceeds
      // it by more than 2^8.  P is formed against the new reference; the O
      // rows are rescaled after P is stored (the logits are dead by then),
      // by the whole warp when any lane must.
      const bool grow = mx > m_used + kRescaleThreshold;
      const bool rescale = grow && m_used != -INFINITY && i > 0;
      const float corr = rescale ? ex2(m_used - mx) : 1.0f;
      if (grow) m_used = mx;
      const float neg_ref = m_used == -INFINITY ? 0.f : -m_used;
      // two columns per packed op: the exponent argument and the row sum
      // (four partial sums, two packed chains)
      float sum4[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
      for (int c = 0; c < BN / 64; ++c) {
        uint32_t pk[32];
#pragma unroll
        for (int e = 0; e < 32; ++e) {
          float t0, t1;
          fma2(t0, t1, x[c * 64 + 2 * e], x[c * 64 + 2 * e + 1], sc, sc, neg_ref, neg_ref);
          const float a0 = ex2(t0), a1 = ex2(t1);
          const int j = 2 * (e & 1);
          fma2(sum4[j], sum4[j + 1], a0, a1, 1.f, 1.f, sum4[j], sum4[j + 1]);
          pk[e] = pack_bf16(a0, a1);
        }
        tmem_st32(s_addr + c * 32, pk);
      }
      l = l * corr + ((sum4[0] + sum4[1]) + (sum4[2] + sum4[3]));
      if (__any_sync(0xffffffffu, rescale)) {
        // the s_full phase just waited for also covers this group's earlier
        // PV products, and the next one is issued only after p_full below

#pragma unroll
        for (int c = 0; c < D / 32; ++c) {
          uint32_t rr[32];
          tmem_ld32(o_addr + c * 32, rr);
          tmem_ld_wait();
          reg_fence32(rr);
#pragma unroll
          for (int e = 0; e < 32; ++e) rr[e] = __float_as_uint(__uint_as_float(rr[e]) * corr);
          tmem_st32(o_addr + c * 32, rr);
        }
      }
      tmem_st_wait();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&p_full[wg]);
      ++i;
    }
    // epilogue: O / l -> global, lse
    if (__all_sync(0xffffffffu, ok && !abort_flag)) {
      bool have = true;
      if (i > 0)
        have = __all_sync(0xffffffffu, mbar_wait(&o_done[wg], 0, &abort_flag, p.status, 33, p.wait_limit));
      tc_fence_after();
      if (have) {
        const float inv = l > 0.f ? 1.f / l : 0.f;
        const bool row_ok = m < p.Sq;
        char* orow = static_cast<char*>(p.o) +
                     (b * p.os[0] + hq * p.os[1] + (int64_t)m * p.os[2]) * (p.out_bf16 ? 2 : 4);
#pragma unroll
        for (int c = 0; c < D / 32; ++c) {
          uint32_t rr[32];
          if (i > 0) {
            tmem_ld32(o_addr + c * 32, rr);
            tmem_ld_wait();
            reg_fence32(rr);
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
          p.lse[((int64_t)b * p.Hq + hq) * p.Sq + m] =
              l > 0.f ? (m_used + log2f(l)) * 0.69314718055994530942f : -INFINITY;
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  // After an abort the copies the producer issued land before the CTA exits;
  // the flag is final here, since every role has left its loop.  (Without
  // an abort the MMA warp has waited for every unit issued.)
  if (warp == kLoadWarp && lane == 0 && abort_flag) {
    mbar_wait_drain(&q_full, 0, 200000000ll);
    for (int s = 0; s < NS; ++s)
      if (uses[s]) mbar_wait_drain(&kv_full[s], (uses[s] - 1) & 1, 200000000ll);
  }
  if (warp == kMmaWarp) tmem_dealloc(tmem, kTmemCols);
}

template <int D>
cudaError_t launch_d(const PrefillLaunch& a, cudaStream_t st) {
  CUtensorMap mq, mk, mv;
  if (!make_map(&mq, a.q, a.B, a.Hq, a.Sq, D, a.qs) || !make_map(&mk, a.k, a.B, a.Hkv, a.Skv, D, a.ks) ||
      !make_map(&mv, a.v, a.B, a.Hkv, a.Skv, D, a.vs))
    return cudaErrorInvalidValue;
  TcParams p;
  memset(&p, 0, sizeof(p));
  p.B = a.B; p.Hq = a.Hq; p.Hkv = a.Hkv; p.group = a.Hq / a.Hkv;
  p.Sq = a.Sq; p.Skv = a.Skv; p.qp0 = a.q_pos0; p.kp0 = a.k_pos0;
  p.n_pairs = (a.Sq + 2 * BM - 1) / (2 * BM);
  {
    // enough KV heads per scheduling group for about kSchedWaves waves of CTAs
    const int per_kv = p.n_pairs * p.group;
    const int n_kv = a.B * a.Hkv;
    int k = (kSchedWaves * sm_count() + per_kv - 1) / per_kv;
    p.kv_per_sched = k < 1 ? 1 : (k > n_kv ? n_kv : k);
  }
  p.mask = a.mask; p.sink = a.sink; p.window = a.window; p.ring_blocks = a.ring_blocks;
  p.cs = (a.ring_blocks > 1 && (a.Skv / a.ring_blocks) % BN != 0) ? 64 : BN;
  p.scale_log2 = a.scale_log2;
  p.o = a.o;
  for (int i = 0; i < 3; ++i) p.os[i] = a.os[i];
  p.lse = a.lse;
  p.out_bf16 = a.out_bf16;
  p.status = device_status_word();
  if (!p.status) return cudaErrorInvalidValue;
  const FaultInjection fi = fault_injection();
  p.wait_limit = fi.wait_limit;
  p.skip_unit = fi.skip_unit;
  const int smem = Cfg<D>::kBytes + 1024;
  cudaError_t e = cudaFuncSetAttribute(prefill_tc_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  const int64_t blocks = (int64_t)p.n_pairs * a.B * a.Hq;
  if (blocks > 0x7fffffff) return cudaErrorInvalidValue;
  prefill_tc_kernel<D><<<(unsigned)blocks, kThreads, smem, st>>>(mq, mk, mv, p);
  return launched(1);
}

}  // namespace

cudaError_t launch_prefill(const PrefillLaunch& a, cudaStream_t st) {
  if (a.ring_blocks > 1 &&
      (a.Sq != a.Skv || a.q_pos0 != 0 || a.k_pos0 != 0 || (a.Skv / a.ring_blocks) % 64 != 0))
    return cudaErrorInvalidValue;
  return a.d == 128 ? launch_d<128>(a, st) : launch_d<64>(a, st);
}

}  // namespace yr
