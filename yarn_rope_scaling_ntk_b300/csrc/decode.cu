// attn_fwd_decode_sinkwindow: one new query token per sequence against a
// cache of `sink` pinned tokens plus a `window`-slot ring buffer ("Context
// Length Extension", Sliding Window + Attention Sinks; "Long-Context
// Scaling", Production defaults).  Keys are stored unrotated and rotated on
// read at their logical cache index; the query sits at n_valid - 1.
//
// HBM-bound: every valid cache entry is read once.  A CTA owns one
// (sequence, kv head) and one slice of the logical entries.  A producer warp
// streams the slice in chunks of CK logical entries into a three-stage
// shared-memory ring with bulk asynchronous copies (a chunk maps to at most
// three physically contiguous runs: sinks, ring up to its wrap, ring after
// the wrap), so the bytes in flight do not depend on registers.  Eight
// compute warps read the stage: TPK threads share a key (each owns 8 rotation
// pairs, one 16-byte vector from each half of the head dimension), rotate it
// at its logical position, and keep an online-softmax state (running max,
// sum, unnormalised output) whose reference max moves lazily.  States are
// merged across the warp by shuffles, across warps in shared memory, and
// across slices by a second kernel.
#include <cuda_fp8.h>
#include <math.h>

#include <mutex>

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
using tc::bulk_g2s;
using tc::smem_u32;

constexpr int kWarps = 8;                    // compute warps
constexpr int kThreads = (kWarps + 1) * 32;  // + one producer warp
constexpr int NSTG = 3;                      // shared-memory stages
constexpr float kRescaleThreshold = 8.0f;    // log2 units
constexpr int kReanchor = 16;                // chunks between exact rotation anchors (FP8 caches)

// PPT rotation pairs per thread: 8 (two 16-byte vectors per key row) when
// one query head shares the key, 4 when several do, so the per-thread query and
// accumulator state fits the registers of nine resident warps.  EB is the
// byte size of a cache element (2: bfloat16, 1: FP8 E4M3); a chunk holds the
// same bytes either way, so an FP8 chunk holds twice the keys.
template <int D, int PPT, int EB>
struct DecodeShape {
  static constexpr int TPK = D / 2 / PPT;     // threads per key
  static constexpr int KPW = 32 / TPK;        // keys per warp step
  static constexpr int KPS = KPW * kWarps;    // keys per CTA step
  static constexpr int CK = (4 / EB) * KPS;   // keys per chunk
  static constexpr int ROW = D * EB;          // bytes per cache row
  static constexpr int STAGE = CK * ROW;      // bytes of K (or V) per stage
  static constexpr int SMEM = 2 * NSTG * STAGE;
};

// 2^x (hardware approximation; relative error about 2^-22, results below
// 2^-126 flushed to 0).
__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

__device__ __forceinline__ float exp2_diff(float a, float b) {
  // 2^(a - b) with a = -inf giving 0.
  return a == -INFINITY ? 0.f : exp2f(a - b);
}

template <int N>
__device__ __forceinline__ void load_bf16(const uint8_t* p, float (&x)[N]) {
  if constexpr (N == 8) {
    const uint4 u = *reinterpret_cast<const uint4*>(p);
    const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
    for (int k = 0; k < 8; ++k) x[k] = (k & 1) ? bf16_hi(w[k >> 1]) : bf16_lo(w[k >> 1]);
  } else {
    const uint2 u = *reinterpret_cast<const uint2*>(p);
    x[0] = bf16_lo(u.x); x[1] = bf16_hi(u.x); x[2] = bf16_lo(u.y); x[3] = bf16_hi(u.y);
  }
}

// N consecutive FP8 E4M3 values (N = 8 or 4) to float, through the hardware
// pair conversion to half precision (exact: every E4M3 value is a half).
template <int N>
__device__ __forceinline__ void load_e4m3(const uint8_t* p, float (&x)[N]) {
  uint32_t w[N / 4];
  if constexpr (N == 8) {
    const uint2 u = *reinterpret_cast<const uint2*>(p);
    w[0] = u.x; w[1] = u.y;
  } else {
    w[0] = *reinterpret_cast<const uint32_t*>(p);
  }
#pragma unroll
  for (int k = 0; k < N / 2; ++k) {
    const __nv_fp8x2_storage_t pair = (__nv_fp8x2_storage_t)((w[k >> 1] >> (16 * (k & 1))) & 0xffffu);
    const __half2 h2 = __half2(__nv_cvt_fp8x2_to_halfraw2(pair, __NV_E4M3));
    const float2 f2 = __half22float2(h2);
    x[2 * k] = f2.x;
    x[2 * k + 1] = f2.y;
  }
}

template <int N, int EB>
__device__ __forceinline__ void load_cache(const uint8_t* p, float (&x)[N]) {
  if constexpr (EB == 2) load_bf16<N>(p, x);
  else load_e4m3<N>(p, x);
}

template <int D, int G, int EB>
__global__ void __launch_bounds__(kThreads, G == 1 ? 2 : 1)
    decode_kernel(const __grid_constant__ DecodeLaunch a, const __grid_constant__ RopeFreqs f) {
  constexpr int PPT = G >= 2 ? 4 : 8;
  constexpr int QROW = D * 2;  // the query is bfloat16
  using Sh = DecodeShape<D, PPT, EB>;
  constexpr int TPK = Sh::TPK, KPW = Sh::KPW, KPS = Sh::KPS, CK = Sh::CK, ROW = Sh::ROW;
  constexpr int HALF = D / 2;
  extern __shared__ __align__(128) uint8_t smem[];
  uint8_t* sK = smem;
  uint8_t* sV = smem + NSTG * Sh::STAGE;
  __shared__ uint64_t full[NSTG], empty[NSTG];
  __shared__ volatile int abort_flag;

  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int bh = blockIdx.x;
  const int b = bh / a.Hkv, hkv = bh % a.Hkv;
  const int hq0 = hkv * (a.Hq / a.Hkv) + blockIdx.z * G;
  const int split = blockIdx.y;
  const int C = a.sink + a.window;
  int* status = a.status;

  int n = a.n_valid[b];
  n = n < 0 ? 0 : (n > C ? C : n);
  int rs = a.ring_start[b];
  rs = ((rs % a.window) + a.window) % a.window;
  const int per = (n + a.splits - 1) / a.splits;
  const int j0 = min(n, split * per);
  const int j1 = min(n, j0 + per);

  if (threadIdx.x == 0) {
    abort_flag = 0;
    for (int s = 0; s < NSTG; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], kWarps);
    }
    tc::fence_mbar_init();
  }
  __syncthreads();

  const uint8_t* kbase = static_cast<const uint8_t*>(a.kc) + (int64_t)bh * C * ROW;
  const uint8_t* vbase = static_cast<const uint8_t*>(a.vc) + (int64_t)bh * C * ROW;

  if (warp == kWarps) {
    // ---------------- producer ----------------
    if (lane == 0) {
      int issued[NSTG] = {0};
      int c = 0;
      for (int jc = j0; jc < j1; jc += CK, ++c) {
        const int s = c % NSTG;
        if (!mbar_wait(&empty[s], ((c / NSTG) & 1) ^ 1, &abort_flag, status, 41, a.wait_limit)) break;
        if (c == a.skip_unit) continue;  // fault injection: this chunk is never loaded
        const int nk = min(CK, j1 - jc);
        mbar_arrive_expect_tx(&full[s], (uint32_t)(2 * nk * ROW));
        for (int j = jc; j < jc + nk;) {
          int phys, stop;
          if (j < a.sink) {
            phys = j;
            stop = min(jc + nk, a.sink);
          } else {
            const int t = (rs + j - a.sink) % a.window;
            phys = a.sink + t;
            stop = min(jc + nk, j + (a.window - t));
          }
          const uint32_t bytes = (uint32_t)((stop - j) * ROW);
          const int off = (j - jc) * ROW;
          bulk_g2s(sK + s * Sh::STAGE + off, kbase + (int64_t)phys * ROW, bytes, &full[s]);
          bulk_g2s(sV + s * Sh::STAGE + off, vbase + (int64_t)phys * ROW, bytes, &full[s]);
          j = stop;
        }
        ++issued[s];
      }
      // Every copy issued lands before the stage buffers are reused for the
      // merge below, also when the compute warps gave up on a chunk after
      // the last one was issued (the last phase of each stage is waited for;
      // the stage's barrier cannot move past it).
      for (int s = 0; s < NSTG; ++s)
        if (issued[s]) mbar_wait_drain(&full[s], (issued[s] - 1) & 1, 200000000ll);
    }
    __syncwarp();
    __syncthreads();
    return;
  }

  // ---------------- compute warps ----------------
  const int c8 = lane % TPK, kg = lane / TPK;
  float2 fr[PPT];
#pragma unroll
  for (int k = 0; k < PPT; ++k) fr[k] = f.f[c8 * PPT + k];
  const bool identity = f.identity != 0;

  // The logit of key position j is <R_m q, R_j k> = <R_(m-j) q, k> with m =
  // n - 1 the query position ("Context Window Scaling ...", Section 2: the
  // inner product depends only on the displacement).  A thread visits its
  // keys at j, j + KPS, j + 2 KPS, ..., so the rotation advances by the fixed
  // angle KPS theta_i per step: one complex multiply per pair, re-anchored
  // exactly (integer displacement, exact turn reduction) at every chunk.
  //  G == 1: the query is rotated backwards, q_hat = R_(m-j) q, and dotted
  //          with the raw key (no per-key rotation of K).
  //  G  > 1: the G query heads share the key, so the key's cos/sin advance
  //          instead and K is rotated once for all of them.
  // The recurrence is used for FP8 caches, where the halved bytes leave the
  // kernel bound by this arithmetic.  For bfloat16 caches the kernel is
  // bound by HBM, and an exact per-key angle keeps consecutive keys
  // independent (more instruction-level parallelism at the same bytes).
  constexpr bool kRecur = EB == 1;
  constexpr bool kRotQ = kRecur && G == 1;
  const int mq = n > 0 ? n - 1 : 0;
  float q1[G][PPT], q2[G][PPT];   // scaled query: raw (kRotQ) or rotated at m
  float stc[PPT], sts[PPT];       // cos / sin of the step angle KPS theta_i
#pragma unroll
  for (int k = 0; k < PPT; ++k) {
    if (identity) { stc[k] = 1.f; sts[k] = 0.f; }
    else turn_cos_sin<true>((float)KPS, fr[k], stc[k], sts[k]);  // precise: the step repeats
  }
  float nsts[PPT];
#pragma unroll
  for (int k = 0; k < PPT; ++k) nsts[k] = -sts[k];
  {
    float cs[PPT], sn[PPT];
#pragma unroll
    for (int k = 0; k < PPT; ++k) {
      if (identity || kRotQ) { cs[k] = 1.f; sn[k] = 0.f; }
      else turn_cos_sin<false>((float)mq, fr[k], cs[k], sn[k]);
    }
#pragma unroll
    for (int g = 0; g < G; ++g) {
      const uint8_t* qp = static_cast<const uint8_t*>(a.q) + ((int64_t)b * a.Hq + hq0 + g) * QROW;
      float x1[PPT], x2[PPT];
      load_bf16<PPT>(qp + c8 * PPT * 2, x1);
      load_bf16<PPT>(qp + HALF * 2 + c8 * PPT * 2, x2);
#pragma unroll
      for (int k = 0; k < PPT; ++k) {
        q1[g][k] = (x1[k] * cs[k] - x2[k] * sn[k]) * a.scale_log2;
        q2[g][k] = (x1[k] * sn[k] + x2[k] * cs[k]) * a.scale_log2;
      }
    }
  }

  // FP8 caches: dequantised value = stored value x scale of the (sequence,
  // KV head).  The rotation is linear, so the key scale multiplies each dot
  // product and the value scale the output.
  const float k_scale = EB == 1 ? a.k_scale[bh] : 1.f;
  const float v_scale = EB == 1 ? a.v_scale[bh] : 1.f;

  float mrun[G], lrun[G], acc1[G][PPT], acc2[G][PPT];
#pragma unroll
  for (int g = 0; g < G; ++g) {
    mrun[g] = -INFINITY;
    lrun[g] = 0.f;
#pragma unroll
    for (int k = 0; k < PPT; ++k) { acc1[g][k] = 0.f; acc2[g][k] = 0.f; }
  }

  bool ok = true;
  int c = 0;
  float rc[PPT], rs_[PPT];   // cos / sin of (m - j) theta (kRotQ) or j theta
  float qh1[PPT], qh2[PPT];  // kRotQ: the backward-rotated query
  for (int jc = j0; jc < j1; jc += CK, ++c) {
    const int s = c % NSTG;
    ok = __all_sync(0xffffffffu, mbar_wait(&full[s], (c / NSTG) & 1, &abort_flag, status, 42, a.wait_limit));
    if (!ok) break;
    const uint8_t* stK = sK + s * Sh::STAGE;
    const uint8_t* stV = sV + s * Sh::STAGE;
    // Anchor: the exact rotation for the thread's first key j_a of this
    // chunk.  The recurrence steps by KPS positions per key, and the thread's
    // first key of the next chunk is KPS after its last key of this one, so
    // it carries over; it is re-anchored every kReanchor chunks, which keeps
    // the drift of the rounded step rotation below about 10^-5.
    if (!kRecur || c % kReanchor == 0) {
      const int j_a = jc + warp * KPW + kg;
#pragma unroll
      for (int k = 0; k < PPT; ++k) {
        if (identity || !kRecur) { rc[k] = 1.f; rs_[k] = 0.f; }
        else turn_cos_sin<false>((float)(kRotQ ? mq - j_a : j_a), f.f[c8 * PPT + k], rc[k], rs_[k]);
      }
      // kRotQ: the backward-rotated query itself is the recurrence state
#pragma unroll
      for (int k = 0; k < PPT; ++k) {
        qh1[k] = q1[0][k] * rc[k] - q2[0][k] * rs_[k];
        qh2[k] = q1[0][k] * rs_[k] + q2[0][k] * rc[k];
      }
    }
#pragma unroll
    for (int u = 0; u < CK / KPS; ++u) {
      const int kk = u * KPS + warp * KPW + kg;  // key within the chunk
      const int j = jc + kk;
      const bool valid = j < j1;
      const uint8_t* kr = stK + kk * ROW + c8 * PPT * EB;
      const uint8_t* vr = stV + kk * ROW + c8 * PPT * EB;
      float x1[PPT], x2[PPT], y1[PPT], y2[PPT];
      load_cache<PPT, EB>(kr, x1);
      load_cache<PPT, EB>(kr + HALF * EB, x2);
      load_cache<PPT, EB>(vr, y1);
      load_cache<PPT, EB>(vr + HALF * EB, y2);
      if constexpr (kRotQ) {
        // raw key against the backward-rotated query, two pairs per packed op
        float d0 = 0.f, d1 = 0.f;
#pragma unroll
        for (int k = 0; k < PPT; k += 2) {
          fma2(d0, d1, qh1[k], qh1[k + 1], x1[k], x1[k + 1], d0, d1);
          fma2(d0, d1, qh2[k], qh2[k + 1], x2[k], x2[k + 1], d0, d1);
          // next key: q_hat <- R(-KPS theta) q_hat
          float n1a, n1b, n2a, n2b;
          mul2(n1a, n1b, qh2[k], qh2[k + 1], sts[k], sts[k + 1]);
          fma2(n1a, n1b, qh1[k], qh1[k + 1], stc[k], stc[k + 1], n1a, n1b);
          mul2(n2a, n2b, qh1[k], qh1[k + 1], nsts[k], nsts[k + 1]);
          fma2(n2a, n2b, qh2[k], qh2[k + 1], stc[k], stc[k + 1], n2a, n2b);
          qh1[k] = n1a; qh1[k + 1] = n1b; qh2[k] = n2a; qh2[k + 1] = n2b;
        }
        float dot = d0 + d1;
#pragma unroll
        for (int o = 1; o < TPK; o <<= 1) dot += __shfl_xor_sync(0xffffffffu, dot, o);
        dot *= k_scale;
        // The rare move of the lazy reference is one warp-uniform branch
        // instead of a divergent one per key.  Keys past the end (only in a
        // slice's last chunk) are skipped: their stage bytes were not loaded.
        const bool grow = valid && dot > mrun[0] + kRescaleThreshold;
        if (__any_sync(0xffffffffu, grow)) {
          const float mnew = grow ? dot : mrun[0];
          const float corr = exp2_diff(mrun[0], mnew);
          lrun[0] *= corr;
#pragma unroll
          for (int k = 0; k < PPT; ++k) { acc1[0][k] *= corr; acc2[0][k] *= corr; }
          mrun[0] = mnew;
        }
        if (valid) {
          const float pr = ex2(dot - mrun[0]);
          lrun[0] += pr;
#pragma unroll
          for (int k = 0; k < PPT; k += 2) {
            fma2(acc1[0][k], acc1[0][k + 1], pr, pr, y1[k], y1[k + 1], acc1[0][k], acc1[0][k + 1]);
            fma2(acc2[0][k], acc2[0][k + 1], pr, pr, y2[k], y2[k + 1], acc2[0][k], acc2[0][k + 1]);
          }
        }
      } else {
        float kr1[PPT], kr2[PPT];   // key as dotted: raw (kRotQ) or rotated at j
        float qa1[G][PPT], qa2[G][PPT];
        if (!kRecur && !identity) {
  #pragma unroll
          for (int k = 0; k < PPT; ++k) turn_cos_sin<false>((float)j, fr[k], rc[k], rs_[k]);
        }
  #pragma unroll
        for (int k = 0; k < PPT; ++k) {
          if (kRotQ) {
            kr1[k] = x1[k];
            kr2[k] = x2[k];
            qa1[0][k] = qh1[k];
            qa2[0][k] = qh2[k];
            // next key: q_hat <- R(-KPS theta) q_hat
            const float a1 = qh1[k], a2 = qh2[k];
            qh1[k] = a1 * stc[k] + a2 * sts[k];
            qh2[k] = a2 * stc[k] - a1 * sts[k];
          } else {
            kr1[k] = x1[k] * rc[k] - x2[k] * rs_[k];
            kr2[k] = x1[k] * rs_[k] + x2[k] * rc[k];
  #pragma unroll
            for (int g = 0; g < G; ++g) { qa1[g][k] = q1[g][k]; qa2[g][k] = q2[g][k]; }
          }
          // advance to the thread's next key: (m - j) decreases (kRotQ) or j
          // increases by KPS
          if (kRecur && !kRotQ) {
            const float c0 = rc[k], s0 = rs_[k];
            rc[k] = c0 * stc[k] - s0 * sts[k];
            rs_[k] = s0 * stc[k] + c0 * sts[k];
          }
        }
  #pragma unroll
        for (int g = 0; g < G; ++g) {
          float dot = 0.f;
  #pragma unroll
          for (int k = 0; k < PPT; ++k) dot = fmaf(qa1[g][k], kr1[k], fmaf(qa2[g][k], kr2[k], dot));
  #pragma unroll
          for (int o = 1; o < TPK; o <<= 1) dot += __shfl_xor_sync(0xffffffffu, dot, o);
          if (EB == 1) dot *= k_scale;
          if (valid) {
            if (dot > mrun[g] + kRescaleThreshold) {  // lazy: the reference moves rarely
              const float corr = exp2_diff(mrun[g], dot);
              lrun[g] *= corr;
  #pragma unroll
              for (int k = 0; k < PPT; ++k) { acc1[g][k] *= corr; acc2[g][k] *= corr; }
              mrun[g] = dot;
            }
            const float pr = exp2f(dot - mrun[g]);
            lrun[g] += pr;
  #pragma unroll
            for (int k = 0; k < PPT; ++k) {
              acc1[g][k] = fmaf(pr, y1[k], acc1[g][k]);
              acc2[g][k] = fmaf(pr, y2[k], acc2[g][k]);
            }
          }
        }
      }
      }
    __syncwarp();
    if (lane == 0) mbar_arrive(&empty[s]);
  }

  // Merge the key groups of the warp (lanes with equal c8).
#pragma unroll
  for (int o = TPK; o < 32; o <<= 1) {
#pragma unroll
    for (int g = 0; g < G; ++g) {
      const float om = __shfl_xor_sync(0xffffffffu, mrun[g], o);
      const float ol = __shfl_xor_sync(0xffffffffu, lrun[g], o);
      const float mn = fmaxf(mrun[g], om);
      const float ca = exp2_diff(mrun[g], mn), cb = exp2_diff(om, mn);
      lrun[g] = lrun[g] * ca + ol * cb;
#pragma unroll
      for (int k = 0; k < PPT; ++k) {
        const float a1 = __shfl_xor_sync(0xffffffffu, acc1[g][k], o);
        const float a2 = __shfl_xor_sync(0xffffffffu, acc2[g][k], o);
        acc1[g][k] = acc1[g][k] * ca + a1 * cb;
        acc2[g][k] = acc2[g][k] * ca + a2 * cb;
      }
      mrun[g] = mn;
    }
  }

  // Merge the warps in shared memory, reusing the stage buffers: every copy
  // the producer issued has been consumed (or drained after an abort) once
  // the block barrier below is passed.
  __syncthreads();
  float* s_acc = reinterpret_cast<float*>(smem);           // [kWarps][G][D]
  float* s_ml = s_acc + kWarps * G * D;                     // [kWarps][G][2]
  if (kg == 0) {
#pragma unroll
    for (int g = 0; g < G; ++g) {
#pragma unroll
      for (int k = 0; k < PPT; ++k) {
        s_acc[(warp * G + g) * D + c8 * PPT + k] = acc1[g][k];
        s_acc[(warp * G + g) * D + HALF + c8 * PPT + k] = acc2[g][k];
      }
      if (c8 == 0) {
        s_ml[(warp * G + g) * 2 + 0] = mrun[g];
        s_ml[(warp * G + g) * 2 + 1] = lrun[g];
      }
    }
  }
  asm volatile("bar.sync 1, %0;" ::"n"(kWarps * 32));  // compute warps only
  if (abort_flag) return;
  for (int t = threadIdx.x; t < G * D; t += kWarps * 32) {
    const int g = t / D, dim = t % D;
    float M = -INFINITY;
#pragma unroll
    for (int w = 0; w < kWarps; ++w) M = fmaxf(M, s_ml[(w * G + g) * 2]);
    float L = 0.f, O = 0.f;
#pragma unroll
    for (int w = 0; w < kWarps; ++w) {
      const float wt = exp2_diff(s_ml[(w * G + g) * 2], M);
      L += s_ml[(w * G + g) * 2 + 1] * wt;
      O += s_acc[(w * G + g) * D + dim] * wt;
    }
    O *= v_scale;
    const int64_t bhq = (int64_t)b * a.Hq + hq0 + g;
    if (a.splits == 1) {
      const float out = L > 0.f ? O / L : 0.f;
      static_cast<__nv_bfloat16*>(a.o)[bhq * D + dim] = __float2bfloat16_rn(out);
      if (dim == 0 && a.lse)
        a.lse[bhq] = L > 0.f ? (M + log2f(L)) * 0.69314718055994530942f : -INFINITY;
    } else {
      const int64_t rows = (int64_t)a.B * a.Hq;
      a.ws[((int64_t)split * rows + bhq) * D + dim] = O;
      if (dim == 0) {
        float* ml = a.ws + (int64_t)a.splits * rows * D;
        ml[((int64_t)split * rows + bhq) * 2 + 0] = M;
        ml[((int64_t)split * rows + bhq) * 2 + 1] = L;
      }
    }
  }
}

// Exact merge of the per-slice softmax states of one (sequence, query head).
__global__ void decode_merge_kernel(DecodeLaunch a) {
  const int64_t rows = (int64_t)a.B * a.Hq;
  const int64_t bhq = blockIdx.x;
  const int D = a.d;
  const float* ml = a.ws + (int64_t)a.splits * rows * D;
  float M = -INFINITY;
  for (int s = 0; s < a.splits; ++s) M = fmaxf(M, ml[((int64_t)s * rows + bhq) * 2]);
  for (int dim = threadIdx.x; dim < D; dim += blockDim.x) {
    float L = 0.f, O = 0.f;
    for (int s = 0; s < a.splits; ++s) {
      const float wt = exp2_diff(ml[((int64_t)s * rows + bhq) * 2], M);
      L += ml[((int64_t)s * rows + bhq) * 2 + 1] * wt;
      O += a.ws[((int64_t)s * rows + bhq) * D + dim] * wt;
    }
    static_cast<__nv_bfloat16*>(a.o)[bhq * D + dim] = __float2bfloat16_rn(L > 0.f ? O / L : 0.f);
    if (dim == 0 && a.lse) a.lse[bhq] = L > 0.f ? (M + log2f(L)) * 0.69314718055994530942f : -INFINITY;
  }
}

template <int D, int G, int EB>
cudaError_t launch_dg(const DecodeLaunch& a, const RopeFreqs& f, cudaStream_t st) {
  const int groups = (a.Hq / a.Hkv) / G;
  dim3 grid((unsigned)(a.B * a.Hkv), (unsigned)a.splits, (unsigned)groups);
  const int smem = DecodeShape<D, (G >= 2 ? 4 : 8), EB>::SMEM;
  cudaError_t e0 = cudaFuncSetAttribute(decode_kernel<D, G, EB>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e0 != cudaSuccess) return e0;
  decode_kernel<D, G, EB><<<grid, kThreads, smem, st>>>(a, f);
  cudaError_t e = launched(1);
  if (e != cudaSuccess || a.splits == 1) return e;
  decode_merge_kernel<<<(unsigned)(a.B * a.Hq), 128, 0, st>>>(a);
  return launched(1);
}

}  // namespace

cudaError_t launch_decode(const DecodeLaunch& a_in, const RopeFreqs& f, cudaStream_t st) {
  DecodeLaunch a = a_in;
  a.status = device_status_word();
  if (!a.status) return cudaErrorInvalidValue;
  const FaultInjection fi = fault_injection();
  a.wait_limit = fi.wait_limit;
  a.skip_unit = fi.skip_unit;
  const int G = a.Hq / a.Hkv;
  if (a.fp8) {
    if (a.d == 128) {
      if (G == 1) return launch_dg<128, 1, 1>(a, f, st);
      if (G == 2) return launch_dg<128, 2, 1>(a, f, st);
      return launch_dg<128, 4, 1>(a, f, st);
    }
    if (G == 1) return launch_dg<64, 1, 1>(a, f, st);
    if (G == 2) return launch_dg<64, 2, 1>(a, f, st);
    return launch_dg<64, 4, 1>(a, f, st);
  }
  if (a.d == 128) {
    if (G == 1) return launch_dg<128, 1, 2>(a, f, st);
    if (G == 2) return launch_dg<128, 2, 2>(a, f, st);
    return launch_dg<128, 4, 2>(a, f, st);  // G = 4 or 8 (two head groups)
  }
  if (G == 1) return launch_dg<64, 1, 2>(a, f, st);
  if (G == 2) return launch_dg<64, 2, 2>(a, f, st);
  return launch_dg<64, 4, 2>(a, f, st);
}

}  // namespace yr

// ---------------------------------------------------------------------------
// Allocation-free decode entry point.
//
// Some callers cannot hand the library a workspace: code that runs where
// device allocation is not allowed at call time (for example an engine's
// per-step enqueue hook that must not allocate, or a process whose memory is
// entirely reserved by another allocator) and callers that have no scratch
// buffer to spare.  For them the split-slice partial states live in one
// fixed array of device memory that belongs to the library: every GPU that
// loads the library holds it until the process exits.
//
// The array is shared by every call on a device and keeps the previous
// call's contents; the decode kernel writes every partial state it later
// merges, so nothing needs clearing between calls.  Calls whose work overlaps
// on the GPU (other streams, or launches not ordered on one stream) race on
// the array.
namespace yr {
namespace {

constexpr size_t kNoAllocScratchBytes = size_t(4) << 20;  // 4 MiB per device
static __device__ __align__(256) float g_decode_scratch[kNoAllocScratchBytes / sizeof(float)];

// Device address of g_decode_scratch on the current device.  In host code
// the array's name is only a host-side stand-in, so the address comes from
// cudaGetSymbolAddress, once per device, with that device current.
float* decode_scratch_address() {
  static std::mutex mu;
  static float* cached[128] = {nullptr};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 128) return nullptr;
  std::lock_guard<std::mutex> lock(mu);
  if (!cached[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_decode_scratch) != cudaSuccess) return nullptr;
    cached[dev] = static_cast<float*>(p);
  }
  return cached[dev];
}

}  // namespace
}  // namespace yr

extern "C" yr_status attn_fwd_decode_sinkwindow_noalloc(
    const yr_rope_cfg* cfg, const void* q, const void* k_cache, const void* v_cache, const int32_t* n_valid,
    const int32_t* ring_start, int32_t B, int32_t Hq, int32_t Hkv, int32_t d, int32_t sink, int32_t window,
    void* o, float* lse, int32_t num_splits, void* stream) {
  yr::clear_error();
  // the same argument errors as the workspace entry point, before the size test
  yr::RopeFreqs f;
  const yr_status st = yr::decode_check_shape("attn_fwd_decode_sinkwindow_noalloc", cfg, B, Hq, Hkv, d, sink,
                                              window, num_splits, &f);
  if (st != YR_OK) return st;
  const size_t need = yr_decode_workspace_bytes(B, Hq, Hkv, d, sink, window, num_splits);
  if (need > yr::kNoAllocScratchBytes) {
    return yr::fail(YR_ERR_INVALID_ARG,
                    "attn_fwd_decode_sinkwindow_noalloc: %zu bytes of split scratch needed, above its fixed "
                    "%zu-byte array; use fewer splits or attn_fwd_decode_sinkwindow with a workspace",
                    need, yr::kNoAllocScratchBytes);
  }
  void* scratch = nullptr;
  if (need > 0) {
    scratch = yr::decode_scratch_address();
    if (!scratch) {
      return yr::fail(YR_ERR_CUDA, "attn_fwd_decode_sinkwindow_noalloc: device scratch address unavailable");
    }
  }
  return attn_fwd_decode_sinkwindow(cfg, q, k_cache, v_cache, n_valid, ring_start, B, Hq, Hkv, d, sink, window,
                                    o, lse, num_splits, scratch, need, stream);
}
