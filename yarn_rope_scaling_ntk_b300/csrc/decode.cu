// attn_fwd_decode_sinkwindow: one new query token per sequence against a
// cache of `sink` pinned tokens plus a `window`-slot ring buffer ("Context
// Length Extension", Sliding Window + Attention Sinks; "Long-Context
// Scaling", Production defaults).  Keys are stored unrotated and rotated on
// read at their logical cache index; the query sits at n_valid - 1.
//
// HBM-bound: every valid cache entry is read once with 16-byte loads.  A CTA
// owns one (sequence, kv head) and one slice of the logical entries; TPK
// threads share a key (each holds 8 rotation pairs: one 16-byte vector from
// each half of the head dimension), and every key group keeps its own
// online-softmax state (running max, sum, unnormalised output) in registers.
// States are merged across the warp by shuffles, across warps in shared
// memory, and across slices by a second kernel.
#include <math.h>

#include <mutex>

#include "common.cuh"
#include "internal.h"

namespace yr {
namespace {

constexpr int kWarps = 8;
constexpr int kThreads = kWarps * 32;

struct OnlineState {
  float m, l;
};

__device__ __forceinline__ float exp2_diff(float a, float b) {
  // 2^(a - b) with a = -inf giving 0.
  return a == -INFINITY ? 0.f : exp2f(a - b);
}

template <int D, int G>
__global__ void __launch_bounds__(kThreads) decode_kernel(DecodeLaunch a, RopeFreqs f) {
  constexpr int TPK = D / 16;     // threads per key
  constexpr int KPW = 32 / TPK;   // keys per warp step
  constexpr int KPS = KPW * kWarps;
  constexpr int HALF = D / 2;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int c = lane % TPK, kg = lane / TPK;
  const int bh = blockIdx.x;
  const int b = bh / a.Hkv, hkv = bh % a.Hkv;
  const int hq0 = hkv * (a.Hq / a.Hkv) + blockIdx.z * G;
  const int split = blockIdx.y;
  const int C = a.sink + a.window;

  int n = a.n_valid[b];
  n = n < 0 ? 0 : (n > C ? C : n);
  int rs = a.ring_start[b];
  rs = ((rs % a.window) + a.window) % a.window;
  const int per = (n + a.splits - 1) / a.splits;
  const int j0 = min(n, split * per);
  const int j1 = min(n, j0 + per);

  float2 fr[8];
#pragma unroll
  for (int k = 0; k < 8; ++k) fr[k] = f.f[c * 8 + k];
  const bool identity = f.identity != 0;

  // Rotated query at position n - 1, pre-multiplied by scale * log2(e) so
  // that the dot product is the logit in base-2 units.
  float q1[G][8], q2[G][8];
  {
    float cs[8], sn[8];
    const float mq = (float)(n > 0 ? n - 1 : 0);
#pragma unroll
    for (int k = 0; k < 8; ++k) {
      if (identity) { cs[k] = 1.f; sn[k] = 0.f; }
      else turn_cos_sin<false>(mq, fr[k], cs[k], sn[k]);
    }
#pragma unroll
    for (int g = 0; g < G; ++g) {
      const __nv_bfloat16* qp = static_cast<const __nv_bfloat16*>(a.q) + ((int64_t)b * a.Hq + hq0 + g) * D;
      const uint4 u1 = *reinterpret_cast<const uint4*>(qp + c * 8);
      const uint4 u2 = *reinterpret_cast<const uint4*>(qp + HALF + c * 8);
      const uint32_t w1[4] = {u1.x, u1.y, u1.z, u1.w}, w2[4] = {u2.x, u2.y, u2.z, u2.w};
#pragma unroll
      for (int k = 0; k < 8; ++k) {
        const float x1 = (k & 1) ? bf16_hi(w1[k >> 1]) : bf16_lo(w1[k >> 1]);
        const float x2 = (k & 1) ? bf16_hi(w2[k >> 1]) : bf16_lo(w2[k >> 1]);
        q1[g][k] = (x1 * cs[k] - x2 * sn[k]) * a.scale_log2;
        q2[g][k] = (x1 * sn[k] + x2 * cs[k]) * a.scale_log2;
      }
    }
  }

  OnlineState st[G];
  float acc1[G][8], acc2[G][8];
#pragma unroll
  for (int g = 0; g < G; ++g) {
    st[g].m = -INFINITY; st[g].l = 0.f;
#pragma unroll
    for (int k = 0; k < 8; ++k) { acc1[g][k] = 0.f; acc2[g][k] = 0.f; }
  }

  const __nv_bfloat16* kbase = static_cast<const __nv_bfloat16*>(a.kc) + (int64_t)bh * C * D + c * 8;
  const __nv_bfloat16* vbase = static_cast<const __nv_bfloat16*>(a.vc) + (int64_t)bh * C * D + c * 8;

  constexpr int U = 2;  // keys in flight per thread
  // jw is warp-uniform, so every lane runs the shuffles; lanes past the end
  // load nothing and skip the update.
  for (int jw = j0 + warp * KPW; jw < j1; jw += U * KPS) {
    const int jb = jw + kg;
    uint4 kd1[U], kd2[U], vd1[U], vd2[U];
    bool ok[U];
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const int j = jb + u * KPS;
      ok[u] = j < j1;
      if (ok[u]) {
        int t = j - a.sink;
        const int phys = j < a.sink ? j : a.sink + ((rs + t) % a.window);
        const int64_t off = (int64_t)phys * D;
        kd1[u] = __ldg(reinterpret_cast<const uint4*>(kbase + off));
        kd2[u] = __ldg(reinterpret_cast<const uint4*>(kbase + off + HALF));
        vd1[u] = __ldg(reinterpret_cast<const uint4*>(vbase + off));
        vd2[u] = __ldg(reinterpret_cast<const uint4*>(vbase + off + HALF));
      } else {
        kd1[u] = kd2[u] = vd1[u] = vd2[u] = make_uint4(0, 0, 0, 0);
      }
    }
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const int j = jb + u * KPS;
      const uint32_t k1w[4] = {kd1[u].x, kd1[u].y, kd1[u].z, kd1[u].w};
      const uint32_t k2w[4] = {kd2[u].x, kd2[u].y, kd2[u].z, kd2[u].w};
      float kr1[8], kr2[8];
#pragma unroll
      for (int k = 0; k < 8; ++k) {
        const float x1 = (k & 1) ? bf16_hi(k1w[k >> 1]) : bf16_lo(k1w[k >> 1]);
        const float x2 = (k & 1) ? bf16_hi(k2w[k >> 1]) : bf16_lo(k2w[k >> 1]);
        float cs = 1.f, sn = 0.f;
        if (!identity) turn_cos_sin<false>((float)j, fr[k], cs, sn);
        kr1[k] = x1 * cs - x2 * sn;
        kr2[k] = x1 * sn + x2 * cs;
      }
      const uint32_t v1w[4] = {vd1[u].x, vd1[u].y, vd1[u].z, vd1[u].w};
      const uint32_t v2w[4] = {vd2[u].x, vd2[u].y, vd2[u].z, vd2[u].w};
#pragma unroll
      for (int g = 0; g < G; ++g) {
        float dot = 0.f;
#pragma unroll
        for (int k = 0; k < 8; ++k) dot = fmaf(q1[g][k], kr1[k], fmaf(q2[g][k], kr2[k], dot));
#pragma unroll
        for (int o = 1; o < TPK; o <<= 1) dot += __shfl_xor_sync(0xffffffffu, dot, o);
        if (ok[u]) {
          const float mn = fmaxf(st[g].m, dot);
          const float corr = exp2_diff(st[g].m, mn);
          const float p = exp2f(dot - mn);
          st[g].l = st[g].l * corr + p;
          st[g].m = mn;
#pragma unroll
          for (int k = 0; k < 8; ++k) {
            const float y1 = (k & 1) ? bf16_hi(v1w[k >> 1]) : bf16_lo(v1w[k >> 1]);
            const float y2 = (k & 1) ? bf16_hi(v2w[k >> 1]) : bf16_lo(v2w[k >> 1]);
            acc1[g][k] = fmaf(p, y1, acc1[g][k] * corr);
            acc2[g][k] = fmaf(p, y2, acc2[g][k] * corr);
          }
        }
      }
    }
  }

  // Merge the key groups of the warp (lanes with equal c).
#pragma unroll
  for (int o = TPK; o < 32; o <<= 1) {
#pragma unroll
    for (int g = 0; g < G; ++g) {
      const float om = __shfl_xor_sync(0xffffffffu, st[g].m, o);
      const float ol = __shfl_xor_sync(0xffffffffu, st[g].l, o);
      const float mn = fmaxf(st[g].m, om);
      const float ca = exp2_diff(st[g].m, mn), cb = exp2_diff(om, mn);
      st[g].l = st[g].l * ca + ol * cb;
#pragma unroll
      for (int k = 0; k < 8; ++k) {
        const float a1 = __shfl_xor_sync(0xffffffffu, acc1[g][k], o);
        const float a2 = __shfl_xor_sync(0xffffffffu, acc2[g][k], o);
        acc1[g][k] = acc1[g][k] * ca + a1 * cb;
        acc2[g][k] = acc2[g][k] * ca + a2 * cb;
      }
      st[g].m = mn;
    }
  }

  // Merge the warps in shared memory.
  __shared__ float s_acc[kWarps][G][D];
  __shared__ float s_ml[kWarps][G][2];
  if (kg == 0) {
#pragma unroll
    for (int g = 0; g < G; ++g) {
#pragma unroll
      for (int k = 0; k < 8; ++k) {
        s_acc[warp][g][c * 8 + k] = acc1[g][k];
        s_acc[warp][g][HALF + c * 8 + k] = acc2[g][k];
      }
      if (c == 0) { s_ml[warp][g][0] = st[g].m; s_ml[warp][g][1] = st[g].l; }
    }
  }
  __syncthreads();
  for (int t = threadIdx.x; t < G * D; t += kThreads) {
    const int g = t / D, dim = t % D;
    float M = -INFINITY;
#pragma unroll
    for (int w = 0; w < kWarps; ++w) M = fmaxf(M, s_ml[w][g][0]);
    float L = 0.f, O = 0.f;
#pragma unroll
    for (int w = 0; w < kWarps; ++w) {
      const float wt = exp2_diff(s_ml[w][g][0], M);
      L += s_ml[w][g][1] * wt;
      O += s_acc[w][g][dim] * wt;
    }
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

template <int D, int G>
cudaError_t launch_dg(const DecodeLaunch& a, const RopeFreqs& f, cudaStream_t st) {
  const int groups = (a.Hq / a.Hkv) / G;
  dim3 grid((unsigned)(a.B * a.Hkv), (unsigned)a.splits, (unsigned)groups);
  decode_kernel<D, G><<<grid, kThreads, 0, st>>>(a, f);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess || a.splits == 1) return e;
  decode_merge_kernel<<<(unsigned)(a.B * a.Hq), 128, 0, st>>>(a);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_decode(const DecodeLaunch& a, const RopeFreqs& f, cudaStream_t st) {
  const int G = a.Hq / a.Hkv;
  if (a.d == 128) {
    if (G == 1) return launch_dg<128, 1>(a, f, st);
    if (G == 2) return launch_dg<128, 2>(a, f, st);
    return launch_dg<128, 4>(a, f, st);  // G = 4 or 8 (two head groups)
  }
  if (G == 1) return launch_dg<64, 1>(a, f, st);
  if (G == 2) return launch_dg<64, 2>(a, f, st);
  return launch_dg<64, 4>(a, f, st);
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
  const size_t need = yr_decode_workspace_bytes(B, Hq, Hkv, d, sink, window, num_splits);
  if (need > yr::kNoAllocScratchBytes) {
    yr::clear_error();
    return yr::fail(YR_ERR_INVALID_ARG,
                    "attn_fwd_decode_sinkwindow_noalloc: %zu bytes of split scratch needed, above its fixed "
                    "%zu-byte array; use fewer splits or attn_fwd_decode_sinkwindow with a workspace",
                    need, yr::kNoAllocScratchBytes);
  }
  void* scratch = nullptr;
  if (need > 0) {
    scratch = yr::decode_scratch_address();
    if (!scratch) {
      yr::clear_error();
      return yr::fail(YR_ERR_CUDA, "attn_fwd_decode_sinkwindow_noalloc: device scratch address unavailable");
    }
  }
  return attn_fwd_decode_sinkwindow(cfg, q, k_cache, v_cache, n_valid, ring_start, B, Hq, Hkv, d, sink, window,
                                    o, lse, num_splits, scratch, need, stream);
}
