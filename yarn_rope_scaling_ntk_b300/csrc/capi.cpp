// Host side of the C ABI: argument checks, the float64 frequency table and
// dispatch to the kernels.  Nothing here allocates device memory.
#include <math.h>
#include <stdarg.h>
#include <stdio.h>
#include <string.h>

#include <algorithm>

#include "internal.h"

namespace yr {

static thread_local char g_msg[512] = {0};

yr_status fail(yr_status st, const char* fmt, ...) {
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(g_msg, sizeof(g_msg), fmt, ap);
  va_end(ap);
  return st;
}

void clear_error() { g_msg[0] = 0; }

yr_status cuda_fail(cudaError_t e, const char* what) {
  return fail(YR_ERR_CUDA, "%s: %s", what, cudaGetErrorString(e));
}

static const double kTwoPi = 6.283185307179586476925286766559;

// Frequencies theta'_i in float64.  Definitions:
//  base      theta_i = b^(-2i/d)         "Context Window Scaling ...", Section 2
//  PI        theta_i / s                 same page, Section 2 (m' = m / s)
//  NTK       b' = b s^(d/(d-2))          "Context Length Extension", NTK-Aware
//                                        Scaling (reading: lowest frequency
//                                        interpolated by s, highest kept)
//  YaRN      (1-g) theta_i/s + g theta_i "Context Window Scaling ...", Section 3
//            g = clamp((r-alpha)/(beta-alpha)), r = L_train / lambda_i,
//            lambda_i = 2 pi b^(2i/d)
//  mscale    0.1 ln s + 1 (YaRN, s > 1)  same page, Section 3 and its listing
//  PERDIM    theta_i / lambda_i          same page, Section 4 (a scale vector
//                                        per dimension, caller-given)
yr_status compute_inv_freq(const yr_rope_cfg* cfg, int d, double* theta, int8_t* cls,
                           double* mscale) {
  if (!cfg) return fail(YR_ERR_INVALID_ARG, "cfg is NULL");
  const int kind = cfg->kind;
  if (kind < YR_ROPE_NONE || kind > YR_ROPE_PERDIM)
    return fail(YR_ERR_INVALID_ARG, "unknown rope kind %d", kind);
  if (d < 2 || (d & 1)) return fail(YR_ERR_INVALID_ARG, "head dimension %d must be even and >= 2", d);
  if (d / 2 > kMaxHalf) return fail(YR_ERR_UNSUPPORTED, "head dimension %d above %d", d, 2 * kMaxHalf);
  if (cfg->head_dim != 0 && cfg->head_dim != d)
    return fail(YR_ERR_INVALID_ARG, "cfg.head_dim %d differs from d %d", cfg->head_dim, d);
  const double b = cfg->theta_base;
  if (!(b > 1.0) || !isfinite(b)) return fail(YR_ERR_INVALID_ARG, "theta_base must be finite and > 1");
  double alpha = cfg->ramp_alpha, beta = cfg->ramp_beta;
  if (alpha == 0.0 && beta == 0.0) { alpha = 1.0; beta = 32.0; }
  if (!(beta > alpha)) return fail(YR_ERR_INVALID_ARG, "ramp_beta must exceed ramp_alpha");
  double s = 1.0;
  const bool scaled = kind == YR_ROPE_PI || kind == YR_ROPE_NTK || kind == YR_ROPE_YARN;
  if (scaled) {
    if (cfg->s > 0.0) {
      if (!isfinite(cfg->s)) return fail(YR_ERR_INVALID_ARG, "s must be finite");
      s = cfg->s;
    } else if (cfg->L_train > 0 && cfg->L_target > 0) {
      s = (double)cfg->L_target / (double)cfg->L_train;
    } else {
      return fail(YR_ERR_INVALID_ARG, "need s > 0 or L_train and L_target > 0");
    }
  }
  if (kind == YR_ROPE_YARN && cfg->L_train <= 0) return fail(YR_ERR_INVALID_ARG, "YaRN needs L_train > 0");
  if (kind == YR_ROPE_PERDIM) {
    if (!cfg->dim_scale) return fail(YR_ERR_INVALID_ARG, "PERDIM needs dim_scale (d/2 factors)");
    for (int i = 0; i < d / 2; ++i)
      if (!(cfg->dim_scale[i] > 0.0) || !isfinite(cfg->dim_scale[i]))
        return fail(YR_ERR_INVALID_ARG, "dim_scale[%d] must be finite and > 0", i);
  }
  if (kind == YR_ROPE_NTK && d <= 2) return fail(YR_ERR_INVALID_ARG, "NTK scaling needs d > 2");

  const int h = d / 2;
  const double bb = kind == YR_ROPE_NTK ? b * pow(s, (double)d / (double)(d - 2)) : b;
  for (int i = 0; i < h; ++i) {
    const double base_i = pow(b, -2.0 * i / d);
    double r = 0.0;
    if (cfg->L_train > 0) r = (double)cfg->L_train / (kTwoPi * pow(b, 2.0 * i / d));
    if (cls) cls[i] = cfg->L_train <= 0 ? 2 : (r < alpha ? 0 : (r > beta ? 2 : 1));
    double t;
    switch (kind) {
      case YR_ROPE_NONE: t = 0.0; break;
      case YR_ROPE_PLAIN: t = base_i; break;
      case YR_ROPE_PI: t = base_i / s; break;
      case YR_ROPE_NTK: t = pow(bb, -2.0 * i / d); break;
      case YR_ROPE_PERDIM: t = base_i / cfg->dim_scale[i]; break;
      default: {
        const double g = std::min(1.0, std::max(0.0, (r - alpha) / (beta - alpha)));
        t = (1.0 - g) * base_i / s + g * base_i;
      }
    }
    theta[i] = t;
  }
  double ms = (kind == YR_ROPE_YARN && s > 1.0) ? 0.1 * log(s) + 1.0 : 1.0;
  if (cfg->mscale_override > 0.0) ms = cfg->mscale_override;
  if (mscale) *mscale = ms;
  return YR_OK;
}

yr_status build_rope_freqs(const yr_rope_cfg* cfg, int d, RopeFreqs* out) {
  double theta[kMaxHalf];
  double ms = 1.0;
  yr_status st = compute_inv_freq(cfg, d, theta, nullptr, &ms);
  if (st != YR_OK) return st;
  memset(out, 0, sizeof(*out));
  out->half = d / 2;
  out->mscale = (float)ms;
  out->identity = cfg->kind == YR_ROPE_NONE;
  for (int i = 0; i < d / 2; ++i) {
    const double f = theta[i] / kTwoPi;  // turns per position
    const float hi = (float)f;
    out->f[i] = make_float2(hi, (float)(f - (double)hi));
  }
  return YR_OK;
}

// The shape and configuration checks of the decode entry points, in the
// order they report errors (no pointer is dereferenced).
yr_status decode_check_shape(const char* who, const yr_rope_cfg* cfg, int32_t B, int32_t Hq, int32_t Hkv,
                             int32_t d, int32_t sink, int32_t window, int32_t num_splits, RopeFreqs* f) {
  if (!cfg) return fail(YR_ERR_INVALID_ARG, "%s: cfg is NULL", who);
  if (B < 0 || Hq < 0 || Hkv < 0) return fail(YR_ERR_INVALID_ARG, "negative shape");
  if (d != 64 && d != 128) return fail(YR_ERR_UNSUPPORTED, "decode head dimension %d (64 or 128)", d);
  if (Hkv <= 0 || Hq <= 0 || Hq % Hkv != 0) return fail(YR_ERR_INVALID_ARG, "Hq %% Hkv != 0");
  const int G = Hq / Hkv;
  if (G != 1 && G != 2 && G != 4 && G != 8)
    return fail(YR_ERR_UNSUPPORTED, "decode supports Hq/Hkv in {1, 2, 4, 8}, got %d", G);
  if (sink < 0 || window < 1) return fail(YR_ERR_INVALID_ARG, "sink must be >= 0 and window >= 1");
  if ((int64_t)sink + window > (1 << 24)) return fail(YR_ERR_INVALID_ARG, "cache above 2^24 entries");
  if (num_splits > 4096) return fail(YR_ERR_INVALID_ARG, "num_splits above 4096");
  return build_rope_freqs(cfg, d, f);
}

}  // namespace yr

using namespace yr;

namespace {

bool aligned16(const void* p) { return ((uintptr_t)p & 15u) == 0; }

bool rows_aligned(const int64_t s[3], int elem) {
  for (int i = 0; i < 3; ++i)
    if (s[i] < 0 || (s[i] * elem) % 16 != 0) return false;
  return true;
}

cudaStream_t as_stream(void* s) { return reinterpret_cast<cudaStream_t>(s); }

}  // namespace

extern "C" {

const char* yr_version(void) { return "yarn_attn 0.1 (sm_103a)"; }

const char* yr_last_error_message(void) { return g_msg; }

yr_status yarn_inv_freq(const yr_rope_cfg* cfg, double* inv_freq, int8_t* cls, double* mscale) {
  clear_error();
  if (!inv_freq) return fail(YR_ERR_INVALID_ARG, "inv_freq is NULL");
  if (!cfg) return fail(YR_ERR_INVALID_ARG, "cfg is NULL");
  return compute_inv_freq(cfg, cfg->head_dim, inv_freq, cls, mscale);
}

yr_status rope_apply(const yr_rope_cfg* cfg, const void* x, void* y, int32_t dtype, int32_t B,
                     int32_t H, int32_t S, int32_t d, const int64_t x_strides[3],
                     const int64_t y_strides[3], int32_t pos0, const int32_t* positions,
                     int32_t apply_mscale, void* stream) {
  clear_error();
  if (dtype != YR_F32 && dtype != YR_BF16) return fail(YR_ERR_INVALID_ARG, "dtype %d", dtype);
  if (B < 0 || H < 0 || S < 0) return fail(YR_ERR_INVALID_ARG, "negative shape");
  if (!x_strides || !y_strides) return fail(YR_ERR_INVALID_ARG, "strides are NULL");
  RopeFreqs f;
  yr_status st = build_rope_freqs(cfg, d, &f);
  if (st != YR_OK) return st;
  const int vec = dtype == YR_BF16 ? 8 : 4;
  const int tpr = d / 2 / vec;
  if ((d / 2) % vec != 0 || (tpr & (tpr - 1)) != 0 || tpr > 32)
    return fail(YR_ERR_UNSUPPORTED, "rope_apply: d=%d not supported (d/2 must be a power-of-two multiple of %d)", d, vec);
  if (pos0 < 0 || (int64_t)pos0 + S > (1 << 24))
    return fail(YR_ERR_INVALID_ARG, "positions must lie in [0, 2^24)");
  if ((int64_t)B * H * S == 0) return YR_OK;
  if (!x || !y) return fail(YR_ERR_INVALID_ARG, "x or y is NULL");
  const int elem = dtype == YR_BF16 ? 2 : 4;
  if (!aligned16(x) || !aligned16(y) || !rows_aligned(x_strides, elem) || !rows_aligned(y_strides, elem))
    return fail(YR_ERR_INVALID_ARG, "pointers and strides must be 16-byte aligned");
  if (x == y && memcmp(x_strides, y_strides, 3 * sizeof(int64_t)) != 0)
    return fail(YR_ERR_INVALID_ARG, "in-place rope_apply needs identical strides");
  RopeLaunch a;
  memset(&a, 0, sizeof(a));
  a.n_seg = 1;
  RopeSegment& sg = a.seg[0];
  sg.x = x; sg.y = y; sg.H = H; sg.S = S; sg.pos0 = pos0;
  for (int i = 0; i < 3; ++i) { sg.xs[i] = x_strides[i]; sg.ys[i] = y_strides[i]; }
  a.in_bf16 = a.out_bf16 = dtype == YR_BF16;
  a.B = B; a.d = d;
  a.positions = positions; a.apply_mscale = apply_mscale != 0;
  cudaError_t e = launch_rope(a, f, as_stream(stream));
  return e == cudaSuccess ? YR_OK : cuda_fail(e, "rope_apply launch");
}

static bool prefill_needs_q_copy(int in_dtype, const yr_rope_cfg* cfg) {
  return in_dtype == YR_F32 || cfg->kind != YR_ROPE_NONE;
}

static size_t prefill_ws_bytes(const yr_rope_cfg* cfg, int in_dtype, int B, int Hq, int Hkv, int Sq, int Skv,
                               int d) {
  if (!cfg || B <= 0 || Hq <= 0 || Hkv <= 0 || Sq <= 0 || Skv <= 0 || d <= 0) return 0;
  size_t bytes = 0;
  if (prefill_needs_q_copy(in_dtype, cfg))
    bytes += (size_t)B * Hq * Sq * d * 2 + (size_t)B * Hkv * Skv * d * 2;
  if (in_dtype == YR_F32) bytes += (size_t)B * Hkv * Skv * d * 2;
  return bytes;
}

size_t yr_prefill_workspace_bytes(const yr_rope_cfg* cfg, int32_t in_dtype, int32_t B, int32_t Hq,
                                  int32_t Hkv, int32_t S, int32_t d) {
  return prefill_ws_bytes(cfg, in_dtype, B, Hq, Hkv, S, S, d);
}

size_t yr_prefill_kv_block_workspace_bytes(const yr_rope_cfg* cfg, int32_t in_dtype, int32_t B, int32_t Hq,
                                           int32_t Hkv, int32_t Sq, int32_t Skv, int32_t d) {
  return prefill_ws_bytes(cfg, in_dtype, B, Hq, Hkv, Sq, Skv, d);
}

// Shared body of attn_fwd_prefill and attn_fwd_prefill_kv_block: query rows
// at positions q_pos0 .. q_pos0 + Sq - 1 against keys at k_pos0 .. k_pos0 +
// Skv - 1 (positions drive both the rotation and the mask).
static yr_status prefill_impl(const char* who, const yr_rope_cfg* cfg, const void* q, const void* k,
                              const void* v, void* o, float* lse, int32_t in_dtype, int32_t out_dtype,
                              int32_t B, int32_t Hq, int32_t Hkv, int32_t Sq, int32_t Skv, int32_t d,
                              int32_t q_pos0, int32_t k_pos0, const int64_t q_strides[3],
                              const int64_t k_strides[3], const int64_t v_strides[3],
                              const int64_t o_strides[3], int32_t mask, int32_t sink, int32_t window,
                              int32_t ring_blocks, float softmax_scale, void* workspace,
                              size_t workspace_bytes, void* stream) {
  if (!cfg) return fail(YR_ERR_INVALID_ARG, "%s: cfg is NULL", who);
  if (in_dtype != YR_F32 && in_dtype != YR_BF16) return fail(YR_ERR_INVALID_ARG, "%s: dtype %d", who, in_dtype);
  if (out_dtype != YR_F32 && out_dtype != YR_BF16) return fail(YR_ERR_INVALID_ARG, "%s: out dtype %d", who, out_dtype);
  if (B < 0 || Hq < 0 || Hkv < 0 || Sq < 0 || Skv < 0) return fail(YR_ERR_INVALID_ARG, "%s: negative shape", who);
  if (d != 64 && d != 128) return fail(YR_ERR_UNSUPPORTED, "attention head dimension %d (64 or 128)", d);
  if (Hkv <= 0 || Hq <= 0 || Hq % Hkv != 0) return fail(YR_ERR_INVALID_ARG, "Hq %% Hkv != 0");
  if (mask < YR_MASK_CAUSAL || mask > YR_MASK_NONE) return fail(YR_ERR_INVALID_ARG, "mask %d", mask);
  if (mask == YR_MASK_SINK_WINDOW && (sink < 0 || window < 1))
    return fail(YR_ERR_INVALID_ARG, "sink must be >= 0 and window >= 1");
  if (ring_blocks < 1) return fail(YR_ERR_INVALID_ARG, "ring_blocks must be >= 1");
  if (q_pos0 < 0 || k_pos0 < 0 || (int64_t)q_pos0 + Sq > (1 << 24) || (int64_t)k_pos0 + Skv > (1 << 24))
    return fail(YR_ERR_INVALID_ARG, "%s: positions must lie in [0, 2^24)", who);
  if (!q_strides || !k_strides || !v_strides || !o_strides) return fail(YR_ERR_INVALID_ARG, "strides are NULL");
  RopeFreqs f;
  yr_status st = build_rope_freqs(cfg, d, &f);
  if (st != YR_OK) return st;
  if (ring_blocks > 1 && Skv % ring_blocks != 0)
    return fail(YR_ERR_INVALID_ARG, "S=%d is not divisible by ring_blocks=%d", Skv, ring_blocks);
  if (ring_blocks > 1 && (Skv / ring_blocks) % 64 != 0)
    return fail(YR_ERR_UNSUPPORTED, "ring blocks must hold a multiple of 64 keys");
  if (B == 0 || Sq == 0) return YR_OK;
  if (!q || !o || (Skv > 0 && (!k || !v))) return fail(YR_ERR_INVALID_ARG, "q, k, v or o is NULL");
  const int elem = in_dtype == YR_BF16 ? 2 : 4;
  const int oelem = out_dtype == YR_BF16 ? 2 : 4;
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(o) || !rows_aligned(q_strides, elem) ||
      !rows_aligned(k_strides, elem) || !rows_aligned(v_strides, elem) || !rows_aligned(o_strides, oelem))
    return fail(YR_ERR_INVALID_ARG, "pointers and strides must be 16-byte aligned");
  const size_t need = prefill_ws_bytes(cfg, in_dtype, B, Hq, Hkv, Sq, Skv, d);
  if (need > 0 && (!workspace || workspace_bytes < need))
    return fail(YR_ERR_INVALID_ARG, "workspace of %zu bytes needed", need);
  if (need > 0 && !aligned16(workspace)) return fail(YR_ERR_INVALID_ARG, "workspace must be 16-byte aligned");

  double ms = f.mscale;
  const double scale = softmax_scale > 0.f ? (double)softmax_scale : ms * ms / sqrt((double)d);
  cudaStream_t cs = as_stream(stream);

  PrefillLaunch p;
  memset(&p, 0, sizeof(p));
  p.q = q; p.k = k; p.v = v; p.o = o; p.lse = lse; p.out_bf16 = out_dtype == YR_BF16;
  p.B = B; p.Hq = Hq; p.Hkv = Hkv; p.d = d;
  p.Sq = Sq; p.Skv = Skv; p.q_pos0 = q_pos0; p.k_pos0 = k_pos0;
  for (int i = 0; i < 3; ++i) {
    p.qs[i] = q_strides[i]; p.ks[i] = k_strides[i]; p.vs[i] = v_strides[i]; p.os[i] = o_strides[i];
  }
  p.mask = mask; p.sink = sink; p.window = window; p.ring_blocks = ring_blocks;
  p.scale_log2 = (float)(scale * 1.4426950408889634073599246810019);

  if (Skv == 0) {
    // no keys: every row is the empty softmax, o = 0 and lse = -inf
    cudaError_t e = launch_fill_empty(o, p.out_bf16, lse, B, Hq, Sq, d, o_strides, cs);
    return e == cudaSuccess ? YR_OK : cuda_fail(e, "attention (empty key set) launch");
  }

  // Rotated bfloat16 copies in the workspace, each [B, H, rows, d]
  // contiguous: Q (rotated at q_pos0 + row), K (rotated at k_pos0 + key),
  // and V (converted) for float32 inputs -- one launch for all of them.
  char* ws = static_cast<char*>(workspace);
  size_t off = 0;
  RopeLaunch ra;
  memset(&ra, 0, sizeof(ra));
  ra.in_bf16 = in_dtype == YR_BF16; ra.out_bf16 = 1;
  ra.B = B; ra.d = d;
  auto prep = [&](const void* src, const int64_t* src_s, int H, int rows, int pos0, bool rotate,
                  const void** dst, int64_t* dst_s) {
    void* out = ws + off;
    const int64_t hs = (int64_t)rows * d;
    off += (size_t)B * H * hs * 2;
    RopeSegment& sg = ra.seg[ra.n_seg++];
    sg.x = src; sg.y = out; sg.H = H; sg.S = rows; sg.pos0 = pos0; sg.identity = rotate ? 0 : 1;
    dst_s[0] = (int64_t)H * hs; dst_s[1] = hs; dst_s[2] = d;
    for (int i = 0; i < 3; ++i) { sg.xs[i] = src_s[i]; sg.ys[i] = dst_s[i]; }
    *dst = out;
  };
  if (prefill_needs_q_copy(in_dtype, cfg)) {
    prep(q, q_strides, Hq, Sq, q_pos0, true, &p.q, p.qs);
    prep(k, k_strides, Hkv, Skv, k_pos0, true, &p.k, p.ks);
    if (in_dtype == YR_F32) prep(v, v_strides, Hkv, Skv, 0, false, &p.v, p.vs);
    cudaError_t e = launch_rope(ra, f, cs);
    if (e != cudaSuccess) return cuda_fail(e, "attention rotation pass");
  }
  cudaError_t e = launch_prefill(p, cs);
  return e == cudaSuccess ? YR_OK : cuda_fail(e, "attention launch");
}

yr_status attn_fwd_prefill(const yr_rope_cfg* cfg, const void* q, const void* k, const void* v,
                           void* o, float* lse, int32_t in_dtype, int32_t B, int32_t Hq,
                           int32_t Hkv, int32_t S, int32_t d, const int64_t q_strides[3],
                           const int64_t k_strides[3], const int64_t v_strides[3],
                           const int64_t o_strides[3], int32_t mask, int32_t sink,
                           int32_t window, int32_t ring_blocks, float softmax_scale,
                           void* workspace, size_t workspace_bytes, void* stream) {
  clear_error();
  if (S > (1 << 24)) return fail(YR_ERR_INVALID_ARG, "S above 2^24");
  return prefill_impl("attn_fwd_prefill", cfg, q, k, v, o, lse, in_dtype, in_dtype, B, Hq, Hkv, S, S, d, 0, 0,
                      q_strides, k_strides, v_strides, o_strides, mask, sink, window, ring_blocks, softmax_scale,
                      workspace, workspace_bytes, stream);
}

yr_status attn_fwd_prefill_kv_block(const yr_rope_cfg* cfg, const void* q, const void* k, const void* v,
                                    void* o, float* lse, int32_t in_dtype, int32_t out_dtype, int32_t B,
                                    int32_t Hq, int32_t Hkv, int32_t Sq, int32_t Skv, int32_t d,
                                    int32_t q_pos0, int32_t k_pos0, const int64_t q_strides[3],
                                    const int64_t k_strides[3], const int64_t v_strides[3],
                                    const int64_t o_strides[3], int32_t mask, int32_t sink, int32_t window,
                                    float softmax_scale, void* workspace, size_t workspace_bytes,
                                    void* stream) {
  clear_error();
  return prefill_impl("attn_fwd_prefill_kv_block", cfg, q, k, v, o, lse, in_dtype, out_dtype, B, Hq, Hkv, Sq,
                      Skv, d, q_pos0, k_pos0, q_strides, k_strides, v_strides, o_strides, mask, sink, window, 1,
                      softmax_scale, workspace, workspace_bytes, stream);
}

yr_status attn_merge_partial(float* o_acc, float* lse_acc, const float* o_part, const float* lse_part,
                             void* o_final, int32_t final_dtype, int32_t B, int32_t H, int32_t S, int32_t d,
                             const int64_t acc_strides[3], const int64_t part_strides[3],
                             const int64_t final_strides[3], void* stream) {
  clear_error();
  if (B < 0 || H < 0 || S < 0) return fail(YR_ERR_INVALID_ARG, "attn_merge_partial: negative shape");
  if (d <= 0 || d % 4 != 0 || d > 1024) return fail(YR_ERR_UNSUPPORTED, "attn_merge_partial: d=%d (a multiple of 4 up to 1024)", d);
  if (final_dtype != YR_F32 && final_dtype != YR_BF16) return fail(YR_ERR_INVALID_ARG, "final dtype %d", final_dtype);
  if ((int64_t)B * H * S == 0) return YR_OK;
  if (!o_acc || !lse_acc || !o_part || !lse_part || !acc_strides || !part_strides)
    return fail(YR_ERR_INVALID_ARG, "attn_merge_partial: a required pointer is NULL");
  if (o_final && !final_strides) return fail(YR_ERR_INVALID_ARG, "attn_merge_partial: final strides are NULL");
  const int felem = final_dtype == YR_BF16 ? 2 : 4;
  if (!aligned16(o_acc) || !aligned16(o_part) || !rows_aligned(acc_strides, 4) || !rows_aligned(part_strides, 4) ||
      (o_final && (((uintptr_t)o_final & 7) != 0 || !rows_aligned(final_strides, felem))))
    return fail(YR_ERR_INVALID_ARG, "attn_merge_partial: pointers and strides must be 16-byte aligned");
  MergeLaunch m;
  memset(&m, 0, sizeof(m));
  m.o_acc = o_acc; m.lse_acc = lse_acc; m.o_part = o_part; m.lse_part = lse_part;
  m.o_final = o_final; m.final_bf16 = final_dtype == YR_BF16;
  m.B = B; m.H = H; m.S = S; m.d = d;
  for (int i = 0; i < 3; ++i) {
    m.as[i] = acc_strides[i]; m.ps[i] = part_strides[i]; m.fs[i] = o_final ? final_strides[i] : 0;
  }
  cudaError_t e = launch_merge(m, as_stream(stream));
  return e == cudaSuccess ? YR_OK : cuda_fail(e, "attn_merge_partial launch");
}

static size_t align16(size_t x) { return (x + 15) & ~(size_t)15; }

size_t yr_bwd_workspace_bytes(const yr_rope_cfg* cfg, int32_t in_dtype, int32_t B, int32_t Hq, int32_t Hkv,
                              int32_t S, int32_t d) {
  if (!cfg || B <= 0 || Hq <= 0 || Hkv <= 0 || S <= 0 || d <= 0) return 0;
  const size_t q = (size_t)B * Hq * S * d * 2, kv = (size_t)B * Hkv * S * d * 2;
  size_t bytes = align16(q) + align16(kv);                   // rotated Q, K
  if (in_dtype == YR_F32) bytes += align16(kv) + align16(q);  // bf16 V, dO
  bytes += 2 * align16((size_t)B * Hq * S * 4);              // D = rowsum(dO * O), -LSE * log2(e)
  return bytes;
}

yr_status attn_bwd(const yr_rope_cfg* cfg, const void* q, const void* k, const void* v, const void* o,
                   const void* dout, const float* lse, void* dq, void* dk, void* dv, int32_t in_dtype,
                   int32_t out_dtype, int32_t B, int32_t Hq, int32_t Hkv, int32_t S, int32_t d,
                   const int64_t q_strides[3], const int64_t k_strides[3], const int64_t v_strides[3],
                   const int64_t o_strides[3], const int64_t do_strides[3], const int64_t dq_strides[3],
                   const int64_t dk_strides[3], const int64_t dv_strides[3], int32_t mask, int32_t sink,
                   int32_t window, float softmax_scale, void* workspace, size_t workspace_bytes, void* stream) {
  clear_error();
  if (!cfg) return fail(YR_ERR_INVALID_ARG, "attn_bwd: cfg is NULL");
  if (in_dtype != YR_F32 && in_dtype != YR_BF16) return fail(YR_ERR_INVALID_ARG, "attn_bwd: dtype %d", in_dtype);
  if (out_dtype != YR_F32 && out_dtype != YR_BF16) return fail(YR_ERR_INVALID_ARG, "attn_bwd: out dtype %d", out_dtype);
  if (B < 0 || Hq < 0 || Hkv < 0 || S < 0) return fail(YR_ERR_INVALID_ARG, "attn_bwd: negative shape");
  if (d != 64 && d != 128) return fail(YR_ERR_UNSUPPORTED, "attn_bwd: head dimension %d (64 or 128)", d);
  if (Hkv <= 0 || Hq <= 0 || Hq % Hkv != 0) return fail(YR_ERR_INVALID_ARG, "attn_bwd: Hq %% Hkv != 0");
  if (S % 128 != 0) return fail(YR_ERR_UNSUPPORTED, "attn_bwd: S=%d must be a multiple of 128", S);
  if (S > (1 << 24)) return fail(YR_ERR_INVALID_ARG, "attn_bwd: S above 2^24");
  if (mask < YR_MASK_CAUSAL || mask > YR_MASK_NONE) return fail(YR_ERR_INVALID_ARG, "attn_bwd: mask %d", mask);
  if (mask == YR_MASK_SINK_WINDOW && (sink < 0 || window < 1))
    return fail(YR_ERR_INVALID_ARG, "attn_bwd: sink must be >= 0 and window >= 1");
  const int64_t* strides[8] = {q_strides, k_strides, v_strides, o_strides, do_strides, dq_strides, dk_strides,
                               dv_strides};
  for (auto st : strides)
    if (!st) return fail(YR_ERR_INVALID_ARG, "attn_bwd: strides are NULL");
  RopeFreqs f;
  yr_status st = build_rope_freqs(cfg, d, &f);
  if (st != YR_OK) return st;
  if (B == 0 || S == 0) return YR_OK;
  if (!q || !k || !v || !o || !dout || !lse || !dq || !dk || !dv)
    return fail(YR_ERR_INVALID_ARG, "attn_bwd: a required pointer is NULL");
  const int elem = in_dtype == YR_BF16 ? 2 : 4, oelem = out_dtype == YR_BF16 ? 2 : 4;
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(o) || !aligned16(dout) || !aligned16(lse) ||
      !aligned16(dq) || !aligned16(dk) || !aligned16(dv) || !rows_aligned(q_strides, elem) ||
      !rows_aligned(k_strides, elem) || !rows_aligned(v_strides, elem) || !rows_aligned(o_strides, elem) ||
      !rows_aligned(do_strides, elem) || !rows_aligned(dq_strides, oelem) || !rows_aligned(dk_strides, oelem) ||
      !rows_aligned(dv_strides, oelem))
    return fail(YR_ERR_INVALID_ARG, "attn_bwd: pointers and strides must be 16-byte aligned");
  const size_t need = yr_bwd_workspace_bytes(cfg, in_dtype, B, Hq, Hkv, S, d);
  if (!workspace || workspace_bytes < need || !aligned16(workspace))
    return fail(YR_ERR_INVALID_ARG, "attn_bwd: workspace of %zu aligned bytes needed", need);

  const double ms = f.mscale;
  const double scale = softmax_scale > 0.f ? (double)softmax_scale : ms * ms / sqrt((double)d);
  cudaStream_t cs = as_stream(stream);
  char* ws = static_cast<char*>(workspace);
  size_t off = 0;
  BwdLaunch a;
  memset(&a, 0, sizeof(a));
  // rotated Q and K (and converted V, dO for float32 inputs): one launch
  RopeLaunch ra;
  memset(&ra, 0, sizeof(ra));
  ra.in_bf16 = in_dtype == YR_BF16; ra.out_bf16 = 1;
  ra.B = B; ra.d = d;
  auto prep = [&](const void* src, const int64_t* src_s, int H, bool rotate, const void** dst, int64_t* dst_s) {
    void* out = ws + off;
    const int64_t hs = (int64_t)S * d;
    off += align16((size_t)B * H * hs * 2);
    RopeSegment& sg = ra.seg[ra.n_seg++];
    sg.x = src; sg.y = out; sg.H = H; sg.S = S; sg.identity = rotate ? 0 : 1;
    dst_s[0] = (int64_t)H * hs; dst_s[1] = hs; dst_s[2] = d;
    for (int i = 0; i < 3; ++i) { sg.xs[i] = src_s[i]; sg.ys[i] = dst_s[i]; }
    *dst = out;
  };
  prep(q, q_strides, Hq, true, &a.q, a.qs);
  prep(k, k_strides, Hkv, true, &a.k, a.ks);
  if (in_dtype == YR_F32) {
    prep(v, v_strides, Hkv, false, &a.v, a.vs);
    prep(dout, do_strides, Hq, false, &a.dout, a.dos);
  } else {
    a.v = v; a.dout = dout;
    for (int i = 0; i < 3; ++i) { a.vs[i] = v_strides[i]; a.dos[i] = do_strides[i]; }
  }
  cudaError_t e = launch_rope(ra, f, cs);
  if (e != cudaSuccess) return cuda_fail(e, "attn_bwd rotation pass");
  float* dsum = reinterpret_cast<float*>(ws + off);
  off += align16((size_t)B * Hq * S * 4);
  float* lse2 = reinterpret_cast<float*>(ws + off);
  e = launch_dsum(dout, o, in_dtype == YR_BF16, dsum, lse, lse2, B, Hq, S, d, do_strides, o_strides, cs);
  if (e != cudaSuccess) return cuda_fail(e, "attn_bwd rowsum(dO * O)");
  a.lse2 = lse2; a.dsum = dsum;
  a.dq = dq; a.dk = dk; a.dv = dv; a.out_bf16 = out_dtype == YR_BF16;
  a.B = B; a.Hq = Hq; a.Hkv = Hkv; a.S = S; a.d = d;
  for (int i = 0; i < 3; ++i) { a.dqs[i] = dq_strides[i]; a.dks[i] = dk_strides[i]; a.dvs[i] = dv_strides[i]; }
  a.mask = mask; a.sink = sink; a.window = window;
  a.scale = (float)scale;
  a.f = f;
  e = launch_bwd(a, cs);
  return e == cudaSuccess ? YR_OK : cuda_fail(e, "attn_bwd launch");
}

int32_t yr_decode_auto_splits(int32_t B, int32_t Hkv, int32_t sink, int32_t window) {
  // Enough CTAs to cover two waves of the 148 SMs, without slices under 512
  // cache entries.
  const int64_t units = (int64_t)B * Hkv;
  const int64_t C = (int64_t)sink + window;
  if (units <= 0 || C <= 0) return 1;
  int64_t want = (2 * 148 + units - 1) / units;
  const int64_t cap = std::max<int64_t>(1, C / 512);
  return (int32_t)std::max<int64_t>(1, std::min<int64_t>({want, cap, 64}));
}

size_t yr_decode_workspace_bytes(int32_t B, int32_t Hq, int32_t Hkv, int32_t d, int32_t sink,
                                 int32_t window, int32_t num_splits) {
  if (B <= 0 || Hq <= 0 || d <= 0) return 0;
  const int splits = num_splits > 0 ? num_splits : yr_decode_auto_splits(B, Hkv, sink, window);
  if (splits <= 1) return 0;
  return (size_t)splits * B * Hq * (d + 2) * sizeof(float);
}


static yr_status decode_impl(const char* who, const yr_rope_cfg* cfg, const void* q, const void* k_cache,
                             const void* v_cache, int fp8, const float* k_scale, const float* v_scale,
                             const int32_t* n_valid, const int32_t* ring_start, int32_t B, int32_t Hq,
                             int32_t Hkv, int32_t d, int32_t sink, int32_t window, void* o, float* lse,
                             int32_t num_splits, void* workspace, size_t workspace_bytes, void* stream) {
  RopeFreqs f;
  yr_status st = decode_check_shape(who, cfg, B, Hq, Hkv, d, sink, window, num_splits, &f);
  if (st != YR_OK) return st;
  if (B == 0) return YR_OK;
  if (!q || !k_cache || !v_cache || !n_valid || !ring_start || !o)
    return fail(YR_ERR_INVALID_ARG, "a required pointer is NULL");
  if (fp8 && (!k_scale || !v_scale)) return fail(YR_ERR_INVALID_ARG, "%s: k_scale and v_scale are required", who);
  if (!aligned16(q) || !aligned16(k_cache) || !aligned16(v_cache) || !aligned16(o))
    return fail(YR_ERR_INVALID_ARG, "pointers must be 16-byte aligned");
  const int splits = num_splits > 0 ? num_splits : yr_decode_auto_splits(B, Hkv, sink, window);
  const size_t need = yr_decode_workspace_bytes(B, Hq, Hkv, d, sink, window, splits);
  if (need > 0 && (!workspace || workspace_bytes < need || !aligned16(workspace)))
    return fail(YR_ERR_INVALID_ARG, "workspace of %zu aligned bytes needed", need);
  const double ms = f.mscale;
  DecodeLaunch a;
  memset(&a, 0, sizeof(a));
  a.q = q; a.kc = k_cache; a.vc = v_cache; a.n_valid = n_valid; a.ring_start = ring_start;
  a.o = o; a.lse = lse; a.ws = splits > 1 ? static_cast<float*>(workspace) : nullptr;
  a.k_scale = k_scale; a.v_scale = v_scale; a.fp8 = fp8;
  a.B = B; a.Hq = Hq; a.Hkv = Hkv; a.d = d; a.sink = sink; a.window = window; a.splits = splits;
  a.scale_log2 = (float)(ms * ms / sqrt((double)d) * 1.4426950408889634073599246810019);
  cudaError_t e = launch_decode(a, f, as_stream(stream));
  return e == cudaSuccess ? YR_OK : cuda_fail(e, "decode launch");
}

yr_status attn_fwd_decode_sinkwindow(const yr_rope_cfg* cfg, const void* q, const void* k_cache,
                                     const void* v_cache, const int32_t* n_valid,
                                     const int32_t* ring_start, int32_t B, int32_t Hq,
                                     int32_t Hkv, int32_t d, int32_t sink, int32_t window,
                                     void* o, float* lse, int32_t num_splits, void* workspace,
                                     size_t workspace_bytes, void* stream) {
  clear_error();
  return decode_impl("attn_fwd_decode_sinkwindow", cfg, q, k_cache, v_cache, 0, nullptr, nullptr, n_valid,
                     ring_start, B, Hq, Hkv, d, sink, window, o, lse, num_splits, workspace, workspace_bytes,
                     stream);
}

yr_status attn_fwd_decode_sinkwindow_fp8(const yr_rope_cfg* cfg, const void* q, const void* k_cache,
                                         const void* v_cache, const float* k_scale, const float* v_scale,
                                         const int32_t* n_valid, const int32_t* ring_start, int32_t B,
                                         int32_t Hq, int32_t Hkv, int32_t d, int32_t sink, int32_t window,
                                         void* o, float* lse, int32_t num_splits, void* workspace,
                                         size_t workspace_bytes, void* stream) {
  clear_error();
  return decode_impl("attn_fwd_decode_sinkwindow_fp8", cfg, q, k_cache, v_cache, 1, k_scale, v_scale, n_valid,
                     ring_start, B, Hq, Hkv, d, sink, window, o, lse, num_splits, workspace, workspace_bytes,
                     stream);
}

yr_status yr_sync_status(void* stream) {
  clear_error();
  cudaError_t e = cudaStreamSynchronize(as_stream(stream));
  if (e != cudaSuccess) return cuda_fail(e, "stream synchronize");
  int* w = device_status_word();
  if (!w) return fail(YR_ERR_CUDA, "device status word unavailable");
  int h = 0;
  e = cudaMemcpy(&h, w, sizeof(int), cudaMemcpyDeviceToHost);
  if (e != cudaSuccess) return cuda_fail(e, "status read");
  if (h != 0) {
    const int zero = 0;
    cudaMemcpy(w, &zero, sizeof(int), cudaMemcpyHostToDevice);
    return fail(YR_ERR_TIMEOUT, "a device-side bounded wait gave up (code %d)", h);
  }
  return YR_OK;
}

}  // extern "C"
