// Private declarations shared by the host entry points and the kernel files.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "yarn_attn.h"

namespace yr {

constexpr int kMaxHalf = 128;  // d/2 upper bound for rope_apply (d <= 256)

// Per-dimension rotation rate in turns per position, theta'_i / (2 pi), split
// into a float hi part and a float lo remainder so that the device can form
// the fractional turn m * f exactly enough for float32 outputs (positions are
// exact integers below 2^24).
struct RopeFreqs {
  float2 f[kMaxHalf];  // x = hi, y = lo
  float mscale;        // temperature factor (1 when not YaRN)
  int32_t half;        // d / 2
  int32_t identity;    // 1 when every frequency is zero (kind NONE)
};

// Host: validate cfg for head dimension d and fill the float64 frequencies.
yr_status compute_inv_freq(const yr_rope_cfg* cfg, int d, double* theta, int8_t* cls,
                           double* mscale);
// Host: the device table built from compute_inv_freq.
yr_status build_rope_freqs(const yr_rope_cfg* cfg, int d, RopeFreqs* out);

// Host: the shape and configuration checks shared by the decode entry points;
// fills the frequency table on success.
yr_status decode_check_shape(const char* who, const yr_rope_cfg* cfg, int32_t B, int32_t Hq, int32_t Hkv,
                             int32_t d, int32_t sink, int32_t window, int32_t num_splits, RopeFreqs* f);

// Error text helpers (thread-local message).
yr_status fail(yr_status st, const char* fmt, ...);
void clear_error();
yr_status cuda_fail(cudaError_t e, const char* what);

// Address of the device status word (per device), set by bounded waits.
int* device_status_word();

// After a kernel launch: the launch status (cudaGetLastError), and on
// success `n` more launches on the library's launch counter.
cudaError_t launched(int n);

// Host-controlled fault injection for the failure-path tests, off unless
// yr_debug_inject_wait_fault() set it: the bound of the decode and prefill
// kernels' first-level waits, and the load unit (a chunk of the decode cache,
// a K/V unit of the attention) whose copies their producer never issues, so
// that the wait on it runs out.  Off: 4e9 cycles and -1.
struct FaultInjection {
  long long wait_limit;
  int skip_unit;
};
FaultInjection fault_injection();

// Number of SMs of the current device.
int sm_count();
// TMA map of a [B, H, S, D] bfloat16 tensor (element strides b, h, s): 4-D,
// 64 x 128 boxes, 128-byte swizzle, zero fill outside the tensor.
bool make_map(CUtensorMap* map, const void* base, int B, int H, int S, int D, const int64_t st[3]);

// ---- launches (kernel files) ----------------------------------------------
// One tensor of a rotation pass: [B, H, S, d] rows at positions pos0 + s
// (or the launch's explicit positions), written to y.
struct RopeSegment {
  const void* x;
  void* y;
  int H, S;
  int64_t xs[3], ys[3];  // element strides (batch, head, position)
  int pos0;
  int identity;  // 1: no rotation (a conversion, and mscale when asked)
  int64_t tile0;  // set by the launcher: first tile of this segment
};
constexpr int kMaxRopeSegments = 4;
struct RopeLaunch {
  RopeSegment seg[kMaxRopeSegments];
  int n_seg;
  int in_bf16, out_bf16;  // float32 -> float32 uses the precise angle path
  int B, d;
  const int32_t* positions;  // explicit positions of row s (one segment), or NULL
  int apply_mscale;
  // set by the launcher
  int rows_per_tile;
  int64_t n_tiles;
  int* status;
};
cudaError_t launch_rope(const RopeLaunch& a, const RopeFreqs& f, cudaStream_t st);

struct DecodeLaunch {
  const void* q;
  const void* kc;
  const void* vc;
  const int32_t* n_valid;
  const int32_t* ring_start;
  void* o;
  float* lse;
  float* ws;  // split partials (NULL when splits == 1)
  const float* k_scale;  // FP8 caches: per (sequence, KV head) scales
  const float* v_scale;
  int fp8;               // 1: caches are FP8 E4M3, 0: bfloat16
  int B, Hq, Hkv, d, sink, window, splits;
  float scale_log2;
  int* status;  // device status word (set by the launcher)
  long long wait_limit;  // first-level wait bound in cycles (set by the launcher)
  int skip_unit;         // fault injection: cache chunk never loaded (-1: none)
};
cudaError_t launch_decode(const DecodeLaunch& a, const RopeFreqs& f, cudaStream_t st);

struct PrefillLaunch {
  const void* q;  // bf16, rotated
  const void* k;  // bf16 rotated
  const void* v;  // bf16
  void* o;
  float* lse;
  int out_bf16;
  int B, Hq, Hkv, d;
  int Sq, Skv;         // query rows and keys
  int q_pos0, k_pos0;  // positions of query row 0 and key 0 (mask)
  int64_t qs[3], ks[3], vs[3], os[3];
  int mask, sink, window, ring_blocks;
  float scale_log2;
};
cudaError_t launch_prefill(const PrefillLaunch& a, cudaStream_t st);

// Attention backward (attn_bwd): q, k rotated bf16 copies, v and dout bf16.
struct BwdLaunch {
  const void* q;
  const void* k;
  const void* v;
  const void* dout;
  const float* lse2;  // -LSE * log2(e)
  const float* dsum;
  void* dq;
  void* dk;
  void* dv;
  int out_bf16;
  int B, Hq, Hkv, S, d;
  int64_t qs[3], ks[3], vs[3], dos[3], dqs[3], dks[3], dvs[3];
  int mask, sink, window;
  float scale;
  RopeFreqs f;
};
cudaError_t launch_bwd(const BwdLaunch& a, cudaStream_t st);
// D = rowsum(dO * O) of [B, H, S, d] tensors (bf16 when bf16 != 0, else f32),
// and lse2 = -lse * log2(e) for the same rows.
cudaError_t launch_dsum(const void* dout, const void* o, int bf16, float* dsum, const float* lse, float* lse2, int B,
                        int H, int S, int d, const int64_t ds[3], const int64_t os[3], cudaStream_t st);

// Exact merge of an attention partial into an accumulator (attn_merge_partial).
struct MergeLaunch {
  float* o_acc;
  float* lse_acc;
  const float* o_part;
  const float* lse_part;
  void* o_final;  // optional output of the merged result (NULL: none)
  int final_bf16;
  int B, H, S, d;
  int64_t as[3], ps[3], fs[3];
};
cudaError_t launch_merge(const MergeLaunch& a, cudaStream_t st);
// o = 0, lse = -inf for every row (attention over an empty key set).
cudaError_t launch_fill_empty(void* o, int out_bf16, float* lse, int B, int H, int S, int d, const int64_t os[3],
                              cudaStream_t st);

}  // namespace yr
