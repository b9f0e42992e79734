/*
 * yarn_attn.h -- C ABI of the B300 (sm_103a) library for rotary position
 * embedding with context-extension rescaling fused into exact blockwise
 * softmax attention.
 *
 * Conventions shared by every entry point
 * ---------------------------------------
 * - Every function returns a yr_status.  Nothing throws across the ABI.  On a
 *   non-zero status, yr_last_error_message() returns a thread-local text.
 * - Arguments are checked on the host before any launch.  A bad argument
 *   returns YR_ERR_INVALID_ARG; a shape or type the kernels do not implement
 *   returns YR_ERR_UNSUPPORTED.  Neither launches anything and there is no
 *   fallback path.
 * - Device pointers are raw CUDA device addresses owned by the caller (for
 *   example from torch tensors).  The library allocates no device memory:
 *   where an entry point needs scratch, the caller passes a device workspace
 *   of at least the size the matching *_workspace_bytes function returns.
 * - Kernels run asynchronously on `stream` (a cudaStream_t passed as void*;
 *   NULL is the legacy default stream).  A launch failure returns
 *   YR_ERR_CUDA.  A device-side bounded wait that gives up records an error
 *   word that yr_sync_status() reports as YR_ERR_TIMEOUT.
 * - Tensor strides are in elements, for the (batch, head, position) axes;
 *   the last (head-dim) axis must be contiguous.  Device pointers and row
 *   strides must be 16-byte aligned.
 * - Positions must be below 2^24 (they are exact in float32).
 *
 * Notation (the pages'): d head dimension, theta_base the RoPE base b,
 * L_train / L_target the trained and desired context lengths, s the scale
 * factor L_target / L_train, sink the number of pinned first tokens and
 * window the sliding-window length.
 */
#ifndef YARN_ATTN_H
#define YARN_ATTN_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  YR_OK = 0,
  YR_ERR_INVALID_ARG = 1,
  YR_ERR_UNSUPPORTED = 2,
  YR_ERR_CUDA = 3,
  YR_ERR_TIMEOUT = 4
} yr_status;

/* Frequency rescaling kinds.
 * NONE : the rotation is the identity (inputs arrive already rotated).
 * PLAIN: theta_i = b^(-2i/d) ("Context Window Scaling: YaRN, LongRoPE, and
 *        RingAttention Architectures", Section 2, Formal RoPE Mechanics).
 * PI   : Position Interpolation, theta_i / s (same page, Section 2, The
 *        Failure of Naive PI; "Context Length Extension", Position
 *        Interpolation).
 * NTK  : NTK-aware base b' = b * s^(d/(d-2)), the base that keeps the
 *        highest frequency and interpolates the lowest one by s ("Context
 *        Length Extension", NTK-Aware Scaling; the page states the effect and
 *        omits the formula, this is the reading adopted).
 * YARN : NTK-by-parts ramp theta'_i = (1-g) theta_i / s + g theta_i with
 *        g = clamp((r - alpha) / (beta - alpha), 0, 1), r = L_train / lambda_i,
 *        lambda_i = 2 pi b^(2i/d), plus the attention temperature
 *        mscale = 0.1 ln s + 1 for s > 1 ("Context Window Scaling ...",
 *        Section 3; "Long-context extension: stretching attention past its
 *        training window", NTK-by-parts).
 * PERDIM: a caller-given factor per dimension, theta'_i = theta_i / lambda_i
 *        (the non-uniform scale vector of LongRoPE, "Context Window Scaling
 *        ...", Section 4 and FAQ 4; the search that finds the vector is not
 *        part of this library).  mscale is 1 unless overridden. */
typedef enum {
  YR_ROPE_NONE = 0,
  YR_ROPE_PLAIN = 1,
  YR_ROPE_PI = 2,
  YR_ROPE_NTK = 3,
  YR_ROPE_YARN = 4,
  YR_ROPE_PERDIM = 5
} yr_rope_kind;

typedef enum { YR_F32 = 0, YR_BF16 = 1 } yr_dtype;

/* Visibility of key position n to query position m.
 * CAUSAL     : n <= m.
 * SINK_WINDOW: n <= m and (n < sink or m - n < window) -- the first `sink`
 *              tokens plus the last `window` tokens up to m ("Context Length
 *              Extension", Sliding Window + Attention Sinks).
 * NONE       : every key. */
typedef enum { YR_MASK_CAUSAL = 0, YR_MASK_SINK_WINDOW = 1, YR_MASK_NONE = 2 } yr_mask;

/* The pages' statement of the problem, as one plain struct.
 * kind            yr_rope_kind.
 * head_dim        d; even.  The attention and decode kernels take 64 or 128.
 * theta_base      b > 1.
 * L_train         trained context length (YaRN needs it; > 0).
 * L_target        desired context length; used when s <= 0.
 * s               scale factor; <= 0 means L_target / L_train.
 * ramp_alpha/beta YaRN ramp bounds on r (defaults 1 and 32 when both are 0).
 * mscale_override > 0 replaces the temperature factor.
 * dim_scale       PERDIM only: host array of d/2 finite factors > 0, read
 *                 during the call (the caller keeps ownership); ignored by
 *                 the other kinds. */
typedef struct {
  int32_t kind;
  int32_t head_dim;
  double theta_base;
  int32_t L_train;
  int32_t L_target;
  double s;
  double ramp_alpha;
  double ramp_beta;
  double mscale_override;
  const double* dim_scale;
} yr_rope_cfg;

/* Rescaled frequencies, host only, float64 (no device work).
 * inv_freq : host array of d/2 doubles receiving theta'_i (radians per
 *            position).  Required.
 * cls      : host array of d/2 int8 receiving the regime of each dimension,
 *            0 interpolated (r < alpha), 1 ramp, 2 kept (r > beta), from
 *            r = L_train / lambda_i of the unscaled frequency; all 2 when
 *            L_train <= 0.  Nullable.
 * mscale   : receives the temperature factor (1 unless YaRN with s > 1, or
 *            the override).  Nullable.
 * Source: "Context Window Scaling ...", Sections 2 and 3; "Context Length
 * Extension", Position Interpolation, NTK-Aware Scaling, YaRN. */
yr_status yarn_inv_freq(const yr_rope_cfg* cfg, double* inv_freq, int8_t* cls, double* mscale);

/* Standalone rotation of a [B, H, S, d] tensor (float32 or bfloat16):
 * each pair (x_i, x_{i+d/2}) at position m is rotated by m * theta'_i,
 *   y_i = x_i cos - x_{i+d/2} sin,   y_{i+d/2} = x_i sin + x_{i+d/2} cos
 * ("Context Window Scaling ...", Section 2), and multiplied by mscale when
 * apply_mscale is non-zero.
 * x, y      : device; y may equal x (in place) when the strides match.
 * x_strides, y_strides : host arrays of 3 int64 (batch, head, position).
 * pos0      : position of row s is pos0 + s when `positions` is NULL.
 * positions : device int32 [S] of explicit positions, or NULL.
 * Memory-bound: one read and one write of x. */
yr_status rope_apply(const yr_rope_cfg* cfg, const void* x, void* y, int32_t dtype,
                     int32_t B, int32_t H, int32_t S, int32_t d,
                     const int64_t x_strides[3], const int64_t y_strides[3],
                     int32_t pos0, const int32_t* positions, int32_t apply_mscale,
                     void* stream);

/* Bytes of device workspace attn_fwd_prefill needs for these shapes
 * (0 when none is needed). */
size_t yr_prefill_workspace_bytes(const yr_rope_cfg* cfg, int32_t in_dtype, int32_t B,
                                  int32_t Hq, int32_t Hkv, int32_t S, int32_t d);

/* Exact softmax attention with the rotation applied to Q and K:
 *   O_m = sum_n softmax_n(scale * <R_m q_m, R_n k_n>) v_n over visible n,
 * scale = mscale^2 / sqrt(d) unless softmax_scale > 0 ("Context Window
 * Scaling ...", Section 1 for the attention, Section 3 for the temperature
 * 1/t = mscale^2).  Keys are folded in 128-key blocks with an online-softmax
 * merge ("Context Length Extension", Ring Attention: partial results are
 * combined with online softmax).  With ring_blocks = N > 1 the sequence is
 * split into N equal logical blocks and query block I folds key blocks in
 * ring order I, I-1, ..., skipping future blocks under a causal or
 * sink-window mask ("Context Window Scaling ...", Section 5 and FAQ 2);
 * ring_blocks = 1 is natural order.  The result is the same up to rounding.
 * q   : device [B, Hq, S, d], in_dtype (F32 or BF16).
 * k,v : device [B, Hkv, S, d], in_dtype; Hq % Hkv == 0, query head h reads
 *       key/value head h / (Hq / Hkv).
 * o   : device [B, Hq, S, d], in_dtype.
 * lse : device float32 [B, Hq, S] (contiguous) receiving the natural-log
 *       sum of exponentials of each row's scaled logits, or NULL.
 * *_strides : host int64[3] (batch, head, position), in elements.
 * d ∈ {64, 128}.  S >= 1 (a ragged last tile is masked).
 * workspace : device scratch of yr_prefill_workspace_bytes(); holds the
 *       rotated bfloat16 copies of Q and K (when kind is not NONE, or the
 *       inputs are float32) and the bfloat16 copy of V (float32 inputs
 *       only); kind NONE with bfloat16 inputs needs none.
 * The matrix products run on bfloat16 operands with float32 accumulation. */
yr_status attn_fwd_prefill(const yr_rope_cfg* cfg, const void* q, const void* k, const void* v,
                           void* o, float* lse, int32_t in_dtype,
                           int32_t B, int32_t Hq, int32_t Hkv, int32_t S, int32_t d,
                           const int64_t q_strides[3], const int64_t k_strides[3],
                           const int64_t v_strides[3], const int64_t o_strides[3],
                           int32_t mask, int32_t sink, int32_t window, int32_t ring_blocks,
                           float softmax_scale, void* workspace, size_t workspace_bytes,
                           void* stream);

/* Bytes of device workspace attn_fwd_prefill_kv_block needs (0 when none). */
size_t yr_prefill_kv_block_workspace_bytes(const yr_rope_cfg* cfg, int32_t in_dtype, int32_t B,
                                           int32_t Hq, int32_t Hkv, int32_t Sq, int32_t Skv, int32_t d);

/* One query block against one key/value block: the computation a device of
 * a ring does for each KV block it holds ("Context Window Scaling ...",
 * Section 5: GPU i computes attention of its query block Q_i with the
 * resident block KV_j; "Context Length Extension", Ring Attention: each GPU
 * computes partial attention with its local keys).  Query row r sits at
 * position q_pos0 + r and key n at k_pos0 + n; positions drive both the
 * rotation and the mask (a block entirely in the future gives o = 0 and
 * lse = -inf for every row, which attn_merge_partial treats as empty).
 * q   : device [B, Hq, Sq, d] in_dtype;  k, v : device [B, Hkv, Skv, d].
 * o   : device [B, Hq, Sq, d] of out_dtype (YR_F32 keeps the partial exact
 *       for merging; YR_BF16 for a single block).
 * lse : device float32 [B, Hq, Sq] contiguous, or NULL (a partial to be
 *       merged needs it).
 * Other arguments as attn_fwd_prefill; ring order is the caller's (one KV
 * block per call).  Skv = 0 gives o = 0 and lse = -inf. */
yr_status attn_fwd_prefill_kv_block(const yr_rope_cfg* cfg, const void* q, const void* k, const void* v,
                                    void* o, float* lse, int32_t in_dtype, int32_t out_dtype, int32_t B,
                                    int32_t Hq, int32_t Hkv, int32_t Sq, int32_t Skv, int32_t d,
                                    int32_t q_pos0, int32_t k_pos0, const int64_t q_strides[3],
                                    const int64_t k_strides[3], const int64_t v_strides[3],
                                    const int64_t o_strides[3], int32_t mask, int32_t sink, int32_t window,
                                    float softmax_scale, void* workspace, size_t workspace_bytes,
                                    void* stream);

/* Exact merge of one attention partial into an accumulator, both over
 * disjoint key sets and normalised over their own keys:
 *   L = ln(e^La + e^Lp),  O = e^(La - L) Oa + e^(Lp - L) Op
 * ("Context Length Extension", Ring Attention: partial results are combined
 * using online softmax).  A side whose lse is -inf is empty: its O is
 * loaded but dropped, never multiplied, so a fresh accumulator needs only
 * lse_acc = -inf (its O buffer must exist; its contents do not matter).
 * o_acc    : device float32 [B, H, S, d] (strides acc_strides), updated.
 * lse_acc  : device float32 [B, H, S] contiguous, updated.
 * o_part, lse_part : the partial, same shapes (o strides part_strides).
 * o_final  : optional device [B, H, S, d] of final_dtype (F32 or BF16)
 *            receiving the merged O as well (NULL: none), strides
 *            final_strides (8-byte aligned for bf16).
 * d a multiple of 4; 16-byte-aligned pointers and rows.  Memory-bound. */
yr_status attn_merge_partial(float* o_acc, float* lse_acc, const float* o_part, const float* lse_part,
                             void* o_final, int32_t final_dtype, int32_t B, int32_t H, int32_t S, int32_t d,
                             const int64_t acc_strides[3], const int64_t part_strides[3],
                             const int64_t final_strides[3], void* stream);

/* Bytes of device workspace attn_bwd needs. */
size_t yr_bwd_workspace_bytes(const yr_rope_cfg* cfg, int32_t in_dtype, int32_t B, int32_t Hq, int32_t Hkv,
                              int32_t S, int32_t d);

/* Gradients of attn_fwd_prefill (natural order, positions 0 .. S - 1) with
 * respect to the unrotated q, k and v, for the fine-tuning that the context
 * extension methods rely on ("Context Window Scaling ...", Section 3:
 * YaRN's brief fine-tune; "Context Length Extension", Position
 * Interpolation: ~1000 fine-tuning steps).  With P the softmax of
 * scale * <R_m q_m, R_n k_n>, dO the gradient of the output and
 * D_m = sum_c dO[m, c] O[m, c]:
 *   dv = P^T dO,  dS = P * (dO V^T - D),
 *   dq = scale R_m^T (dS Kr),  dk = scale R_n^T (dS^T Qr).
 * q, o, dout : device [B, Hq, S, d] in_dtype;  k, v : [B, Hkv, S, d].
 * lse  : device float32 [B, Hq, S] contiguous, the forward's row log-sum-exp.
 * dq   : device [B, Hq, S, d];  dk, dv : [B, Hkv, S, d], out_dtype (F32 or
 *        BF16).  GQA: dk and dv sum over the query heads of their group.
 * Supported: d in {64, 128}, S a multiple of 128.  mask, sink, window and
 * softmax_scale as in attn_fwd_prefill.  The products run on bfloat16
 * operands (the rotated q and k, v, dO, P and dS) with float32 accumulation.
 * workspace: device scratch of yr_bwd_workspace_bytes(). */
yr_status attn_bwd(const yr_rope_cfg* cfg, const void* q, const void* k, const void* v, const void* o,
                   const void* dout, const float* lse, void* dq, void* dk, void* dv, int32_t in_dtype,
                   int32_t out_dtype, int32_t B, int32_t Hq, int32_t Hkv, int32_t S, int32_t d,
                   const int64_t q_strides[3], const int64_t k_strides[3], const int64_t v_strides[3],
                   const int64_t o_strides[3], const int64_t do_strides[3], const int64_t dq_strides[3],
                   const int64_t dk_strides[3], const int64_t dv_strides[3], int32_t mask, int32_t sink,
                   int32_t window, float softmax_scale, void* workspace, size_t workspace_bytes, void* stream);

/* Split count the decode entry point uses when num_splits <= 0. */
int32_t yr_decode_auto_splits(int32_t B, int32_t Hkv, int32_t sink, int32_t window);

/* Bytes of device workspace attn_fwd_decode_sinkwindow needs (0 when the
 * chosen split count is 1). */
size_t yr_decode_workspace_bytes(int32_t B, int32_t Hq, int32_t Hkv, int32_t d, int32_t sink,
                                 int32_t window, int32_t num_splits);

/* One new query token per sequence against a cache of `sink` pinned tokens
 * plus a `window`-slot ring buffer ("Context Length Extension", Sliding
 * Window + Attention Sinks: s + w entries regardless of length; "Long-Context
 * Scaling", Production defaults: 4 pinned sinks).
 * q        : device bf16 [B, Hq, d], already written at the newest position.
 * k_cache, v_cache : device bf16 [B, Hkv, sink + window, d]; keys stored
 *            unrotated.  Slots 0..sink-1 hold the sinks; logical window entry
 *            t (0 = oldest) lives in slot sink + (ring_start + t) mod window.
 * n_valid  : device int32 [B], number of valid logical entries (<= sink +
 *            window; the query is entry n_valid - 1).  0 gives o = 0 and
 *            lse = -inf.
 * ring_start : device int32 [B], in [0, window).
 * Positions are logical cache indices: entry j at j, the query at
 * n_valid - 1 (the cache is used without changing RoPE).
 * o        : device bf16 [B, Hq, d].  lse: device float32 [B, Hq] or NULL.
 * num_splits : <= 0 picks yr_decode_auto_splits(); otherwise the cache is cut
 *            into that many slices per (sequence, kv head) whose partial
 *            softmax states are merged exactly in a second kernel.
 * workspace : device scratch of yr_decode_workspace_bytes() (may be NULL
 *            when that is 0).
 * Memory-bound: one read of each valid cache entry. */
yr_status attn_fwd_decode_sinkwindow(const yr_rope_cfg* cfg, const void* q, const void* k_cache,
                                     const void* v_cache, const int32_t* n_valid,
                                     const int32_t* ring_start, int32_t B, int32_t Hq,
                                     int32_t Hkv, int32_t d, int32_t sink, int32_t window,
                                     void* o, float* lse, int32_t num_splits, void* workspace,
                                     size_t workspace_bytes, void* stream);

/* attn_fwd_decode_sinkwindow over an FP8 cache: k_cache and v_cache hold
 * OCP FP8 E4M3 values (1 byte each, [B, Hkv, sink + window, d]) and the
 * dequantised entry is the stored value times the float32 scale of its
 * (sequence, KV head): k_scale[b * Hkv + h] for keys, v_scale[...] for
 * values (device arrays of B * Hkv).  Quantising the cache to FP8 halves the
 * bytes the memory-bound decode reads ("Context Window Scaling ...", FAQ 3:
 * KV-cache quantisation to FP8 or INT4).  Keys are stored unrotated; the
 * rotation, mask, positions, splits, workspace and outputs are those of
 * attn_fwd_decode_sinkwindow (q and o stay bfloat16). */
yr_status attn_fwd_decode_sinkwindow_fp8(const yr_rope_cfg* cfg, const void* q, const void* k_cache,
                                         const void* v_cache, const float* k_scale, const float* v_scale,
                                         const int32_t* n_valid, const int32_t* ring_start, int32_t B,
                                         int32_t Hq, int32_t Hkv, int32_t d, int32_t sink, int32_t window,
                                         void* o, float* lse, int32_t num_splits, void* workspace,
                                         size_t workspace_bytes, void* stream);

/* attn_fwd_decode_sinkwindow without a workspace argument, for callers that
 * cannot allocate device memory when they call (for example an engine's
 * per-step hook that must not allocate, or a process whose device memory is
 * all reserved by another allocator) or have no scratch buffer to pass.  The
 * pages have no counterpart: this is an interface convenience only.
 * Arguments, layouts and results are those of attn_fwd_decode_sinkwindow.
 * The split partial states go to one fixed 4 MiB array of device memory that
 * the library holds on every GPU that loads it, until the process exits; the
 * call itself allocates nothing.  Its first call on a device looks up that
 * array's device address (cudaGetSymbolAddress, with the device current), so
 * make that first call before any stream capture.  Every call on a device
 * shares the array and it keeps the last call's contents (each call writes
 * every partial state before reading it); calls that overlap on the GPU
 * race.  A split count whose scratch would exceed 4 MiB
 * (num_splits * B * Hq * (d + 2) * 4 bytes) returns YR_ERR_INVALID_ARG with
 * a message; a split count of 1 needs no scratch. */
yr_status attn_fwd_decode_sinkwindow_noalloc(const yr_rope_cfg* cfg, const void* q,
                                             const void* k_cache, const void* v_cache,
                                             const int32_t* n_valid, const int32_t* ring_start,
                                             int32_t B, int32_t Hq, int32_t Hkv, int32_t d,
                                             int32_t sink, int32_t window, void* o, float* lse,
                                             int32_t num_splits, void* stream);

/* Synchronises `stream`, then reads and clears the device error word that
 * bounded waits set; returns YR_ERR_TIMEOUT if one gave up, YR_ERR_CUDA on a
 * CUDA error, YR_OK otherwise. */
yr_status yr_sync_status(void* stream);

/* Test hook for the failure path: host-controlled fault injection (the pages
 * have no counterpart; not for production use).  While set, the decode and
 * prefill kernels bound their first-level waits by wait_limit_cycles SM
 * cycles (0: the default, 4e9, about 2 s at the maximum clock) and, when
 * skip_unit >= 0, their load producers never issue the copies of that load
 * unit (decode: cache chunk skip_unit of each slice; prefill: K/V load unit
 * skip_unit of each CTA, unit 0 being the first K tile), so the wait on it
 * runs out.  A kernel whose wait runs out records the code that
 * yr_sync_status() reports as YR_ERR_TIMEOUT, lets the copies and products
 * it issued finish, frees its tensor memory and returns; the outputs of that
 * call are undefined and the device stays usable.  The setting is process-wide and stays
 * until changed: yr_debug_inject_wait_fault(0, -1) turns it off.
 * wait_limit_cycles < 0 or skip_unit < -1 returns YR_ERR_INVALID_ARG. */
yr_status yr_debug_inject_wait_fault(int64_t wait_limit_cycles, int32_t skip_unit);

/* Number of kernels the library has launched in this process so far, over
 * every entry point and device (each successful launch counts once).  Host
 * only; for counting the launches inside a timed region.  Not part of the
 * method: the pages have no counterpart. */
uint64_t yr_kernel_launch_count(void);

/* Thread-local text of the last error (empty when none). */
const char* yr_last_error_message(void);

/* Library version string. */
const char* yr_version(void);

#ifdef __cplusplus
}
#endif

#endif /* YARN_ATTN_H */
