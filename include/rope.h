/*
 * rope.h -- C ABI of librope: rotary position embedding (RoPE) on the GPU.
 *
 * What the library computes.  For a token at table row r and pair index i,
 * the pair (x1, x2) of a query or key head row becomes
 *     (x1 cos t - x2 sin t,  x1 sin t + x2 cos t),   t = angle(r, i)
 * ("Rotary Embedding (RoPE) Kernel Optimization", Overview).  Queries and
 * keys are rotated in one launch ("How Unsloth Optimizes RoPE Embedding
 * Computations in Triton Kernels", Triton Kernel Architecture for RoPE:
 * the fused Q+K kernel), and the backward pass is the same rotation by -t
 * (same page, Frequently Asked Questions: gradients use the same kernel
 * with the backward flag).
 *
 * Conventions shared by every entry point:
 *   - Pointers marked "device" must point to memory of the current CUDA
 *     device.  The caller owns every buffer; the library allocates nothing
 *     and never synchronises the stream, except in rope_check_errors.
 *   - `stream` is a cudaStream_t passed as void*; NULL is the default stream.
 *     Work is enqueued asynchronously on that stream.
 *   - Tensors are dense and contiguous.  seq_before_head = 0: [B, H, S, D]
 *     (Unsloth page, Usage Examples; "rotary-embedding-torch", Input Tensor
 *     Shapes); seq_before_head = 1: [B, S, H, D] ("rotary-embedding-torch",
 *     RotaryEmbedding / Key Parameters: seq_before_head_dim).
 *   - Element types: ROPE_F32, ROPE_BF16, ROPE_F16.  Arithmetic is fp32;
 *     each output element is rounded once to the element type.
 *   - Pair layouts ("Rotary Embedding (RoPE) Kernel Optimization", Core
 *     Technique / Paired Element Layout): ROPE_SPLIT_HALF pairs
 *     (x[i], x[i + rotary_dim/2]); ROPE_INTERLEAVED pairs (x[2i], x[2i+1]).
 *   - Partial rotation ("rotary-embedding-torch", RotaryEmbedding / Key
 *     Parameters: dim is the size of the rotated part): only the first
 *     rotary_dim features of each head row are rotated; features
 *     [rotary_dim, D) are neither read nor written.
 *   - Errors detected on the host are returned before anything is enqueued;
 *     nothing is modified then.
 */
#ifndef ROPE_H
#define ROPE_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    ROPE_OK = 0,
    ROPE_ERR_INVALID_ARG = 1,      /* bad size, null pointer, overlap, ...       */
    ROPE_ERR_UNSUPPORTED = 2,      /* dtype or layout value outside the enums    */
    ROPE_ERR_CUDA = 3,             /* a CUDA call failed (launch, sync, ...)     */
    ROPE_ERR_POS_OUT_OF_RANGE = 4, /* a position index was outside the table     */
    ROPE_ERR_KERNEL_TIMEOUT = 5    /* a bounded wait inside a kernel expired      */
} rope_status;

typedef enum { ROPE_SPLIT_HALF = 0, ROPE_INTERLEAVED = 1 } rope_layout;
typedef enum { ROPE_F32 = 0, ROPE_BF16 = 1, ROPE_F16 = 2 } rope_dtype;
/* attention masks ("rotary-embedding-torch", flash_attn_with_rotary / Input
 * Tensor Shapes: attn_mask (batch, seq_len_k) or (batch, seq_len_q, seq_len_k)) */
typedef enum {
    ROPE_MASK_NONE = 0,
    ROPE_MASK_KEYS = 1,        /* uint8 [B, Sk]: one entry per key (key padding) */
    ROPE_MASK_QUERY_KEYS = 2   /* uint8 [B, Sq, Sk]: one entry per query and key */
} rope_mask_kind;
/* frequency modes ("rotary-embedding-torch", RotaryEmbedding: freqs_for) */
typedef enum { ROPE_FREQ_LANG = 0, ROPE_FREQ_PIXEL = 1, ROPE_FREQ_CONSTANT = 2 } rope_freq_mode;

/*
 * rope_tables_build -- fill the cos/sin table.
 *
 * Source: "rotary-embedding-torch", RotaryEmbedding / Key Parameters (theta
 * is the frequency base, default 10000; interpolate_factor scales sequence
 * positions, default 1.0); "Rotary Embedding (RoPE) Kernel Optimization",
 * Common Pitfalls (cos/sin are [seq_len, D/2] and broadcast over batch and
 * heads).  The pages do not print the frequency formula; the library uses
 * the standard one: for row m and pair i (0 <= i < rotary_dim/2)
 *     angle = (m / interpolate_factor) * theta^(-2i / rotary_dim),
 * evaluated in fp64, and stores cos(angle), sin(angle) rounded to fp32.
 *
 * cos_out, sin_out: device, caller-owned, float[max_pos * rotary_dim/2]
 *   each, row-major [max_pos, rotary_dim/2].
 * Errors: ROPE_ERR_INVALID_ARG if theta <= 0, interpolate_factor <= 0 (or
 *   either is not finite), rotary_dim < 2 or odd, max_pos < 0, a null
 *   output with max_pos > 0, or overlapping outputs.  max_pos = 0 is a
 *   no-op.  ROPE_ERR_CUDA if the launch fails.
 */
rope_status rope_tables_build(double theta, int32_t rotary_dim, int64_t max_pos,
                              double interpolate_factor, float *cos_out, float *sin_out,
                              void *stream);

/*
 * rope_tables_build_ex -- the cos/sin table of a frequency mode, at given
 * row positions, optionally with the XPOS scale folded in.
 *
 * Source: "rotary-embedding-torch", RotaryEmbedding / Key Parameters names
 * freqs_for = 'lang' (default) | 'pixel' | 'constant' and use_xpos (length
 * extrapolation) without formulas; the published definitions are used.  For
 * row m and pair i (0 <= i < h = rotary_dim/2):
 *     p     = pos_offset + m / pos_divisor
 *     w_i   = theta^(-2i / rotary_dim)                     ROPE_FREQ_LANG
 *           = pi * (1 + i * (max_freq/2 - 1) / (h - 1))    ROPE_FREQ_PIXEL
 *             (pi when h = 1; Perceiver's Fourier features, positions
 *             usually in [-1, 1]: pos_offset = -1, pos_divisor = (rows-1)/2)
 *           = 1                                            ROPE_FREQ_CONSTANT
 *     s     = 1 when xpos_sign = 0, else (XPOS, Sun et al. 2022)
 *             zeta_i^(xpos_sign * (p - xpos_center) / xpos_scale_base),
 *             zeta_i = (2i/rotary_dim + xpos_gamma) / (1 + xpos_gamma)
 *     cos_out[m][i] = s * cos(p * w_i), sin_out[m][i] = s * sin(p * w_i),
 * all in fp64, each stored rounded once to fp32.  XPOS scales the query by
 * zeta^(+n/B) and the key by zeta^(-n/B): build one table with xpos_sign =
 * +1 for Q and one with -1 for K and rotate each with rope_apply_q (the
 * backward flag, which negates the sine, then gives the XPOS gradient too).
 * ROPE_FREQ_LANG with pos_offset = 0 and pos_divisor = interpolate_factor
 * reproduces rope_tables_build bit for bit.
 *
 * cos_out, sin_out: device, caller-owned, float[rows * rotary_dim/2] each.
 * Errors: ROPE_ERR_UNSUPPORTED for an unknown mode; ROPE_ERR_INVALID_ARG if
 *   rotary_dim < 2 or odd, rows < 0, theta <= 0 (lang), max_freq <= 0
 *   (pixel), pos_divisor <= 0, a non-finite pos_offset / pos_divisor,
 *   xpos_sign outside {-1, 0, 1}, and with xpos_sign != 0 a scale base or
 *   gamma <= 0 or a non-finite centre; null or overlapping outputs with
 *   rows > 0.  rows = 0 is a no-op.  ROPE_ERR_CUDA if the launch fails.
 */
rope_status rope_tables_build_ex(int32_t freq_mode, double theta, double max_freq,
                                 int32_t rotary_dim, int64_t rows, double pos_offset,
                                 double pos_divisor, int32_t xpos_sign, double xpos_scale_base,
                                 double xpos_gamma, double xpos_center, float *cos_out,
                                 float *sin_out, void *stream);

/*
 * rope_apply_qk -- rotate Q and K in place, in one launch.
 *
 * Source: Unsloth page, Triton Kernel Architecture for RoPE (Q and K in one
 * kernel) and Usage Examples (fast_rope_embedding(Q, K, cos, sin,
 * position_ids)); "rotary-embedding-torch", flash_attn_with_rotary / Key
 * Features (heads_q != heads_kv for GQA/MQA).
 *
 * q: device, [B, Hq, S, D] or [B, S, Hq, D] of `dtype`, updated in place.
 * k: device, [B, Hk, S, D] or [B, S, Hk, D] of `dtype`, updated in place;
 *    may be NULL when Hk = 0.  q and k must not overlap each other or the
 *    tables.
 * cos, sin: device, float[table_rows, rotary_dim/2] (as written by
 *    rope_tables_build with max_pos = table_rows).
 * pos_idx: device int32[S] or NULL.  Token s (in every batch) uses table
 *    row pos_idx[s] (Unsloth page, Support for Custom Position IDs;
 *    "rotary-embedding-torch", Input Tensor Shapes: rotary_pos_emb_indices
 *    (seq_len,)).  The value -1 leaves the token unrotated (the pos_mask of
 *    "rotary-embedding-torch", flash_attn_with_rotary): its rows are not
 *    written.  With NULL, token s uses row s and S <= table_rows is required.
 *    Any other value outside [0, table_rows) leaves that token unrotated and
 *    raises a device-side flag reported by rope_check_errors as
 *    ROPE_ERR_POS_OUT_OF_RANGE.
 * B, S >= 0; Hq, Hk >= 0; D >= 1; rotary_dim even, 2 <= rotary_dim <= D.
 *    An empty problem (B, S or Hq + Hk zero) returns ROPE_OK and enqueues
 *    nothing.
 * layout: rope_layout.  seq_before_head, backward: 0 or 1.  backward = 1
 *    rotates by the negated angle (the gradient of the forward rotation).
 * dtype: rope_dtype of q and k.
 * table_rows: rows of cos and sin (>= 1 for a non-empty problem).
 * Errors: ROPE_ERR_UNSUPPORTED for dtype/layout outside the enums;
 *    ROPE_ERR_INVALID_ARG for the size, flag, pointer and overlap rules
 *    above; ROPE_ERR_CUDA if the launch fails.  Pointers or rows that are
 *    not 16-byte aligned take a slower element-wise kernel, same results.
 */
rope_status rope_apply_qk(void *q, void *k, const float *cos, const float *sin,
                          const int32_t *pos_idx, int64_t B, int32_t Hq, int32_t Hk, int64_t S,
                          int32_t D, int32_t rotary_dim, int32_t layout, int32_t seq_before_head,
                          int32_t backward, int32_t dtype, int64_t table_rows, void *stream);

/*
 * rope_apply_qk_out -- rotate Q and K out of place (or in place), with
 * optional per-sequence position indices.
 *
 * Same computation as rope_apply_qk, reading q and k and writing q_out and
 * k_out.  An output may be exactly its input (that tensor is rotated in
 * place); otherwise it must not overlap any input, the tables, pos_idx or
 * the other output.  Out of place, the output receives every element: the
 * rotated span, the tail [rotary_dim, D) copied unchanged, and the rows of
 * unrotated tokens (position -1 or out of range) copied unchanged.
 *
 * Position indices (Unsloth page, Support for Custom Position IDs:
 * prefix-tuning and context shifting; "rotary-embedding-torch", Input Tensor
 * Shapes: indices into a padded frequency buffer):
 *   pos_batch_stride = 0: pos_idx is int32[S], shared by every batch (as in
 *     rope_apply_qk);
 *   pos_batch_stride >= S: pos_idx is int32[B][pos_batch_stride] and token
 *     (b, s) uses pos_idx[b * pos_batch_stride + s] -- one position vector per
 *     sequence, e.g. sequences decoded at different offsets.
 * Other strides return ROPE_ERR_INVALID_ARG.  Everything else (sizes, flags,
 * errors, range flag) as for rope_apply_qk.
 */
rope_status rope_apply_qk_out(const void *q, const void *k, void *q_out, void *k_out,
                              const float *cos, const float *sin, const int32_t *pos_idx,
                              int64_t pos_batch_stride, int64_t B, int32_t Hq, int32_t Hk,
                              int64_t S, int32_t D, int32_t rotary_dim, int32_t layout,
                              int32_t seq_before_head, int32_t backward, int32_t dtype,
                              int64_t table_rows, void *stream);

/*
 * rope_apply_q -- rotate one tensor in place (the query-only kernel of the
 * Unsloth page, Triton Kernel Architecture for RoPE).  Same rules as
 * rope_apply_qk with x in place of q, H in place of Hq, and no k.
 */
rope_status rope_apply_q(void *x, const float *cos, const float *sin, const int32_t *pos_idx,
                         int64_t B, int32_t H, int64_t S, int32_t D, int32_t rotary_dim,
                         int32_t layout, int32_t seq_before_head, int32_t backward, int32_t dtype,
                         int64_t table_rows, void *stream);

/*
 * rope_attention_fwd -- attention forward with the rotation fused into the
 * loads of Q and K ("rotary-embedding-torch", flash_attn_with_rotary: the
 * rotary transformation is applied to the loaded Q and K blocks inside the
 * attention kernel, so rotated Q and K are never written to global memory).
 *
 *   o = softmax(scale * rot(q) rot(k)^T + mask) v
 *
 * q: device [B, Hq, Sq, D]; k, v: device [B, Hk, Sk, D]; o: device
 *    [B, Hq, Sq, D], written; all of `dtype` (ROPE_BF16 or ROPE_F16), dense.
 *    Hq must be a multiple of Hk (GQA/MQA: query head h uses key/value head
 *    h / (Hq/Hk)).
 * cos, sin: the rotation table (rope_tables_build or rope_tables_build_ex, any
 *    frequency mode), [table_rows, rotary_dim/2].
 * pos_q, pos_k: device int32 [Sq], [Sk] or NULL (row = index); -1 leaves a
 *    token unrotated (pos_mask); other out-of-range values are not rotated and
 *    raise the flag that rope_check_errors reports.
 * rotary_dim: multiple of 16, 16 <= rotary_dim <= D; D is 64 or 128.
 * layout: pair layout of the rotation.  causal: 0 or 1; the mask is aligned
 *    to the bottom right (query i sees key j when j <= i + Sk - Sq); a query
 *    row that sees no key gets zeros.
 * softmax_scale: > 0, or <= 0 for 1/sqrt(D).
 * k_workspace: NULL, or a device buffer of workspace_bytes >= B * Hk * Sk *
 *    D * 2 bytes, 16-byte aligned, overlapping no other argument; owned by
 *    the caller and overwritten.  NULL: every CTA rotates the key tiles it
 *    reads in shared memory, and rot(K) is never written.  Given: rot(K) is
 *    written there once per call by the rotation kernel (rope_apply_qk's
 *    arithmetic, so the same bits), then the attention kernel reads the
 *    rotated keys (for D = 128 on pairs of SMs, with no CTA rotating key
 *    tiles).  Under GQA every key tile is read by many CTAs, so for long
 *    sequences the workspace path is the faster one; both give the same
 *    result bit for bit.  Q is rotated inside the attention kernel either way.
 * Arithmetic: the rotated q and k rows are rounded to `dtype`, S = q k^T is
 *    accumulated in fp32 in tensor memory, P is rounded to `dtype` for the
 *    P v product (fp32 accumulation), o is rounded once.
 * Errors: ROPE_ERR_UNSUPPORTED for other dtypes, D, rotary_dim, layouts or
 *    pointers not 16-byte aligned; ROPE_ERR_INVALID_ARG for bad sizes, null
 *    pointers, o overlapping an input, a workspace too small or overlapping;
 *    ROPE_ERR_CUDA if the launch fails, which includes more than 65535
 *    query tiles per head -- Sq > 65535 * 128 when Hq / Hk is even, else
 *    Sq > 65535 * 256.  B, Hq or Sq zero: nothing to do, ROPE_OK.  Asynchronous on `stream`; rope_check_errors later reports
 *    out-of-range positions and, should a wait inside the kernel expire (about
 *    2 s; o is then not written), ROPE_ERR_KERNEL_TIMEOUT.
 */
rope_status rope_attention_fwd(const void *q, const void *k, const void *v, void *o,
                               const float *cos, const float *sin, const int32_t *pos_q,
                               const int32_t *pos_k, int64_t B, int32_t Hq, int32_t Hk, int64_t Sq,
                               int64_t Sk, int32_t D, int32_t rotary_dim, int32_t layout,
                               int32_t causal, float softmax_scale, int32_t dtype,
                               int64_t table_rows, void *k_workspace, int64_t workspace_bytes,
                               void *stream);

/*
 * rope_attention_fwd_masked -- rope_attention_fwd with a boolean attention
 * mask ("rotary-embedding-torch", flash_attn_with_rotary / Input Tensor
 * Shapes: attn_mask, batch x seq_len_k or batch x seq_len_q x seq_len_k,
 * whose False entries are excluded like masked scores):
 *
 *   o = softmax(scale * rot(q) rot(k)^T + causal mask + attn_mask) v
 *
 * attn_mask: device bytes, 0 = the key is hidden from the query (its score
 *    becomes -inf), any other value = visible (torch.bool tensors qualify):
 *      mask_kind ROPE_MASK_KEYS:       [B, Sk], the same for every query
 *                                      (padded batches: key padding);
 *      mask_kind ROPE_MASK_QUERY_KEYS: [B, Sq, Sk], one row per query (read
 *                                      as 16-byte vectors when the pointer
 *                                      is 16-byte aligned and Sk % 16 == 0,
 *                                      else byte by byte);
 *      mask_kind ROPE_MASK_NONE:       ignored (may be NULL): rope_attention_fwd.
 *    Dense, contiguous, shared by all heads; it must not overlap o or the
 *    workspace.  The mask applies together with `causal`; a query row that
 *    sees no key gets zeros.
 * Key tiles a [B, Sk] mask hides entirely: with a k_workspace of at least
 *    W + 4 B bytes, W = B * Hk * Sk * D * 2 rounded up to a multiple of 16,
 *    the call also writes there (from byte W) the number of 128-key tiles up
 *    to each batch entry's last visible key, and the attention kernels skip
 *    the tiles past it (the result is the same bit for bit: hidden keys only
 *    add exact zeros).  With a smaller workspace, or none, every tile is
 *    computed.
 * Padding: with at least W + 8 B bytes, the call also writes (from byte
 *    W + 4 B) each entry's prefix length, L when its mask shows exactly the
 *    keys [0, L), else -1; the attention kernels of the workspace path
 *    then compute such an entry as an unmasked one with L keys, without
 *    reading its mask (the same bits).
 * Everything else as rope_attention_fwd.
 * Errors: as rope_attention_fwd; also ROPE_ERR_UNSUPPORTED for a mask_kind
 *    outside the enum and ROPE_ERR_INVALID_ARG for a NULL mask (with Sk > 0)
 *    or one that overlaps o or the workspace.
 */
rope_status rope_attention_fwd_masked(const void *q, const void *k, const void *v, void *o,
                                      const float *cos, const float *sin, const int32_t *pos_q,
                                      const int32_t *pos_k, int64_t B, int32_t Hq, int32_t Hk,
                                      int64_t Sq, int64_t Sk, int32_t D, int32_t rotary_dim,
                                      int32_t layout, int32_t causal, float softmax_scale,
                                      int32_t dtype, int64_t table_rows, const uint8_t *attn_mask,
                                      int32_t mask_kind, void *k_workspace,
                                      int64_t workspace_bytes, void *stream);

/*
 * rope_attention_fwd_noalloc -- rope_attention_fwd with the key workspace
 * taken from a fixed device array inside this library (32 MiB), for callers
 * that cannot allocate device memory at call time: an engine that has
 * reserved the device's memory for its own pool, plugin code limited to the
 * buffers its host framework hands it, or a latency-critical path that
 * cannot afford cudaMalloc.  The pages have no counterpart of this entry
 * point; it is an addition of this library.
 *
 * Arguments, result and errors: as rope_attention_fwd with k_workspace set,
 * except that rot(K) goes to the library's array.  The arguments are checked
 * first, exactly as rope_attention_fwd checks them (its error, if any, is
 * returned); then ROPE_ERR_UNSUPPORTED when B * Hk * Sk * D * 2 bytes exceed
 * 32 MiB (33554432 bytes).  Both happen before anything touches the device.
 * Nothing is allocated or freed, and no allocating library routine is called.
 * Set-up: the first call on a device (with that device current) looks up the
 *    array's device address once (cudaGetSymbolAddress) and caches it; make
 *    that first call before any stream capture.  The cached address belongs
 *    to the device's context as it was then: after cudaDeviceReset (or any
 *    reset of the primary context) the process must be restarted before this
 *    entry point is called again.
 * Sharing: every device that loads the library holds the 32 MiB array until
 *    the process exits.  All calls on a device share it; each call rewrites
 *    the part it uses before reading it (nothing needs to start at zero), and
 *    calls whose work overlaps on the GPU (on streams not ordered with each
 *    other) race on it.
 */
rope_status rope_attention_fwd_noalloc(const void *q, const void *k, const void *v, void *o,
                                       const float *cos, const float *sin, const int32_t *pos_q,
                                       const int32_t *pos_k, int64_t B, int32_t Hq, int32_t Hk,
                                       int64_t Sq, int64_t Sk, int32_t D, int32_t rotary_dim,
                                       int32_t layout, int32_t causal, float softmax_scale,
                                       int32_t dtype, int64_t table_rows, void *stream);

/*
 * rope_check_errors -- synchronise `stream`, then report and clear the
 * current device's error flag.
 * Returns ROPE_ERR_CUDA if the stream reports an error, else
 * ROPE_ERR_KERNEL_TIMEOUT if a wait inside an attention kernel expired
 * (about 2 s; that launch stopped early and its output is incomplete), else
 * ROPE_ERR_POS_OUT_OF_RANGE if any launch since the last check met an
 * out-of-range position index, else ROPE_OK.  The flag is shared by all
 * streams of the device.
 */
rope_status rope_check_errors(void *stream);

/*
 * rope_probe_wait_expiry -- diagnostic: exercise the path an expired wait
 * takes, without stalling any real kernel.  One thread of one CTA waits,
 * with the bounded mbarrier wait that the attention kernels use, on a barrier that nothing arrives at; after `cycles` SM clock cycles
 * (1 .. 4e9; 2e6 is about a millisecond) the wait gives up and sets the
 * timeout bit of the device error flag, as an expired wait inside those
 * kernels does.  The next rope_check_errors then returns
 * ROPE_ERR_KERNEL_TIMEOUT and clears the flag.  The pages have no
 * counterpart; this is an addition of this library, for tests and for
 * callers that want to check their error handling.
 * Errors: ROPE_ERR_INVALID_ARG for cycles outside 1 .. 4e9 (nothing is
 *    launched); ROPE_ERR_CUDA if the launch fails.  Asynchronous on `stream`.
 */
rope_status rope_probe_wait_expiry(int64_t cycles, void *stream);

/* rope_status_string -- static, NUL-terminated name of a status value. */
const char *rope_status_string(rope_status status);

/*
 * rope_qk_kernel_variant -- which kernel rope_apply_qk would launch for
 * these arguments, without launching anything or touching the device.
 * Returns 0 when nothing would be launched (error or empty problem),
 * 2 for the element-wise kernel (any shape or alignment),
 * 3 for the register-staged 16-byte vector kernel (the automatic choice
 * for 16-byte aligned shapes whose rotary span is whole pairs of vectors).
 * Useful for tests and for callers checking that their tensors are aligned.
 */
int32_t rope_qk_kernel_variant(const void *q, const void *k, const float *cos, const float *sin,
                               const int32_t *pos_idx, int64_t B, int32_t Hq, int32_t Hk,
                               int64_t S, int32_t D, int32_t rotary_dim, int32_t layout,
                               int32_t seq_before_head, int32_t backward, int32_t dtype,
                               int64_t table_rows);

/*
 * rope_force_kernel_variant -- process-wide choice of the rotation kernel,
 * for tests and tuning: 0 = automatic (default), 2 or 3 as returned by
 * rope_qk_kernel_variant.  While 3 is forced, calls whose shapes or pointers
 * do not qualify for it return ROPE_ERR_UNSUPPORTED.  Both kernels compute
 * bit-identical results.  ROPE_ERR_INVALID_ARG for other values.
 */
rope_status rope_force_kernel_variant(int32_t variant);

/*
 * rope_tune_rotation_launch -- process-wide grid sizing of the vector
 * rotation kernel, for tuning and measurement; the results do not depend on
 * it.  The kernel splits its work, units of (TT consecutive tokens, one
 * head), into balanced contiguous runs, one per lane group of TT rows.
 *   ctas_per_sm: cap the grid at this many CTAs per SM (0 = as many as can
 *     be resident at once, the default; 1 .. 64 otherwise);
 *   min_units: the fewest units a run holds before the grid grows (0 = the
 *     default, 1);
 *   prefetch_next: 1 or 0 = while rotating a tile, prefetch the first heads
 *     of the run's next tile into L2 (the default); -1 = do not.
 * ROPE_ERR_INVALID_ARG for values outside these ranges (nothing changes).
 * The pages have no counterpart; this is an addition of this library.
 */
rope_status rope_tune_rotation_launch(int32_t ctas_per_sm, int32_t min_units,
                                      int32_t prefetch_next);

#ifdef __cplusplus
}
#endif

#endif /* ROPE_H */
