// rope_internal.cuh -- declarations shared by the translation units of librope.
// Not part of the public ABI (include/rope.h is).
#pragma once

#include <cstdint>
#include <cuda_runtime.h>

namespace rope {

// One rotated tensor: base pointer and element strides of its batch, head and
// sequence dimensions (the feature dimension is contiguous).
struct TensorRef {
    void *base;
    int32_t heads;
    int64_t stride_b;
    int64_t stride_h;
    int64_t stride_s;
};

// Everything a rotation launch needs.  Passed by value as a kernel parameter.
struct ApplyArgs {
    TensorRef t[2];            // Q then K; ntensors of them are valid
    void *out[2];              // output base of each tensor (same strides); == t[i].base in place
    int32_t ntensors;
    int32_t copy_through[2];   // 1: tensor written out of place (pass-through values are copied)
    const float *cos;          // [table_rows, rotary_dim/2]
    const float *sin;
    const int32_t *pos_idx;    // [S], [B, pos_stride_b] or nullptr
    int64_t pos_stride_b;      // 0: one position vector shared by all batches
    int64_t B;
    int64_t S;
    int32_t D;
    int32_t rotary_dim;
    int64_t table_rows;
    int32_t backward;          // 1: rotate by the negated angle
    int32_t *range_flag;       // device word set when a position is out of range
};

// Kernel variants: kVector moves 16-byte vectors through registers (the
// automatic choice for aligned shapes), kScalar handles any shape one pair at
// a time.  The values are those rope_qk_kernel_variant reports.
enum Variant : int32_t { kNone = 0, kScalar = 2, kVector = 3 };

// Threads per CTA of the vectorised kernel and heads in flight per thread.
#ifndef ROPE_VEC_THREADS
#define ROPE_VEC_THREADS 128
#endif
#ifndef ROPE_VEC_UNROLL
#define ROPE_VEC_UNROLL 4
#endif
// Resident CTAs per SM the register allocation must allow (launch bounds).
#ifndef ROPE_VEC_MIN_BLOCKS
#define ROPE_VEC_MIN_BLOCKS 4
#endif
// Launch the hot kernels with programmatic dependent launch.
#ifndef ROPE_PDL
#define ROPE_PDL 1
#endif
// Register kernel: keep the next batch of heads' loads in flight while
// rotating the current batch.
#ifndef ROPE_VEC_PIPELINE
#define ROPE_VEC_PIPELINE 1
#endif
constexpr bool kVecPipeline = ROPE_VEC_PIPELINE != 0;
// Cache hints of the register kernel's Q/K loads (see load_stream).
#ifndef ROPE_VEC_LOAD_MODE
#define ROPE_VEC_LOAD_MODE 2
#endif
constexpr int kVecLoadMode = ROPE_VEC_LOAD_MODE;
// Loads of rotary spans that are not whole 256-byte rows: 0 = ld.global.cs,
// 1 = ld.global.cs.L2::64B.
#ifndef ROPE_VEC_PART_HINT
#define ROPE_VEC_PART_HINT 1
#endif
constexpr int kVecPartHint = ROPE_VEC_PART_HINT;
constexpr bool kPdl = ROPE_PDL != 0;
// Head rows of its first units each thread row prefetches into L2 before
// waiting for the previous grid (0: none; default: one batch of heads).
#ifndef ROPE_VEC_PREFETCH_HEADS
#define ROPE_VEC_PREFETCH_HEADS ROPE_VEC_UNROLL
#endif
constexpr int kVecPrefetchHeads = ROPE_VEC_PREFETCH_HEADS;
// L2 prefetches of head rows: a bulk prefetch of the rotary span's exact
// bytes per row (cp.async.bulk.prefetch.L2) or prefetch.global.L2 of the
// lines under each thread's two vectors (whole lines): 0 = lines always,
// 1 = bulk always, 2 = bulk for spans that are not whole rows (a partial
// rotary span, where whole lines would fetch the tail too), else lines.
#ifndef ROPE_VEC_PREFETCH_BULK
#define ROPE_VEC_PREFETCH_BULK 2
#endif
constexpr int kVecPrefetchBulk = ROPE_VEC_PREFETCH_BULK;
constexpr int kVecThreads = ROPE_VEC_THREADS;
constexpr int kVecUnroll = ROPE_VEC_UNROLL;
constexpr int kVecMinBlocks = ROPE_VEC_MIN_BLOCKS;
// NJ (16-byte vectors per half span) must fit in one CTA row: the register
// kernel takes rotary spans of up to 32 * kVecThreads bytes.
constexpr int kMaxVectorsPerHalf = kVecThreads;

// Attention with rotary Q/K (rope_attention.cuh).
struct AttnArgs {
    const void *q, *k, *v;
    const void *k_rot;               // k rotated beforehand (rot(K), same layout), or nullptr
    void *o;
    const float *cos, *sin;
    const int32_t *pos_q, *pos_k;    // [Sq], [Sk] or nullptr (-1 = not rotated)
    int64_t B;
    int32_t Hq, Hk;
    int64_t Sq, Sk;
    int32_t rotary_dim;
    int64_t table_rows;
    float scale_log2;                // softmax scale * log2(e)
    int32_t causal;
    int32_t *flag;
    const uint8_t *mask;             // attn_mask bytes (0 = hidden), or nullptr
    int32_t mask_kind;               // 0: none, 1: [B, Sk], 2: [B, Sq, Sk]
    int32_t mask_vec16;              // kind 2: rows 16-byte aligned (read as vectors)
    const int32_t *kv_tiles;         // [B]: key tiles up to the last key a [B, Sk] mask
                                     // shows (0: none), or nullptr (no skipping)
    const int32_t *kv_len;           // [B]: L when a [B, Sk] mask shows exactly the keys
                                     // [0, L), else -1; or nullptr
};
// Writes kv_tiles, and kv_len when lens is not null, for a [B, Sk]
// attn_mask (rope_api.cu).
cudaError_t launch_mask_tiles(const uint8_t *mask, int64_t B, int64_t Sk, int32_t *tiles,
                              int32_t *lens, cudaStream_t st);
cudaError_t launch_attention(const AttnArgs &a, int32_t D, int32_t layout, int32_t dtype,
                             cudaStream_t st);
// The same for calls with an attn_mask (rope_attention_masked.cu).
cudaError_t launch_attention_masked(const AttnArgs &a, int32_t D, int32_t layout, int32_t dtype,
                                    cudaStream_t st);
// One bounded mbarrier wait that expires after `cycles` clock cycles and sets
// bit 1 of *flag (rope_probe_wait_expiry).
cudaError_t launch_wait_probe(int32_t *flag, long long cycles, cudaStream_t st);

// Grid sizing of the register kernel (rope_tune_rotation_launch; 0 = the
// default of each field).  ctas_per_sm caps the grid at that many CTAs per SM
// (default: as many as are resident at once); min_units is the fewest
// (token tile, head) units a lane group takes before the grid grows (default
// 1); prefetch_next > 0 prefetches the first heads of a lane group's next tile
// into L2 while it rotates the current one (default on; -1 turns it off).
struct VecLaunchTuning {
    int32_t ctas_per_sm;
    int32_t min_units;
    int32_t prefetch_next;
};
VecLaunchTuning vec_launch_tuning();

// Per element type launchers (rope_apply_f32.cu, rope_apply_bf16.cu, rope_apply_f16.cu).
cudaError_t launch_apply_f32(const ApplyArgs &a, int32_t layout, Variant v, cudaStream_t st);
cudaError_t launch_apply_bf16(const ApplyArgs &a, int32_t layout, Variant v, cudaStream_t st);
cudaError_t launch_apply_f16(const ApplyArgs &a, int32_t layout, Variant v, cudaStream_t st);

}  // namespace rope
