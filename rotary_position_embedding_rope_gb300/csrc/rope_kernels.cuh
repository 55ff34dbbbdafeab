// rope_kernels.cuh -- the rotation kernels of librope (sm_103a).
//
// What is computed ("Rotary Embedding (RoPE) Kernel Optimization", Overview):
// each pair (x1, x2) of a head row at table row r becomes
//     (x1 c - x2 s, x1 s + x2 c),  c = cos[r][i], s = sin[r][i]
// and the backward pass uses -s ("How Unsloth Optimizes RoPE Embedding
// Computations in Triton Kernels", Frequently Asked Questions).
//
// Design (GB300): RoPE moves 4 bytes per bf16 pair each way and does a few
// flops, so it is bound by HBM bandwidth.  The vectorised kernel therefore:
//   * gives each token a row of the CTA (NJ threads) and keeps that token's
//     cos/sin values in registers for all Hq + Hk heads, so the table row is
//     read once per token (the Unsloth page motivates head grouping, Triton
//     Kernel Architecture for RoPE; here the group is all heads);
//   * moves data in 16-byte vectors: thread j owns vector j of the first
//     half of the rotary span and vector j of the second half.  For
//     split-half pairs (x[i], x[i+rd/2]) the partner of every element is the
//     same lane of the other vector; for interleaved pairs (x[2i], x[2i+1])
//     both elements sit in one vector.  Pairing is a register swizzle, no
//     strided scalar loads and no shuffles;
//   * issues the loads of kVecUnroll heads before any arithmetic so each
//     thread has 2 * kVecUnroll 16-byte requests in flight;
//   * uses streaming (evict-first) loads and stores: every byte is touched
//     exactly once;
//   * never reads or writes features past rotary_dim, nor tokens whose
//     position is -1 (pass-through without arithmetic).
// The element-wise kernel handles shapes and pointers the vector kernel
// cannot (rotary span not a multiple of 32 bytes, rows or pointers not
// 16-byte aligned).  Both use the same arithmetic, so their results are
// bit-identical.
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include <atomic>

#include "rope_internal.cuh"

namespace rope {

// ---------------------------------------------------------------------------
// Element types: number of elements in a 16-byte vector and conversions.
// Widening to fp32 is exact; narrowing rounds to nearest even, once.
// ---------------------------------------------------------------------------
template <typename T> struct Elt;

template <> struct Elt<float> {
    static constexpr int V = 4;
    __device__ __forceinline__ static float to_f(float x) { return x; }
    __device__ __forceinline__ static float from_f(float x) { return x; }
    __device__ __forceinline__ static void unpack(const uint4 &u, float (&f)[V]) {
        f[0] = __uint_as_float(u.x); f[1] = __uint_as_float(u.y);
        f[2] = __uint_as_float(u.z); f[3] = __uint_as_float(u.w);
    }
    __device__ __forceinline__ static uint4 pack(const float (&f)[V]) {
        return make_uint4(__float_as_uint(f[0]), __float_as_uint(f[1]),
                          __float_as_uint(f[2]), __float_as_uint(f[3]));
    }
};

template <> struct Elt<__nv_bfloat16> {
    static constexpr int V = 8;
    __device__ __forceinline__ static float to_f(__nv_bfloat16 x) { return __bfloat162float(x); }
    __device__ __forceinline__ static __nv_bfloat16 from_f(float x) { return __float2bfloat16_rn(x); }
    __device__ __forceinline__ static float2 word_to_f2(uint32_t w) {
        __nv_bfloat162 h;
        memcpy(&h, &w, 4);
        return __bfloat1622float2(h);
    }
    __device__ __forceinline__ static uint32_t f2_to_word(float a, float b) {
        __nv_bfloat162 h = __floats2bfloat162_rn(a, b);   // a -> low half, b -> high half
        uint32_t w;
        memcpy(&w, &h, 4);
        return w;
    }
    __device__ __forceinline__ static void unpack(const uint4 &u, float (&f)[V]) {
        float2 p;
        p = word_to_f2(u.x); f[0] = p.x; f[1] = p.y;
        p = word_to_f2(u.y); f[2] = p.x; f[3] = p.y;
        p = word_to_f2(u.z); f[4] = p.x; f[5] = p.y;
        p = word_to_f2(u.w); f[6] = p.x; f[7] = p.y;
    }
    __device__ __forceinline__ static uint4 pack(const float (&f)[V]) {
        return make_uint4(f2_to_word(f[0], f[1]), f2_to_word(f[2], f[3]),
                          f2_to_word(f[4], f[5]), f2_to_word(f[6], f[7]));
    }
};

template <> struct Elt<__half> {
    static constexpr int V = 8;
    __device__ __forceinline__ static float to_f(__half x) { return __half2float(x); }
    __device__ __forceinline__ static __half from_f(float x) { return __float2half_rn(x); }
    __device__ __forceinline__ static float2 word_to_f2(uint32_t w) {
        __half2 h;
        memcpy(&h, &w, 4);
        return __half22float2(h);
    }
    __device__ __forceinline__ static uint32_t f2_to_word(float a, float b) {
        __half2 h = __floats2half2_rn(a, b);
        uint32_t w;
        memcpy(&w, &h, 4);
        return w;
    }
    __device__ __forceinline__ static void unpack(const uint4 &u, float (&f)[V]) {
        float2 p;
        p = word_to_f2(u.x); f[0] = p.x; f[1] = p.y;
        p = word_to_f2(u.y); f[2] = p.x; f[3] = p.y;
        p = word_to_f2(u.z); f[4] = p.x; f[5] = p.y;
        p = word_to_f2(u.w); f[6] = p.x; f[7] = p.y;
    }
    __device__ __forceinline__ static uint4 pack(const float (&f)[V]) {
        return make_uint4(f2_to_word(f[0], f[1]), f2_to_word(f[2], f[3]),
                          f2_to_word(f[4], f[5]), f2_to_word(f[6], f[7]));
    }
};

// ---------------------------------------------------------------------------
// a*b - c*d with Kahan's fma-based compensation: the rounding error of c*d
// is recovered exactly by an fma and added back, so the result has a
// relative error of at most 2 units in the last place of fp32 (Jeannerod,
// Louvet & Muller, "Further analysis of Kahan's algorithm for the accurate
// computation of 2x2 determinants", Math. Comp. 82, 2013).  That keeps a
// bf16/fp16 output within one unit of the correctly rounded value even when
// the two products nearly cancel.  Explicit _rn intrinsics keep the compiler
// from contracting or reordering the steps.
// ---------------------------------------------------------------------------
__device__ __forceinline__ float diff_of_products(float a, float b, float c, float d) {
    const float w = __fmul_rn(c, d);
    const float e = __fmaf_rn(-c, d, w);      // w - c*d, exact
    const float f = __fmaf_rn(a, b, -w);      // a*b - w, one rounding
    return __fadd_rn(f, e);
}

// (x1, x2) <- (x1 c - x2 s, x1 s + x2 c)
__device__ __forceinline__ void rotate_pair(float &x1, float &x2, float c, float s) {
    const float y1 = diff_of_products(x1, c, x2, s);
    const float y2 = diff_of_products(x1, s, -x2, c);
    x1 = y1;
    x2 = y2;
}

// ---------------------------------------------------------------------------
// Programmatic dependent launch.  The hot kernels are launched with the
// programmatic-stream-serialisation attribute: the next launch in the stream
// may become resident while this one drains.  Every kernel waits for the
// previous grid to complete (and its memory to be visible) before it reads or
// writes global memory, so results do not depend on the overlap.
// ---------------------------------------------------------------------------
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_trigger()
{
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

template <typename Kernel, typename... Args>
cudaError_t launch_hot(Kernel kernel, dim3 grid, dim3 block, size_t smem, cudaStream_t st,
                       Args... args)
{
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = kPdl ? 1 : 0;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kernel, args...);
}

// Streaming 16-byte accesses of Q/K.  Every byte is read once and written
// once, so nothing is kept in L1; kVecLoadMode picks the cache hints:
//   0: ld/st.global.cs (evict-first streaming)
//   1: ld.global.L1::no_allocate.L2::256B (fetch the whole 256-byte segment
//      into L2, so the second-half load of a row hits L2) / st.global.cs
//   2: ld.global.cs.L2::256B / st.global.cs
// The 256-byte fetch is used only when `whole` says the rotary spans tile
// whole 256-byte segments; otherwise it would pull in bytes (the tail past
// rotary_dim, neighbouring rows) the kernel never touches.
__device__ __forceinline__ uint4 load_stream(const uint4 *p, bool whole = false)
{
    if (!whole) {
        if constexpr (kVecPartHint == 1) {
            uint4 v;
            asm volatile("ld.global.cs.L2::64B.v4.u32 {%0, %1, %2, %3}, [%4];"
                         : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                         : "l"(p));
            return v;
        } else {
            return __ldcs(p);
        }
    }
    if constexpr (kVecLoadMode == 1) {
        uint4 v;
        asm volatile("ld.global.L1::no_allocate.L2::256B.v4.u32 {%0, %1, %2, %3}, [%4];"
                     : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                     : "l"(p));
        return v;
    } else if constexpr (kVecLoadMode == 2) {
        uint4 v;
        asm volatile("ld.global.cs.L2::256B.v4.u32 {%0, %1, %2, %3}, [%4];"
                     : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                     : "l"(p));
        return v;
    } else {
        return __ldcs(p);
    }
}
__device__ __forceinline__ void store_stream(uint4 *p, const uint4 &v) { __stcs(p, v); }

// Rotate the rotary spans of heads [lo, hi) of one token, whose head 0 row
// starts at in0 (read) and out0 (written; == in0 in place), heads stride_h
// elements apart.  U heads' loads are issued before any arithmetic; with
// kVecPipeline the loads of the next U heads are issued before the current
// ones are rotated, so two batches are in flight.
template <typename T, int LAYOUT>
__device__ __forceinline__ void rotate_vectors(uint4 &va, uint4 &vb, const float *c,
                                               const float *sn)
{
    constexpr int V = Elt<T>::V;
    float fa[V], fb[V];
    Elt<T>::unpack(va, fa);
    Elt<T>::unpack(vb, fb);
    if constexpr (LAYOUT == 0) {
#pragma unroll
        for (int e = 0; e < V; ++e)
            rotate_pair(fa[e], fb[e], c[e], sn[e]);
    } else {
#pragma unroll
        for (int e = 0; e < V / 2; ++e) {
            rotate_pair(fa[2 * e], fa[2 * e + 1], c[e], sn[e]);
            rotate_pair(fb[2 * e], fb[2 * e + 1], c[V / 2 + e], sn[V / 2 + e]);
        }
    }
    va = Elt<T>::pack(fa);
    vb = Elt<T>::pack(fb);
}

template <typename T, int LAYOUT, int U>
__device__ __forceinline__ void rotate_heads(const T *in0, T *out0, int64_t stride_h, int32_t lo,
                                             int32_t hi, int j, int NJ, const float *c,
                                             const float *sn, bool whole)
{
    if constexpr (!kVecPipeline) {
        for (int32_t h0 = lo; h0 < hi; h0 += U) {
            uint4 va[U], vb[U];
#pragma unroll
            for (int u = 0; u < U; ++u) {
                if (h0 + u < hi) {
                    const uint4 *ptr = reinterpret_cast<const uint4 *>(in0 + (int64_t)(h0 + u) * stride_h);
                    va[u] = load_stream(ptr + j, whole);
                    vb[u] = load_stream(ptr + j + NJ, whole);
                }
            }
#pragma unroll
            for (int u = 0; u < U; ++u) {
                if (h0 + u < hi) {
                    rotate_vectors<T, LAYOUT>(va[u], vb[u], c, sn);
                    uint4 *ptr = reinterpret_cast<uint4 *>(out0 + (int64_t)(h0 + u) * stride_h);
                    store_stream(ptr + j, va[u]);
                    store_stream(ptr + j + NJ, vb[u]);
                }
            }
        }
    } else {
        uint4 ca[U], cb[U], na[U], nb[U];
#pragma unroll
        for (int u = 0; u < U; ++u) {
            if (lo + u < hi) {
                const uint4 *ptr = reinterpret_cast<const uint4 *>(in0 + (int64_t)(lo + u) * stride_h);
                ca[u] = load_stream(ptr + j, whole);
                cb[u] = load_stream(ptr + j + NJ, whole);
            }
        }
        for (int32_t h0 = lo; h0 < hi; h0 += U) {
            const int32_t h1 = h0 + U;
#pragma unroll
            for (int u = 0; u < U; ++u) {
                if (h1 + u < hi) {
                    const uint4 *ptr = reinterpret_cast<const uint4 *>(in0 + (int64_t)(h1 + u) * stride_h);
                    na[u] = load_stream(ptr + j, whole);
                    nb[u] = load_stream(ptr + j + NJ, whole);
                }
            }
#pragma unroll
            for (int u = 0; u < U; ++u) {
                if (h0 + u < hi) {
                    rotate_vectors<T, LAYOUT>(ca[u], cb[u], c, sn);
                    uint4 *ptr = reinterpret_cast<uint4 *>(out0 + (int64_t)(h0 + u) * stride_h);
                    store_stream(ptr + j, ca[u]);
                    store_stream(ptr + j + NJ, cb[u]);
                }
            }
#pragma unroll
            for (int u = 0; u < U; ++u) {
                ca[u] = na[u];
                cb[u] = nb[u];
            }
        }
    }
}

// Out of place only: copy 16-byte vectors [v0, v1) of head rows [lo, hi)
// from in0 to out0 unchanged (the tail past rotary_dim, or whole rows of
// tokens that are not rotated); the CTA row's NJ threads stride the vectors.
template <typename T>
__device__ __forceinline__ void copy_heads(const T *in0, T *out0, int64_t stride_h, int32_t lo,
                                           int32_t hi, int j, int NJ, int32_t v0, int32_t v1)
{
    for (int32_t hd = lo; hd < hi; ++hd) {
        const uint4 *src = reinterpret_cast<const uint4 *>(in0 + (int64_t)hd * stride_h);
        uint4 *dst = reinterpret_cast<uint4 *>(out0 + (int64_t)hd * stride_h);
        for (int32_t v = v0 + j; v < v1; v += NJ)
            store_stream(dst + v, load_stream(src + v));
    }
}

// ---------------------------------------------------------------------------
// Register-staged vector kernel.
//   blockDim = (NJ, TS): NJ = 16-byte vectors per half of the rotary span,
//   TS token rows, a whole number of lane groups.  A lane group is
//   TT = max(1, 32 / NJ) consecutive rows: one warp when NJ <= 32 (TT tokens side by side), else
//   one row of NJ threads.  It works on tiles of TT consecutive tokens of the
//   flattened (batch, sequence) order, row r taking token tile * TT + r.
//   The work is the list of units (tile, head), the P = Hq + Hk heads of a
//   tile in order (Q heads, then K heads).  Lane group g of the grid takes a
//   balanced contiguous run of units [u0, u1): every lane group does the same
//   work to within one unit whatever the grid size, so the grid is sized to
//   the CTAs that are resident at once and no partial last wave idles the
//   GPU.  A run walks its tiles in order: for each, every row loads its
//   token's cos/sin values once into registers and rotates the run's heads
//   of that tile, the loads of the next kU heads issued before the current
//   ones are rotated.  All rows of a lane group share the run, so their
//   control flow is the same (except past the last token and for unrotated
//   tokens).
//   Split-half: vector j holds elements [jV, jV+V) and vector j+NJ holds
//   their partners [rd/2 + jV, ...); cos/sin columns [jV, jV+V).
//   Interleaved: vector j holds pairs [jV/2, jV/2 + V/2) and vector j+NJ
//   holds pairs [(j+NJ)V/2, ...); the thread keeps both column ranges.
// ---------------------------------------------------------------------------

// Prefetch into L2 the row vectors of thread j of heads [hb, he) (unit head
// indices: Q heads first, then K heads) of token (b, s); WHOLE: the kernel
// instance for rotary spans that are whole rows (kVecPrefetchBulk picks the
// form of the prefetch).
template <typename T, bool WHOLE>
__device__ __forceinline__ void prefetch_heads(const ApplyArgs &p, int64_t b, int64_t s,
                                               int32_t hb, int32_t he, int j, int NJ)
{
    constexpr bool bulk = kVecPrefetchBulk == 1 || (kVecPrefetchBulk == 2 && !WHOLE);
#pragma unroll
    for (int ti = 0; ti < 2; ++ti) {
        if (ti >= p.ntensors)
            break;
        const TensorRef t = p.t[ti];
        const int32_t off = ti ? p.t[0].heads : 0;
        const int32_t lo = (hb > off ? hb : off) - off;
        const int32_t hi = (he < off + t.heads ? he : off + t.heads) - off;
        const T *in0 = static_cast<const T *>(t.base) + b * t.stride_b + s * t.stride_s;
        for (int32_t hd = lo; hd < hi; ++hd) {
            const uint4 *row = reinterpret_cast<const uint4 *>(in0 + (int64_t)hd * t.stride_h);
            if constexpr (bulk) {
                // the rotary span exactly (2 NJ 16-byte vectors), one request
                if (j == 0)
                    asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;"
                                 ::"l"(row), "r"((uint32_t)(32 * NJ)) : "memory");
            } else {
                asm volatile("prefetch.global.L2 [%0];" ::"l"(row + j));
                asm volatile("prefetch.global.L2 [%0];" ::"l"(row + j + NJ));
            }
        }
    }
}

// WHOLE: the rotary spans are whole rows of a multiple of 256 bytes
// (rotary_dim == D, D elements a multiple of 256 bytes); the launcher picks
// the instance.  The other instance still tests this at run time: with the
// test folded away its code measured slower on partial rotary spans.
// NJC: NJ known at compile time (then TT and the lane groups per CTA are
// too), or 0: NJ = blockDim.x and TT as passed.
template <typename T, int LAYOUT, int U, bool WHOLE, int NJC>
__global__ void __launch_bounds__(kVecThreads, kVecMinBlocks)
rope_vec_kernel(const ApplyArgs p, int64_t n_units, int32_t TT_arg, int32_t prefetch_next)
{
    constexpr int V = Elt<T>::V;
    const int NJ = NJC > 0 ? NJC : (int)blockDim.x;
    const int32_t TT = NJC > 0 ? (NJC >= 32 ? 1 : 32 / NJC) : TT_arg;
    const int j = threadIdx.x;
    const int h = p.rotary_dim >> 1;
    const int32_t P = p.t[0].heads + (p.ntensors > 1 ? p.t[1].heads : 0);
    const bool whole = WHOLE || (p.rotary_dim == p.D && (p.D * (int32_t)sizeof(T)) % 256 == 0);
    const int64_t total_tokens = p.B * p.S;

    // this lane group's run of units
    const int lgs = NJC > 0 ? (NJC >= kVecThreads ? 1 : (kVecThreads / NJC) / TT)
                            : (int)blockDim.y / TT;
    const int lg = threadIdx.y / TT;
    const int row = threadIdx.y - lg * TT;
    const int64_t G = (int64_t)gridDim.x * lgs;
    const int64_t g = (int64_t)blockIdx.x * lgs + lg;
    const int64_t share = n_units / G;
    const int64_t extra = n_units - share * G;
    const int64_t u0 = g * share + (g < extra ? g : extra);
    const int64_t u1 = u0 + share + (g < extra ? 1 : 0);

    if constexpr (kVecPrefetchHeads > 0) {
        // Before waiting for the previous grid: pull the first head rows of
        // this row's run into L2.  A prefetch only fills L2, the coherence
        // point that the previous grid's writes also reach, so it cannot make
        // a later load see stale data; it overlaps DRAM latency with the
        // previous launch's tail.
        if (u0 < u1) {
            const int64_t tile = u0 / P;
            const int32_t hb = (int32_t)(u0 - tile * P);
            int64_t he = hb + kVecPrefetchHeads;
            he = he < P ? he : P;
            he = he < hb + (u1 - u0) ? he : hb + (u1 - u0);
            const int64_t tok = tile * TT + row;
            if (tok < total_tokens) {
                const int64_t b = tok / p.S;
                prefetch_heads<T, WHOLE>(p, b, tok - b * p.S, hb, (int32_t)he, j, NJ);
            }
        }
    }

    pdl_wait();
    pdl_trigger();

    // the run, tile by tile (the launcher keeps every run below 2^30 units)
    const int64_t tile0 = u0 / P;
    int32_t hb = (int32_t)(u0 - tile0 * P);
    int64_t tok = tile0 * TT + row;
    for (int32_t left = (int32_t)(u1 - u0); left > 0; tok += TT, hb = 0) {
        const int32_t he = P - hb < left ? P : hb + left;
        left -= he - hb;
        if (tok >= total_tokens)
            continue;
        const int64_t b = tok / p.S;
        const int64_t s = tok - b * p.S;

        // the next tile of the run: its first heads into L2 now, so its
        // first loads do not start the pipeline from DRAM latency
        if (prefetch_next > 0 && left > 0 && tok + TT < total_tokens) {
            const int64_t nt = tok + TT;
            const int64_t nb = nt / p.S;
            const int32_t nhe = (int32_t)(U < left ? U : left);
            prefetch_heads<T, WHOLE>(p, nb, nt - nb * p.S, 0, nhe < P ? nhe : P, j, NJ);
        }

        // position of this token: table row, -1 = leave unrotated
        int64_t r = s;
        bool rotate = true;
        if (p.pos_idx != nullptr) {
            r = __ldg(p.pos_idx + b * p.pos_stride_b + s);
            if (r != -1 && (r < 0 || r >= p.table_rows)) {
                if (j == 0)
                    atomicOr(p.range_flag, 1);
                rotate = false;
            }
            rotate = rotate && r != -1;
        }
        if (!rotate) {
            {                                         // out of place: pass whole rows through
#pragma unroll
                for (int ti = 0; ti < 2; ++ti) {
                    if (ti >= p.ntensors)
                        break;
                    if (!p.copy_through[ti])
                        continue;
                    const TensorRef t = p.t[ti];
                    const int32_t off = ti ? p.t[0].heads : 0;
                    const int32_t lo = (hb > off ? hb : off) - off;
                    const int32_t hi = (he < off + t.heads ? he : off + t.heads) - off;
                    const int64_t o = b * t.stride_b + s * t.stride_s;
                    if (lo < hi)
                        copy_heads<T>(static_cast<const T *>(t.base) + o,
                                      static_cast<T *>(p.out[ti]) + o, t.stride_h, lo, hi, j, NJ,
                                      0, (p.D * (int32_t)sizeof(T)) / 16);
                }
            }
            continue;
        }

        // this thread's cos/sin values, kept in registers for the tile's heads
        float c[V], sn[V];
        const float *crow = p.cos + r * h;
        const float *srow = p.sin + r * h;
        if constexpr (LAYOUT == 0) {
#pragma unroll
            for (int q = 0; q < V / 4; ++q) {
                const float4 cv = __ldg(reinterpret_cast<const float4 *>(crow + j * V) + q);
                const float4 sv = __ldg(reinterpret_cast<const float4 *>(srow + j * V) + q);
                c[4 * q] = cv.x; c[4 * q + 1] = cv.y; c[4 * q + 2] = cv.z; c[4 * q + 3] = cv.w;
                sn[4 * q] = sv.x; sn[4 * q + 1] = sv.y; sn[4 * q + 2] = sv.z; sn[4 * q + 3] = sv.w;
            }
        } else if constexpr (V == 8) {
            const float4 c0 = __ldg(reinterpret_cast<const float4 *>(crow + j * 4));
            const float4 c1 = __ldg(reinterpret_cast<const float4 *>(crow + (j + NJ) * 4));
            const float4 s0 = __ldg(reinterpret_cast<const float4 *>(srow + j * 4));
            const float4 s1 = __ldg(reinterpret_cast<const float4 *>(srow + (j + NJ) * 4));
            c[0] = c0.x; c[1] = c0.y; c[2] = c0.z; c[3] = c0.w;
            c[4] = c1.x; c[5] = c1.y; c[6] = c1.z; c[7] = c1.w;
            sn[0] = s0.x; sn[1] = s0.y; sn[2] = s0.z; sn[3] = s0.w;
            sn[4] = s1.x; sn[5] = s1.y; sn[6] = s1.z; sn[7] = s1.w;
        } else {
            const float2 c0 = __ldg(reinterpret_cast<const float2 *>(crow + j * 2));
            const float2 c1 = __ldg(reinterpret_cast<const float2 *>(crow + (j + NJ) * 2));
            const float2 s0 = __ldg(reinterpret_cast<const float2 *>(srow + j * 2));
            const float2 s1 = __ldg(reinterpret_cast<const float2 *>(srow + (j + NJ) * 2));
            c[0] = c0.x; c[1] = c0.y; c[2] = c1.x; c[3] = c1.y;
            sn[0] = s0.x; sn[1] = s0.y; sn[2] = s1.x; sn[3] = s1.y;
        }
        if (p.backward) {
#pragma unroll
            for (int e = 0; e < V; ++e)
                sn[e] = -sn[e];
        }

#pragma unroll
        for (int ti = 0; ti < 2; ++ti) {
            if (ti >= p.ntensors)
                break;
            const TensorRef t = p.t[ti];                  // static index after unrolling
            const int32_t off = ti ? p.t[0].heads : 0;
            const int32_t lo = (hb > off ? hb : off) - off;
            const int32_t hi = (he < off + t.heads ? he : off + t.heads) - off;
            if (lo >= hi)
                continue;
            const int64_t o = b * t.stride_b + s * t.stride_s;
            const T *in0 = static_cast<const T *>(t.base) + o;
            T *out0 = static_cast<T *>(p.out[ti]) + o;
            rotate_heads<T, LAYOUT, U>(in0, out0, t.stride_h, lo, hi, j, NJ, c, sn, whole);
            if (p.copy_through[ti] && p.rotary_dim < p.D)  // pass the tail through
                copy_heads<T>(in0, out0, t.stride_h, lo, hi, j, NJ,
                              (p.rotary_dim * (int32_t)sizeof(T)) / 16,
                              (p.D * (int32_t)sizeof(T)) / 16);
        }
    }
}

// ---------------------------------------------------------------------------
// Element-wise kernel: any alignment and any even rotary_dim.  Rows are
// enumerated tensor by tensor as (b, head, s), s fastest; each row has
// rotary_dim/2 pair units and, out of place, D - rotary_dim tail units
// (copied).  One unit per loop iteration.
// ---------------------------------------------------------------------------
template <typename T, int LAYOUT>
__global__ void rope_scalar_kernel(const ApplyArgs p, int64_t rows0, int64_t total_units,
                                   int32_t units_per_row)
{
    const int h = p.rotary_dim >> 1;
    const int64_t stride = (int64_t)gridDim.x * blockDim.x;
    pdl_wait();
    pdl_trigger();
    for (int64_t idx = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; idx < total_units;
         idx += stride) {
        const int64_t unit = idx % units_per_row;
        int64_t row = idx / units_per_row;
        const int ti = row < rows0 ? 0 : 1;
        if (ti)
            row -= rows0;
        const int32_t heads = ti ? p.t[1].heads : p.t[0].heads;
        const int64_t sb = ti ? p.t[1].stride_b : p.t[0].stride_b;
        const int64_t sh = ti ? p.t[1].stride_h : p.t[0].stride_h;
        const int64_t ss = ti ? p.t[1].stride_s : p.t[0].stride_s;
        const int64_t s = row % p.S;
        row /= p.S;
        const int64_t head = row % heads;
        const int64_t b = row / heads;
        const int64_t o = b * sb + head * sh + s * ss;
        const T *x = static_cast<const T *>(ti ? p.t[1].base : p.t[0].base) + o;
        T *y = static_cast<T *>(ti ? p.out[1] : p.out[0]) + o;

        if (unit >= h) {                              // tail element, out of place only
            if (!(ti ? p.copy_through[1] : p.copy_through[0]))
                continue;
            const int64_t d = p.rotary_dim + (unit - h);
            y[d] = x[d];
            continue;
        }
        const int64_t i = unit;
        const int64_t i1 = LAYOUT == 0 ? i : 2 * i;
        const int64_t i2 = LAYOUT == 0 ? i + h : 2 * i + 1;
        int64_t r = s;
        if (p.pos_idx != nullptr) {
            r = __ldg(p.pos_idx + b * p.pos_stride_b + s);
            if (r == -1 || r < 0 || r >= p.table_rows) {
                if (r != -1 && i == 0)
                    atomicOr(p.range_flag, 1);
                if (ti ? p.copy_through[1] : p.copy_through[0]) {   // pass the pair through
                    y[i1] = x[i1];
                    y[i2] = x[i2];
                }
                continue;
            }
        }
        const float c = __ldg(p.cos + r * h + i);
        float sn = __ldg(p.sin + r * h + i);
        if (p.backward)
            sn = -sn;
        float x1 = Elt<T>::to_f(x[i1]);
        float x2 = Elt<T>::to_f(x[i2]);
        rotate_pair(x1, x2, c, sn);
        y[i1] = Elt<T>::from_f(x1);
        y[i2] = Elt<T>::from_f(x2);
    }
}

// ---------------------------------------------------------------------------
// SM count and resident CTAs per SM of a kernel on the current device, looked
// up once per device and pair layout and then cached.  The cache has internal
// linkage: each translation unit (one element type) keeps its own, and two
// copies of the library in one process never share one.
// ---------------------------------------------------------------------------
namespace {
constexpr int kCacheDevices = 64;
std::atomic<int> g_cache_sms[kCacheDevices];
constexpr int kVecInstances = 6;               // pair layout x (partial, whole, whole with NJ = 8)
std::atomic<int> g_cache_occ[kVecInstances][kCacheDevices];

// inst: the kernel instance, 0 .. kVecInstances - 1
cudaError_t resident_ctas(const void *kernel, int inst, int *sms, int *per_sm)
{
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess)
        return e;
    if (dev < 0 || dev >= kCacheDevices || inst < 0 || inst >= kVecInstances)
        return cudaErrorInvalidDevice;
    const int li = inst;
    int n = g_cache_sms[dev].load(std::memory_order_relaxed);
    int o = g_cache_occ[li][dev].load(std::memory_order_relaxed);
    if (n <= 0 || o <= 0) {
        e = cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
        if (e != cudaSuccess)
            return e;
        e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&o, kernel, kVecThreads, 0);
        if (e != cudaSuccess)
            return e;
        g_cache_sms[dev].store(n, std::memory_order_relaxed);
        g_cache_occ[li][dev].store(o, std::memory_order_relaxed);
    }
    *sms = n;
    *per_sm = o;
    return cudaSuccess;
}
}  // namespace

// ---------------------------------------------------------------------------
// Host-side launcher for one element type.
// ---------------------------------------------------------------------------
template <typename T>
cudaError_t launch_apply(const ApplyArgs &a, int32_t layout, Variant v, cudaStream_t st)
{
    if (v == kVector) {
        constexpr int V = Elt<T>::V;
        const int NJ = (a.rotary_dim / 2) / V;                 // vectors per half span
        const int TT = NJ >= 32 ? 1 : 32 / NJ;                 // tokens per lane group
        const int lgs = NJ >= kVecThreads ? 1 : (kVecThreads / NJ) / TT;   // lane groups per CTA
        const int TS = lgs * TT;                               // token rows per CTA
        const int32_t P = a.t[0].heads + (a.ntensors > 1 ? a.t[1].heads : 0);
        const int64_t tiles = (a.B * a.S + TT - 1) / TT;
        const int64_t units = tiles * P;
        // rotary spans that are whole rows of a multiple of 256 bytes; the
        // commonest of them (8 vectors per half: 16-bit D = 128, fp32 D = 64)
        // with NJ fixed at compile time
        const bool whole = a.rotary_dim == a.D && (a.D * (int32_t)sizeof(T)) % 256 == 0;
        const int kind = whole ? (NJ == 8 ? 2 : 1) : 0;
        using Kernel = void (*)(const ApplyArgs, int64_t, int32_t, int32_t);
        const Kernel kernels[2][3] = {
            {rope_vec_kernel<T, 0, kVecUnroll, false, 0>, rope_vec_kernel<T, 0, kVecUnroll, true, 0>,
             rope_vec_kernel<T, 0, kVecUnroll, true, 8>},
            {rope_vec_kernel<T, 1, kVecUnroll, false, 0>, rope_vec_kernel<T, 1, kVecUnroll, true, 0>,
             rope_vec_kernel<T, 1, kVecUnroll, true, 8>}};
        const Kernel kernel = kernels[layout ? 1 : 0][kind];
        // The grid.  Calls with at least one tile per lane group that can be
        // resident at once take one tile (all P heads of TT tokens) per lane
        // group, as many CTAs as that makes: the hardware hands the CTAs out
        // as resident ones finish, which balances the load better than a
        // fixed persistent split (measured).  Smaller calls cut their units
        // into as many balanced runs as there are resident lane groups (at
        // least one unit each), so a few tokens still occupy every SM.  The
        // tuning entry point can force the cap and the run length instead.
        const VecLaunchTuning tune = vec_launch_tuning();
        int sms = 0, per_sm = 0;
        cudaError_t e = resident_ctas(reinterpret_cast<const void *>(kernel),
                                      (layout ? 3 : 0) + kind, &sms, &per_sm);
        if (e != cudaSuccess)
            return e;
        const int64_t resident = (int64_t)sms * (per_sm > 0 ? per_sm : 1);
        const bool big = tiles >= resident * lgs;
        int64_t runs;
        if (tune.min_units > 0)
            runs = (units + tune.min_units - 1) / tune.min_units;
        else
            runs = big ? tiles : (units < resident * lgs ? units : resident * lgs);
        int64_t grid = (runs + lgs - 1) / lgs;
        const int64_t cap = tune.ctas_per_sm > 0 ? (int64_t)sms * tune.ctas_per_sm
                                                 : (big ? grid : resident);
        if (grid > cap)
            grid = cap;
        const int64_t min_grid = units / ((int64_t)lgs << 30) + 1;   // runs below 2^30 units
        if (grid < min_grid)
            grid = min_grid;
        if (grid > 0x7fffffffLL)
            grid = 0x7fffffffLL;
        return launch_hot(kernel, dim3((unsigned)grid), dim3(NJ, TS), 0, st, a, units, TT,
                          tune.prefetch_next >= 0 ? 1 : 0);
    }
    const int64_t rows0 = a.B * a.S * a.t[0].heads;
    const int64_t rows1 = a.ntensors > 1 ? a.B * a.S * a.t[1].heads : 0;
    const bool any_copy = a.copy_through[0] || (a.ntensors > 1 && a.copy_through[1]);
    const int32_t units_per_row = a.rotary_dim / 2 + (any_copy ? a.D - a.rotary_dim : 0);
    const int64_t total = (rows0 + rows1) * units_per_row;
    const int threads = 256;
    int64_t blocks = (total + threads - 1) / threads;
    if (blocks > 152LL * 64)
        blocks = 152LL * 64;                                   // grid-stride beyond this
    auto kernel = layout == 0 ? rope_scalar_kernel<T, 0> : rope_scalar_kernel<T, 1>;
    return launch_hot(kernel, dim3((unsigned)blocks), dim3(threads), 0, st, a, rows0, total,
                      units_per_row);
}

}  // namespace rope
