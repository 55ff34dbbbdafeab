// rope_attention.cuh -- attention forward with the rotation fused into the
// loads of the Q and K tiles, on the sm_103a tensor cores (tcgen05, TMEM, TMA).
//
// "rotary-embedding-torch", flash_attn_with_rotary: the rotary transformation
// is applied to the loaded blocks of Q and K inside the attention kernel, so
// the rotated tensors are never written back to global memory; GQA/MQA
// (heads_q != heads_kv), a causal mask and per-token positions (-1 = not
// rotated, the pos_mask) are supported.
//
//   O = softmax(scale * rot(Q) rot(K)^T + mask) V
//
// Three kernels share the helpers of this file:
//   * rope_attn_kernel (described here): the key tiles are rotated in shared
//     memory by every CTA that reads them (no key workspace);
//   * rope_attn_pp_kernel and rope_attn_2sm_kernel (described at their
//     definitions): the keys were rotated once beforehand into a workspace
//     by the rotation kernel; D = 64 and D = 128 (pairs of SMs).
//
// rope_attn_kernel: one CTA = two row blocks of 128 query rows that read the same key/value
// head: two query heads of one GQA group (same rows), or, when the group
// size is odd, two consecutive query tiles of one head.  288 threads: warps
// 4j .. 4j+3 own row block j (thread t: row t mod 128, which is also TMEM lane
// t mod 128 of block j's accumulators, S in columns [256j, 256j+128), O in
// [256j+128, 256j+128+D)); warp 8 issues every TMA copy and MMA.  The roles
// meet only through mbarriers, never a CTA-wide barrier inside the loop.
//
// Key tile kt, in shared memory:
//   * K rows arrive by TMA (cp.async.bulk.tensor, boxes of 64 elements x 128
//     rows, 128-byte swizzle: the K-major SW128 operand layout); the table
//     rows of the keys arrive the same way (boxes of 32 fp32 values), when
//     the keys sit at their own indices and rotary_dim is a multiple of 64.
//     Both are requested as soon as the previous tile's S is done, so their
//     latency hides behind that tile's softmax.
//   * The 256 row-block threads rotate the key tile in place (rotate_pair:
//     Kahan-compensated, one rounding to the element type, as in the
//     rotation kernels).
//   * Warp 8 issues S = Q K^T per row block (tcgen05.mma, fp32 in TMEM).
//   * Each thread reads its S row (tcgen05.ld), applies the mask and the
//     online softmax in the exp2 domain and writes P as bf16/fp16 back into
//     the first 64 columns of its S row (tcgen05.st); O is rescaled in TMEM
//     when the reference max moved.
//   * Warp 8 issues O += P V per row block with P read from TMEM and V (TMA,
//     two buffers, MN-major SW128) from shared memory.  That product overlaps
//     the next tile's rotation.
// The epilogue divides by the softmax sum and writes O.  Causal tiles past
// the diagonal are skipped.  Every mbarrier wait is bounded (~2 s of clock):
// a role whose wait expires raises a shared abort flag that ends the other
// roles' waits; warp 8 then waits (bounded) for its copies and MMAs in
// flight, TMEM is freed and the timeout flag is raised.
#pragma once

#include <atomic>
#include <cstring>
#include <type_traits>

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include "rope_kernels.cuh"

namespace rope {

constexpr int kAttnRows = 128;
constexpr int kAttnKeys = 128;
constexpr int kAttnBlocks = 2;                 // row blocks per CTA
constexpr int kMathThreads = kAttnRows * kAttnBlocks;   // row-block warps 0 .. 7
constexpr int kIssueWarp = kMathThreads / 32;              // warp 8: TMA and MMA issue
constexpr int kAttnThreads = kMathThreads + 32;
constexpr uint32_t kBlockCols = 256;           // TMEM columns of one row block (S + O)
constexpr uint32_t kTmemCols = kBlockCols * kAttnBlocks;
constexpr uint32_t kChunkBytes = kAttnKeys * 16;   // one 16-byte column of a 128-row tile
constexpr uint32_t kBoxBytes = kAttnKeys * 128;    // one 128-byte-wide swizzled box of 128 rows
constexpr uint32_t kSwizzle128 = 2;                // descriptor layout type: 128-byte swizzle
constexpr long long kAttnWaitCycles = 4000000000LL;

// Tensor maps of one call, all with 128-byte swizzle: K and V as
// [B * Hk][Sk][D] and Q as [B * Hq][Sq][D] (box: 64 elements x 128 rows; Q
// only for rope_attn_pp_kernel), the cos and sin tables as
// [table_rows][rotary_dim / 2] fp32 (box: 32 values x 128 rows).  A box lands
// as 128 rows of 128 bytes, the 16-byte chunk c of row r at chunk c ^ (r & 7).
struct AttnMaps {
    CUtensorMap k, v, cos, sin, q, o;             // o: rope_attn_2sm_kernel's output tiles
};

__device__ __forceinline__ uint32_t attn_smem_u32(const void *p)
{
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

// Shared-memory matrix descriptor.  Without swizzle (layout 0): core
// matrices of 8 rows x 16 bytes, K-major lbo = bytes between core matrices
// along K, sbo = along M/N.  128-byte swizzle (layout 2): K-major sbo = bytes
// between 8-row groups (lbo unused), the start moving 32 bytes per 16-element
// step inside a 64-element row; MN-major lbo = bytes between 64-element
// atoms along N, sbo = bytes between 8-row groups along K.
__device__ __forceinline__ uint64_t umma_desc(uint32_t saddr, uint32_t lbo, uint32_t sbo,
                                              uint32_t layout = 0)
{
    uint64_t d = 0;
    d |= (uint64_t)((saddr >> 4) & 0x3FFF);
    d |= (uint64_t)((lbo >> 4) & 0x3FFF) << 16;
    d |= (uint64_t)((sbo >> 4) & 0x3FFF) << 32;
    d |= (uint64_t)1 << 46;                        // descriptor version for tcgen05
    d |= (uint64_t)layout << 61;
    return d;
}

// Byte offset of 16-byte chunk c of row r in a 128-row tile of swizzled
// 128-byte-wide boxes (eight chunks per box row).
__device__ __forceinline__ uint32_t sw128(int r, int c)
{
    return (uint32_t)(c >> 3) * kBoxBytes + (uint32_t)r * 128u + (uint32_t)((c ^ r) & 7) * 16u;
}

// Instruction descriptor of kind::f16: fp32 accumulator, A and B of the same
// 16-bit type (bf16 = 1, f16 = 0), A K-major, B K-major or MN-major.
__device__ __forceinline__ uint32_t umma_idesc(int M, int N, uint32_t ab_format, int b_mn_major)
{
    return (1u << 4) | (ab_format << 7) | (ab_format << 10) | ((uint32_t)b_mn_major << 16) |
           ((uint32_t)(N >> 3) << 17) | ((uint32_t)(M >> 4) << 24);
}

// D (TMEM) (+)= A (shared memory) * B (shared memory)
__device__ __forceinline__ void umma_ss(uint32_t d_tmem, uint64_t a, uint64_t b, uint32_t idesc,
                                        uint32_t accumulate)
{
    asm volatile("{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
                 "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}"
                 ::"r"(d_tmem), "l"(a), "l"(b), "r"(idesc), "r"(accumulate)
                 : "memory");
}

// D (TMEM) (+)= A (TMEM: lane = row, two 16-bit elements per column, the
// even one in the low half) * B (shared memory)
__device__ __forceinline__ void umma_ts(uint32_t d_tmem, uint32_t a_tmem, uint64_t b,
                                        uint32_t idesc, uint32_t accumulate)
{
    asm volatile("{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
                 "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}"
                 ::"r"(d_tmem), "r"(a_tmem), "l"(b), "r"(idesc), "r"(accumulate)
                 : "memory");
}

__device__ __forceinline__ void umma_commit(uint64_t *bar)
{
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];"
                 ::"r"(attn_smem_u32(bar))
                 : "memory");
}

__device__ __forceinline__ void mbar_init(uint64_t *bar, uint32_t count)
{
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(attn_smem_u32(bar)), "r"(count)
                 : "memory");
}

__device__ __forceinline__ void mbar_expect_tx(uint64_t *bar, uint32_t bytes)
{
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;"
                 ::"r"(attn_smem_u32(bar)), "r"(bytes)
                 : "memory");
}

__device__ __forceinline__ void tma_load_3d(void *dst, const CUtensorMap *map, int x, int y, int z,
                                            uint64_t *bar)
{
    asm volatile("cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
                 " [%0], [%1, {%2, %3, %4}], [%5];"
                 ::"r"(attn_smem_u32(dst)), "l"(map), "r"(x), "r"(y), "r"(z),
                   "r"(attn_smem_u32(bar))
                 : "memory");
}

__device__ __forceinline__ void tma_load_2d(void *dst, const CUtensorMap *map, int x, int y,
                                            uint64_t *bar)
{
    asm volatile("cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
                 " [%0], [%1, {%2, %3}], [%4];"
                 ::"r"(attn_smem_u32(dst)), "l"(map), "r"(x), "r"(y), "r"(attn_smem_u32(bar))
                 : "memory");
}

// Bounded wait for the phase of the given parity; false on expiry (after
// `limit` clock cycles, ~2 s by default) or once another thread of the CTA
// has raised *abort.
__device__ __forceinline__ bool attn_wait(uint64_t *bar, uint32_t parity,
                                          const volatile int *abort = nullptr,
                                          long long limit = kAttnWaitCycles)
{
    const long long t0 = clock64();
    while (true) {
        uint32_t done;
        asm volatile("{\n\t.reg .pred p;\n\t"
                     "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
                     "selp.u32 %0, 1, 0, p;\n\t}"
                     : "=r"(done)
                     : "r"(attn_smem_u32(bar)), "r"(parity)
                     : "memory");
        if (done)
            return true;
        if ((abort != nullptr && *abort) || clock64() - t0 > limit)
            return false;
    }
}

__device__ __forceinline__ void mbar_arrive(uint64_t *bar)
{
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(attn_smem_u32(bar)) : "memory");
}

__device__ __forceinline__ void tmem_ld32(uint32_t addr, float (&v)[32])
{
    uint32_t r[32];
    asm volatile("tcgen05.ld.sync.aligned.32x32b.x32.b32 "
                 "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
                 "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]),
                   "=r"(r[6]), "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]),
                   "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]),
                   "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]),
                   "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]),
                   "=r"(r[30]), "=r"(r[31])
                 : "r"(addr)
                 : "memory");
    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
    for (int i = 0; i < 32; ++i)
        v[i] = __uint_as_float(r[i]);
}

// Like tmem_ld32 but without the wait: several loads can be in flight
// before one tcgen05.wait::ld.
__device__ __forceinline__ void tmem_ld32_nowait(uint32_t addr, float *v)
{
    uint32_t *r = reinterpret_cast<uint32_t *>(v);
    asm volatile("tcgen05.ld.sync.aligned.32x32b.x32.b32 "
                 "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
                 "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]),
                   "=r"(r[6]), "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]),
                   "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]),
                   "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]),
                   "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]),
                   "=r"(r[30]), "=r"(r[31])
                 : "r"(addr)
                 : "memory");
}

__device__ __forceinline__ void tmem_st32(uint32_t addr, const float (&v)[32])
{
    asm volatile("tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], "
                 "{%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,"
                 "%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32};"
                 ::"r"(addr), "r"(__float_as_uint(v[0])), "r"(__float_as_uint(v[1])),
                   "r"(__float_as_uint(v[2])), "r"(__float_as_uint(v[3])),
                   "r"(__float_as_uint(v[4])), "r"(__float_as_uint(v[5])),
                   "r"(__float_as_uint(v[6])), "r"(__float_as_uint(v[7])),
                   "r"(__float_as_uint(v[8])), "r"(__float_as_uint(v[9])),
                   "r"(__float_as_uint(v[10])), "r"(__float_as_uint(v[11])),
                   "r"(__float_as_uint(v[12])), "r"(__float_as_uint(v[13])),
                   "r"(__float_as_uint(v[14])), "r"(__float_as_uint(v[15])),
                   "r"(__float_as_uint(v[16])), "r"(__float_as_uint(v[17])),
                   "r"(__float_as_uint(v[18])), "r"(__float_as_uint(v[19])),
                   "r"(__float_as_uint(v[20])), "r"(__float_as_uint(v[21])),
                   "r"(__float_as_uint(v[22])), "r"(__float_as_uint(v[23])),
                   "r"(__float_as_uint(v[24])), "r"(__float_as_uint(v[25])),
                   "r"(__float_as_uint(v[26])), "r"(__float_as_uint(v[27])),
                   "r"(__float_as_uint(v[28])), "r"(__float_as_uint(v[29])),
                   "r"(__float_as_uint(v[30])), "r"(__float_as_uint(v[31]))
                 : "memory");
}

__device__ __forceinline__ void tmem_st16(uint32_t addr, const uint32_t (&v)[16])
{
    asm volatile("tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], "
                 "{%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16};"
                 ::"r"(addr), "r"(v[0]), "r"(v[1]), "r"(v[2]), "r"(v[3]), "r"(v[4]), "r"(v[5]),
                   "r"(v[6]), "r"(v[7]), "r"(v[8]), "r"(v[9]), "r"(v[10]), "r"(v[11]),
                   "r"(v[12]), "r"(v[13]), "r"(v[14]), "r"(v[15])
                 : "memory");
}

// 2^x with the SFU's approximate exponential (relative error ~2^-22, far
// below the bf16/fp16 rounding of P that follows).
__device__ __forceinline__ float fast_exp2(float x)
{
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// Byte offset of element (r, k) in a K-major no-swizzle tile of 128 rows.
__device__ __forceinline__ uint32_t kmajor128(int r, int k)
{
    return (uint32_t)(k >> 3) * kChunkBytes + (uint32_t)(r >> 3) * 128u + (uint32_t)(r & 7) * 16u +
           (uint32_t)(k & 7) * 2u;
}

// Table row of a token: its index, or its position; -1 when not rotated.
__device__ __forceinline__ int64_t attn_row(const int32_t *pos, int64_t s, int64_t table_rows,
                                            int32_t *flag, bool report = true)
{
    if (pos == nullptr)
        return s;
    const int64_t r = __ldg(pos + s);
    if (r == -1)
        return -1;
    if (r < 0 || r >= table_rows) {
        if (report)
            atomicOr(flag, 1);
        return -1;
    }
    return r;
}

// Warp-cooperative load of the 32 query-tile rows [32 * warp, 32 * warp + 32)
// from global memory, rotated.  Lane l takes row (l & 7) of an 8-row group and
// chunk (l >> 3) of a group of four 16-byte chunks, so every shared-memory
// store instruction writes four runs of 128 contiguous bytes (8 rows of one
// chunk): no bank conflicts.  Each pass issues the loads of all four rows of
// the lane (data and table) before any arithmetic.  Rows whose token index
// (tok0 + row) is not below n_tok are stored as zeros.  The first rotary_dim
// features are rotated with the row's table row (its position; -1 = not
// rotated): split-half pairs a chunk with its partner chunk (+ rd/16),
// interleaved pairs sit inside one chunk.  Features past rotary_dim are copied.
template <typename T, int LAYOUT, int D>
__device__ __forceinline__ void warp_load_tile(const T *rows, int64_t tok0, int64_t n_tok,
                                               const int32_t *pos, const AttnArgs &a, uint8_t *tile,
                                               int warp, int lane)
{
    constexpr int CPR = D / 8;                     // 16-byte chunks per row
    constexpr int G = 4;                           // 8-row groups per warp
    const int rr = lane & 7, cc = lane >> 3;
    const int rd = a.rotary_dim;
    const int h = rd >> 1;
    const int h8 = rd / 16;                        // chunks per half span
    int r[G];
    bool valid[G];
    int64_t trow[G];
    const uint4 *src[G];
#pragma unroll
    for (int g = 0; g < G; ++g) {
        r[g] = warp * 32 + g * 8 + rr;
        valid[g] = tok0 + r[g] < n_tok;
        src[g] = reinterpret_cast<const uint4 *>(rows + (int64_t)r[g] * D);
        trow[g] = valid[g] ? attn_row(pos, tok0 + r[g], a.table_rows, a.flag, cc == 0) : -1;
    }
    const int rot_chunks = LAYOUT == 0 ? h8 : rd / 8;
#pragma unroll 1
    for (int c = cc; c < rot_chunks; c += 4) {
        if constexpr (LAYOUT == 0) {
            uint4 x1[G], x2[G];
            float4 cv[G][2], sv[G][2];
#pragma unroll
            for (int g = 0; g < G; ++g) {
                x1[g] = valid[g] ? __ldg(src[g] + c) : make_uint4(0, 0, 0, 0);
                x2[g] = valid[g] ? __ldg(src[g] + c + h8) : make_uint4(0, 0, 0, 0);
                const int64_t tr = trow[g] < 0 ? 0 : trow[g];
#pragma unroll
                for (int q = 0; q < 2; ++q) {
                    cv[g][q] = __ldg(reinterpret_cast<const float4 *>(a.cos + tr * h + c * 8) + q);
                    sv[g][q] = __ldg(reinterpret_cast<const float4 *>(a.sin + tr * h + c * 8) + q);
                }
            }
#pragma unroll
            for (int g = 0; g < G; ++g) {
                uint4 y1 = x1[g], y2 = x2[g];
                if (trow[g] >= 0) {
                    float f1[8], f2[8];
                    const float cs[8] = {cv[g][0].x, cv[g][0].y, cv[g][0].z, cv[g][0].w,
                                         cv[g][1].x, cv[g][1].y, cv[g][1].z, cv[g][1].w};
                    const float sn[8] = {sv[g][0].x, sv[g][0].y, sv[g][0].z, sv[g][0].w,
                                         sv[g][1].x, sv[g][1].y, sv[g][1].z, sv[g][1].w};
                    Elt<T>::unpack(x1[g], f1);
                    Elt<T>::unpack(x2[g], f2);
#pragma unroll
                    for (int e = 0; e < 8; ++e)
                        rotate_pair(f1[e], f2[e], cs[e], sn[e]);
                    y1 = Elt<T>::pack(f1);
                    y2 = Elt<T>::pack(f2);
                }
                *reinterpret_cast<uint4 *>(tile + kmajor128(r[g], c * 8)) = y1;
                *reinterpret_cast<uint4 *>(tile + kmajor128(r[g], (c + h8) * 8)) = y2;
            }
        } else {
            uint4 x[G];
            float4 cv[G], sv[G];
#pragma unroll
            for (int g = 0; g < G; ++g) {
                x[g] = valid[g] ? __ldg(src[g] + c) : make_uint4(0, 0, 0, 0);
                const int64_t tr = trow[g] < 0 ? 0 : trow[g];
                cv[g] = __ldg(reinterpret_cast<const float4 *>(a.cos + tr * h + c * 4));
                sv[g] = __ldg(reinterpret_cast<const float4 *>(a.sin + tr * h + c * 4));
            }
#pragma unroll
            for (int g = 0; g < G; ++g) {
                uint4 y = x[g];
                if (trow[g] >= 0) {
                    float f[8];
                    Elt<T>::unpack(x[g], f);
                    rotate_pair(f[0], f[1], cv[g].x, sv[g].x);
                    rotate_pair(f[2], f[3], cv[g].y, sv[g].y);
                    rotate_pair(f[4], f[5], cv[g].z, sv[g].z);
                    rotate_pair(f[6], f[7], cv[g].w, sv[g].w);
                    y = Elt<T>::pack(f);
                }
                *reinterpret_cast<uint4 *>(tile + kmajor128(r[g], c * 8)) = y;
            }
        }
    }
    // chunks copied unchanged: past the rotary span
#pragma unroll 1
    for (int c = rd / 8 + cc; c < CPR; c += 4) {
        uint4 x[G];
#pragma unroll
        for (int g = 0; g < G; ++g)
            x[g] = valid[g] ? __ldg(src[g] + c) : make_uint4(0, 0, 0, 0);
#pragma unroll
        for (int g = 0; g < G; ++g)
            *reinterpret_cast<uint4 *>(tile + kmajor128(r[g], c * 8)) = x[g];
    }
}

// One (row, chunk) item of the key-tile rotation: the data chunk(s), their
// shared-memory offsets and the cos/sin values.
struct KeyItem {
    uint4 x1, x2;
    uint32_t o1, o2;
    float cs[8], sn[8];
    bool rot;
};

// Loads item i of a tile rotation (row i mod 128, chunk i / 128) from a
// tile of swizzled boxes whose row r holds token k0 + r of a sequence of S
// tokens with positions pos (NULL: the token index).
template <typename T, int LAYOUT, bool STAGED>
__device__ __forceinline__ void load_key_item(KeyItem &it, int i, const uint8_t *sK,
                                              const uint8_t *sT, int64_t k0, const int32_t *pos,
                                              int64_t S, const AttnArgs &a)
{
    constexpr int NQ = LAYOUT == 0 ? 2 : 1;        // float4 table reads per item
    const int rd = a.rotary_dim, h = rd >> 1, h8 = rd / 16;
    const int r = i & (kAttnKeys - 1), p = i >> 7;
    it.o1 = sw128(r, p);
    it.o2 = sw128(r, p + h8);
    it.x1 = *reinterpret_cast<const uint4 *>(sK + it.o1);
    if (LAYOUT == 0)
        it.x2 = *reinterpret_cast<const uint4 *>(sK + it.o2);
    it.rot = true;
    if constexpr (STAGED) {
        const uint8_t *sC = sT, *sS = sT + (size_t)(rd / 64) * kBoxBytes;
#pragma unroll
        for (int q = 0; q < NQ; ++q) {
            const float4 c4 = *reinterpret_cast<const float4 *>(sC + sw128(r, NQ * p + q));
            const float4 s4 = *reinterpret_cast<const float4 *>(sS + sw128(r, NQ * p + q));
            it.cs[4 * q] = c4.x; it.cs[4 * q + 1] = c4.y; it.cs[4 * q + 2] = c4.z; it.cs[4 * q + 3] = c4.w;
            it.sn[4 * q] = s4.x; it.sn[4 * q + 1] = s4.y; it.sn[4 * q + 2] = s4.z; it.sn[4 * q + 3] = s4.w;
        }
    } else {
        const int64_t tok = k0 + r;
        const int64_t tr = tok < S ? attn_row(pos, tok, a.table_rows, a.flag, p == 0) : -1;
        it.rot = tr >= 0;
        const int64_t trc = tr < 0 ? 0 : tr;
        const float4 *cr = reinterpret_cast<const float4 *>(a.cos + trc * h + p * 4 * NQ);
        const float4 *sr = reinterpret_cast<const float4 *>(a.sin + trc * h + p * 4 * NQ);
#pragma unroll
        for (int q = 0; q < NQ; ++q) {
            const float4 c4 = __ldg(cr + q);
            const float4 s4 = __ldg(sr + q);
            it.cs[4 * q] = c4.x; it.cs[4 * q + 1] = c4.y; it.cs[4 * q + 2] = c4.z; it.cs[4 * q + 3] = c4.w;
            it.sn[4 * q] = s4.x; it.sn[4 * q + 1] = s4.y; it.sn[4 * q + 2] = s4.z; it.sn[4 * q + 3] = s4.w;
        }
    }
}

// Rotates a loaded item and writes it back (unrotated rows stay as they are).
template <typename T, int LAYOUT>
__device__ __forceinline__ void store_key_item(KeyItem &it, uint8_t *sK)
{
    if (!it.rot)
        return;
    if constexpr (LAYOUT == 0) {
        float f1[8], f2[8];
        Elt<T>::unpack(it.x1, f1);
        Elt<T>::unpack(it.x2, f2);
#pragma unroll
        for (int e = 0; e < 8; ++e)
            rotate_pair(f1[e], f2[e], it.cs[e], it.sn[e]);
        *reinterpret_cast<uint4 *>(sK + it.o1) = Elt<T>::pack(f1);
        *reinterpret_cast<uint4 *>(sK + it.o2) = Elt<T>::pack(f2);
    } else {
        float f[8];
        Elt<T>::unpack(it.x1, f);
#pragma unroll
        for (int e = 0; e < 4; ++e)
            rotate_pair(f[2 * e], f[2 * e + 1], it.cs[e], it.sn[e]);
        *reinterpret_cast<uint4 *>(sK + it.o1) = Elt<T>::pack(f);
    }
}

// Rotates a 128-row tile in place (rows k0 .. k0 + 127 of a sequence of S
// tokens with positions pos, in swizzled 128-byte boxes as the TMA left them;
// rows past S hold zeros) by NT threads, tid in [0, NT).  Item i = (row i mod
// 128, chunk i / 128): consecutive lanes take consecutive rows of one chunk,
// which the swizzle spreads over eight distinct 16-byte bank groups.  NF
// items are loaded before any is rotated.  STAGED: the tokens sit at their
// own indices and their table rows were staged the same way next to the
// tile (cos: rd / 64 boxes, then sin); otherwise each row's position is read
// and its table row fetched from global memory.
template <typename T, int LAYOUT, bool STAGED, int NT, int NF>
__device__ __forceinline__ void rotate_tile(uint8_t *sK, const uint8_t *sT, int64_t k0,
                                            const int32_t *pos, int64_t S, const AttnArgs &a,
                                            int tid)
{
    const int per_row = LAYOUT == 0 ? a.rotary_dim / 16 : a.rotary_dim / 8;
    const int items = kAttnKeys * per_row;
#pragma unroll 1
    for (int i = tid; i < items; i += NF * NT) {
        KeyItem x[NF];
#pragma unroll
        for (int f = 0; f < NF; ++f)
            if (f == 0 || i + f * NT < items)
                load_key_item<T, LAYOUT, STAGED>(x[f], i + f * NT, sK, sT, k0, pos, S, a);
#pragma unroll
        for (int f = 0; f < NF; ++f)
            if (f == 0 || i + f * NT < items)
                store_key_item<T, LAYOUT>(x[f], sK);
    }
}

// Issue warp: request key tile k0 (and its staged table rows) into sK / sT,
// completion on bar.  Lane 0 arms the barrier with the byte count first.
template <int D, bool STAGED>
__device__ __forceinline__ void issue_key_tile(const AttnMaps &m, uint8_t *sK, uint8_t *sT, int k0,
                                               int zkv, int tboxes, uint64_t *bar, int lane)
{
    const uint32_t bytes = (uint32_t)(D / 64) * kBoxBytes + (STAGED ? 2u * tboxes * kBoxBytes : 0u);
    if (lane == 0)
        mbar_expect_tx(bar, bytes);
    __syncwarp();
    if (lane < D / 64)
        tma_load_3d(sK + lane * kBoxBytes, &m.k, lane * 64, k0, zkv, bar);
    if (STAGED && lane >= 8 && lane < 8 + 2 * tboxes) {
        const int t = lane - 8;
        const bool is_cos = t < tboxes;
        tma_load_2d(sT + t * kBoxBytes, is_cos ? &m.cos : &m.sin, (is_cos ? t : t - tboxes) * 32,
                    k0, bar);
    }
}

// Issue warp: request value tile k0 into sV (MN-major SW128: columns 64 b ..
// 64 b + 63 in box b, key r at row r), completion on bar.
template <int D>
__device__ __forceinline__ void issue_value_tile(const AttnMaps &m, uint8_t *sV, int k0, int zkv,
                                                 uint64_t *bar, int lane)
{
    if (lane == 0)
        mbar_expect_tx(bar, (uint32_t)(D / 64) * kBoxBytes);
    __syncwarp();
    if (lane < D / 64)
        tma_load_3d(sV + lane * kBoxBytes, &m.v, lane * 64, k0, zkv, bar);
}

// The work of one CTA (or CTA pair) on query tile qtile of (batch, head)
// unit `unit`: batch b and key/value head zkv = b * Hk + hk; row
// block j holds query head hq_first + j * hq_step, rows q0_first + j * q_step
// .. + 127 (two query heads of one GQA group when pair_heads, else two
// consecutive query tiles of one head); n_tiles = the key tiles those rows
// can see.  The one-unit-per-CTA kernels take unit = blockIdx.x and the query
// tiles last first along blockIdx.y: the hardware hands out blocks x fastest,
// so under a causal mask every CTA of the longest query tiles starts before
// any of the shorter ones (longest job first; the short ones fill the end).
struct AttnWork {
    int64_t b, q0_first, q_step, n_tiles;
    int32_t hq_first, hq_step, zkv;
};

__device__ __forceinline__ AttnWork attn_work(const AttnArgs &a, int32_t pair_heads,
                                              uint32_t unit, int64_t qtile)
{
    AttnWork w;
    if (pair_heads) {
        const int32_t pairs = a.Hq / 2;
        w.b = unit / pairs;
        w.hq_first = (int32_t)(unit - w.b * pairs) * 2;
        w.hq_step = 1;
        w.q0_first = qtile * kAttnRows;
        w.q_step = 0;
    } else {
        w.b = unit / a.Hq;
        w.hq_first = (int32_t)(unit - w.b * a.Hq);
        w.hq_step = 0;
        w.q0_first = qtile * 2 * kAttnRows;
        w.q_step = kAttnRows;
    }
    w.zkv = (int32_t)(w.b * a.Hk + w.hq_first / (a.Hq / a.Hk));
    const int64_t shift = a.Sk - a.Sq;             // bottom-right aligned causal mask
    w.n_tiles = (a.Sk + kAttnKeys - 1) / kAttnKeys;
    if (a.causal) {
        int64_t last_row = w.q0_first + (kAttnBlocks - 1) * w.q_step + kAttnRows - 1;
        if (last_row > a.Sq - 1)
            last_row = a.Sq - 1;
        const int64_t last = last_row + shift;     // last key visible to the CTA
        const int64_t t = last < 0 ? 0 : last / kAttnKeys + 1;
        if (t < w.n_tiles)
            w.n_tiles = t;
    }
    // key tiles past the last key the batch entry's attn_mask shows hold only
    // hidden keys: every role reads the same count, so all skip them alike
    if (a.kv_tiles != nullptr) {
        const int64_t t = __ldg(a.kv_tiles + w.b);
        if (t < w.n_tiles)
            w.n_tiles = t;
    }
    return w;
}

// Packed pairs of fp32 values (Blackwell's f32x2 arithmetic: one instruction
// for two lanes' worth of fma or add, each rounded as its scalar form).
__device__ __forceinline__ uint64_t f32x2(float lo, float hi)
{
    uint64_t r;
    asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(lo), "f"(hi));
    return r;
}

__device__ __forceinline__ void f32x2_split(uint64_t r, float &lo, float &hi)
{
    asm("mov.b64 {%0, %1}, %2;" : "=f"(lo), "=f"(hi) : "l"(r));
}

__device__ __forceinline__ uint64_t fma_f32x2(uint64_t a, uint64_t b, uint64_t c)
{
    uint64_t d;
    asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
    return d;
}

__device__ __forceinline__ uint64_t add_f32x2(uint64_t a, uint64_t b)
{
    uint64_t d;
    asm("add.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
    return d;
}

// max(a, b, c) in one instruction
__device__ __forceinline__ float fmax3(float a, float b, float c)
{
    float d;
    asm("max.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
    return d;
}

// One online-softmax step of query row qi on the key tile at k0.  The row's
// S = Q K^T sits in TMEM columns [acc, acc + 128) of its lane and its O in
// [o_base, o_base + D).  The 128 S values are read once and held in
// registers.  Computes the row max over the visible keys, moves the lazy
// reference max m_ref when needed, writes P = 2^(s * scale * log2(e) -
// m_ref) as packed 16-bit values over the first 64 columns of S, updates the
// running sum l_run and rescales O when the reference moved (not on the first
// tile: O holds nothing yet).  The max and the sum keep eight and four
// partial results, so no long chain of dependent instructions sets the
// latency.  Warp-collective; the caller waits for the TMEM stores before
// signalling that P is ready.
//
// PACKED: the scale-and-subtract and the partial sums use f32x2 pairs (one
// instruction per two keys); otherwise the same operations one lane at a
// time, in the same order, so both forms give the same bits (the scalar one
// needs fewer registers: rope_attn_kernel, whose key rotation holds more
// values live, would spill with the pairs).
struct ONoWait {
    __device__ __forceinline__ bool operator()() const { return true; }
};

// Bytes b0..b3 of x that are nonzero, as bits 0..3.
__device__ __forceinline__ uint32_t nonzero_bytes4(uint32_t x)
{
    // 0x80 in each nonzero byte, moved to bit 0 of its byte; one multiply
    // then gathers bits 0, 8, 16, 24 into bits 21..24 (no two partial
    // products overlap, so nothing carries)
    const uint32_t t = (__vcmpne4(x, 0u) & 0x80808080u) >> 7;
    return (t * 0x00204081u) >> 21 & 0xFu;
}

// attn_mask of the 128 keys k0 .. k0 + 127 for query row qi of batch b
// (warp-collective): bit (i & 31) of vis[i >> 5] set when key k0 + i is
// visible.  Keys at or past Sk, and rows at or past Sq, read as visible (the
// tile's key count and the row's own bound hide them).
//   a.mask_kind 1, [B, Sk]: lane l reads keys k0 + 32e + l (e = 0..3), four
//     coalesced 32-byte reads shared by every row of the batch, and a ballot
//     per e gives word e to all lanes;
//   a.mask_kind 2, [B, Sq, Sk]: each row reads its own 128 bytes, as eight
//     16-byte vectors when the rows are 16-byte aligned (a.mask_vec16), else
//     byte by byte.
// The softmax step calls it after the tensor-memory loads of S: holding the
// mask's bytes across them costs registers the step does not have (spills),
// and an L1 prefetch of the next tile's bytes one step ahead measured slower
// than none.
__device__ __forceinline__ void mask_bits(const AttnArgs &a, int64_t b, int64_t qi, int64_t k0,
                                          uint32_t (&vis)[4])
{
    if (a.mask_kind == 1) {
        const int lane = threadIdx.x & 31;
        const uint8_t *row = a.mask + b * a.Sk;
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            const int64_t kk = k0 + 32 * e + lane;
            const bool on = kk >= a.Sk || __ldg(row + kk) != 0;
            vis[e] = __ballot_sync(0xffffffffu, on);
        }
        return;
    }
#pragma unroll
    for (int e = 0; e < 4; ++e)
        vis[e] = 0xffffffffu;
    if (qi >= a.Sq)
        return;
    const uint8_t *row = a.mask + (b * a.Sq + qi) * a.Sk + k0;
    const int64_t nk = a.Sk - k0;                   // keys of this row from k0 on
    if (a.mask_vec16) {
#pragma unroll
        for (int c = 0; c < 8; ++c) {               // chunk c: keys 16c .. 16c + 15
            if (16 * c < nk) {
                const uint4 x = __ldg(reinterpret_cast<const uint4 *>(row) + c);
                const uint32_t m16 = nonzero_bytes4(x.x) | nonzero_bytes4(x.y) << 4 |
                                     nonzero_bytes4(x.z) << 8 | nonzero_bytes4(x.w) << 12;
                vis[c >> 1] &= ~(0xFFFFu << (16 * (c & 1))) | (m16 << (16 * (c & 1)));
            }
        }
    } else {
#pragma unroll 8
        for (int i = 0; i < kAttnKeys; ++i) {
            if (i < nk && row[i] == 0)
                vis[i >> 5] &= ~(1u << (i & 31));
        }
    }
}

// sk: keys the row may see at most (a [B, Sk] mask that shows a prefix of
// the keys), -1: all Sk.
template <typename T, int D, bool PACKED, bool MASK, typename OReady = ONoWait>
__device__ __forceinline__ void softmax_tile(uint32_t acc_base, uint32_t o_base, int64_t qi,
                                             int64_t k0, int64_t shift, const AttnArgs &a,
                                             int64_t b, bool not_first, float &m_ref,
                                             float &l_run, const OReady &o_ready = OReady(),
                                             int64_t sk = -1)
{
    // columns of this tile visible to this row: [0, nvis)
    int64_t vis_end = sk >= 0 ? sk : a.Sk;   // first invisible key
    if (a.causal && qi + shift + 1 < vis_end)
        vis_end = qi + shift + 1;
    const int64_t nv = vis_end - k0;
    const int nvis = nv < 0 ? 0 : (nv > kAttnKeys ? kAttnKeys : (int)nv);
    const bool full = __all_sync(0xffffffffu, nvis == kAttnKeys);   // no causal/length mask
    float sv[kAttnKeys];
#pragma unroll
    for (int c0 = 0; c0 < kAttnKeys; c0 += 32)
        tmem_ld32_nowait(acc_base + c0, sv + c0);
    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
    uint32_t vis[4];
    bool unmasked = true;                  // no attn_mask bit clear in this tile
    if constexpr (MASK) {
        mask_bits(a, b, qi, k0, vis);
        unmasked = __all_sync(0xffffffffu, (vis[0] & vis[1] & vis[2] & vis[3]) == 0xffffffffu);
    }
    if (!full) {
#pragma unroll
        for (int i = 0; i < kAttnKeys; ++i)
            sv[i] = i < nvis ? sv[i] : -INFINITY;  // masked keys: 2^-inf = 0 below
    }
    if constexpr (MASK) {
        if (!unmasked) {
#pragma unroll
            for (int i = 0; i < kAttnKeys; ++i)
                sv[i] = (vis[i >> 5] >> (i & 31)) & 1u ? sv[i] : -INFINITY;
        }
    }
    float m8[8];
#pragma unroll
    for (int r = 0; r < 8; ++r)
        m8[r] = sv[r];
#pragma unroll
    for (int i = 8; i < kAttnKeys; i += 2)
        m8[(i >> 1) & 7] = fmax3(m8[(i >> 1) & 7], sv[i], sv[i + 1]);
    float mx = fmax3(fmax3(m8[0], m8[1], m8[2]), fmax3(m8[3], m8[4], m8[5]), fmaxf(m8[6], m8[7]));
    mx *= a.scale_log2;                    // scale > 0: max commutes with it
    // The exponentials use a reference max m_ref that only moves when the
    // row max exceeds it by more than 8 (factor 256): P stays <= 256, exact
    // in fp32 and bf16/fp16 range, and O is rescaled only then.
    float alpha = 1.0f;
    if (mx > m_ref + 8.0f) {
        alpha = m_ref == -INFINITY ? 0.0f : fast_exp2(m_ref - mx);
        m_ref = mx;
    }
    // m_ref is -inf only while the row has seen no visible key; every key
    // of this tile is then masked (-inf) and gives 2^-inf = 0
    const float neg_m = m_ref == -INFINITY ? 0.0f : -m_ref;
    // s * scale - m and the partial sums of the even and the odd keys,
    // four of each
    uint32_t w[kAttnKeys / 2];
    float s4[4];
    if constexpr (PACKED) {
        const uint64_t scale2 = f32x2(a.scale_log2, a.scale_log2), neg_m2 = f32x2(neg_m, neg_m);
        uint64_t sum2[4] = {0, 0, 0, 0};           // (even, odd) pairs of +0.0f
#pragma unroll
        for (int i = 0; i < kAttnKeys; i += 2) {
            float t0, t1;
            f32x2_split(fma_f32x2(f32x2(sv[i], sv[i + 1]), scale2, neg_m2), t0, t1);
            const float p0 = fast_exp2(t0);
            const float p1 = fast_exp2(t1);
            sum2[(i >> 1) & 3] = add_f32x2(sum2[(i >> 1) & 3], f32x2(p0, p1));
            w[i >> 1] = Elt<T>::f2_to_word(p0, p1);
        }
#pragma unroll
        for (int r = 0; r < 4; ++r) {
            float e, o;
            f32x2_split(sum2[r], e, o);
            s4[r] = e + o;
        }
    } else {
        float se[4] = {0.0f, 0.0f, 0.0f, 0.0f}, so[4] = {0.0f, 0.0f, 0.0f, 0.0f};
#pragma unroll
        for (int i = 0; i < kAttnKeys; i += 2) {
            const float p0 = fast_exp2(fmaf(sv[i], a.scale_log2, neg_m));
            const float p1 = fast_exp2(fmaf(sv[i + 1], a.scale_log2, neg_m));
            se[(i >> 1) & 3] += p0;
            so[(i >> 1) & 3] += p1;
            w[i >> 1] = Elt<T>::f2_to_word(p0, p1);
        }
#pragma unroll
        for (int r = 0; r < 4; ++r)
            s4[r] = se[r] + so[r];
    }
    // keys 2c, 2c + 1 -> column c (the even key in the low half)
#pragma unroll
    for (int c = 0; c < kAttnKeys / 2; c += 16)
        tmem_st16(acc_base + c, *reinterpret_cast<const uint32_t(*)[16]>(w + c));
    l_run = l_run * alpha + ((s4[0] + s4[1]) + (s4[2] + s4[3]));
    // rescale O rows of this warp; o_ready() waits until no product still
    // writes O (a warp-uniform false, its wait expired, skips the rescale)
    if (not_first && __any_sync(0xffffffffu, alpha != 1.0f) && o_ready()) {
        asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
#pragma unroll 1
        for (int c0 = 0; c0 < D; c0 += 32) {
            float ov[32];
            tmem_ld32(o_base + c0, ov);
#pragma unroll
            for (int i = 0; i < 32; ++i)
                ov[i] *= alpha;
            tmem_st32(o_base + c0, ov);
        }
    }
}

// Epilogue of query row qi: O / l from TMEM columns [o_base, o_base + D),
// rounded once, to the row of O (zeros when the row saw no key).  TMEM
// loads are warp-wide; rows at or past Sq store nothing.
template <typename T, int D>
__device__ __forceinline__ void store_o_row(uint32_t o_base, T *O, int64_t qi, int64_t Sq,
                                            bool any_key, float l_run)
{
    const float inv = (any_key && l_run > 0.0f) ? 1.0f / l_run : 0.0f;
    uint4 *dst = reinterpret_cast<uint4 *>(O + qi * D);
#pragma unroll
    for (int c0 = 0; c0 < D; c0 += 32) {
        float ov[32];
        if (any_key) {
            tmem_ld32(o_base + c0, ov);
        } else {
#pragma unroll
            for (int i = 0; i < 32; ++i)
                ov[i] = 0.0f;
        }
        if (qi < Sq) {
#pragma unroll
            for (int c = 0; c < 4; ++c) {
                float f[8];
#pragma unroll
                for (int e = 0; e < 8; ++e)
                    f[e] = ov[c * 8 + e] * inv;
                dst[(c0 + c * 8) / 8] = Elt<T>::pack(f);
            }
        }
    }
}

// Row r of a 128-row output block, as store_o_row computes it, into a
// staging tile of D / 64 swizzled 128-byte boxes (features 0 .. 63, then
// 64 .. 127) for a TMA store: in each 16-byte store of a warp, the rows r and
// r + 8 share a bank group and the eight row residues fill all eight, the
// fewest shared-memory wavefronts for 512 bytes.
template <typename T, int D>
__device__ __forceinline__ void stage_o_row(uint32_t o_base, uint8_t *sO, int r, bool any_key,
                                            float l_run)
{
    const float inv = (any_key && l_run > 0.0f) ? 1.0f / l_run : 0.0f;
#pragma unroll
    for (int c0 = 0; c0 < D; c0 += 32) {
        float ov[32];
        if (any_key) {
            tmem_ld32(o_base + c0, ov);
        } else {
#pragma unroll
            for (int i = 0; i < 32; ++i)
                ov[i] = 0.0f;
        }
#pragma unroll
        for (int c = 0; c < 4; ++c) {
            float f[8];
#pragma unroll
            for (int e = 0; e < 8; ++e)
                f[e] = ov[c * 8 + e] * inv;
            *reinterpret_cast<uint4 *>(sO + sw128(r, c0 / 8 + c)) = Elt<T>::pack(f);
        }
    }
}

// TMA store of one swizzled box from shared memory (bulk-group completion).
// Rows past the tensor's extent are not written.
__device__ __forceinline__ void tma_store_3d(const CUtensorMap *map, const void *src, int x, int y,
                                             int z)
{
    asm volatile("cp.async.bulk.tensor.3d.global.shared::cta.bulk_group [%0, {%2, %3, %4}], [%1];"
                 ::"l"(map), "r"(attn_smem_u32(src)), "r"(x), "r"(y), "r"(z)
                 : "memory");
}

// Epilogue of one row warp (warp-collective): its 32 rows 32 wq .. 32 wq + 31
// of a 128-row output block (row r of this thread) staged in the block's
// 128 x D staging tile sO once the warp's previous store from it has read
// it, then one TMA store per 64 features from lane 0 (a 64 x 32 box of map:
// O as [B Hq][Sq][D]).  where(q0, z) gives the block's first query row and
// its output head; it is called after the staging (fewer values live across
// it).  Only the warp's own bulk group is waited for, so no warp waits on
// another.
template <typename T, int D, typename Where>
__device__ __forceinline__ void store_o_warp(const CUtensorMap *map, uint32_t o_base, uint8_t *sO,
                                             int r, int wq, int64_t Sq, bool any_key, float l_run,
                                             const Where &where)
{
    const bool lead = (threadIdx.x & 31) == 0;
    if (lead)
        asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory");
    __syncwarp();
    stage_o_row<T, D>(o_base, sO, r, any_key, l_run);
    // O's columns are read (the caller's next tensor-core work may follow)
    // and the staged rows are visible to the copy engine
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
    __syncwarp();
    int64_t q0;
    int z;
    where(q0, z);
    const int64_t y0 = q0 + wq * 32;
    if (lead && y0 < Sq) {
#pragma unroll
        for (int bx = 0; bx < D / 64; ++bx)
            tma_store_3d(map, sO + bx * kBoxBytes + wq * 32 * 128, bx * 64, (int)y0, z);
        asm volatile("cp.async.bulk.commit_group;" ::: "memory");
    }
}

// Before a CTA ends: the warp's output stores have completed.
__device__ __forceinline__ void drain_o_stores()
{
    if ((threadIdx.x & 31) == 0)
        asm volatile("cp.async.bulk.wait_group 0;" ::: "memory");
    __syncwarp();
}

template <typename T, int LAYOUT, int D, bool STAGED, bool MASK>
__global__ void __launch_bounds__(kAttnThreads, 1)
    rope_attn_kernel(const AttnArgs a, const __grid_constant__ AttnMaps maps, const int32_t pair_heads)
{
    constexpr uint32_t kTile = kAttnRows * D * 2;  // bytes of a 128 x D tile
    constexpr uint32_t ab_format = std::is_same<T, __nv_bfloat16>::value ? 1u : 0u;
    extern __shared__ __align__(1024) uint8_t smem[];
    // [Q_0][Q_1][K][V_0][V_1][table staging]
    uint8_t *sQ = smem;
    uint8_t *sK = sQ + kAttnBlocks * kTile;
    uint8_t *sV = sK + kTile;
    uint8_t *sT = sV + 2 * kTile;
    // completions: key tile + table landed (TMA), value tile landed (TMA, per
    // buffer), S ready and O += P V done (MMA commits, per row block), key
    // tile rotated (the kMathThreads row-block threads arrive) and P ready
    // (the block's 128 threads arrive)
    __shared__ __align__(8) uint64_t bar_k, bar_v[2], bar_s[2], bar_o[2], bar_krot, bar_p[2];
    __shared__ uint32_t tmem_base;
    __shared__ int abort_flag;

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const bool math = warp < kIssueWarp;           // a row-block warp (else the issue warp)
    const int j = math ? warp >> 2 : 0;            // row block of this warp
    const int wq = warp & 3;                       // TMEM lane quarter
    const int row = tid & (kAttnRows - 1);
    const AttnWork w = attn_work(a, pair_heads, blockIdx.x, gridDim.y - 1 - blockIdx.y);
    const int32_t hq = w.hq_first + j * w.hq_step;
    const int zkv = w.zkv;
    const int64_t q0 = w.q0_first + j * w.q_step;
    const int64_t qi = q0 + row;
    const T *Qh = static_cast<const T *>(a.q) + ((w.b * a.Hq + hq) * a.Sq) * D;
    T *O = static_cast<T *>(a.o) + ((w.b * a.Hq + hq) * a.Sq) * D;
    const int tboxes = a.rotary_dim / 64;          // table boxes of cos (and of sin)
    const int64_t shift = a.Sk - a.Sq;             // bottom-right aligned causal mask
    const int64_t n_tiles = w.n_tiles;

    if (warp == 0) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;"
                     ::"r"(attn_smem_u32(&tmem_base)), "r"(kTmemCols)
                     : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    }
    if (tid == 0) {
        mbar_init(&bar_k, 1);
        mbar_init(&bar_v[0], 1);
        mbar_init(&bar_v[1], 1);
        for (int blk = 0; blk < kAttnBlocks; ++blk) {
            mbar_init(&bar_s[blk], 1);
            mbar_init(&bar_o[blk], 1);
            mbar_init(&bar_p[blk], kAttnRows);
        }
        mbar_init(&bar_krot, kMathThreads);
        abort_flag = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    __syncthreads();
    // the first key tile and the first two value tiles, while Q is loaded
    if (warp == kIssueWarp && n_tiles > 0) {
        issue_key_tile<D, STAGED>(maps, sK, sT, 0, zkv, tboxes, &bar_k, lane);
        issue_value_tile<D>(maps, sV, 0, zkv, &bar_v[0], lane);
        if (n_tiles > 1)
            issue_value_tile<D>(maps, sV + kTile, kAttnKeys, zkv, &bar_v[1], lane);
    }
    // the query tile of each row block, rotated (by that block's four warps)
    if (math)
        warp_load_tile<T, LAYOUT, D>(Qh + q0 * D, q0, a.Sq, a.pos_q, a, sQ + j * kTile, wq, lane);
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
    __syncthreads();
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
    const uint32_t tmem = tmem_base;
    volatile int *abort = &abort_flag;
    bool ok = true;

    if (math) {
        // ---- row-block warps: rotate each key tile, then the softmax of row qi
        const uint32_t acc_base = tmem + (uint32_t)j * kBlockCols + ((uint32_t)(wq * 32) << 16);
        float m_ref = -INFINITY, l_run = 0.0f;     // reference max (log2 domain), sum
        uint32_t ph = 0;                           // parity of tile kt's phases
        for (int64_t kt = 0; kt < n_tiles; ++kt, ph ^= 1) {
            const int64_t k0 = kt * kAttnKeys;
            // 1. the key tile (and its table rows) has landed: rotate it in place
            ok = __all_sync(0xffffffffu, attn_wait(&bar_k, ph, abort));
            if (!ok)
                break;
            // one item at a time: with the softmax's 128 S values this
            // kernel has no registers left for a second item in flight
            rotate_tile<T, LAYOUT, STAGED, kMathThreads, 1>(sK, sT, k0, a.pos_k, a.Sk, a, tid);
            asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
            mbar_arrive(&bar_krot);
            // 2. this block's S = Q K^T is ready; its O += P V of the previous
            //    tile has finished (the issue warp waits for it before S)
            ok = __all_sync(0xffffffffu, attn_wait(&bar_s[j], ph, abort) &&
                                             (kt == 0 || attn_wait(&bar_o[j], ph ^ 1, abort)));
            if (!ok)
                break;
            asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
            // 3. online softmax; P goes back into TMEM over S
            softmax_tile<T, D, false, MASK>(acc_base, acc_base + kAttnKeys, qi, k0, shift, a, w.b,
                                      kt > 0, m_ref, l_run);
            asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
            asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
            mbar_arrive(&bar_p[j]);
        }
        // the last O += P V
        if (ok && n_tiles > 0)
            ok = __all_sync(0xffffffffu, attn_wait(&bar_o[j], ph ^ 1, abort));
        asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
        if (!ok) {
            *abort = 1;
        } else if (n_tiles > 0) {
            // epilogue: O / l of the warp's rows, staged in the block's query
            // tile (no S product reads it any more) and stored by TMA
            store_o_warp<T, D>(&maps.o, acc_base + kAttnKeys, sQ + j * kTile, row, wq, a.Sq, true,
                               l_run, [&](int64_t &q0r, int &z) {
                                   q0r = q0;
                                   z = (int)(w.b * a.Hq + hq);
                               });
            drain_o_stores();
        } else {
            // no key tile (nor, without keys, a tensor map): zeros
            store_o_row<T, D>(acc_base + kAttnKeys, O, qi, a.Sq, false, l_run);
        }
    } else {
        // ---- issue warp: TMA copies one tile ahead, the MMAs (lane 0)
        const uint32_t idesc_s = umma_idesc(128, kAttnKeys, ab_format, 0);
        const uint32_t idesc_o = umma_idesc(128, D, ab_format, 1);
        // copies in flight (bar_k; bar_v bit b) and the parities they complete
        // next; every commit covers all earlier MMAs, so the last one covers them all
        bool pend_k = n_tiles > 0, pend_mma = false;
        uint32_t pend_v = (n_tiles > 0 ? 1u : 0u) | (n_tiles > 1 ? 2u : 0u);
        uint32_t ph_k = 0, ph_v = 0, last_ph = 0;
        uint64_t *last_bar = &bar_s[0];
        for (int64_t kt = 0; kt < n_tiles; ++kt) {
            const int64_t k0 = kt * kAttnKeys;
            const bool next = kt + 1 < n_tiles;
            const uint32_t ph = (uint32_t)(kt & 1);
            // the key tile is rotated
            ok = __all_sync(0xffffffffu, attn_wait(&bar_krot, ph, abort));
            if (!ok)
                break;
            ph_k ^= 1;                             // the math warps waited for it
            pend_k = false;
            // S = Q K^T per row block, once the block's previous O += P V has
            // finished (P shares S's columns)
            for (int blk = 0; blk < kAttnBlocks; ++blk) {
                if (kt > 0) {
                    ok = __all_sync(0xffffffffu, attn_wait(&bar_o[blk], ph ^ 1, abort));
                    if (!ok)
                        break;
                }
                asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
                if (lane == 0) {
#pragma unroll
                    for (int kk = 0; kk < D / 16; ++kk)
                        umma_ss(tmem + blk * kBlockCols,
                                umma_desc(attn_smem_u32(sQ + blk * kTile) + kk * 2u * kChunkBytes,
                                          kChunkBytes, 128u),
                                umma_desc(attn_smem_u32(sK) + (kk >> 2) * kBoxBytes + (kk & 3) * 32u,
                                          16u, 1024u, kSwizzle128),
                                idesc_s, kk > 0);
                    umma_commit(&bar_s[blk]);
                }
                __syncwarp();
                pend_mma = true;
                last_bar = &bar_s[blk];
                last_ph = ph;
            }
            if (!ok)
                break;
            // the value tile after the next one, into the buffer both products
            // of the previous tile have released
            if (next && kt > 0) {
                issue_value_tile<D>(maps, sV + ((kt + 1) & 1) * kTile, (int)(k0 + kAttnKeys), zkv,
                                    &bar_v[(kt + 1) & 1], lane);
                pend_v |= 1u << ((kt + 1) & 1);
            }
            // both S are ready: the key buffer and the table staging are free
            ok = __all_sync(0xffffffffu, attn_wait(&bar_s[kAttnBlocks - 1], ph, abort));
            if (!ok)
                break;
            if (next) {
                issue_key_tile<D, STAGED>(maps, sK, sT, (int)(k0 + kAttnKeys), zkv, tboxes, &bar_k,
                                          lane);
                pend_k = true;
            }
            // O += P V per row block as its P becomes ready
            const int vb = (int)(kt & 1);
            ok = __all_sync(0xffffffffu, attn_wait(&bar_v[vb], (ph_v >> vb) & 1u, abort));
            if (!ok)
                break;
            ph_v ^= 1u << vb;
            pend_v &= ~(1u << vb);
            const uint32_t v_addr = attn_smem_u32(sV + vb * kTile);
            for (int blk = 0; blk < kAttnBlocks; ++blk) {
                ok = __all_sync(0xffffffffu, attn_wait(&bar_p[blk], ph, abort));
                if (!ok)
                    break;
                asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
                if (lane == 0) {
#pragma unroll
                    for (int kk = 0; kk < kAttnKeys / 16; ++kk)
                        umma_ts(tmem + blk * kBlockCols + kAttnKeys, tmem + blk * kBlockCols + kk * 8,
                                umma_desc(v_addr + kk * 2048u, kBoxBytes, 1024u, kSwizzle128),
                                idesc_o, (kt > 0 || kk > 0) ? 1u : 0u);
                    umma_commit(&bar_o[blk]);
                }
                __syncwarp();
                last_bar = &bar_o[blk];
                last_ph = ph;
            }
            if (!ok)
                break;
        }
        if (ok && pend_mma) {
            ok = __all_sync(0xffffffffu, attn_wait(last_bar, last_ph, abort));
            if (ok)
                pend_mma = false;
        }
        if (!ok) {
            *abort = 1;
            // give every copy and MMA still in flight one more bounded wait
            if (pend_k)
                (void)attn_wait(&bar_k, ph_k);
            if (pend_mma)
                (void)attn_wait(last_bar, last_ph);
            if (pend_v & 1u)
                (void)attn_wait(&bar_v[0], ph_v & 1u);
            if (pend_v & 2u)
                (void)attn_wait(&bar_v[1], (ph_v >> 1) & 1u);
        }
    }
    // every role has left its loop; a copy or an MMA that did not complete in
    // time is reported and nothing was written
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
    __syncthreads();
    if (tid == 0 && abort_flag)
        atomicOr(a.flag, 2);
    if (warp == 0)
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem),
                     "r"(kTmemCols)
                     : "memory");
}

// ---------------------------------------------------------------------------
// Attention over keys rotated beforehand (rope_attention_fwd with a key
// workspace: the rotation kernel writes rot(K) there once per call, so no
// CTA spends issue slots rotating key tiles).  Q is still rotated as its
// tile is loaded.  Freed of the joint key rotation, the two row blocks run
// out of step: while one block's warps compute the softmax of a key tile,
// the tensor cores run the other block's products.
//
// 352 threads: warps 0-7 the two row blocks (as in rope_attn_kernel), warps
// 8 and 9 issue the MMAs of row block 0 and 1, warp 10 the TMA copies.  One
// issuing warp per block: a warp that issues MMAs stalls while the tensor
// pipe is full, and a shared issuer would hold one block's ready P behind
// the other block's products.  Shared memory: Q_0, Q_1, two key stages, two
// value stages (6 tiles of 128 x D).  Block j's issuer runs, per key tile kt,
//   O_j += P_j V(kt) (once P_j is in TMEM); S_j = Q_j K(kt+1) (once that
//   product has finished: P_j sits in the columns S_j overwrites)
// and both issuers release a key or value stage (arrival count 2).  Every
// wait is bounded as in rope_attn_kernel.
// ---------------------------------------------------------------------------
constexpr int kPpMmaWarp = kMathThreads / 32;      // warps 8, 9: MMA issue of blocks 0, 1
constexpr int kPpTmaWarp = kPpMmaWarp + kAttnBlocks;   // warp 10
constexpr int kPpThreads = kMathThreads + 32 * (kAttnBlocks + 1);
constexpr int kPpStages = 2;                       // key and value stages

template <typename T, int LAYOUT, int D, bool STAGED_Q, bool MASK>
__global__ void __launch_bounds__(kPpThreads, 1)
    rope_attn_pp_kernel(const AttnArgs a, const __grid_constant__ AttnMaps maps,
                        const int32_t pair_heads)
{
    constexpr uint32_t kTile = kAttnRows * D * 2;  // bytes of a 128 x D tile
    constexpr uint32_t ab_format = std::is_same<T, __nv_bfloat16>::value ? 1u : 0u;
    extern __shared__ __align__(1024) uint8_t smem[];
    // [Q_0][Q_1][K stage 0][V stage 0][K stage 1][V stage 1].  STAGED_Q: the
    // table rows of the query tiles (both blocks hold the same rows) land in
    // stage 1 first (cos: rd / 64 boxes, then sin; at most 2 tiles' bytes),
    // which receives its key and value tiles once Q is rotated.
    uint8_t *sQ = smem;
    uint8_t *sKV = sQ + kAttnBlocks * kTile;
    auto sK = [&](int stage) { return sKV + stage * 2 * kTile; };
    auto sV = [&](int stage) { return sKV + stage * 2 * kTile + kTile; };
    const int tboxes = a.rotary_dim / 64;          // table boxes of cos (and of sin)
    // stage landed (TMA) / stage free (one MMA commit from each issuer), per
    // stage; S ready and O += P V done (MMA commits), P ready (the block's
    // 128 threads), per block
    __shared__ __align__(8) uint64_t bar_kfull[kPpStages], bar_kfree[kPpStages],
        bar_vfull[kPpStages], bar_vfree[kPpStages], bar_s[kAttnBlocks], bar_o[kAttnBlocks],
        bar_p[kAttnBlocks], bar_q, bar_sm[kAttnBlocks];
    __shared__ uint32_t tmem_base;
    __shared__ int abort_flag;

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const bool math = warp < kPpMmaWarp;
    const int j = math ? warp >> 2 : 0;
    const int wq = warp & 3;
    const int row = tid & (kAttnRows - 1);
    const AttnWork w = attn_work(a, pair_heads, blockIdx.x, gridDim.y - 1 - blockIdx.y);
    const int32_t hq = w.hq_first + j * w.hq_step;
    const int64_t q0 = w.q0_first + j * w.q_step;
    const int64_t qi = q0 + row;
    T *O = static_cast<T *>(a.o) + ((w.b * a.Hq + hq) * a.Sq) * D;
    const int64_t shift = a.Sk - a.Sq;
    const int64_t n_tiles = w.n_tiles;

    if (warp == 0) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;"
                     ::"r"(attn_smem_u32(&tmem_base)), "r"(kTmemCols)
                     : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    }
    if (tid == 0) {
        for (int s = 0; s < kPpStages; ++s) {
            mbar_init(&bar_kfull[s], 1);
            mbar_init(&bar_kfree[s], kAttnBlocks);
            mbar_init(&bar_vfull[s], 1);
            mbar_init(&bar_vfree[s], kAttnBlocks);
        }
        for (int blk = 0; blk < kAttnBlocks; ++blk) {
            mbar_init(&bar_s[blk], 1);
            mbar_init(&bar_o[blk], 1);
            mbar_init(&bar_p[blk], kAttnRows);
            mbar_init(&bar_sm[blk], kAttnRows);
        }
        mbar_init(&bar_q, 1);
        abort_flag = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    __syncthreads();
    // both query tiles (and their table rows), then the key and value tiles
    // of stage 0 (and of stage 1 when it holds no table rows)
    const int64_t first_stages = STAGED_Q ? 1 : kPpStages;
    if (warp == kPpTmaWarp) {
        constexpr int kBoxes = D / 64;             // 64-element boxes per row
        if (lane == 0)
            mbar_expect_tx(&bar_q, (uint32_t)(kAttnBlocks * kBoxes + (STAGED_Q ? 2 * tboxes : 0)) *
                                       kBoxBytes);
        __syncwarp();
        if (lane < kAttnBlocks * kBoxes) {
            const int blk = lane / kBoxes, box = lane % kBoxes;
            tma_load_3d(sQ + blk * kTile + box * kBoxBytes, &maps.q, box * 64,
                        (int)(w.q0_first + blk * w.q_step),
                        (int)(w.b * a.Hq + w.hq_first + blk * w.hq_step), &bar_q);
        }
        if (STAGED_Q && lane >= 8 && lane < 8 + 2 * tboxes) {
            const int t = lane - 8;
            const bool is_cos = t < tboxes;
            tma_load_2d(sK(1) + t * kBoxBytes, is_cos ? &maps.cos : &maps.sin,
                        (is_cos ? t : t - tboxes) * 32, (int)w.q0_first, &bar_q);
        }
        for (int64_t kt = 0; kt < first_stages && kt < n_tiles; ++kt) {
            issue_key_tile<D, false>(maps, sK((int)kt), nullptr, (int)(kt * kAttnKeys), w.zkv, 0,
                                     &bar_kfull[kt], lane);
            issue_value_tile<D>(maps, sV((int)kt), (int)(kt * kAttnKeys), w.zkv, &bar_vfull[kt],
                                lane);
        }
    }
    // each row block rotates its query tile in place (rows past Sq: zeros)
    bool q_ok = true;
    if (math) {
        q_ok = __all_sync(0xffffffffu, attn_wait(&bar_q, 0u));
        if (q_ok)
            rotate_tile<T, LAYOUT, STAGED_Q, kAttnRows, 1>(sQ + j * kTile, sK(1), q0, a.pos_q,
                                                           a.Sq, a, row);
        else
            abort_flag = 1;
    }
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
    __syncthreads();
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
    const uint32_t tmem = tmem_base;
    volatile int *abort = &abort_flag;
    bool ok = !*abort;                             // false: the query tiles never landed

    if (math) {
        // ---- row-block warps: the softmax of row qi, tile after tile
        const uint32_t acc_base = tmem + (uint32_t)j * kBlockCols + ((uint32_t)(wq * 32) << 16);
        float m_ref = -INFINITY, l_run = 0.0f;
        // the key tiles; M: the softmax reads the attn_mask's bytes, else the
        // row sees at most the first sk keys (-1: all)
        auto key_tiles = [&](auto m_tag, int64_t sk) {
            constexpr bool M = decltype(m_tag)::value;
            for (int64_t kt = 0; kt < n_tiles; ++kt) {
                // S of this block is ready (its previous O += P V has finished:
                // the issuer waited for it before issuing S), and it is this
                // block's turn: the softmax steps alternate between the blocks
                // (block 0 on tile kt after block 1 on tile kt - 1, block 1 after
                // block 0 on the same tile), so each has the exponential unit to
                // itself while the tensor cores run the other block's products
                ok = __all_sync(0xffffffffu,
                                attn_wait(&bar_s[j], (uint32_t)(kt & 1), abort) &&
                                    (j == 0 ? kt == 0 || attn_wait(&bar_sm[1], (uint32_t)((kt - 1) & 1),
                                                                   abort)
                                            : attn_wait(&bar_sm[0], (uint32_t)(kt & 1), abort)));
                if (!ok)
                    break;
                asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
                softmax_tile<T, D, true, M>(acc_base, acc_base + kAttnKeys, qi, kt * kAttnKeys, shift, a,
                                      w.b, kt > 0, m_ref, l_run, ONoWait(), sk);
                mbar_arrive(&bar_sm[j]);
                asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
                asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
                mbar_arrive(&bar_p[j]);
            }
        };
        if constexpr (MASK) {
            // a [B, Sk] mask that shows exactly the keys [0, L) of this batch
            // entry (padding): the unmasked softmax over L keys
            const int64_t len = a.kv_len != nullptr ? __ldg(a.kv_len + w.b) : -1;
            if (len >= 0)
                key_tiles(std::false_type(), len);
            else
                key_tiles(std::true_type(), (int64_t)-1);
        } else {
            key_tiles(std::false_type(), (int64_t)-1);
        }
        // the last O += P V
        if (ok && n_tiles > 0)
            ok = __all_sync(0xffffffffu,
                            attn_wait(&bar_o[j], (uint32_t)((n_tiles - 1) & 1), abort));
        asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
        if (!ok) {
            *abort = 1;
        } else if (n_tiles > 0) {
            // O / l of the warp's rows, staged in the block's query tile (no
            // S product reads it any more) and stored by TMA
            store_o_warp<T, D>(&maps.o, acc_base + kAttnKeys, sQ + j * kTile, row, wq, a.Sq, true,
                               l_run, [&](int64_t &q0r, int &z) {
                                   q0r = q0;
                                   z = (int)(w.b * a.Hq + hq);
                               });
            drain_o_stores();
        } else {
            store_o_row<T, D>(acc_base + kAttnKeys, O, qi, a.Sq, false, l_run);
        }
    } else if (warp < kPpTmaWarp) {
        // ---- MMA issue of row block jb (lane 0 issues; the waits are warp-wide)
        const int jb = warp - kPpMmaWarp;
        const uint32_t idesc_s = umma_idesc(128, kAttnKeys, ab_format, 0);
        const uint32_t idesc_o = umma_idesc(128, D, ab_format, 1);
        const uint32_t acc = tmem + (uint32_t)jb * kBlockCols;
        const uint32_t q_addr = attn_smem_u32(sQ + jb * kTile);
        uint64_t *last_bar = nullptr;              // the last commit covers every MMA before it
        uint32_t last_ph = 0;
        // S = Q_jb K(stage), completion on bar_s[jb]; releases the key stage
        auto issue_s = [&](int stage) {
            if (lane == 0) {
                const uint32_t k_addr = attn_smem_u32(sK(stage));
#pragma unroll
                for (int kk = 0; kk < D / 16; ++kk)
                    umma_ss(acc,
                            umma_desc(q_addr + (kk >> 2) * kBoxBytes + (kk & 3) * 32u, 16u, 1024u,
                                      kSwizzle128),
                            umma_desc(k_addr + (kk >> 2) * kBoxBytes + (kk & 3) * 32u, 16u, 1024u,
                                      kSwizzle128),
                            idesc_s, kk > 0);
                umma_commit(&bar_s[jb]);
                umma_commit(&bar_kfree[stage]);
            }
            __syncwarp();
        };
        if (n_tiles > 0) {
            ok = __all_sync(0xffffffffu, attn_wait(&bar_kfull[0], 0u, abort));
            if (ok) {
                asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
                issue_s(0);
                last_bar = &bar_s[jb];
                last_ph = 0;
            }
        }
        for (int64_t kt = 0; ok && kt < n_tiles; ++kt) {
            const int st = (int)(kt % kPpStages);
            const uint32_t use_ph = (uint32_t)((kt / kPpStages) & 1);
            const int nst = (int)((kt + 1) % kPpStages);
            const uint32_t nuse_ph = (uint32_t)(((kt + 1) / kPpStages) & 1);
            // O_jb += P_jb V(kt) once the value tile has landed and P is in TMEM
            ok = __all_sync(0xffffffffu, attn_wait(&bar_vfull[st], use_ph, abort) &&
                                             attn_wait(&bar_p[jb], (uint32_t)(kt & 1), abort));
            if (!ok)
                break;
            asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
            if (lane == 0) {
                const uint32_t v_addr = attn_smem_u32(sV(st));
#pragma unroll
                for (int kk = 0; kk < kAttnKeys / 16; ++kk)
                    umma_ts(acc + kAttnKeys, acc + kk * 8,
                            umma_desc(v_addr + kk * 2048u, kBoxBytes, 1024u, kSwizzle128), idesc_o,
                            (kt > 0 || kk > 0) ? 1u : 0u);
                umma_commit(&bar_o[jb]);
                umma_commit(&bar_vfree[st]);
            }
            __syncwarp();
            last_bar = &bar_o[jb];
            last_ph = (uint32_t)(kt & 1);
            if (kt + 1 >= n_tiles)
                break;
            // S_jb of the next key tile, once that tile has landed and this
            // block's O += P V has released the columns of P
            ok = __all_sync(0xffffffffu, attn_wait(&bar_kfull[nst], nuse_ph, abort) &&
                                             attn_wait(&bar_o[jb], (uint32_t)(kt & 1), abort));
            if (!ok)
                break;
            asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
            issue_s(nst);
            last_bar = &bar_s[jb];
            last_ph = (uint32_t)((kt + 1) & 1);
        }
        if (ok && last_bar != nullptr)
            ok = __all_sync(0xffffffffu, attn_wait(last_bar, last_ph, abort));
        if (!ok) {
            *abort = 1;
            if (last_bar != nullptr)
                (void)attn_wait(last_bar, last_ph);   // the MMAs in flight
        }
    } else {
        // ---- TMA warp: tile kt into stage kt mod 2 once the products of
        // tile kt - 2 have released it
        int64_t k_last[kPpStages], v_last[kPpStages];   // last tile copied into a stage (-1: none)
#pragma unroll
        for (int s = 0; s < kPpStages; ++s) {
            k_last[s] = s < n_tiles && s < first_stages ? s : -1;
            v_last[s] = k_last[s];
        }
        // stage 1 held the query tiles' table rows until the rotation above
        for (int64_t kt = first_stages; ok && kt < kPpStages && kt < n_tiles; ++kt) {
            issue_key_tile<D, false>(maps, sK((int)kt), nullptr, (int)(kt * kAttnKeys), w.zkv, 0,
                                     &bar_kfull[kt], lane);
            issue_value_tile<D>(maps, sV((int)kt), (int)(kt * kAttnKeys), w.zkv, &bar_vfull[kt],
                                lane);
            k_last[kt] = v_last[kt] = kt;
        }
        for (int64_t kt = kPpStages; ok && kt < n_tiles; ++kt) {
            const int st = (int)(kt % kPpStages);
            const uint32_t free_ph = (uint32_t)(((kt / kPpStages) - 1) & 1);
            ok = __all_sync(0xffffffffu, attn_wait(&bar_kfree[st], free_ph, abort));
            if (!ok)
                break;
            issue_key_tile<D, false>(maps, sK(st), nullptr, (int)(kt * kAttnKeys), w.zkv, 0,
                                     &bar_kfull[st], lane);
            k_last[st] = kt;
            ok = __all_sync(0xffffffffu, attn_wait(&bar_vfree[st], free_ph, abort));
            if (!ok)
                break;
            issue_value_tile<D>(maps, sV(st), (int)(kt * kAttnKeys), w.zkv, &bar_vfull[st],
                                lane);
            v_last[st] = kt;
        }
        if (!ok) {
            *abort = 1;
            // one more bounded wait for the query tiles and the last copies
            // into each stage
            (void)attn_wait(&bar_q, 0u);
#pragma unroll
            for (int s = 0; s < kPpStages; ++s) {
                if (k_last[s] >= 0)
                    (void)attn_wait(&bar_kfull[s], (uint32_t)((k_last[s] / kPpStages) & 1));
                if (v_last[s] >= 0)
                    (void)attn_wait(&bar_vfull[s], (uint32_t)((v_last[s] / kPpStages) & 1));
            }
        }
    }
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
    __syncthreads();
    if (tid == 0 && abort_flag)
        atomicOr(a.flag, 2);
    if (warp == 0)
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem),
                     "r"(kTmemCols)
                     : "memory");
}

// ---------------------------------------------------------------------------
// Attention over keys rotated beforehand, on pairs of SMs (a cluster of two
// CTAs and tcgen05 MMAs with cta_group::2: M = 256, the two CTAs' row blocks
// stacked).  Each CTA owns one 128-row block (two heads of a GQA group, or
// two consecutive query tiles of one head, as the row blocks of
// rope_attn_pp_kernel) and holds half of every key tile (64 keys) and half of
// every value tile (64 of the 128 feature columns); the leader CTA (rank 0)
// issues the MMAs of both.  One instruction now covers 256 rows, half as
// many per flop as with M = 128, and with one row block per CTA its TMEM has
// room for three S buffers: S(kt + 1) and S(kt + 2) are computed while the
// softmax of S(kt) runs, and no S waits for the previous O += P V.
//
// 224 threads per CTA: warps 0-3 the row block (thread t = row t), warp 4 the
// leader's S issue, warp 5 the leader's O += P V issue, warp 6 the TMA copies
// of its CTA (the follower's count their bytes on the leader's barriers).
// TMEM columns: S buffers at 0, 128 and 256, O at 384.  Shared memory: the query
// tile, three stages of (key half, value half), the query tile's table rows.
// The CTAs meet through mbarriers: multicast MMA commits reach both, the
// follower's arrivals and copies reach the leader's barriers.  Every wait is
// bounded; a role whose wait expires raises the abort flag of both CTAs.
// ---------------------------------------------------------------------------
constexpr int k2Stages = 3;
constexpr int k2SIssueWarp = 4;                    // leader: S issue
constexpr int k2PVIssueWarp = 5;
constexpr int k2TmaWarp = 6;
constexpr int k2Threads = 7 * 32;
constexpr int k2SBufs = 3;                         // S buffers in TMEM
constexpr uint32_t k2OCol = k2SBufs * kAttnKeys;   // TMEM column of O (384)
constexpr uint32_t k2Half = 16384;                 // bytes of a CTA's half key or value tile
// Key / value stage g mod 3 is released by the commits that complete S
// buffer g mod 3 (S(g) has read the key half) and its O barrier (O += P V
// has read the value half): one commit per issuing thread and tile.
static_assert(k2Stages == k2SBufs, "stages and S buffers advance together");

__device__ __forceinline__ uint32_t peer_addr(const void *p, uint32_t cta)
{
    uint32_t r;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(attn_smem_u32(p)), "r"(cta));
    return r;
}

// Arrival on a barrier of the peer CTA (default semantics: release at CTA
// scope; a cluster-scope release fence costs ~1.4 k cycles inside this
// kernel).  Used after tcgen05.wait::st and tcgen05.fence::before_thread_sync
// (the tensor-memory stores it announces have completed) or after
// fence.proxy.async (the shared-memory stores are visible to the tensor cores).
__device__ __forceinline__ void mbar_arrive_remote(uint32_t cluster_addr)
{
    asm volatile("mbarrier.arrive.shared::cluster.b64 _, [%0];" ::"r"(cluster_addr) : "memory");
}

// TMA load into this CTA's shared memory whose completion (bytes) is
// counted on a barrier of the CTA pair's leader (cluster address).
__device__ __forceinline__ void tma_load_3d_to_leader(void *dst, const CUtensorMap *map, int x, int y,
                                                      int z, uint32_t leader_bar)
{
    asm volatile("cp.async.bulk.tensor.3d.cta_group::2.shared::cluster.global.tile.mbarrier::"
                 "complete_tx::bytes [%0], [%1, {%2, %3, %4}], [%5];"
                 ::"r"(attn_smem_u32(dst)), "l"(map), "r"(x), "r"(y), "r"(z), "r"(leader_bar)
                 : "memory");
}

__device__ __forceinline__ void umma2_ss(uint32_t d_tmem, uint64_t a, uint64_t b, uint32_t idesc,
                                         uint32_t accumulate)
{
    asm volatile("{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
                 "tcgen05.mma.cta_group::2.kind::f16 [%0], %1, %2, %3, p;\n\t}"
                 ::"r"(d_tmem), "l"(a), "l"(b), "r"(idesc), "r"(accumulate)
                 : "memory");
}

__device__ __forceinline__ void umma2_ts(uint32_t d_tmem, uint32_t a_tmem, uint64_t b,
                                         uint32_t idesc, uint32_t accumulate)
{
    asm volatile("{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
                 "tcgen05.mma.cta_group::2.kind::f16 [%0], [%1], %2, %3, p;\n\t}"
                 ::"r"(d_tmem), "r"(a_tmem), "l"(b), "r"(idesc), "r"(accumulate)
                 : "memory");
}

// Commit of the issuing thread's earlier MMAs to the barrier at the same
// shared-memory offset in every CTA of cta_mask.
__device__ __forceinline__ void umma2_commit(uint64_t *bar, uint16_t cta_mask)
{
    asm volatile("tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.multicast::"
                 "cluster.b64 [%0], %1;"
                 ::"r"(attn_smem_u32(bar)), "h"(cta_mask)
                 : "memory");
}

__device__ __forceinline__ void cluster_sync_all()
{
    asm volatile("barrier.cluster.arrive.release.aligned;\n\t"
                 "barrier.cluster.wait.acquire.aligned;" ::: "memory");
}

template <typename T, int LAYOUT, bool STAGED_Q, bool MASK>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(k2Threads, 1)
    rope_attn_2sm_kernel(const AttnArgs a, const __grid_constant__ AttnMaps maps,
                         const int32_t pair_heads)
{
    constexpr int D = 128;
    constexpr uint32_t kTile = kAttnRows * D * 2;  // the query tile
    constexpr uint32_t ab_format = std::is_same<T, __nv_bfloat16>::value ? 1u : 0u;
    extern __shared__ __align__(1024) uint8_t smem[];
    uint8_t *sQ = smem;
    uint8_t *sStages = sQ + kTile;
    uint8_t *sT = sStages + k2Stages * 2 * k2Half;     // the query tile's table rows
    uint8_t *sO = sT + 4 * kBoxBytes;                  // the output block, staged for TMA
    auto sK = [&](int st) { return sStages + st * 2 * k2Half; };
    auto sV = [&](int st) { return sStages + st * 2 * k2Half + k2Half; };
    // both CTAs' key / value halves landed (leader only: TMA bytes of both);
    // S buffer ready, which also releases key stage b (multicast); P
    // ready (leader only: each row warp of both CTAs arrives); the O += P V
    // that read P from S buffer b done, which also releases value stage b
    // (multicast); query tile landed; both
    // query tiles rotated (leader only: each row warp arrives); every MMA of
    // the S / the P V issuer finished (leader, once at the end).
    // A parity wait is only sound for the phase right after the last one
    // known to have completed (a barrier two phases away from the awaited one
    // reads as complete, or as never completing): every barrier below is
    // waited for that way, which is why O += P V completes one barrier per S
    // buffer.
    __shared__ __align__(8) uint64_t bar_kfull[k2Stages], bar_vfull[k2Stages], bar_s[k2SBufs],
        bar_p[k2SBufs], bar_o[k2SBufs], bar_q, bar_qr, bar_drain[2];
    __shared__ uint32_t tmem_base;
    __shared__ int abort_flag;

    uint32_t rank;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(rank));
    const bool leader = rank == 0;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const bool math = warp < 4;
    // the work units, longest query tile first: unit L is query tile
    // ytiles - 1 - L / heads_units of (batch, head) unit L mod heads_units;
    // cluster c takes units c, c + clusters, ...
    const int64_t qtiles = (a.Sq + kAttnRows - 1) / kAttnRows;
    const int64_t heads_units = a.B * (pair_heads ? a.Hq / 2 : a.Hq);
    const int64_t ytiles = pair_heads ? qtiles : (qtiles + 1) / 2;
    const int64_t n_units = heads_units * ytiles;
    const int64_t clusters = gridDim.x >> 1, cid = blockIdx.x >> 1;
    auto unit_work = [&](int64_t L) {
        return attn_work(a, pair_heads, (uint32_t)(L % heads_units), ytiles - 1 - L / heads_units);
    };
    const int64_t shift = a.Sk - a.Sq;
    const int tboxes = a.rotary_dim / 64;

    if (warp == 0) {
        asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;"
                     ::"r"(attn_smem_u32(&tmem_base)), "r"(kTmemCols)
                     : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;" ::: "memory");
    }
    if (tid == 0) {
        for (int s = 0; s < k2Stages; ++s) {
            mbar_init(&bar_kfull[s], 1);
            mbar_init(&bar_vfull[s], 1);
        }
        for (int b = 0; b < k2SBufs; ++b) {
            mbar_init(&bar_s[b], 1);
            mbar_init(&bar_p[b], 2 * (kAttnRows / 32));
            mbar_init(&bar_o[b], 1);
        }
        mbar_init(&bar_q, 1);
        mbar_init(&bar_qr, 2 * (kAttnRows / 32));
        mbar_init(&bar_drain[0], 1);
        mbar_init(&bar_drain[1], 1);
        abort_flag = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
    cluster_sync_all();                            // barriers and TMEM of both CTAs ready
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
    const uint32_t tmem = tmem_base;
    volatile int *abort = &abort_flag;
    const uint32_t peer_abort = peer_addr(&abort_flag, rank ^ 1u);
    auto raise_abort = [&]() {
        *abort = 1;
        asm volatile("st.shared::cluster.u32 [%0], %1;" ::"r"(peer_abort), "r"(1) : "memory");
    };
    bool ok = true;

    if (math) {
        // ---- the row block: per unit, rotate the query tile, then the
        // softmax of row qi on S buffer g mod 3 (g counts this CTA's tiles)
        const uint32_t lanes = (uint32_t)(warp * 32) << 16;
        const uint32_t o_base = tmem + k2OCol + lanes;
        int64_t g = 0;
        uint32_t sb = 0, s_ph = 0;                 // S buffer g mod 3 and its phase parity
        uint32_t ob = 0, o_ph = 0;                 // the same for tile g - 1 (O barriers)
        uint32_t qn = 0;                           // units with key tiles so far
        // Pass L: the key tiles of unit L, then the query tile of unit
        // L + clusters, then the epilogue of unit L.  The next unit's query
        // tile is loaded once unit L's last S has finished; rotated before
        // unit L's epilogue, it lets the next unit's first S products run
        // while the epilogue waits for the last O += P V and stores O.  The
        // first pass (L = cid - clusters) only rotates the first query tile.
        for (int64_t L = cid - clusters; ok && L < n_units; L += clusters) {
            const bool real = L >= cid;
            const AttnWork w = unit_work(real ? L : cid);
            const int64_t qi = w.q0_first + (int64_t)rank * w.q_step + tid;
            const int64_t n_tiles = real ? w.n_tiles : 0;     // the same in both CTAs
            float m_ref = -INFINITY, l_run = 0.0f;
            // the key tiles; M: the softmax reads the attn_mask's bytes, else
            // the row sees at most the first sk keys (-1: all)
            auto key_tiles = [&](auto m_tag, int64_t sk) {
                constexpr bool M = decltype(m_tag)::value;
                for (int64_t kt = 0; kt < n_tiles; ++kt, ++g) {
                    const uint32_t b = sb;
                    ok = __all_sync(0xffffffffu, attn_wait(&bar_s[b], s_ph, abort));
                    if (!ok)
                        break;
                    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
                    // O may still be updated by the products of tiles g - 2 and
                    // g - 1 (that of g - 3 had finished before S(g) was issued): a
                    // rescale waits for the later one, which finishes after the
                    // earlier (rare: the row max moved by more than 8)
                    bool o_ok = true;
                    auto o_ready = [&]() {
                        o_ok = __all_sync(0xffffffffu, attn_wait(&bar_o[ob], o_ph, abort));
                        return o_ok;
                    };
                    softmax_tile<T, D, true, M>(tmem + (uint32_t)b * kAttnKeys + lanes, o_base, qi,
                                          kt * kAttnKeys, shift, a, w.b, kt > 0, m_ref, l_run, o_ready,
                                          sk);
                    ok = o_ok;
                    asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
                    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
                    // this warp's P rows are in TMEM: one arrival per row warp of
                    // both CTAs on the leader's barrier
                    __syncwarp();
                    if (lane == 0) {
                        if (leader)
                            mbar_arrive(&bar_p[b]);
                        else
                            mbar_arrive_remote(peer_addr(&bar_p[b], 0));
                    }
                    // tile g becomes the "previous" tile; advance to g + 1
                    ob = sb;
                    o_ph = s_ph;
                    if (++sb == k2SBufs) {
                        sb = 0;
                        s_ph ^= 1u;
                    }
                    if (!ok)
                        break;
                }
            };
            if constexpr (MASK) {
                // a [B, Sk] mask that shows exactly the keys [0, L) of this
                // batch entry (padding): the unmasked softmax over L keys
                const int64_t len = real && a.kv_len != nullptr ? __ldg(a.kv_len + w.b) : -1;
                if (len >= 0)
                    key_tiles(std::false_type(), len);
                else
                    key_tiles(std::true_type(), (int64_t)-1);
            } else {
                key_tiles(std::false_type(), (int64_t)-1);
            }
            if (!ok)
                break;
            // the next unit's query tile, once it has landed: rotated in
            // place, then one arrival per row warp of both CTAs on the
            // leader's barrier
            if (L + clusters < n_units && unit_work(L + clusters).n_tiles > 0) {
                const AttnWork wn = unit_work(L + clusters);
                ok = __all_sync(0xffffffffu, attn_wait(&bar_q, qn & 1u, abort));
                if (!ok)
                    break;
                // items in flight per thread: 2 (1 in the masked kernel),
                // which frees the registers the tile loop needs (4 spilled
                // and measured 5 % slower)
                rotate_tile<T, LAYOUT, STAGED_Q, kAttnRows, MASK ? 1 : 2>(
                    sQ, sT, wn.q0_first + (int64_t)rank * wn.q_step, a.pos_q, a.Sq, a, tid);
                asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
                __syncwarp();
                if (lane == 0)
                    mbar_arrive_remote(peer_addr(&bar_qr, 0));
                ++qn;
            }
            if (!real)
                continue;
            // the unit's last O += P V (products finish in order), then O / l
            if (n_tiles > 0)
                ok = __all_sync(0xffffffffu, attn_wait(&bar_o[ob], o_ph, abort));
            asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
            if (!ok)
                break;
            // O / l of the warp's 32 rows: staged in shared memory once the
            // warp's store of the previous unit has read it, then one TMA
            // store per 64 features (rows past Sq are not written)
            // (store_o_warp's steps, written out: this kernel's register
            // allocation spills more with the shared helper)
            if (lane == 0)
                asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory");
            __syncwarp();
            stage_o_row<T, D>(o_base, sO, tid, n_tiles > 0, l_run);
            asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
            asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
            __syncwarp();
            const AttnWork we = unit_work(L);     // recomputed: fewer values live across the rotation
            const int64_t y0 = we.q0_first + (int64_t)rank * we.q_step + warp * 32;
            if (lane == 0 && y0 < a.Sq) {
                const int z = (int)(we.b * a.Hq + we.hq_first + (int32_t)rank * we.hq_step);
                tma_store_3d(&maps.o, sO + warp * 32 * 128, 0, (int)y0, z);
                tma_store_3d(&maps.o, sO + kBoxBytes + warp * 32 * 128, 64, (int)y0, z);
                asm volatile("cp.async.bulk.commit_group;" ::: "memory");
            }
        }
        drain_o_stores();
        if (!ok)
            raise_abort();
    } else if (warp == k2SIssueWarp && leader) {
        // ---- S = Q K^T for both CTAs into S buffer g mod 3
        const uint32_t idesc = umma_idesc(256, kAttnKeys, ab_format, 0);
        const uint32_t q_addr = attn_smem_u32(sQ);
        int64_t g = 0;
        uint32_t qn = 0;
        for (int64_t L = cid; ok && L < n_units; L += clusters) {
            const int64_t n_tiles = unit_work(L).n_tiles;
            if (n_tiles == 0)
                continue;
            // both CTAs' query tiles of this unit are rotated
            ok = __all_sync(0xffffffffu, attn_wait(&bar_qr, qn & 1u, abort));
            ++qn;
            for (int64_t kt = 0; ok && kt < n_tiles; ++kt, ++g) {
                const int st = (int)(g % k2Stages), b = (int)(g % k2SBufs);
                // both key halves landed; the product that read P from this S
                // buffer (tile g - 3) has finished
                ok = __all_sync(0xffffffffu,
                                attn_wait(&bar_kfull[st], (uint32_t)((g / k2Stages) & 1), abort) &&
                                    (g < k2SBufs ||
                                     attn_wait(&bar_o[b], (uint32_t)(((g / k2SBufs) - 1) & 1),
                                                  abort)));
                if (!ok)
                    break;
                asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
                if (lane == 0) {
                    const uint32_t k_addr = attn_smem_u32(sK(st));
#pragma unroll
                    for (int kk = 0; kk < D / 16; ++kk)
                        umma2_ss(tmem + (uint32_t)b * kAttnKeys,
                                 umma_desc(q_addr + (kk >> 2) * kBoxBytes + (kk & 3) * 32u, 16u,
                                           1024u, kSwizzle128),
                                 umma_desc(k_addr + (kk >> 2) * (k2Half / 2) + (kk & 3) * 32u, 16u,
                                           1024u, kSwizzle128),
                                 idesc, kk > 0);
                    umma2_commit(&bar_s[b], 3);
                }
                __syncwarp();
            }
        }
        // every MMA this thread issued has finished (one commit, phase 0)
        if (lane == 0)
            umma2_commit(&bar_drain[0], 1);
        __syncwarp();
        if (!__all_sync(0xffffffffu, attn_wait(&bar_drain[0], 0u)))
            ok = false;
        if (!ok)
            raise_abort();
    } else if (warp == k2PVIssueWarp && leader) {
        // ---- O += P V for both CTAs once both P are in TMEM
        const uint32_t idesc = umma_idesc(256, D, ab_format, 1);
        int64_t g = 0;
        for (int64_t L = cid; ok && L < n_units; L += clusters) {
            const int64_t n_tiles = unit_work(L).n_tiles;
            for (int64_t kt = 0; ok && kt < n_tiles; ++kt, ++g) {
                const int st = (int)(g % k2Stages), b = (int)(g % k2SBufs);
                ok = __all_sync(0xffffffffu,
                                attn_wait(&bar_p[b], (uint32_t)((g / k2SBufs) & 1), abort) &&
                                    attn_wait(&bar_vfull[st], (uint32_t)((g / k2Stages) & 1),
                                                 abort));
                if (!ok)
                    break;
                asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
                if (lane == 0) {
                    const uint32_t v_addr = attn_smem_u32(sV(st));
#pragma unroll
                    for (int kk = 0; kk < kAttnKeys / 16; ++kk)
                        umma2_ts(tmem + k2OCol, tmem + (uint32_t)b * kAttnKeys + kk * 8,
                                 umma_desc(v_addr + kk * 2048u, kBoxBytes, 1024u, kSwizzle128),
                                 idesc, (kt > 0 || kk > 0) ? 1u : 0u);
                    umma2_commit(&bar_o[b], 3);
                }
                __syncwarp();
            }
        }
        // every MMA this thread issued has finished (one commit, phase 0)
        if (lane == 0)
            umma2_commit(&bar_drain[1], 1);
        __syncwarp();
        if (!__all_sync(0xffffffffu, attn_wait(&bar_drain[1], 0u)))
            ok = false;
        if (!ok)
            raise_abort();
    } else if (warp == k2TmaWarp) {
        // ---- per unit: the query tile (and its table rows) once the
        // previous unit's last S has read the old one (its key stage's
        // release: S products finish in order, and that stage's previous
        // release, of tile g - 3, has been waited for), then this CTA's halves
        // of key and value tile g into stage g mod 3 once tile g - 3 released it
        int64_t k_last[k2Stages], v_last[k2Stages];
#pragma unroll
        for (int s = 0; s < k2Stages; ++s)
            k_last[s] = v_last[s] = -1;
        bool q_pending = false;
        int64_t g = 0, g_prev = -1;                // g_prev: the previous unit's last tile
        for (int64_t L = cid; ok && L < n_units; L += clusters) {
            const AttnWork w = unit_work(L);
            const int64_t n_tiles = w.n_tiles;
            if (n_tiles == 0)
                continue;
            const int32_t hq = w.hq_first + (int32_t)rank * w.hq_step;
            const int64_t q0 = w.q0_first + (int64_t)rank * w.q_step;
            if (g_prev >= 0)
                ok = __all_sync(0xffffffffu,
                                attn_wait(&bar_s[g_prev % k2Stages],
                                             (uint32_t)((g_prev / k2Stages) & 1), abort));
            if (!ok)
                break;
            if (lane == 0)
                mbar_expect_tx(&bar_q,
                               (uint32_t)(D / 64 + (STAGED_Q ? 2 * tboxes : 0)) * kBoxBytes);
            __syncwarp();
            if (lane < D / 64)
                tma_load_3d(sQ + lane * kBoxBytes, &maps.q, lane * 64, (int)q0,
                            (int)(w.b * a.Hq + hq), &bar_q);
            if (STAGED_Q && lane >= 8 && lane < 8 + 2 * tboxes) {
                const int t = lane - 8;
                const bool is_cos = t < tboxes;
                tma_load_2d(sT + t * kBoxBytes, is_cos ? &maps.cos : &maps.sin,
                            (is_cos ? t : t - tboxes) * 32, (int)q0, &bar_q);
            }
            q_pending = true;
            for (int64_t kt = 0; ok && kt < n_tiles; ++kt, ++g) {
                const int st = (int)(g % k2Stages);
                const int k0 = (int)(kt * kAttnKeys);
                const uint32_t free_ph = (uint32_t)(((g / k2Stages) - 1) & 1);
                if (g >= k2Stages)
                    ok = __all_sync(0xffffffffu, attn_wait(&bar_s[st], free_ph, abort));
                if (!ok)
                    break;
                // this CTA's half of key tile k0: keys k0 + 64 rank .. + 63;
                // both CTAs' bytes complete the leader's barrier
                if (leader && lane == 0)
                    mbar_expect_tx(&bar_kfull[st], 2 * k2Half);
                __syncwarp();
                if (lane < D / 64) {
                    if (leader)
                        tma_load_3d(sK(st) + lane * (k2Half / 2), &maps.k, lane * 64, k0, w.zkv,
                                    &bar_kfull[st]);
                    else
                        tma_load_3d_to_leader(sK(st) + lane * (k2Half / 2), &maps.k, lane * 64,
                                              k0 + 64, w.zkv, peer_addr(&bar_kfull[st], 0));
                }
                k_last[st] = g;
                if (g >= k2Stages)
                    ok = __all_sync(0xffffffffu, attn_wait(&bar_o[st], free_ph, abort));
                if (!ok)
                    break;
                // this CTA's half of value tile k0: feature columns 64 rank ..
                // + 63 of its 128 keys
                if (lane == 0) {
                    if (leader) {
                        mbar_expect_tx(&bar_vfull[st], 2 * k2Half);
                        tma_load_3d(sV(st), &maps.v, 0, k0, w.zkv, &bar_vfull[st]);
                    } else {
                        tma_load_3d_to_leader(sV(st), &maps.v, 64, k0, w.zkv,
                                              peer_addr(&bar_vfull[st], 0));
                    }
                }
                __syncwarp();
                v_last[st] = g;
            }
            g_prev = g - 1;
        }
        if (!ok) {
            raise_abort();
            // one more bounded wait for the last query tile and, in the
            // leader, the last copies into each stage (its barriers count both
            // CTAs' bytes; the follower's memory stays valid until the pair's
            // final barrier below, which the leader reaches after these waits)
            (void)q_pending;
#pragma unroll
            for (int s = 0; s < k2Stages; ++s) {
                if (leader && k_last[s] >= 0)
                    (void)attn_wait(&bar_kfull[s], (uint32_t)((k_last[s] / k2Stages) & 1));
                if (leader && v_last[s] >= 0)
                    (void)attn_wait(&bar_vfull[s], (uint32_t)((v_last[s] / k2Stages) & 1));
            }
        }
    }
    // every role has left its loops; the pair meets once more before TMEM is
    // freed, so no MMA of the leader still reads the follower's memory
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
    cluster_sync_all();
    if (tid == 0 && *abort)
        atomicOr(a.flag, 2);
    if (warp == 0)
        asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;" ::"r"(tmem),
                     "r"(kTmemCols)
                     : "memory");
}

// ---------------------------------------------------------------------------
// host side

typedef CUresult (*EncodeTiledFn)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *,
                                  const cuuint64_t *, const cuuint64_t *, const cuuint32_t *,
                                  const cuuint32_t *, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

// The driver's tensor-map encoder, looked up once.
static EncodeTiledFn encode_tiled()
{
    static std::atomic<EncodeTiledFn> fn{nullptr};
    EncodeTiledFn f = fn.load(std::memory_order_acquire);
    if (f == nullptr) {
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                             &q) != cudaSuccess ||
            q != cudaDriverEntryPointSuccess || p == nullptr)
            return nullptr;
        f = reinterpret_cast<EncodeTiledFn>(p);
        fn.store(f, std::memory_order_release);
    }
    return f;
}

// [heads][rows][D] 16-bit elements; box 64 elements x box_rows rows x 1
// head, 128-byte swizzle.
static bool encode_kv(EncodeTiledFn enc, CUtensorMap *m, const void *base, CUtensorMapDataType dt,
                      int64_t heads, int64_t rows, int32_t D, uint32_t box_rows = kAttnKeys)
{
    const cuuint64_t dims[3] = {(cuuint64_t)D, (cuuint64_t)rows, (cuuint64_t)heads};
    const cuuint64_t strides[2] = {(cuuint64_t)D * 2, (cuuint64_t)rows * D * 2};
    const cuuint32_t box[3] = {64, box_rows, 1};
    const cuuint32_t estr[3] = {1, 1, 1};
    return enc(m, dt, 3, const_cast<void *>(base), dims, strides, box, estr,
               CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
               CU_TENSOR_MAP_L2_PROMOTION_L2_128B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// [table_rows][rotary_dim / 2] fp32; box 32 values x 128 rows, 128-byte
// swizzle (rotary_dim a multiple of 64).
static bool encode_table(EncodeTiledFn enc, CUtensorMap *m, const float *base, int64_t rows,
                         int32_t half)
{
    const cuuint64_t dims[2] = {(cuuint64_t)half, (cuuint64_t)rows};
    const cuuint64_t strides[1] = {(cuuint64_t)half * 4};
    const cuuint32_t box[2] = {32, (cuuint32_t)kAttnKeys};
    const cuuint32_t estr[2] = {1, 1};
    return enc(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, const_cast<float *>(base), dims, strides, box,
               estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
               CU_TENSOR_MAP_L2_PROMOTION_L2_128B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Dynamic shared memory of one CTA.  rope_attn_kernel: two query tiles, the
// key tile, two value tiles and the table staging (two 128 x rotary_dim / 2
// fp32 blocks at most); rope_attn_pp_kernel: two query tiles and two stages
// of key and value tiles.  With D = 64 the request is raised so that one CTA
// holds an SM (its 512 TMEM columns are the whole SM's).
// rope_attn_2sm_kernel (D = 128): the query tile, three stages of a key
// half and a value half, the query tile's table rows, the output block
// (224 KB).
static size_t attn_2sm_smem_bytes()
{
    return (size_t)kAttnRows * 128 * 2 + (size_t)k2Stages * 2 * k2Half + 4 * (size_t)kBoxBytes +
           (size_t)kAttnRows * 128 * 2;
}

static size_t attn_smem_bytes(int D, bool prerotated)
{
    const size_t tile = (size_t)kAttnRows * D * 2;
    const size_t need = prerotated
                            ? kAttnBlocks * tile + 2 * kPpStages * tile
                            : kAttnBlocks * tile + tile + 2 * tile + (size_t)2 * (D / 64) * kBoxBytes;
    const size_t one_per_sm = 120 * 1024;
    return need > one_per_sm ? need : one_per_sm;
}

// rope_attn_pp_kernel stages the query tiles' table rows when both row
// blocks hold the same rows (two heads of a GQA group), the rows sit at
// their own indices and rotary_dim is a multiple of 64 (whole table boxes).
static bool pp_staged_q(const AttnArgs &a, int pair_heads)
{
    return pair_heads && a.pos_q == nullptr && a.rotary_dim % 64 == 0;
}

// Launches one attention kernel instance over (head units, query tiles).
template <auto Kernel>
static cudaError_t launch_attn(int threads, size_t smem, const AttnArgs &a, const AttnMaps &maps,
                               int pair_heads, cudaStream_t st)
{
    const int64_t qtiles = (a.Sq + kAttnRows - 1) / kAttnRows;
    const int64_t heads = a.B * (pair_heads ? a.Hq / 2 : a.Hq);
    const int64_t ytiles = pair_heads ? qtiles : (qtiles + 1) / 2;
    if (ytiles > 65535 || heads > 0x7fffffff)
        return cudaErrorInvalidConfiguration;      // grid.y / grid.x limits
    const dim3 grid((unsigned)heads, (unsigned)ytiles);
    // the shared-memory limit is raised once per kernel instance and device
    static std::atomic<uint64_t> raised{0};       // bit d: done on device d (d < 64)
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess)
        return e;
    const uint64_t bit = dev < 64 ? (uint64_t)1 << dev : 0;
    if (bit == 0 || !(raised.load(std::memory_order_acquire) & bit)) {
        e = cudaFuncSetAttribute(Kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        if (e != cudaSuccess)
            return e;
        raised.fetch_or(bit, std::memory_order_acq_rel);
    }
    Kernel<<<grid, threads, smem, st>>>(a, maps, pair_heads);
    return cudaGetLastError();
}

// Launches the persistent rope_attn_2sm_kernel: one cluster of two CTAs per
// pair of SMs (at most one per work unit).
template <auto Kernel>
static cudaError_t launch_attn_2sm(const AttnArgs &a, const AttnMaps &maps, int pair_heads,
                                   cudaStream_t st)
{
    static std::atomic<uint64_t> raised{0};       // bit d: shared-memory limit raised on device d
    static std::atomic<int> sm_count[64];         // multiprocessors of device d (0: not read yet)
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess)
        return e;
    if (dev < 0 || dev >= 64)
        return cudaErrorInvalidDevice;
    int sms = sm_count[dev].load(std::memory_order_acquire);
    if (sms == 0) {
        e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
        if (e != cudaSuccess)
            return e;
        sm_count[dev].store(sms, std::memory_order_release);
    }
    const uint64_t bit = (uint64_t)1 << dev;
    if (!(raised.load(std::memory_order_acquire) & bit)) {
        e = cudaFuncSetAttribute(Kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 (int)attn_2sm_smem_bytes());
        if (e != cudaSuccess)
            return e;
        raised.fetch_or(bit, std::memory_order_acq_rel);
    }
    const int64_t qtiles = (a.Sq + kAttnRows - 1) / kAttnRows;
    const int64_t units = a.B * (pair_heads ? a.Hq / 2 : a.Hq) * (pair_heads ? qtiles : (qtiles + 1) / 2);
    const int64_t clusters = units < sms / 2 ? units : sms / 2;
    if (clusters < 1)
        return cudaSuccess;
    Kernel<<<dim3((unsigned)(2 * clusters)), k2Threads, attn_2sm_smem_bytes(), st>>>(a, maps,
                                                                                      pair_heads);
    return cudaGetLastError();
}

template <typename T, int LAYOUT, int D, bool MASK>
static cudaError_t launch_attn_layout(const AttnArgs &a, const AttnMaps &maps, int pair_heads,
                                      cudaStream_t st)
{
    // keys rotated beforehand: pairs of SMs for D = 128, one SM for D = 64
    if constexpr (D == 128) {
        if (a.k_rot != nullptr) {
            if (a.pos_q == nullptr && a.rotary_dim % 64 == 0)
                return launch_attn_2sm<rope_attn_2sm_kernel<T, LAYOUT, true, MASK>>(a, maps, pair_heads,
                                                                              st);
            return launch_attn_2sm<rope_attn_2sm_kernel<T, LAYOUT, false, MASK>>(a, maps, pair_heads, st);
        }
    } else {
        if (a.k_rot != nullptr) {
            if (pp_staged_q(a, pair_heads))
                return launch_attn<rope_attn_pp_kernel<T, LAYOUT, D, true, MASK>>(
                    kPpThreads, attn_smem_bytes(D, true), a, maps, pair_heads, st);
            return launch_attn<rope_attn_pp_kernel<T, LAYOUT, D, false, MASK>>(
                kPpThreads, attn_smem_bytes(D, true), a, maps, pair_heads, st);
        }
    }
    const size_t smem = attn_smem_bytes(D, false);
    if (a.pos_k == nullptr && a.rotary_dim % 64 == 0)
        return launch_attn<rope_attn_kernel<T, LAYOUT, D, true, MASK>>(kAttnThreads, smem, a, maps,
                                                                 pair_heads, st);
    return launch_attn<rope_attn_kernel<T, LAYOUT, D, false, MASK>>(kAttnThreads, smem, a, maps,
                                                              pair_heads, st);
}

template <typename T, int D, bool MASK>
static cudaError_t launch_attn_d(const AttnArgs &a, const AttnMaps &maps, int32_t layout,
                                 int pair_heads, cudaStream_t st)
{
    return layout == 0 ? launch_attn_layout<T, 0, D, MASK>(a, maps, pair_heads, st)
                       : launch_attn_layout<T, 1, D, MASK>(a, maps, pair_heads, st);
}

// Tensor maps of the call, then the kernel for its shape, element type and
// key path; MASK: the kernels that apply an attn_mask.
template <bool MASK>
cudaError_t launch_attention_t(const AttnArgs &a, int32_t D, int32_t layout, int32_t dtype,
                               cudaStream_t st)
{
    AttnMaps maps;
    memset(&maps, 0, sizeof maps);
    // two heads of one GQA group per CTA when the group size is even, else
    // two consecutive query tiles of one head
    const int pair_heads = (a.Hq / a.Hk) % 2 == 0 ? 1 : 0;
    if (a.Sk > 0) {
        EncodeTiledFn enc = encode_tiled();
        if (enc == nullptr)
            return cudaErrorNotSupported;
        const CUtensorMapDataType dt =
            dtype == 1 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16;
        const int64_t heads = a.B * a.Hk;
        // keys rotated beforehand are read from the workspace (by
        // rope_attn_2sm_kernel in halves of 64 keys), else from k; the query
        // tiles arrive by TMA only when the keys were rotated beforehand
        const bool two_sm = a.k_rot != nullptr && D == 128;
        if (!encode_kv(enc, &maps.k, a.k_rot != nullptr ? a.k_rot : a.k, dt, heads, a.Sk, D,
                       two_sm ? 64u : (uint32_t)kAttnKeys) ||
            !encode_kv(enc, &maps.v, a.v, dt, heads, a.Sk, D) ||
            (a.k_rot != nullptr && !encode_kv(enc, &maps.q, a.q, dt, a.B * a.Hq, a.Sq, D)) ||
            !encode_kv(enc, &maps.o, a.o, dt, a.B * a.Hq, a.Sq, D, 32u))
            return cudaErrorInvalidValue;
        // the table boxes: of the key tiles (keys rotated in the kernel) or
        // of the query tiles (keys rotated beforehand)
        const bool stage_table =
            a.k_rot == nullptr ? a.pos_k == nullptr && a.rotary_dim % 64 == 0
                               : (two_sm ? a.pos_q == nullptr && a.rotary_dim % 64 == 0
                                         : pp_staged_q(a, pair_heads));
        if (stage_table &&
            (!encode_table(enc, &maps.cos, a.cos, a.table_rows, a.rotary_dim / 2) ||
             !encode_table(enc, &maps.sin, a.sin, a.table_rows, a.rotary_dim / 2)))
            return cudaErrorInvalidValue;
    }
    if (dtype == 1)
        return D == 64 ? launch_attn_d<__nv_bfloat16, 64, MASK>(a, maps, layout, pair_heads, st)
                       : launch_attn_d<__nv_bfloat16, 128, MASK>(a, maps, layout, pair_heads, st);
    return D == 64 ? launch_attn_d<__half, 64, MASK>(a, maps, layout, pair_heads, st)
                   : launch_attn_d<__half, 128, MASK>(a, maps, layout, pair_heads, st);
}

}  // namespace rope
