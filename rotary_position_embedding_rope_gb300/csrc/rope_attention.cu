// rope_attention.cu -- attention forward with the rotation fused into the
// loads of the Q and K tiles, on the sm_103a tensor cores (tcgen05, TMEM).
//
// "rotary-embedding-torch", flash_attn_with_rotary: the rotary transformation
// is applied to the loaded blocks of Q and K inside the attention kernel, so
// the rotated tensors are never written back to global memory; GQA/MQA
// (heads_q != heads_kv), a causal mask and per-token positions (-1 = not
// rotated, the pos_mask) are supported.
//
//   O = softmax(scale * rot(Q) rot(K)^T + mask) V
//
// One CTA = 128 query rows of one (batch, query head); thread t owns query
// row t, which is also TMEM lane t of the accumulators.  Per key tile of 128:
//   1. every thread loads one key row and one value row, rotates the key row
//      in fp32 (rotate_pair: Kahan-compensated, one rounding) and stores both
//      to shared memory in the canonical no-swizzle layouts (K: K-major,
//      V: MN-major, so V rows are stored as they are read);
//   2. thread 0 issues S = Q K^T (tcgen05.mma, M = N = 128, K = 16 steps,
//      fp32 in TMEM columns [0, 128)) and commits to an mbarrier;
//   3. each thread reads its S row back (tcgen05.ld), applies the mask and
//      the online softmax in the exp2 domain, writes P as bf16/fp16 to shared
//      memory and rescales its O row in TMEM when the running max moved;
//   4. thread 0 issues O += P V (M = 128, N = D, K = 16 steps, TMEM columns
//      [128, 128 + D)) and commits.
// The epilogue divides by the softmax sum and writes O.  Causal tiles past
// the diagonal are skipped.  Every mbarrier wait is bounded (~2 s of clock):
// on expiry the CTA raises the timeout flag, waits (bounded) for its MMAs,
// frees its TMEM and returns.
#include <type_traits>

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include "rope_kernels.cuh"

namespace rope {

constexpr int kAttnRows = 128;
constexpr int kAttnKeys = 128;
constexpr uint32_t kTmemCols = 256;        // S: 128 columns, O: up to 128
constexpr long long kAttnWaitCycles = 4000000000LL;

__device__ __forceinline__ uint32_t attn_smem_u32(const void *p)
{
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

// Shared-memory matrix descriptor, canonical layout without swizzle: core
// matrices of 8 rows x 16 bytes; lbo = bytes between core matrices along K,
// sbo = bytes between core matrices along M/N.
__device__ __forceinline__ uint64_t umma_desc(uint32_t saddr, uint32_t lbo, uint32_t sbo)
{
    uint64_t d = 0;
    d |= (uint64_t)((saddr >> 4) & 0x3FFF);
    d |= (uint64_t)((lbo >> 4) & 0x3FFF) << 16;
    d |= (uint64_t)((sbo >> 4) & 0x3FFF) << 32;
    d |= (uint64_t)1 << 46;                        // descriptor version for tcgen05
    return d;
}

// Instruction descriptor of kind::f16: fp32 accumulator, A and B of the same
// 16-bit type (bf16 = 1, f16 = 0), A K-major, B K-major or MN-major.
__device__ __forceinline__ uint32_t umma_idesc(int M, int N, uint32_t ab_format, int b_mn_major)
{
    return (1u << 4) | (ab_format << 7) | (ab_format << 10) | ((uint32_t)b_mn_major << 16) |
           ((uint32_t)(N >> 3) << 17) | ((uint32_t)(M >> 4) << 24);
}

__device__ __forceinline__ void umma(uint32_t d_tmem, uint64_t a, uint64_t b, uint32_t idesc,
                                     uint32_t accumulate)
{
    asm volatile("{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
                 "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}"
                 ::"r"(d_tmem), "l"(a), "l"(b), "r"(idesc), "r"(accumulate)
                 : "memory");
}

__device__ __forceinline__ void umma_commit(uint64_t *bar)
{
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];"
                 ::"r"(attn_smem_u32(bar))
                 : "memory");
}

__device__ __forceinline__ bool attn_wait(uint64_t *bar, uint32_t parity)
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
        if (clock64() - t0 > kAttnWaitCycles)
            return false;
    }
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
    return (uint32_t)(k >> 3) * 2048u + (uint32_t)(r >> 3) * 128u + (uint32_t)(r & 7) * 16u +
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

// Warp-cooperative load of the 32 tile rows [32 * warp, 32 * warp + 32).
// Lane l takes row (l & 7) of an 8-row group and chunk (l >> 3) of a group of
// four 16-byte chunks, so every shared-memory store instruction writes four
// runs of 128 contiguous bytes (8 rows of one chunk): the minimum number of
// wavefronts, no bank conflicts, in both canonical layouts.  Global reads are
// 64-byte runs per row.  Rows whose token index (tok0 + row) is not below
// n_tok are stored as zeros.
//   ROT: the first rotary_dim features are rotated with the row's table row
//        (its position; -1 = not rotated).  Split-half: the lane loads the
//        first-half chunk and its partner chunk (+ rd/16) and rotates both
//        (the same arithmetic as the row-wise kernels); interleaved: pairs
//        sit inside one chunk.  Features past rotary_dim are copied.
template <typename T, int LAYOUT, int D, bool ROT>
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
        trow[g] = (ROT && valid[g]) ? attn_row(pos, tok0 + r[g], a.table_rows, a.flag, cc == 0) : -1;
    }
    // rotated chunks: each pass issues the loads of all four rows of the lane
    // (data and table) before any arithmetic, so a pass costs one round trip
    const int rot_chunks = ROT ? (LAYOUT == 0 ? h8 : rd / 8) : 0;
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
    // chunks copied unchanged: past the rotary span (or all, without ROT)
    const int first_copy = ROT ? rd / 8 : 0;
#pragma unroll 1
    for (int c = first_copy + cc; c < CPR; c += 4) {
        uint4 x[G];
#pragma unroll
        for (int g = 0; g < G; ++g)
            x[g] = valid[g] ? __ldg(src[g] + c) : make_uint4(0, 0, 0, 0);
#pragma unroll
        for (int g = 0; g < G; ++g)
            *reinterpret_cast<uint4 *>(tile + kmajor128(r[g], c * 8)) = x[g];
    }
}

// Value tile rows [32 * warp, 32 * warp + 32) straight into the MN-major
// tile with cp.async (16-byte global -> shared copies, no registers; rows past
// n_tok are zero-filled).  Completion: cp.async.wait_group by the caller.
template <int D>
__device__ __forceinline__ void warp_copy_vtile(const void *rows, int64_t tok0, int64_t n_tok,
                                                uint8_t *tile, int warp, int lane)
{
    constexpr int CPR = D / 8;
    const int rr = lane & 7, cc = lane >> 3;       // 8 rows x 4 chunks: 512 contiguous bytes
#pragma unroll
    for (int g = 0; g < 4; ++g) {
        const int r = warp * 32 + g * 8 + rr;
        const bool valid = tok0 + r < n_tok;
#pragma unroll
        for (int c = cc; c < CPR; c += 4) {
            const uint8_t *src = static_cast<const uint8_t *>(rows) +
                                 (valid ? ((int64_t)r * D * 2 + c * 16) : 0);
            const uint32_t dst = attn_smem_u32(tile + (uint32_t)(r >> 3) * CPR * 128u +
                                               (uint32_t)c * 128u + (uint32_t)(r & 7) * 16u);
            asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(dst), "l"(src),
                         "r"(valid ? 16 : 0)
                         : "memory");
        }
    }
    asm volatile("cp.async.commit_group;" ::: "memory");
}

template <typename T, int LAYOUT, int D>
__global__ void __launch_bounds__(kAttnRows, 2) rope_attn_kernel(const AttnArgs a)
{
    constexpr uint32_t kTile = kAttnRows * D * 2;  // bytes of a 128 x D tile
    constexpr uint32_t ab_format = std::is_same<T, __nv_bfloat16>::value ? 1u : 0u;
    extern __shared__ __align__(1024) uint8_t smem[];
    uint8_t *sQ = smem;
    uint8_t *sK = sQ + kTile;
    uint8_t *sV = sK + kTile;
    // P (128 x 128) reuses the K tile once S = Q K^T has been read out of it
    // (the K tile is exactly P's size when D = 128)
    uint8_t *sP = D == kAttnKeys ? sK : sV + kTile;
    __shared__ __align__(8) uint64_t bar;
    __shared__ uint32_t tmem_base;

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int64_t bh = blockIdx.y;
    const int64_t b = bh / a.Hq;
    const int32_t hq = static_cast<int32_t>(bh - b * a.Hq);
    const int32_t hk = hq / (a.Hq / a.Hk);
    const int64_t q0 = (int64_t)blockIdx.x * kAttnRows;
    const int64_t qi = q0 + tid;
    const T *Q = static_cast<const T *>(a.q) + ((b * a.Hq + hq) * a.Sq) * D;
    const T *K = static_cast<const T *>(a.k) + ((b * a.Hk + hk) * a.Sk) * D;
    const T *Vg = static_cast<const T *>(a.v) + ((b * a.Hk + hk) * a.Sk) * D;
    T *O = static_cast<T *>(a.o) + ((b * a.Hq + hq) * a.Sq) * D;

    if (warp == 0) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;"
                     ::"r"(attn_smem_u32(&tmem_base)), "r"(kTmemCols)
                     : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    }
    if (tid == 0) {
        asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" ::"r"(attn_smem_u32(&bar)) : "memory");
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }

    // the query tile, rotated
    warp_load_tile<T, LAYOUT, D, true>(Q + q0 * D, q0, a.Sq, a.pos_q, a, sQ, warp, lane);

    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
    __syncthreads();
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
    const uint32_t tmem = tmem_base;
    const uint32_t lane_base = tmem + ((uint32_t)(warp * 32) << 16);
    const uint32_t idesc_s = umma_idesc(128, kAttnKeys, ab_format, 0);
    const uint32_t idesc_o = umma_idesc(128, D, ab_format, 1);

    // key tiles this query tile can see
    const int64_t shift = a.Sk - a.Sq;             // bottom-right aligned causal mask
    int64_t n_tiles = (a.Sk + kAttnKeys - 1) / kAttnKeys;
    if (a.causal) {
        const int64_t last = q0 + kAttnRows - 1 + shift;   // last key visible to this tile
        const int64_t t = last < 0 ? 0 : last / kAttnKeys + 1;
        if (t < n_tiles)
            n_tiles = t;
    }

    float m_ref = -INFINITY, l_run = 0.0f;         // reference max (log2 domain), sum
    uint32_t phase = 0;
    bool ok = true;                                // CTA-uniform
    for (int64_t kt = 0; kt < n_tiles; ++kt) {
        // 1. key tile (rotated) and value tile, loaded warp-cooperatively
        const int64_t k0 = kt * kAttnKeys;
        warp_copy_vtile<D>(Vg + k0 * D, k0, a.Sk, sV, warp, lane);
        warp_load_tile<T, LAYOUT, D, true>(K + k0 * D, k0, a.Sk, a.pos_k, a, sK, warp, lane);
        asm volatile("cp.async.wait_group 0;" ::: "memory");
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
        asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
        __syncthreads();
        asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");

        // 2. S = Q K^T
        if (tid == 0) {
#pragma unroll
            for (int kk = 0; kk < D / 16; ++kk)
                umma(tmem, umma_desc(attn_smem_u32(sQ) + kk * 4096u, 2048u, 128u),
                     umma_desc(attn_smem_u32(sK) + kk * 4096u, 2048u, 128u), idesc_s, kk > 0);
            umma_commit(&bar);
        }
        // while the MMAs run: pull the next tile's key and value rows into L2
        if (kt + 1 < n_tiles) {
            const int64_t nk = (kt + 1) * kAttnKeys + tid;
            if (nk < a.Sk) {
#pragma unroll
                for (int off = 0; off < D; off += 64) {
                    asm volatile("prefetch.global.L2 [%0];" ::"l"(K + nk * D + off));
                    asm volatile("prefetch.global.L2 [%0];" ::"l"(Vg + nk * D + off));
                }
            }
        }
        ok = __syncthreads_and(attn_wait(&bar, phase));
        if (!ok)
            break;
        phase ^= 1;
        asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");

        // 3. online softmax of this thread's row (TMEM loads are warp-wide)
        // columns of this tile visible to this row: [0, nvis)
        int64_t vis_end = a.Sk;                    // first invisible key
        if (a.causal && qi + shift + 1 < vis_end)
            vis_end = qi + shift + 1;
        const int64_t nv = vis_end - kt * kAttnKeys;
        const int nvis = nv < 0 ? 0 : (nv > kAttnKeys ? kAttnKeys : (int)nv);
        float mx = -INFINITY;
        const bool full = __all_sync(0xffffffffu, nvis == kAttnKeys);   // no mask in this tile
#pragma unroll 1
        for (int c0 = 0; c0 < kAttnKeys; c0 += 32) {
            float sv[32];
            tmem_ld32(lane_base + c0, sv);
            if (full) {
#pragma unroll
                for (int i = 0; i < 32; ++i)
                    mx = fmaxf(mx, sv[i]);
            } else {
#pragma unroll
                for (int i = 0; i < 32; ++i)
                    if (c0 + i < nvis)
                        mx = fmaxf(mx, sv[i]);
            }
        }
        mx *= a.scale_log2;                        // scale > 0: max commutes with it
        // The exponentials use a reference max m_ref that only moves when the
        // row max exceeds it by more than 8 (factor 256): P stays <= 256,
        // exact in fp32 and bf16/fp16 range, and O is rescaled only then.
        float alpha = 1.0f;
        if (mx > m_ref + 8.0f) {
            alpha = m_ref == -INFINITY ? 0.0f : fast_exp2(m_ref - mx);
            m_ref = mx;
        }
        const float m_new = m_ref;
        float sum = 0.0f;
#pragma unroll 1
        for (int c0 = 0; c0 < kAttnKeys; c0 += 32) {
            float sv[32];
            tmem_ld32(lane_base + c0, sv);
            float pv[32];
            if (full) {
#pragma unroll
                for (int i = 0; i < 32; ++i) {
                    pv[i] = fast_exp2(fmaf(sv[i], a.scale_log2, -m_new));
                    sum += pv[i];
                }
            } else {
#pragma unroll
                for (int i = 0; i < 32; ++i) {
                    pv[i] = c0 + i < nvis ? fast_exp2(fmaf(sv[i], a.scale_log2, -m_new)) : 0.0f;
                    sum += pv[i];
                }
            }
#pragma unroll
            for (int c = 0; c < 4; ++c) {
                float f[8];
#pragma unroll
                for (int e = 0; e < 8; ++e)
                    f[e] = pv[c * 8 + e];
                *reinterpret_cast<uint4 *>(sP + kmajor128(tid, c0 + c * 8)) = Elt<T>::pack(f);
            }
        }
        l_run = l_run * alpha + sum;
        if (kt > 0 && __any_sync(0xffffffffu, alpha != 1.0f)) {   // rescale O rows of this warp
#pragma unroll 1
            for (int c0 = 0; c0 < D; c0 += 32) {
                float ov[32];
                tmem_ld32(lane_base + kAttnKeys + c0, ov);
#pragma unroll
                for (int i = 0; i < 32; ++i)
                    ov[i] *= alpha;
                tmem_st32(lane_base + kAttnKeys + c0, ov);
            }
            asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
        }
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
        asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
        __syncthreads();
        asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");

        // 4. O += P V
        if (tid == 0) {
#pragma unroll
            for (int kk = 0; kk < kAttnKeys / 16; ++kk)
                umma(tmem + kAttnKeys, umma_desc(attn_smem_u32(sP) + kk * 4096u, 2048u, 128u),
                     umma_desc(attn_smem_u32(sV) + kk * 2u * (D / 8) * 128u, (D / 8) * 128u, 128u),
                     idesc_o, (kt > 0 || kk > 0) ? 1u : 0u);
            umma_commit(&bar);
        }
        ok = __syncthreads_and(attn_wait(&bar, phase));
        if (!ok)
            break;
        phase ^= 1;
        asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
    }

    if (!ok) {
        // an MMA did not complete in time: report, give it one more bounded
        // wait, free TMEM and leave without writing
        if (tid == 0)
            atomicOr(a.flag, 2);
        (void)attn_wait(&bar, phase);
    } else {
        // epilogue: O / l for this row (zeros when no key is visible); TMEM
        // loads are warp-wide, stores only for rows inside the sequence
        const float inv = (n_tiles > 0 && l_run > 0.0f) ? 1.0f / l_run : 0.0f;
        uint4 *dst = reinterpret_cast<uint4 *>(O + qi * D);
#pragma unroll
        for (int c0 = 0; c0 < D; c0 += 32) {
            float ov[32];
            if (n_tiles > 0) {
                tmem_ld32(lane_base + kAttnKeys + c0, ov);
            } else {
#pragma unroll
                for (int i = 0; i < 32; ++i)
                    ov[i] = 0.0f;
            }
            if (qi < a.Sq) {
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
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
    __syncthreads();
    if (warp == 0)
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem),
                     "r"(kTmemCols)
                     : "memory");
}

template <typename T>
static cudaError_t launch_attn_t(const AttnArgs &a, int32_t D, int32_t layout, cudaStream_t st)
{
    const dim3 grid((unsigned)((a.Sq + kAttnRows - 1) / kAttnRows), (unsigned)(a.B * a.Hq));
    auto go = [&](auto kernel, int d) -> cudaError_t {
        const size_t smem = (size_t)3 * kAttnRows * d * 2 +
                            (d == kAttnKeys ? 0 : (size_t)kAttnRows * kAttnKeys * 2);
        cudaError_t e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             (int)smem);
        if (e != cudaSuccess)
            return e;
        kernel<<<grid, kAttnRows, smem, st>>>(a);
        return cudaGetLastError();
    };
    if (D == 64)
        return layout == 0 ? go(rope_attn_kernel<T, 0, 64>, 64) : go(rope_attn_kernel<T, 1, 64>, 64);
    return layout == 0 ? go(rope_attn_kernel<T, 0, 128>, 128) : go(rope_attn_kernel<T, 1, 128>, 128);
}

cudaError_t launch_attention(const AttnArgs &a, int32_t D, int32_t layout, int32_t dtype,
                             cudaStream_t st)
{
    return dtype == 1 ? launch_attn_t<__nv_bfloat16>(a, D, layout, st)
                      : launch_attn_t<__half>(a, D, layout, st);
}

}  // namespace rope
