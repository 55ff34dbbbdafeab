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

// Warp-cooperative load of the 32 tile rows [32 * warp, 32 * warp + 32):
// every load instruction covers RPI = 32 / CPR whole rows (CPR = D / 8
// chunks of 16 bytes per row), so global reads are fully coalesced.  Lane l
// holds chunk l % CPR of row l / CPR of each group.  Rows whose token index
// (tok0 + row) is not below n_tok are stored as zeros.
//   ROT: the first rotary_dim features are rotated with the row's table row
//        (its position; -1 = not rotated).  Split-half: the partner chunk of a
//        first-half chunk c is chunk c + rd/16 of the same row, fetched from
//        that lane with a shuffle; each lane computes the pair and keeps its
//        own element (the same arithmetic as the row-wise kernels).
//   VTILE: store to the MN-major value tile instead of a K-major tile.
template <typename T, int LAYOUT, int D, bool ROT, bool VTILE>
__device__ __forceinline__ void warp_load_tile(const T *rows, int64_t tok0, int64_t n_tok,
                                               const int32_t *pos, const AttnArgs &a, uint8_t *tile,
                                               int warp, int lane)
{
    constexpr int CPR = D / 8;
    constexpr int RPI = 32 / CPR;
    constexpr int ITERS = 32 / RPI;
    constexpr int BATCH = ITERS;                   // every load of the warp in flight at once
    const int c = lane % CPR;
    const int rsub = lane / CPR;
    const int rd = a.rotary_dim;
    const int h8 = rd / 16;                        // chunks per half span (split-half)
#pragma unroll 1
    for (int i0 = 0; i0 < ITERS; i0 += BATCH) {
        uint4 x[BATCH];
#pragma unroll
        for (int u = 0; u < BATCH; ++u) {
            const int r = warp * 32 + (i0 + u) * RPI + rsub;
            const bool valid = tok0 + r < n_tok;
            x[u] = valid ? __ldg(reinterpret_cast<const uint4 *>(rows + (int64_t)r * D) + c)
                         : make_uint4(0, 0, 0, 0);
        }
#pragma unroll
        for (int u = 0; u < BATCH; ++u) {
            const int r = warp * 32 + (i0 + u) * RPI + rsub;
            uint4 y = x[u];
            if constexpr (ROT) {
                const int64_t tok = tok0 + r;
                const int64_t trow =
                    tok < n_tok ? attn_row(pos, tok, a.table_rows, a.flag, c == 0) : -1;
                if constexpr (LAYOUT == 0) {
                    const int src = c < h8 ? lane + h8 : (c < 2 * h8 ? lane - h8 : lane);
                    uint4 partner;
                    partner.x = __shfl_sync(0xffffffffu, x[u].x, src);
                    partner.y = __shfl_sync(0xffffffffu, x[u].y, src);
                    partner.z = __shfl_sync(0xffffffffu, x[u].z, src);
                    partner.w = __shfl_sync(0xffffffffu, x[u].w, src);
                    if (trow >= 0 && c < 2 * h8) {
                        const bool first = c < h8;
                        const int pi = (first ? c : c - h8) * 8;    // pair index of element 0
                        const float *crow = a.cos + trow * (rd >> 1) + pi;
                        const float *srow = a.sin + trow * (rd >> 1) + pi;
                        float f1[8], f2[8], cc[8], ss[8];
                        Elt<T>::unpack(first ? x[u] : partner, f1);
                        Elt<T>::unpack(first ? partner : x[u], f2);
#pragma unroll
                        for (int q = 0; q < 2; ++q) {
                            const float4 cv = __ldg(reinterpret_cast<const float4 *>(crow) + q);
                            const float4 sv = __ldg(reinterpret_cast<const float4 *>(srow) + q);
                            cc[4 * q] = cv.x; cc[4 * q + 1] = cv.y; cc[4 * q + 2] = cv.z; cc[4 * q + 3] = cv.w;
                            ss[4 * q] = sv.x; ss[4 * q + 1] = sv.y; ss[4 * q + 2] = sv.z; ss[4 * q + 3] = sv.w;
                        }
#pragma unroll
                        for (int e = 0; e < 8; ++e)
                            rotate_pair(f1[e], f2[e], cc[e], ss[e]);
                        y = Elt<T>::pack(first ? f1 : f2);
                    }
                } else {
                    if (trow >= 0 && c < rd / 8) {
                        const float4 cv = __ldg(reinterpret_cast<const float4 *>(a.cos + trow * (rd >> 1) + c * 4));
                        const float4 sv = __ldg(reinterpret_cast<const float4 *>(a.sin + trow * (rd >> 1) + c * 4));
                        float f[8];
                        Elt<T>::unpack(x[u], f);
                        rotate_pair(f[0], f[1], cv.x, sv.x);
                        rotate_pair(f[2], f[3], cv.y, sv.y);
                        rotate_pair(f[4], f[5], cv.z, sv.z);
                        rotate_pair(f[6], f[7], cv.w, sv.w);
                        y = Elt<T>::pack(f);
                    }
                }
            }
            if constexpr (VTILE)
                *reinterpret_cast<uint4 *>(tile + (uint32_t)(r >> 3) * CPR * 128u + (uint32_t)c * 128u +
                                           (uint32_t)(r & 7) * 16u) = y;
            else
                *reinterpret_cast<uint4 *>(tile + kmajor128(r, c * 8)) = y;
        }
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
    constexpr int RPI = 32 / CPR;
    const int c = lane % CPR;
    const int rsub = lane / CPR;
#pragma unroll
    for (int it = 0; it < 32 / RPI; ++it) {
        const int r = warp * 32 + it * RPI + rsub;
        const bool valid = tok0 + r < n_tok;
        const uint8_t *src = static_cast<const uint8_t *>(rows) +
                             (valid ? ((int64_t)r * D * 2 + c * 16) : 0);
        const uint32_t dst = attn_smem_u32(tile + (uint32_t)(r >> 3) * CPR * 128u +
                                           (uint32_t)c * 128u + (uint32_t)(r & 7) * 16u);
        asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(dst), "l"(src),
                     "r"(valid ? 16 : 0)
                     : "memory");
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
    warp_load_tile<T, LAYOUT, D, true, false>(Q + q0 * D, q0, a.Sq, a.pos_q, a, sQ, warp, lane);

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
        warp_load_tile<T, LAYOUT, D, true, false>(K + k0 * D, k0, a.Sk, a.pos_k, a, sK, warp, lane);
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
        const int64_t lim = a.causal ? qi + shift : INT64_MAX;
        float mx = -INFINITY;
#pragma unroll 1
        for (int c0 = 0; c0 < kAttnKeys; c0 += 32) {
            float sv[32];
            tmem_ld32(lane_base + c0, sv);
#pragma unroll
            for (int i = 0; i < 32; ++i) {
                const int64_t key = kt * kAttnKeys + c0 + i;
                if (key < a.Sk && key <= lim)
                    mx = fmaxf(mx, sv[i] * a.scale_log2);
            }
        }
        // The exponentials use a reference max m_ref that only moves when the
        // row max exceeds it by more than 8 (factor 256): P stays <= 256,
        // exact in fp32 and bf16/fp16 range, and O is rescaled only then.
        float alpha = 1.0f;
        if (mx > m_ref + 8.0f) {
            alpha = m_ref == -INFINITY ? 0.0f : exp2f(m_ref - mx);
            m_ref = mx;
        }
        const float m_new = m_ref;
        float sum = 0.0f;
#pragma unroll 1
        for (int c0 = 0; c0 < kAttnKeys; c0 += 32) {
            float sv[32];
            tmem_ld32(lane_base + c0, sv);
            float pv[32];
#pragma unroll
            for (int i = 0; i < 32; ++i) {
                const int64_t key = kt * kAttnKeys + c0 + i;
                pv[i] = (key < a.Sk && key <= lim) ? exp2f(sv[i] * a.scale_log2 - m_new) : 0.0f;
                sum += pv[i];
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
