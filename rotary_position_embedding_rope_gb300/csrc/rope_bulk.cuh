// rope_bulk.cuh -- the bulk-copy (TMA) staged rotation kernel of librope.
//
// Same arithmetic as the register kernel (rotate_pair, one rounding), but the
// head rows travel between HBM and shared memory through the Blackwell bulk
// copy engine (cp.async.bulk with mbarrier completion) instead of through
// registers.  Bytes in flight are then bounded by shared memory, not by the
// register file, which is what an HBM-bound kernel needs on GB300 to keep
// ~7 TB/s of requests outstanding.
//
// Work decomposition.  A unit is (token tile, head): the rotary spans of TS
// consecutive tokens of one batch, for one of the Hq + Hk heads.  Units are
// ordered tile-major, head-minor, and split into balanced contiguous ranges
// over a persistent grid (SM count x resident CTAs), so every SM gets the
// same amount of work in one wave.  The CTA thread (j, y) owns token row y of
// the current tile and 16-byte vectors j and j + NJ of its rotary span; it
// loads that token's cos/sin values into registers once per tile and reuses
// them for every head of the tile (the head grouping that the Unsloth page,
// Triton Kernel Architecture for RoPE, motivates; here all heads).
//
// Pipeline (NST stages of TS rows each, in dynamic shared memory):
//   warp 0 issues the loads of the next NST - 1 units ahead (one bulk copy
//   for a contiguous block of rows, or one per row), each stage completing
//   an mbarrier with the byte count; all threads wait for the stage, rotate
//   it in place in shared memory, fence the generic proxy against the async
//   proxy, synchronise, and warp 0 writes the stage back with bulk stores
//   (rows at position -1 or out of range are neither loaded nor stored).
//   A stage is refilled ROPE_BULK_STORE_LAG - 1 iterations after its store
//   was issued, once that store has finished reading it
//   (cp.async.bulk.wait_group.read), so stores drain while later loads land.
// Every mbarrier wait is bounded (~2 s of clock cycles): on expiry the CTA
// raises bit 2 of the device flag, waits (bounded) for its own copies and
// returns without writing further.
#pragma once

#include "rope_kernels.cuh"

namespace rope {

#ifndef ROPE_BULK_STAGES
#define ROPE_BULK_STAGES 6
#endif
#ifndef ROPE_BULK_THREADS
#define ROPE_BULK_THREADS 256
#endif
// Stores in flight per issuing lane before a stage is refilled.
#ifndef ROPE_BULK_STORE_LAG
#define ROPE_BULK_STORE_LAG 2
#endif
constexpr int kBulkStages = ROPE_BULK_STAGES;
constexpr int kBulkStoreLag = ROPE_BULK_STORE_LAG;
static_assert(kBulkStoreLag >= 1 && kBulkStoreLag < kBulkStages, "store lag must leave a load stage");
constexpr int kBulkThreads = ROPE_BULK_THREADS;
constexpr long long kWaitBudgetCycles = 4000000000LL;   // ~2 s at 2 GHz
constexpr int32_t kFlagTimeout = 2;

// Launch geometry computed on the host.
struct BulkPlan {
    int32_t nj;              // 16-byte vectors per half span
    int32_t ts;              // token rows per tile (and per stage)
    int32_t span;            // rotary span bytes of one row (rotary_dim * elt)
    int32_t heads;           // Hq + Hk
    int64_t tiles_per_b;
    int64_t units;           // tiles * heads
    int32_t contiguous[2];   // rows of tensor t are back to back and span == row
};

// ---- PTX wrappers -----------------------------------------------------------
__device__ __forceinline__ uint32_t smem_u32(const void *p)
{
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}
__device__ __forceinline__ void mbar_init(uint64_t *bar, uint32_t count)
{
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count)
                 : "memory");
}
__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t *bar, uint32_t bytes)
{
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)),
                 "r"(bytes)
                 : "memory");
}
__device__ __forceinline__ bool mbar_try_wait(uint64_t *bar, uint32_t parity)
{
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(smem_u32(bar)), "r"(parity)
        : "memory");
    return ok != 0;
}
// Wait for the phase with the given parity to complete; false after the budget.
__device__ __forceinline__ bool mbar_wait_bounded(uint64_t *bar, uint32_t parity)
{
    if (mbar_try_wait(bar, parity))
        return true;
    const long long t0 = clock64();
    while (!mbar_try_wait(bar, parity)) {
        if (clock64() - t0 > kWaitBudgetCycles)
            return false;
    }
    return true;
}
__device__ __forceinline__ void bulk_load(void *smem_dst, const void *gmem_src, uint32_t bytes,
                                          uint64_t *bar)
{
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];"
        ::"r"(smem_u32(smem_dst)), "l"(gmem_src), "r"(bytes), "r"(smem_u32(bar))
        : "memory");
}
__device__ __forceinline__ void bulk_store(void *gmem_dst, const void *smem_src, uint32_t bytes)
{
    asm volatile("cp.async.bulk.global.shared::cta.bulk_group [%0], [%1], %2;" ::"l"(gmem_dst),
                 "r"(smem_u32(smem_src)), "r"(bytes)
                 : "memory");
}
__device__ __forceinline__ void bulk_commit() { asm volatile("cp.async.bulk.commit_group;" ::: "memory"); }
// Wait until at most kBulkStoreLag - 1 of this thread's store groups still read shared memory.
__device__ __forceinline__ void bulk_wait_read_lag()
{
    asm volatile("cp.async.bulk.wait_group.read %0;" ::"n"(kBulkStoreLag - 1) : "memory");
}
__device__ __forceinline__ void bulk_wait_all() { asm volatile("cp.async.bulk.wait_group 0;" ::: "memory"); }
__device__ __forceinline__ void fence_proxy_async_smem()
{
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}
__device__ __forceinline__ void fence_mbarrier_init()
{
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

// ---- unit geometry ------------------------------------------------------------
// Position in the unit sequence (tile-major, head-minor), advanced without
// divisions; only the starting unit of a CTA is divided out.
struct UnitIter {
    int64_t tile;     // global tile index
    int64_t b;        // batch of the tile
    int64_t tib;      // tile within the batch
    int32_t head;     // 0 .. Hq + Hk - 1
};

__device__ __forceinline__ UnitIter unit_iter(const BulkPlan &bp, int64_t u)
{
    UnitIter it;
    it.tile = u / bp.heads;
    it.head = static_cast<int32_t>(u - it.tile * bp.heads);
    it.b = it.tile / bp.tiles_per_b;
    it.tib = it.tile - it.b * bp.tiles_per_b;
    return it;
}

__device__ __forceinline__ void unit_next(const BulkPlan &bp, UnitIter &it)
{
    if (++it.head == bp.heads) {
        it.head = 0;
        ++it.tile;
        if (++it.tib == bp.tiles_per_b) {
            it.tib = 0;
            ++it.b;
        }
    }
}

struct Unit {
    int32_t t;              // tensor: 0 = Q, 1 = K
    int64_t b;              // batch
    int64_t s0;             // first token of the tile
    int32_t rows;           // rows in this tile (TS, or fewer at the end of a batch)
    const uint8_t *row0;    // address of the first row's rotary span
    int64_t row_stride;     // bytes between consecutive rows
};

__device__ __forceinline__ Unit unit_of(const ApplyArgs &p, const BulkPlan &bp, const UnitIter &it,
                                        int32_t elt)
{
    Unit x;
    x.t = it.head < p.t[0].heads ? 0 : 1;
    const int32_t hh = x.t ? it.head - p.t[0].heads : it.head;
    x.b = it.b;
    x.s0 = it.tib * bp.ts;
    const int64_t left = p.S - x.s0;
    x.rows = static_cast<int32_t>(left < bp.ts ? left : bp.ts);
    // field-wise selects keep the parameter struct out of local memory
    const void *base = x.t ? p.t[1].base : p.t[0].base;
    const int64_t sb = x.t ? p.t[1].stride_b : p.t[0].stride_b;
    const int64_t sh = x.t ? p.t[1].stride_h : p.t[0].stride_h;
    const int64_t ss = x.t ? p.t[1].stride_s : p.t[0].stride_s;
    x.row0 = static_cast<const uint8_t *>(base) + (it.b * sb + (int64_t)hh * sh + x.s0 * ss) * elt;
    x.row_stride = ss * elt;
    return x;
}

// Table row of token (b, s): s itself, or its position index; -1 when the row must not be
// touched (masked or out of range).  Out-of-range positions raise the flag.
__device__ __forceinline__ int64_t token_row(const ApplyArgs &p, int64_t b, int64_t s, bool report)
{
    if (p.pos_idx == nullptr)
        return s;
    const int64_t r = __ldg(p.pos_idx + b * p.pos_stride_b + s);
    if (r == -1)
        return -1;
    if (r < 0 || r >= p.table_rows) {
        if (report)
            atomicOr(p.range_flag, 1);
        return -1;
    }
    return r;
}

// Lane-level validity of rows lane, lane + 32, ... of a unit (bit i: row lane + 32 i).
__device__ __forceinline__ uint32_t lane_rows_valid(const ApplyArgs &p, const Unit &x, int lane)
{
    uint32_t m = 0;
    for (int r = lane, i = 0; r < x.rows; r += 32, ++i)
        if (token_row(p, x.b, x.s0 + r, false) >= 0)
            m |= 1u << i;
    return m;
}

// Warp 0: issue the loads of unit x into stage `dst`, completing `bar`.
__device__ __forceinline__ void issue_unit_load(const ApplyArgs &p, const BulkPlan &bp,
                                                const Unit &x, uint8_t *dst, uint64_t *bar,
                                                int lane)
{
    const uint32_t valid = lane_rows_valid(p, x, lane);
    uint32_t lane_all = 0;
    for (int r = lane, i = 0; r < x.rows; r += 32, ++i)
        lane_all |= 1u << i;
    const bool all_valid = __all_sync(0xffffffffu, valid == lane_all);
    const int n_valid = __reduce_add_sync(0xffffffffu, __popc(valid));
    if (lane == 0)
        mbar_arrive_expect_tx(bar, static_cast<uint32_t>(n_valid) * bp.span);
    __syncwarp();
    if (all_valid && (x.t ? bp.contiguous[1] : bp.contiguous[0])) {
        if (lane == 0 && x.rows > 0)
            bulk_load(dst, x.row0, static_cast<uint32_t>(x.rows) * bp.span, bar);
    } else {
        for (int r = lane, i = 0; r < x.rows; r += 32, ++i)
            if (valid & (1u << i))
                bulk_load(dst + (int64_t)r * bp.span, x.row0 + r * x.row_stride, bp.span, bar);
    }
}

// Warp 0: write stage `src` of unit x back (valid rows only); one bulk group per lane.
__device__ __forceinline__ void issue_unit_store(const ApplyArgs &p, const BulkPlan &bp,
                                                 const Unit &x, const uint8_t *src, int lane)
{
    const uint32_t valid = lane_rows_valid(p, x, lane);
    uint32_t lane_all = 0;
    for (int r = lane, i = 0; r < x.rows; r += 32, ++i)
        lane_all |= 1u << i;
    const bool all_valid = __all_sync(0xffffffffu, valid == lane_all);
    if (all_valid && (x.t ? bp.contiguous[1] : bp.contiguous[0])) {
        if (lane == 0 && x.rows > 0)
            bulk_store(const_cast<uint8_t *>(x.row0), src, static_cast<uint32_t>(x.rows) * bp.span);
    } else {
        for (int r = lane, i = 0; r < x.rows; r += 32, ++i)
            if (valid & (1u << i))
                bulk_store(const_cast<uint8_t *>(x.row0 + r * x.row_stride), src + (int64_t)r * bp.span,
                           bp.span);
    }
    bulk_commit();
}

template <typename T, int LAYOUT>
__global__ void __launch_bounds__(kBulkThreads)
rope_bulk_kernel(const ApplyArgs p, const BulkPlan bp)
{
    constexpr int V = Elt<T>::V;
    constexpr int32_t elt = sizeof(T);
    extern __shared__ __align__(128) uint8_t stages[];
    __shared__ uint64_t full[kBulkStages];

    const int NJ = blockDim.x;
    const int j = threadIdx.x;
    const int y = threadIdx.y;
    const int tid = threadIdx.y * blockDim.x + threadIdx.x;
    const int warp = tid >> 5;
    const int lane = tid & 31;
    const int h = p.rotary_dim >> 1;
    const int64_t stage_bytes = (int64_t)bp.ts * bp.span;

    // balanced contiguous range of units for this CTA
    const int64_t G = gridDim.x, c = blockIdx.x;
    const int64_t share = bp.units / G, extra = bp.units - share * G;
    const int64_t u0 = c * share + (c < extra ? c : extra);
    const int64_t n = share + (c < extra ? 1 : 0);
    if (n == 0)
        return;

    if (tid == 0) {
        for (int s = 0; s < kBulkStages; ++s)
            mbar_init(&full[s], 1);
        fence_mbarrier_init();
    }
    __syncthreads();
    pdl_wait();
    pdl_trigger();

    int64_t issued = 0;                               // units whose loads were issued (warp 0)
    UnitIter prod = unit_iter(bp, u0);                // next unit to load (warp 0)
    if (warp == 0) {
        for (; issued < n && issued < kBulkStages; ++issued) {
            issue_unit_load(p, bp, unit_of(p, bp, prod, elt),
                            stages + (issued % kBulkStages) * stage_bytes,
                            &full[issued % kBulkStages], lane);
            unit_next(bp, prod);
        }
    }
    UnitIter cons = unit_iter(bp, u0);                // unit being rotated

    float cs[V], sn[V];
    int64_t cur_tile = -1;
    int64_t my_row = -1;                              // table row of token y, -1 = skip
    bool aborted = false;

    for (int64_t k = 0; k < n; ++k, unit_next(bp, cons)) {
        const Unit x = unit_of(p, bp, cons, elt);
        const int s = static_cast<int>(k % kBulkStages);
        const uint32_t parity = static_cast<uint32_t>((k / kBulkStages) & 1);
        if (cons.tile != cur_tile) {                  // new tile: this token's cos/sin
            cur_tile = cons.tile;
            my_row = y < x.rows ? token_row(p, x.b, x.s0 + y, j == 0) : -1;
            if (my_row >= 0) {
                const float *crow = p.cos + my_row * h;
                const float *srow = p.sin + my_row * h;
                if constexpr (LAYOUT == 0) {
#pragma unroll
                    for (int q = 0; q < V / 4; ++q) {
                        const float4 cv = __ldg(reinterpret_cast<const float4 *>(crow + j * V) + q);
                        const float4 sv = __ldg(reinterpret_cast<const float4 *>(srow + j * V) + q);
                        cs[4 * q] = cv.x; cs[4 * q + 1] = cv.y; cs[4 * q + 2] = cv.z; cs[4 * q + 3] = cv.w;
                        sn[4 * q] = sv.x; sn[4 * q + 1] = sv.y; sn[4 * q + 2] = sv.z; sn[4 * q + 3] = sv.w;
                    }
                } else if constexpr (V == 8) {
                    const float4 c0 = __ldg(reinterpret_cast<const float4 *>(crow + j * 4));
                    const float4 c1 = __ldg(reinterpret_cast<const float4 *>(crow + (j + NJ) * 4));
                    const float4 s0 = __ldg(reinterpret_cast<const float4 *>(srow + j * 4));
                    const float4 s1 = __ldg(reinterpret_cast<const float4 *>(srow + (j + NJ) * 4));
                    cs[0] = c0.x; cs[1] = c0.y; cs[2] = c0.z; cs[3] = c0.w;
                    cs[4] = c1.x; cs[5] = c1.y; cs[6] = c1.z; cs[7] = c1.w;
                    sn[0] = s0.x; sn[1] = s0.y; sn[2] = s0.z; sn[3] = s0.w;
                    sn[4] = s1.x; sn[5] = s1.y; sn[6] = s1.z; sn[7] = s1.w;
                } else {
                    const float2 c0 = __ldg(reinterpret_cast<const float2 *>(crow + j * 2));
                    const float2 c1 = __ldg(reinterpret_cast<const float2 *>(crow + (j + NJ) * 2));
                    const float2 s0 = __ldg(reinterpret_cast<const float2 *>(srow + j * 2));
                    const float2 s1 = __ldg(reinterpret_cast<const float2 *>(srow + (j + NJ) * 2));
                    cs[0] = c0.x; cs[1] = c0.y; cs[2] = c1.x; cs[3] = c1.y;
                    sn[0] = s0.x; sn[1] = s0.y; sn[2] = s1.x; sn[3] = s1.y;
                }
                if (p.backward) {
#pragma unroll
                    for (int e = 0; e < V; ++e)
                        sn[e] = -sn[e];
                }
            }
        }

        const bool ready = mbar_wait_bounded(&full[s], parity);
        uint8_t *stage = stages + (int64_t)s * stage_bytes;
        if (ready && my_row >= 0) {
            uint4 *row = reinterpret_cast<uint4 *>(stage + (int64_t)y * bp.span);
            float fa[V], fb[V];
            Elt<T>::unpack(row[j], fa);
            Elt<T>::unpack(row[j + NJ], fb);
            if constexpr (LAYOUT == 0) {
#pragma unroll
                for (int e = 0; e < V; ++e)
                    rotate_pair(fa[e], fb[e], cs[e], sn[e]);
            } else {
#pragma unroll
                for (int e = 0; e < V / 2; ++e) {
                    rotate_pair(fa[2 * e], fa[2 * e + 1], cs[e], sn[e]);
                    rotate_pair(fb[2 * e], fb[2 * e + 1], cs[V / 2 + e], sn[V / 2 + e]);
                }
            }
            row[j] = Elt<T>::pack(fa);
            row[j + NJ] = Elt<T>::pack(fb);
        }
        fence_proxy_async_smem();
        if (__syncthreads_or(!ready)) {
            aborted = true;
            break;
        }
        if (warp == 0) {
            issue_unit_store(p, bp, x, stage, lane);
            // refill the stage consumed kBulkStoreLag - 1 iterations ago, once its
            // store has finished reading it
            if (k >= kBulkStoreLag - 1 && issued < n) {
                bulk_wait_read_lag();
                __syncwarp();
                const int s_prev = static_cast<int>(issued % kBulkStages);
                issue_unit_load(p, bp, unit_of(p, bp, prod, elt),
                                stages + (int64_t)s_prev * stage_bytes, &full[s_prev], lane);
                unit_next(bp, prod);
                ++issued;
            }
        }
    }

    if (warp == 0) {
        if (aborted) {
            if (lane == 0)
                atomicOr(p.range_flag, kFlagTimeout);
            // wait (bounded) for the last load issued on each stage to land
            for (int64_t k = issued > kBulkStages ? issued - kBulkStages : 0; k < issued; ++k)
                (void)mbar_wait_bounded(&full[k % kBulkStages],
                                        static_cast<uint32_t>((k / kBulkStages) & 1));
        }
        bulk_wait_all();
    }
}

// Host: launch the bulk-staged kernel.
template <typename T>
cudaError_t launch_bulk(const ApplyArgs &a, int32_t layout, cudaStream_t st)
{
    constexpr int V = Elt<T>::V;
    BulkPlan bp;
    bp.nj = (a.rotary_dim / 2) / V;
    bp.ts = bp.nj >= kBulkThreads ? 1 : kBulkThreads / bp.nj;
    bp.span = a.rotary_dim * (int32_t)sizeof(T);
    bp.heads = a.t[0].heads + (a.ntensors > 1 ? a.t[1].heads : 0);
    bp.tiles_per_b = (a.S + bp.ts - 1) / bp.ts;
    bp.units = a.B * bp.tiles_per_b * bp.heads;
    for (int t = 0; t < 2; ++t)
        bp.contiguous[t] = t < a.ntensors && a.t[t].stride_s == a.D && a.rotary_dim == a.D;
    const size_t smem = (size_t)kBulkStages * bp.ts * bp.span;
    auto kernel = layout == 0 ? rope_bulk_kernel<T, 0> : rope_bulk_kernel<T, 1>;
    cudaError_t e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)smem);
    if (e != cudaSuccess)
        return e;
    int dev = 0, sms = 0, per_sm = 0;
    e = cudaGetDevice(&dev);
    if (e == cudaSuccess)
        e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (e == cudaSuccess)
        e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kernel, bp.nj * bp.ts, smem);
    if (e != cudaSuccess)
        return e;
    int64_t grid = (int64_t)sms * (per_sm > 0 ? per_sm : 1);
    if (grid > bp.units)
        grid = bp.units;
    const dim3 block(bp.nj, bp.ts);
    return launch_hot(kernel, dim3((unsigned)grid), block, smem, st, a, bp);
}

}  // namespace rope
