// rope_api.cu -- the C ABI of librope (include/rope.h): argument checks,
// kernel selection, the cos/sin table kernel and the device range flag.
#include <cmath>
#include <cstdint>
#include <cstring>
#include <atomic>
#include <mutex>

#include <cuda_runtime.h>

#include "rope.h"
#include "rope_internal.cuh"

namespace rope {

// ---------------------------------------------------------------------------
// Device flag word: bit 0 is set (atomicOr) by the rotation kernels when a
// position index is outside [0, table_rows) and not -1; bit 1 when a wait of
// an attention kernel (or of rope_probe_wait_expiry) ran out of its time
// budget.  One word per device; the kernels get its address as an argument.
// g_flag_taken receives the value read-and-cleared by rope_check_errors.
// ---------------------------------------------------------------------------
__device__ int32_t g_range_flag;
__device__ int32_t g_flag_taken;

constexpr int kMaxDevices = 64;
static int32_t *g_flag_addr[kMaxDevices];
static int32_t *g_taken_addr[kMaxDevices];
static std::mutex g_flag_mutex;

static cudaError_t flag_addresses(int32_t **flag, int32_t **taken)
{
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess)
        return e;
    if (dev < 0 || dev >= kMaxDevices)
        return cudaErrorInvalidDevice;
    std::lock_guard<std::mutex> lock(g_flag_mutex);
    if (g_flag_addr[dev] == nullptr) {
        void *a = nullptr, *t = nullptr;
        e = cudaGetSymbolAddress(&a, g_range_flag);
        if (e != cudaSuccess)
            return e;
        e = cudaGetSymbolAddress(&t, g_flag_taken);
        if (e != cudaSuccess)
            return e;
        g_flag_addr[dev] = static_cast<int32_t *>(a);
        g_taken_addr[dev] = static_cast<int32_t *>(t);
    }
    *flag = g_flag_addr[dev];
    *taken = g_taken_addr[dev];
    return cudaSuccess;
}

__global__ void take_flag_kernel(int32_t *flag, int32_t *taken)
{
    *taken = atomicExch(flag, 0);
}

// Key tiles of 128 up to the last visible key of each batch entry of a
// [B, Sk] attn_mask, and (lens not null) the entry's prefix length: L when
// the mask shows exactly the keys [0, L) (its first hidden key comes after
// its last visible one: padding), else -1.  One CTA per entry reads the
// whole row once, 16 bytes per load when the row is 16-byte aligned, with no
// early exit (so the loads do not wait on one another), keeping the last
// visible and the first hidden key; the CTA then takes the max and the min.
constexpr int kMaskTileKeys = 128;         // the attention kernels' key tile
__global__ void mask_tiles_kernel(const uint8_t *mask, int64_t Sk, int32_t *tiles, int32_t *lens)
{
    __shared__ int32_t warp_last[8], warp_first[8];
    const uint8_t *row = mask + (int64_t)blockIdx.x * Sk;
    int32_t last = -1, first = (int32_t)Sk;    // last visible, first hidden key
    const int64_t nvec = (reinterpret_cast<uintptr_t>(row) & 15) == 0 ? Sk / 16 : 0;
    for (int64_t c = threadIdx.x; c < nvec; c += blockDim.x) {
        const uint4 x = __ldg(reinterpret_cast<const uint4 *>(row) + c);
        const uint32_t wd[4] = {x.x, x.y, x.z, x.w};
#pragma unroll
        for (int e = 0; e < 16; ++e) {
            const int32_t i = (int32_t)(c * 16 + e);
            if ((wd[e >> 2] >> (8 * (e & 3))) & 0xFFu)
                last = i;                      // increasing i: the last one wins
            else
                first = first < i ? first : i;
        }
    }
    for (int64_t i = nvec * 16 + threadIdx.x; i < Sk; i += blockDim.x) {
        if (row[i] != 0)
            last = (int32_t)i;
        else
            first = first < (int32_t)i ? first : (int32_t)i;
    }
    last = __reduce_max_sync(0xffffffffu, last);
    first = __reduce_min_sync(0xffffffffu, first);
    if ((threadIdx.x & 31) == 0) {
        warp_last[threadIdx.x >> 5] = last;
        warp_first[threadIdx.x >> 5] = first;
    }
    __syncthreads();
    if (threadIdx.x == 0) {
        int32_t m = -1, f = (int32_t)Sk;
        for (int w = 0; w < (int)(blockDim.x >> 5); ++w) {
            m = warp_last[w] > m ? warp_last[w] : m;
            f = warp_first[w] < f ? warp_first[w] : f;
        }
        tiles[blockIdx.x] = m < 0 ? 0 : m / kMaskTileKeys + 1;
        if (lens != nullptr)
            lens[blockIdx.x] = f > m ? m + 1 : -1;
    }
}

cudaError_t launch_mask_tiles(const uint8_t *mask, int64_t B, int64_t Sk, int32_t *tiles,
                              int32_t *lens, cudaStream_t st)
{
    mask_tiles_kernel<<<(unsigned)B, 256, 0, st>>>(mask, Sk, tiles, lens);
    return cudaGetLastError();
}

// ---------------------------------------------------------------------------
// cos/sin table ("rotary-embedding-torch", RotaryEmbedding / Key Parameters:
// theta base, interpolate_factor scales positions; "Rotary Embedding (RoPE)
// Kernel Optimization", Common Pitfalls: [seq_len, D/2] tables).
// Column i = blockIdx.x * 32 + threadIdx.x computes its inverse frequency
// theta^(-2i/rd) once, then walks rows m; every angle is formed and reduced
// in fp64 (angles reach ~2.6e5 rad for long contexts, where fp32 would be
// off by ~1e-2 rad) and the results are rounded once to fp32.
// ---------------------------------------------------------------------------
__global__ void rope_table_kernel(double theta, int32_t rotary_dim, int64_t max_pos,
                                  double interpolate_factor, float *cos_out, float *sin_out)
{
    const int32_t h = rotary_dim / 2;
    const int32_t i = blockIdx.x * blockDim.x + threadIdx.x;
    if (i >= h)
        return;
    const double inv_freq = pow(theta, -(2.0 * (double)i) / (double)rotary_dim);
    for (int64_t m = (int64_t)blockIdx.y * blockDim.y + threadIdx.y; m < max_pos;
         m += (int64_t)gridDim.y * blockDim.y) {
        const double angle = ((double)m / interpolate_factor) * inv_freq;
        double sv, cv;
        sincos(angle, &sv, &cv);
        cos_out[m * h + i] = __double2float_rn(cv);
        sin_out[m * h + i] = __double2float_rn(sv);
    }
}

// Tables of a frequency mode at row positions pos_offset + m / pos_divisor,
// scaled by zeta_i^(xpos_sign (p - centre) / base) when xpos_sign != 0 (the
// XPOS query/key scale folded into the table).  One column per thread: the
// frequency and zeta are computed once, then fp64 sincos and pow per entry.
__global__ void rope_table_ex_kernel(int32_t mode, double theta, double max_freq,
                                     int32_t rotary_dim, int64_t rows, double pos_offset,
                                     double pos_divisor, int32_t xpos_sign, double xpos_base,
                                     double xpos_gamma, double xpos_center, float *cos_out,
                                     float *sin_out)
{
    const int32_t h = rotary_dim / 2;
    const int32_t i = blockIdx.x * blockDim.x + threadIdx.x;
    if (i >= h)
        return;
    double w;
    if (mode == ROPE_FREQ_PIXEL)
        w = h == 1 ? M_PI : M_PI * (1.0 + (double)i * (max_freq / 2.0 - 1.0) / (double)(h - 1));
    else if (mode == ROPE_FREQ_CONSTANT)
        w = 1.0;
    else
        w = pow(theta, -(2.0 * (double)i) / (double)rotary_dim);
    const double zeta = (2.0 * (double)i / (double)rotary_dim + xpos_gamma) / (1.0 + xpos_gamma);
    for (int64_t m = (int64_t)blockIdx.y * blockDim.y + threadIdx.y; m < rows;
         m += (int64_t)gridDim.y * blockDim.y) {
        const double p = pos_offset + (double)m / pos_divisor;
        const double angle = p * w;
        const double sc =
            xpos_sign == 0 ? 1.0 : pow(zeta, (double)xpos_sign * (p - xpos_center) / xpos_base);
        double sv, cv;
        sincos(angle, &sv, &cv);
        cos_out[m * h + i] = __double2float_rn(sc * cv);
        sin_out[m * h + i] = __double2float_rn(sc * sv);
    }
}

// ---------------------------------------------------------------------------
// Argument checks and kernel choice (host only; no CUDA calls).
// ---------------------------------------------------------------------------
static bool mul_ok(int64_t a, int64_t b, int64_t *out)
{
    return !__builtin_mul_overflow(a, b, out);
}

static bool ranges_overlap(const void *a, int64_t abytes, const void *b, int64_t bbytes)
{
    if (a == nullptr || b == nullptr || abytes <= 0 || bbytes <= 0)
        return false;
    const uintptr_t a0 = reinterpret_cast<uintptr_t>(a), b0 = reinterpret_cast<uintptr_t>(b);
    return a0 < b0 + (uintptr_t)bbytes && b0 < a0 + (uintptr_t)abytes;
}

static bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// Kernel variant forced by rope_force_kernel_variant (0 = automatic choice).
static std::atomic<int32_t> g_forced_variant{0};

// Grid sizing of the register kernel (rope_tune_rotation_launch).
static std::atomic<int32_t> g_tune_ctas_per_sm{0}, g_tune_min_units{0}, g_tune_prefetch_next{0};

VecLaunchTuning vec_launch_tuning()
{
    VecLaunchTuning t;
    t.ctas_per_sm = g_tune_ctas_per_sm.load(std::memory_order_relaxed);
    t.min_units = g_tune_min_units.load(std::memory_order_relaxed);
    t.prefetch_next = g_tune_prefetch_next.load(std::memory_order_relaxed);
    return t;
}

struct Plan {
    ApplyArgs args;
    int32_t layout;
    int32_t dtype;
    Variant variant;
};

// All arguments of a rotation call (in place: q_out == q, k_out == k).
struct CallArgs {
    const void *q, *k;
    void *q_out, *k_out;
    const float *cos, *sin;
    const int32_t *pos_idx;
    int64_t pos_stride_b;
    int64_t B;
    int32_t Hq, Hk;
    int64_t S;
    int32_t D, rotary_dim, layout, seq_before_head, backward, dtype;
    int64_t table_rows;
};

static rope_status plan_apply(const CallArgs &c, Plan *plan)
{
    std::memset(plan, 0, sizeof *plan);
    plan->variant = kNone;
    if (c.dtype != ROPE_F32 && c.dtype != ROPE_BF16 && c.dtype != ROPE_F16)
        return ROPE_ERR_UNSUPPORTED;
    if (c.layout != ROPE_SPLIT_HALF && c.layout != ROPE_INTERLEAVED)
        return ROPE_ERR_UNSUPPORTED;
    if ((c.seq_before_head != 0 && c.seq_before_head != 1) || (c.backward != 0 && c.backward != 1))
        return ROPE_ERR_INVALID_ARG;
    if (c.B < 0 || c.S < 0 || c.Hq < 0 || c.Hk < 0 || c.D < 1 || c.table_rows < 0)
        return ROPE_ERR_INVALID_ARG;
    if (c.rotary_dim < 2 || (c.rotary_dim & 1) || c.rotary_dim > c.D)
        return ROPE_ERR_INVALID_ARG;
    if (c.pos_stride_b != 0 && c.pos_stride_b < c.S)
        return ROPE_ERR_INVALID_ARG;

    const int64_t elt = c.dtype == ROPE_F32 ? 4 : 2;
    const int64_t h = c.rotary_dim / 2;
    int64_t tok = 0, nq = 0, nk = 0, qbytes = 0, kbytes = 0, tab = 0, tabbytes = 0, posn = 0;
    if (!mul_ok(c.B, c.S, &tok) || !mul_ok(tok, (int64_t)c.Hq * c.D, &nq) ||
        !mul_ok(tok, (int64_t)c.Hk * c.D, &nk) || !mul_ok(nq, elt, &qbytes) ||
        !mul_ok(nk, elt, &kbytes) || !mul_ok(c.table_rows, h, &tab) || !mul_ok(tab, 4, &tabbytes) ||
        !mul_ok(c.B > 0 ? c.B - 1 : 0, c.pos_stride_b, &posn))
        return ROPE_ERR_INVALID_ARG;
    if (tok == 0 || (int64_t)c.Hq + c.Hk == 0)
        return ROPE_OK;                                  // empty: nothing to launch

    if ((c.Hq > 0 && (c.q == nullptr || c.q_out == nullptr)) ||
        (c.Hk > 0 && (c.k == nullptr || c.k_out == nullptr)) || c.cos == nullptr || c.sin == nullptr)
        return ROPE_ERR_INVALID_ARG;
    if (c.table_rows < 1 || (c.pos_idx == nullptr && c.S > c.table_rows))
        return ROPE_ERR_INVALID_ARG;
    const int64_t posbytes = c.pos_idx ? (posn + c.S) * 4 : 0;
    const void *q = c.Hq > 0 ? c.q : nullptr, *k = c.Hk > 0 ? c.k : nullptr;
    const void *qo = c.Hq > 0 ? c.q_out : nullptr, *ko = c.Hk > 0 ? c.k_out : nullptr;
    // every written range must be disjoint from every other range, except an
    // output that is exactly its own input (in place)
    const struct { const void *p; int64_t n; } ins[5] = {
        {q, qbytes}, {k, kbytes}, {c.cos, tabbytes}, {c.sin, tabbytes}, {c.pos_idx, posbytes}};
    const struct { const void *p; int64_t n; const void *self; } outs[2] = {
        {qo, qbytes, q}, {ko, kbytes, k}};
    for (int o = 0; o < 2; ++o) {
        const bool in_place = outs[o].p == outs[o].self;
        for (int i = 0; i < 5; ++i) {
            if (in_place && ins[i].p == outs[o].self)
                continue;                              // the tensor rotated in place
            if (ranges_overlap(outs[o].p, outs[o].n, ins[i].p, ins[i].n))
                return ROPE_ERR_INVALID_ARG;
        }
    }
    if (ranges_overlap(qo, qbytes, ko, kbytes))
        return ROPE_ERR_INVALID_ARG;
    if (qo == q && ranges_overlap(q, qbytes, k, kbytes))
        return ROPE_ERR_INVALID_ARG;

    ApplyArgs &a = plan->args;
    int n = 0;
    const int32_t heads[2] = {c.Hq, c.Hk};
    const void *bases[2] = {c.q, c.k};
    void *outp[2] = {c.q_out, c.k_out};
    for (int t = 0; t < 2; ++t) {
        if (heads[t] == 0)
            continue;
        TensorRef &r = a.t[n];
        r.base = const_cast<void *>(bases[t]);
        r.heads = heads[t];
        if (c.seq_before_head) {                    // [B, S, H, D]
            r.stride_h = c.D;
            r.stride_s = (int64_t)heads[t] * c.D;
            r.stride_b = c.S * r.stride_s;
        } else {                                    // [B, H, S, D]
            r.stride_s = c.D;
            r.stride_h = c.S * c.D;
            r.stride_b = (int64_t)heads[t] * r.stride_h;
        }
        a.out[n] = outp[t];
        a.copy_through[n] = outp[t] != bases[t];
        ++n;
    }
    a.ntensors = n;
    a.cos = c.cos;
    a.sin = c.sin;
    a.pos_idx = c.pos_idx;
    a.pos_stride_b = c.pos_idx ? c.pos_stride_b : 0;
    a.B = c.B;
    a.S = c.S;
    a.D = c.D;
    a.rotary_dim = c.rotary_dim;
    a.table_rows = c.table_rows;
    a.backward = c.backward;
    plan->layout = c.layout;
    plan->dtype = c.dtype;

    // 16-byte vectors need: a rotary span of whole vector pairs, 16-byte
    // aligned rows, aligned base pointers and tables, and NJ within a CTA.
    const int64_t span_bytes = c.rotary_dim * elt;
    bool vec = (span_bytes % 32) == 0 && ((int64_t)c.D * elt) % 16 == 0 && aligned16(c.cos) &&
               aligned16(c.sin) && span_bytes / 32 <= kMaxVectorsPerHalf;
    for (int t = 0; t < n; ++t)
        vec = vec && aligned16(a.t[t].base) && aligned16(a.out[t]);
    const int32_t forced = g_forced_variant.load(std::memory_order_relaxed);
    if (forced == kScalar)
        plan->variant = kScalar;
    else if (forced == kVector) {
        if (!vec)
            return ROPE_ERR_UNSUPPORTED;
        plan->variant = kVector;
    } else
        plan->variant = vec ? kVector : kScalar;
    return ROPE_OK;
}

static rope_status launch_plan(const Plan &plan, cudaStream_t st)
{
    cudaError_t e;
    switch (plan.dtype) {
    case ROPE_F32: e = launch_apply_f32(plan.args, plan.layout, plan.variant, st); break;
    case ROPE_BF16: e = launch_apply_bf16(plan.args, plan.layout, plan.variant, st); break;
    default: e = launch_apply_f16(plan.args, plan.layout, plan.variant, st); break;
    }
    return e == cudaSuccess ? ROPE_OK : ROPE_ERR_CUDA;
}

}  // namespace rope

using namespace rope;

extern "C" {

rope_status rope_tables_build(double theta, int32_t rotary_dim, int64_t max_pos,
                              double interpolate_factor, float *cos_out, float *sin_out,
                              void *stream)
{
    if (!(theta > 0.0) || !std::isfinite(theta) || !(interpolate_factor > 0.0) ||
        !std::isfinite(interpolate_factor) || rotary_dim < 2 || (rotary_dim & 1) || max_pos < 0)
        return ROPE_ERR_INVALID_ARG;
    if (max_pos == 0)
        return ROPE_OK;
    const int64_t h = rotary_dim / 2;
    int64_t n = 0, bytes = 0;
    if (!mul_ok(max_pos, h, &n) || !mul_ok(n, 4, &bytes))
        return ROPE_ERR_INVALID_ARG;
    if (cos_out == nullptr || sin_out == nullptr || ranges_overlap(cos_out, bytes, sin_out, bytes))
        return ROPE_ERR_INVALID_ARG;
    const dim3 block(32, 8);
    const int64_t rows_blocks = (max_pos + block.y - 1) / block.y;
    const dim3 grid((unsigned)((h + 31) / 32), (unsigned)(rows_blocks < 8192 ? rows_blocks : 8192));
    rope_table_kernel<<<grid, block, 0, static_cast<cudaStream_t>(stream)>>>(
        theta, rotary_dim, max_pos, interpolate_factor, cos_out, sin_out);
    return cudaGetLastError() == cudaSuccess ? ROPE_OK : ROPE_ERR_CUDA;
}

rope_status rope_tables_build_ex(int32_t freq_mode, double theta, double max_freq,
                                 int32_t rotary_dim, int64_t rows, double pos_offset,
                                 double pos_divisor, int32_t xpos_sign, double xpos_scale_base,
                                 double xpos_gamma, double xpos_center, float *cos_out,
                                 float *sin_out, void *stream)
{
    if (freq_mode != ROPE_FREQ_LANG && freq_mode != ROPE_FREQ_PIXEL &&
        freq_mode != ROPE_FREQ_CONSTANT)
        return ROPE_ERR_UNSUPPORTED;
    if (rotary_dim < 2 || (rotary_dim & 1) || rows < 0)
        return ROPE_ERR_INVALID_ARG;
    if (freq_mode == ROPE_FREQ_LANG && !(theta > 0.0 && std::isfinite(theta)))
        return ROPE_ERR_INVALID_ARG;
    if (freq_mode == ROPE_FREQ_PIXEL && !(max_freq > 0.0 && std::isfinite(max_freq)))
        return ROPE_ERR_INVALID_ARG;
    if (!std::isfinite(pos_offset) || !(pos_divisor > 0.0 && std::isfinite(pos_divisor)))
        return ROPE_ERR_INVALID_ARG;
    if (xpos_sign < -1 || xpos_sign > 1)
        return ROPE_ERR_INVALID_ARG;
    if (xpos_sign != 0 &&
        !(xpos_scale_base > 0.0 && std::isfinite(xpos_scale_base) && xpos_gamma > 0.0 &&
          std::isfinite(xpos_gamma) && std::isfinite(xpos_center)))
        return ROPE_ERR_INVALID_ARG;
    if (rows == 0)
        return ROPE_OK;
    const int64_t h = rotary_dim / 2;
    int64_t n = 0, bytes = 0;
    if (!mul_ok(rows, h, &n) || !mul_ok(n, 4, &bytes))
        return ROPE_ERR_INVALID_ARG;
    if (cos_out == nullptr || sin_out == nullptr || ranges_overlap(cos_out, bytes, sin_out, bytes))
        return ROPE_ERR_INVALID_ARG;
    const dim3 block(32, 8);
    const int64_t rows_blocks = (rows + block.y - 1) / block.y;
    const dim3 grid((unsigned)((h + 31) / 32), (unsigned)(rows_blocks < 8192 ? rows_blocks : 8192));
    rope_table_ex_kernel<<<grid, block, 0, static_cast<cudaStream_t>(stream)>>>(
        freq_mode, theta, max_freq, rotary_dim, rows, pos_offset, pos_divisor, xpos_sign,
        xpos_scale_base, xpos_gamma, xpos_center, cos_out, sin_out);
    return cudaGetLastError() == cudaSuccess ? ROPE_OK : ROPE_ERR_CUDA;
}

static rope_status apply_call(const CallArgs &c, void *stream)
{
    Plan plan;
    rope_status st = plan_apply(c, &plan);
    if (st != ROPE_OK || plan.variant == kNone)
        return st;
    int32_t *taken = nullptr;
    if (flag_addresses(&plan.args.range_flag, &taken) != cudaSuccess)
        return ROPE_ERR_CUDA;
    return launch_plan(plan, static_cast<cudaStream_t>(stream));
}

rope_status rope_apply_qk(void *q, void *k, const float *cos, const float *sin,
                          const int32_t *pos_idx, int64_t B, int32_t Hq, int32_t Hk, int64_t S,
                          int32_t D, int32_t rotary_dim, int32_t layout, int32_t seq_before_head,
                          int32_t backward, int32_t dtype, int64_t table_rows, void *stream)
{
    const CallArgs c = {q, k, q, k, cos, sin, pos_idx, 0, B, Hq, Hk, S, D, rotary_dim, layout,
                        seq_before_head, backward, dtype, table_rows};
    return apply_call(c, stream);
}

rope_status rope_apply_q(void *x, const float *cos, const float *sin, const int32_t *pos_idx,
                         int64_t B, int32_t H, int64_t S, int32_t D, int32_t rotary_dim,
                         int32_t layout, int32_t seq_before_head, int32_t backward, int32_t dtype,
                         int64_t table_rows, void *stream)
{
    return rope_apply_qk(x, nullptr, cos, sin, pos_idx, B, H, 0, S, D, rotary_dim, layout,
                         seq_before_head, backward, dtype, table_rows, stream);
}

rope_status rope_apply_qk_out(const void *q, const void *k, void *q_out, void *k_out,
                              const float *cos, const float *sin, const int32_t *pos_idx,
                              int64_t pos_batch_stride, int64_t B, int32_t Hq, int32_t Hk,
                              int64_t S, int32_t D, int32_t rotary_dim, int32_t layout,
                              int32_t seq_before_head, int32_t backward, int32_t dtype,
                              int64_t table_rows, void *stream)
{
    const CallArgs c = {q, k, q_out, k_out, cos, sin, pos_idx, pos_batch_stride, B, Hq, Hk, S, D,
                        rotary_dim, layout, seq_before_head, backward, dtype, table_rows};
    return apply_call(c, stream);
}

int32_t rope_qk_kernel_variant(const void *q, const void *k, const float *cos, const float *sin,
                               const int32_t *pos_idx, int64_t B, int32_t Hq, int32_t Hk,
                               int64_t S, int32_t D, int32_t rotary_dim, int32_t layout,
                               int32_t seq_before_head, int32_t backward, int32_t dtype,
                               int64_t table_rows)
{
    const CallArgs c = {q, k, const_cast<void *>(q), const_cast<void *>(k), cos, sin, pos_idx, 0,
                        B, Hq, Hk, S, D, rotary_dim, layout, seq_before_head, backward, dtype,
                        table_rows};
    Plan plan;
    return plan_apply(c, &plan) == ROPE_OK ? (int32_t)plan.variant : 0;
}

}  // extern "C"

namespace rope {

// All arguments of an attention call.
struct AttnCall {
    const void *q, *k, *v;
    void *o;
    const float *cos, *sin;
    const int32_t *pos_q, *pos_k;
    int64_t B;
    int32_t Hq, Hk;
    int64_t Sq, Sk;
    int32_t D, rotary_dim, layout, causal;
    float softmax_scale;
    int32_t dtype;
    int64_t table_rows;
    const uint8_t *mask;
    int32_t mask_kind;
    void *k_workspace;
    int64_t workspace_bytes;
};

// Bytes of the key workspace a call uses: rot(K) (kb bytes); with a [B, Sk]
// mask and room for them, then B int32 key-tile counts from the first
// 16-byte boundary after rot(K), and with room for them too, B int32 prefix
// lengths right after the counts.
static int64_t mask_tiles_offset(int64_t kb) { return (kb + 15) / 16 * 16; }

static int64_t workspace_extent(const AttnCall &c, int64_t kb)
{
    if (c.mask_kind != ROPE_MASK_KEYS || c.Sk > 0x7fffffffLL || c.B > 0x7fffffffLL)
        return kb;
    const int64_t tiles_end = mask_tiles_offset(kb) + 4 * c.B;
    if (c.workspace_bytes >= tiles_end + 4 * c.B)
        return tiles_end + 4 * c.B;
    if (c.workspace_bytes >= tiles_end)
        return tiles_end;
    return kb;
}

// Host checks of an attention call, in order; *empty is set when the call
// has no output rows (nothing to do).  No CUDA calls.
static rope_status attention_check(const AttnCall &c, bool *empty, int64_t *kbytes)
{
    *empty = false;
    if (c.dtype != ROPE_BF16 && c.dtype != ROPE_F16)
        return ROPE_ERR_UNSUPPORTED;
    if (c.layout != ROPE_SPLIT_HALF && c.layout != ROPE_INTERLEAVED)
        return ROPE_ERR_UNSUPPORTED;
    if (c.D != 64 && c.D != 128)
        return ROPE_ERR_UNSUPPORTED;
    if (c.rotary_dim < 16 || c.rotary_dim > c.D || (c.rotary_dim % 16) != 0)
        return ROPE_ERR_UNSUPPORTED;
    if (c.mask_kind < ROPE_MASK_NONE || c.mask_kind > ROPE_MASK_QUERY_KEYS)
        return ROPE_ERR_UNSUPPORTED;
    if ((c.causal != 0 && c.causal != 1) || c.B < 0 || c.Sq < 0 || c.Sk < 0 || c.Hq < 0 ||
        c.Hk < 0 || c.table_rows < 0 || !(c.softmax_scale == c.softmax_scale))
        return ROPE_ERR_INVALID_ARG;
    if (c.Hq > 0 && (c.Hk == 0 || c.Hq % c.Hk != 0))
        return ROPE_ERR_INVALID_ARG;
    int64_t nq = 0, nk = 0, qb = 0, kb = 0, tab = 0, tabb = 0, mb = 0;
    if (!mul_ok(c.B * (int64_t)c.Hq, c.Sq, &nq) || !mul_ok(nq, (int64_t)c.D * 2, &qb) ||
        !mul_ok(c.B * (int64_t)c.Hk, c.Sk, &nk) || !mul_ok(nk, (int64_t)c.D * 2, &kb) ||
        !mul_ok(c.table_rows, c.rotary_dim / 2, &tab) || !mul_ok(tab, 4, &tabb) ||
        !mul_ok(c.B, c.Sk, &mb) ||
        (c.mask_kind == ROPE_MASK_QUERY_KEYS && !mul_ok(mb, c.Sq, &mb)))
        return ROPE_ERR_INVALID_ARG;
    if (c.mask_kind == ROPE_MASK_NONE)
        mb = 0;
    *kbytes = kb;
    if (c.B == 0 || c.Hq == 0 || c.Sq == 0) {
        *empty = true;                                   // no output rows
        return ROPE_OK;
    }
    if (!c.q || !c.o || !c.cos || !c.sin || (c.Sk > 0 && (!c.k || !c.v)) ||
        (c.Sk > 0 && c.mask_kind != ROPE_MASK_NONE && !c.mask))
        return ROPE_ERR_INVALID_ARG;
    if (c.table_rows < 1 || (!c.pos_q && c.Sq > c.table_rows) || (!c.pos_k && c.Sk > c.table_rows))
        return ROPE_ERR_INVALID_ARG;
    if (!aligned16(c.q) || !aligned16(c.k) || !aligned16(c.v) || !aligned16(c.o) ||
        !aligned16(c.cos) || !aligned16(c.sin))
        return ROPE_ERR_UNSUPPORTED;
    const void *o = c.o;
    if (ranges_overlap(o, qb, c.q, qb) || ranges_overlap(o, qb, c.k, kb) ||
        ranges_overlap(o, qb, c.v, kb) || ranges_overlap(o, qb, c.cos, tabb) ||
        ranges_overlap(o, qb, c.sin, tabb) || ranges_overlap(o, qb, c.pos_q, c.Sq * 4) ||
        ranges_overlap(o, qb, c.pos_k, c.Sk * 4) || ranges_overlap(o, qb, c.mask, mb))
        return ROPE_ERR_INVALID_ARG;
    // the key workspace receives rot(K): at least kb bytes, aligned, and
    // disjoint from every other buffer of the call (with the key tiles of a
    // [B, Sk] mask after them when it has room for those too)
    const void *ws = c.Sk > 0 ? c.k_workspace : nullptr;
    if (ws != nullptr) {
        if (c.workspace_bytes < kb)
            return ROPE_ERR_INVALID_ARG;
        if (!aligned16(ws))
            return ROPE_ERR_UNSUPPORTED;
        const int64_t used = workspace_extent(c, kb);
        if (ranges_overlap(ws, used, c.q, qb) || ranges_overlap(ws, used, c.k, kb) ||
            ranges_overlap(ws, used, c.v, kb) || ranges_overlap(ws, used, o, qb) ||
            ranges_overlap(ws, used, c.cos, tabb) || ranges_overlap(ws, used, c.sin, tabb) ||
            ranges_overlap(ws, used, c.pos_q, c.Sq * 4) ||
            ranges_overlap(ws, used, c.pos_k, c.Sk * 4) || ranges_overlap(ws, used, c.mask, mb))
            return ROPE_ERR_INVALID_ARG;
    }
    return ROPE_OK;
}

static rope_status attention_call(const AttnCall &c, void *stream)
{
    bool empty = false;
    int64_t kb = 0;
    const rope_status st = attention_check(c, &empty, &kb);
    if (st != ROPE_OK || empty)
        return st;
    void *ws = c.Sk > 0 ? c.k_workspace : nullptr;
    AttnArgs a;
    std::memset(&a, 0, sizeof a);
    a.q = c.q; a.k = c.k; a.v = c.v; a.o = c.o;
    a.k_rot = ws;
    a.cos = c.cos; a.sin = c.sin;
    a.pos_q = c.pos_q; a.pos_k = c.pos_k;
    a.B = c.B; a.Hq = c.Hq; a.Hk = c.Hk; a.Sq = c.Sq; a.Sk = c.Sk;
    a.rotary_dim = c.rotary_dim;
    a.table_rows = c.table_rows;
    const double scale = c.softmax_scale > 0.0f ? c.softmax_scale : 1.0 / std::sqrt((double)c.D);
    a.scale_log2 = (float)(scale * 1.4426950408889634);
    a.causal = c.causal;
    a.mask_kind = c.Sk > 0 ? c.mask_kind : ROPE_MASK_NONE;
    a.mask = a.mask_kind != ROPE_MASK_NONE ? c.mask : nullptr;
    a.mask_vec16 = a.mask_kind == ROPE_MASK_QUERY_KEYS && aligned16(c.mask) && c.Sk % 16 == 0;
    int32_t *taken = nullptr;
    if (flag_addresses(&a.flag, &taken) != cudaSuccess)
        return ROPE_ERR_CUDA;
    if (ws != nullptr) {
        // rot(K) into the workspace, by the rotation kernel on the same stream
        // (out of place: -1 and out-of-range positions copy the key unchanged)
        const CallArgs r = {nullptr, c.k, nullptr, ws, c.cos, c.sin, c.pos_k, 0, c.B, 0, c.Hk, c.Sk,
                            c.D, c.rotary_dim, c.layout, 0, 0, c.dtype, c.table_rows};
        const rope_status s = apply_call(r, stream);
        if (s != ROPE_OK)
            return s;
        // a [B, Sk] mask: the key tiles each batch entry shows, after rot(K),
        // then (room permitting) the entries' prefix lengths
        const int64_t used = workspace_extent(c, kb);
        if (a.mask_kind == ROPE_MASK_KEYS && used > kb) {
            int32_t *tiles = reinterpret_cast<int32_t *>(static_cast<uint8_t *>(ws) +
                                                         mask_tiles_offset(kb));
            int32_t *lens = used > mask_tiles_offset(kb) + 4 * c.B ? tiles + c.B : nullptr;
            if (launch_mask_tiles(c.mask, c.B, c.Sk, tiles, lens,
                                  static_cast<cudaStream_t>(stream)) != cudaSuccess)
                return ROPE_ERR_CUDA;
            a.kv_tiles = tiles;
            a.kv_len = lens;
        }
    }
    return launch_attention(a, c.D, c.layout, c.dtype, static_cast<cudaStream_t>(stream)) ==
                   cudaSuccess
               ? ROPE_OK
               : ROPE_ERR_CUDA;
}

rope_status attention_args_status(const void *q, const void *k, const void *v, void *o,
                                  const float *cos, const float *sin, const int32_t *pos_q,
                                  const int32_t *pos_k, int64_t B, int32_t Hq, int32_t Hk,
                                  int64_t Sq, int64_t Sk, int32_t D, int32_t rotary_dim,
                                  int32_t layout, int32_t causal, float softmax_scale,
                                  int32_t dtype, int64_t table_rows)
{
    const AttnCall c = {q, k, v, o, cos, sin, pos_q, pos_k, B, Hq, Hk, Sq, Sk, D, rotary_dim, layout,
                        causal, softmax_scale, dtype, table_rows, nullptr, ROPE_MASK_NONE, nullptr,
                        0};
    bool empty = false;
    int64_t kb = 0;
    return attention_check(c, &empty, &kb);
}

}  // namespace rope

extern "C" {

rope_status rope_attention_fwd(const void *q, const void *k, const void *v, void *o,
                               const float *cos, const float *sin, const int32_t *pos_q,
                               const int32_t *pos_k, int64_t B, int32_t Hq, int32_t Hk, int64_t Sq,
                               int64_t Sk, int32_t D, int32_t rotary_dim, int32_t layout,
                               int32_t causal, float softmax_scale, int32_t dtype,
                               int64_t table_rows, void *k_workspace, int64_t workspace_bytes,
                               void *stream)
{
    const AttnCall c = {q, k, v, o, cos, sin, pos_q, pos_k, B, Hq, Hk, Sq, Sk, D, rotary_dim, layout,
                        causal, softmax_scale, dtype, table_rows, nullptr, ROPE_MASK_NONE,
                        k_workspace, workspace_bytes};
    return attention_call(c, stream);
}

rope_status rope_attention_fwd_masked(const void *q, const void *k, const void *v, void *o,
                                      const float *cos, const float *sin, const int32_t *pos_q,
                                      const int32_t *pos_k, int64_t B, int32_t Hq, int32_t Hk,
                                      int64_t Sq, int64_t Sk, int32_t D, int32_t rotary_dim,
                                      int32_t layout, int32_t causal, float softmax_scale,
                                      int32_t dtype, int64_t table_rows, const uint8_t *attn_mask,
                                      int32_t mask_kind, void *k_workspace,
                                      int64_t workspace_bytes, void *stream)
{
    const AttnCall c = {q, k, v, o, cos, sin, pos_q, pos_k, B, Hq, Hk, Sq, Sk, D, rotary_dim, layout,
                        causal, softmax_scale, dtype, table_rows, attn_mask, mask_kind,
                        k_workspace, workspace_bytes};
    return attention_call(c, stream);
}

rope_status rope_check_errors(void *stream)
{
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    if (cudaStreamSynchronize(st) != cudaSuccess)
        return ROPE_ERR_CUDA;
    int32_t *flag = nullptr, *taken = nullptr;
    if (flag_addresses(&flag, &taken) != cudaSuccess)
        return ROPE_ERR_CUDA;
    take_flag_kernel<<<1, 1, 0, st>>>(flag, taken);
    if (cudaGetLastError() != cudaSuccess)
        return ROPE_ERR_CUDA;
    int32_t value = 0;
    if (cudaMemcpyAsync(&value, taken, sizeof value, cudaMemcpyDeviceToHost, st) != cudaSuccess ||
        cudaStreamSynchronize(st) != cudaSuccess)
        return ROPE_ERR_CUDA;
    if (value & 2)
        return ROPE_ERR_KERNEL_TIMEOUT;
    return value ? ROPE_ERR_POS_OUT_OF_RANGE : ROPE_OK;
}

// Longest wait the probe may take: the kernels' own bound (~2 s of clock).
static constexpr int64_t kMaxProbeCycles = 4000000000LL;

rope_status rope_probe_wait_expiry(int64_t cycles, void *stream)
{
    if (cycles <= 0 || cycles > kMaxProbeCycles)
        return ROPE_ERR_INVALID_ARG;
    int32_t *flag = nullptr, *taken = nullptr;
    if (flag_addresses(&flag, &taken) != cudaSuccess)
        return ROPE_ERR_CUDA;
    return launch_wait_probe(flag, (long long)cycles, static_cast<cudaStream_t>(stream)) ==
                   cudaSuccess
               ? ROPE_OK
               : ROPE_ERR_CUDA;
}

rope_status rope_force_kernel_variant(int32_t variant)
{
    if (variant != kNone && variant != kScalar && variant != kVector)
        return ROPE_ERR_INVALID_ARG;
    g_forced_variant.store(variant, std::memory_order_relaxed);
    return ROPE_OK;
}

rope_status rope_tune_rotation_launch(int32_t ctas_per_sm, int32_t min_units,
                                      int32_t prefetch_next)
{
    if (ctas_per_sm < 0 || ctas_per_sm > 64 || min_units < 0 || prefetch_next < -1 ||
        prefetch_next > 1)
        return ROPE_ERR_INVALID_ARG;
    g_tune_ctas_per_sm.store(ctas_per_sm, std::memory_order_relaxed);
    g_tune_min_units.store(min_units, std::memory_order_relaxed);
    g_tune_prefetch_next.store(prefetch_next, std::memory_order_relaxed);
    return ROPE_OK;
}

const char *rope_status_string(rope_status status)
{
    switch (status) {
    case ROPE_OK: return "ROPE_OK";
    case ROPE_ERR_INVALID_ARG: return "ROPE_ERR_INVALID_ARG";
    case ROPE_ERR_UNSUPPORTED: return "ROPE_ERR_UNSUPPORTED";
    case ROPE_ERR_CUDA: return "ROPE_ERR_CUDA";
    case ROPE_ERR_POS_OUT_OF_RANGE: return "ROPE_ERR_POS_OUT_OF_RANGE";
    case ROPE_ERR_KERNEL_TIMEOUT: return "ROPE_ERR_KERNEL_TIMEOUT";
    default: return "ROPE_STATUS_UNKNOWN";
    }
}

}  // extern "C"
