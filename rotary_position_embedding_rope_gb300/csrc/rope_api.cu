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
// the bulk-staged kernel ran out of its time budget.  One word per device; the
// kernels get its address as an argument.  g_flag_taken receives the value
// read-and-cleared by rope_check_errors.
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

struct Plan {
    ApplyArgs args;
    int32_t layout;
    int32_t dtype;
    Variant variant;
};

static rope_status plan_apply(void *q, void *k, const float *cos, const float *sin,
                              const int32_t *pos_idx, int64_t B, int32_t Hq, int32_t Hk, int64_t S,
                              int32_t D, int32_t rotary_dim, int32_t layout,
                              int32_t seq_before_head, int32_t backward, int32_t dtype,
                              int64_t table_rows, Plan *plan)
{
    std::memset(plan, 0, sizeof *plan);
    plan->variant = kNone;
    if (dtype != ROPE_F32 && dtype != ROPE_BF16 && dtype != ROPE_F16)
        return ROPE_ERR_UNSUPPORTED;
    if (layout != ROPE_SPLIT_HALF && layout != ROPE_INTERLEAVED)
        return ROPE_ERR_UNSUPPORTED;
    if ((seq_before_head != 0 && seq_before_head != 1) || (backward != 0 && backward != 1))
        return ROPE_ERR_INVALID_ARG;
    if (B < 0 || S < 0 || Hq < 0 || Hk < 0 || D < 1 || table_rows < 0)
        return ROPE_ERR_INVALID_ARG;
    if (rotary_dim < 2 || (rotary_dim & 1) || rotary_dim > D)
        return ROPE_ERR_INVALID_ARG;

    const int64_t elt = dtype == ROPE_F32 ? 4 : 2;
    const int64_t h = rotary_dim / 2;
    int64_t tok = 0, nq = 0, nk = 0, qbytes = 0, kbytes = 0, tab = 0, tabbytes = 0;
    if (!mul_ok(B, S, &tok) || !mul_ok(tok, (int64_t)Hq * D, &nq) ||
        !mul_ok(tok, (int64_t)Hk * D, &nk) || !mul_ok(nq, elt, &qbytes) ||
        !mul_ok(nk, elt, &kbytes) || !mul_ok(table_rows, h, &tab) || !mul_ok(tab, 4, &tabbytes))
        return ROPE_ERR_INVALID_ARG;
    if (tok == 0 || (int64_t)Hq + Hk == 0)
        return ROPE_OK;                                  // empty: nothing to launch

    if ((Hq > 0 && q == nullptr) || (Hk > 0 && k == nullptr) || cos == nullptr || sin == nullptr)
        return ROPE_ERR_INVALID_ARG;
    if (table_rows < 1 || (pos_idx == nullptr && S > table_rows))
        return ROPE_ERR_INVALID_ARG;
    if (ranges_overlap(q, qbytes, k, kbytes) || ranges_overlap(q, qbytes, cos, tabbytes) ||
        ranges_overlap(q, qbytes, sin, tabbytes) || ranges_overlap(k, kbytes, cos, tabbytes) ||
        ranges_overlap(k, kbytes, sin, tabbytes) || ranges_overlap(q, qbytes, pos_idx, S * 4) ||
        ranges_overlap(k, kbytes, pos_idx, S * 4))
        return ROPE_ERR_INVALID_ARG;

    ApplyArgs &a = plan->args;
    int n = 0;
    const int32_t heads[2] = {Hq, Hk};
    void *bases[2] = {q, k};
    for (int t = 0; t < 2; ++t) {
        if (heads[t] == 0)
            continue;
        TensorRef &r = a.t[n++];
        r.base = bases[t];
        r.heads = heads[t];
        if (seq_before_head) {                      // [B, S, H, D]
            r.stride_h = D;
            r.stride_s = (int64_t)heads[t] * D;
            r.stride_b = S * r.stride_s;
        } else {                                    // [B, H, S, D]
            r.stride_s = D;
            r.stride_h = S * D;
            r.stride_b = (int64_t)heads[t] * r.stride_h;
        }
    }
    a.ntensors = n;
    a.cos = cos;
    a.sin = sin;
    a.pos_idx = pos_idx;
    a.B = B;
    a.S = S;
    a.D = D;
    a.rotary_dim = rotary_dim;
    a.table_rows = table_rows;
    a.backward = backward;
    plan->layout = layout;
    plan->dtype = dtype;

    // 16-byte vectors need: a rotary span of whole vector pairs, 16-byte
    // aligned rows, aligned base pointers and tables, and NJ within a CTA.
    const int64_t span_bytes = rotary_dim * elt;
    bool vec = (span_bytes % 32) == 0 && ((int64_t)D * elt) % 16 == 0 && aligned16(cos) &&
               aligned16(sin) && span_bytes / 32 <= kMaxVectorsPerHalf;
    for (int t = 0; t < n; ++t)
        vec = vec && aligned16(a.t[t].base);
    const int32_t forced = g_forced_variant.load(std::memory_order_relaxed);
    if (forced == kScalar)
        plan->variant = kScalar;
    else if (forced == kBulk || forced == kVector) {
        if (!vec)
            return ROPE_ERR_UNSUPPORTED;
        plan->variant = static_cast<Variant>(forced);
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

rope_status rope_apply_qk(void *q, void *k, const float *cos, const float *sin,
                          const int32_t *pos_idx, int64_t B, int32_t Hq, int32_t Hk, int64_t S,
                          int32_t D, int32_t rotary_dim, int32_t layout, int32_t seq_before_head,
                          int32_t backward, int32_t dtype, int64_t table_rows, void *stream)
{
    Plan plan;
    rope_status st = plan_apply(q, k, cos, sin, pos_idx, B, Hq, Hk, S, D, rotary_dim, layout,
                                seq_before_head, backward, dtype, table_rows, &plan);
    if (st != ROPE_OK || plan.variant == kNone)
        return st;
    int32_t *taken = nullptr;
    if (flag_addresses(&plan.args.range_flag, &taken) != cudaSuccess)
        return ROPE_ERR_CUDA;
    return launch_plan(plan, static_cast<cudaStream_t>(stream));
}

rope_status rope_apply_q(void *x, const float *cos, const float *sin, const int32_t *pos_idx,
                         int64_t B, int32_t H, int64_t S, int32_t D, int32_t rotary_dim,
                         int32_t layout, int32_t seq_before_head, int32_t backward, int32_t dtype,
                         int64_t table_rows, void *stream)
{
    return rope_apply_qk(x, nullptr, cos, sin, pos_idx, B, H, 0, S, D, rotary_dim, layout,
                         seq_before_head, backward, dtype, table_rows, stream);
}

int32_t rope_qk_kernel_variant(const void *q, const void *k, const float *cos, const float *sin,
                               const int32_t *pos_idx, int64_t B, int32_t Hq, int32_t Hk,
                               int64_t S, int32_t D, int32_t rotary_dim, int32_t layout,
                               int32_t seq_before_head, int32_t backward, int32_t dtype,
                               int64_t table_rows)
{
    Plan plan;
    rope_status st = plan_apply(const_cast<void *>(q), const_cast<void *>(k), cos, sin, pos_idx,
                                B, Hq, Hk, S, D, rotary_dim, layout, seq_before_head, backward,
                                dtype, table_rows, &plan);
    return st == ROPE_OK ? (int32_t)plan.variant : 0;
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

rope_status rope_force_kernel_variant(int32_t variant)
{
    if (variant < 0 || variant > 3)
        return ROPE_ERR_INVALID_ARG;
    g_forced_variant.store(variant, std::memory_order_relaxed);
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
