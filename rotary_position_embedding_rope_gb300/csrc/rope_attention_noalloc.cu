// rope_attention_noalloc.cu -- rope_attention_fwd_noalloc: the rotary
// attention with its key workspace in a fixed device array of this library,
// for callers that cannot allocate device memory when they call it.
//
// Who needs it: a serving engine or framework that reserves (nearly) all of
// the device's memory for its own pool at start-up, plugin code that may only
// use memory handed to it by its host framework, and code on a
// latency-critical path where a cudaMalloc (which can synchronise the device)
// is not acceptable.  Such a caller still passes q, k, v, o and the tables;
// the rot(K) buffer that rope_attention_fwd takes as k_workspace comes from
// g_key_scratch below instead.
//
// The array has a fixed size (kKeyScratchBytes, 32 MiB) and is held by every
// device that loads this library, until the process exits.  Calls share it:
// each call overwrites the B * Hk * Sk * D elements it uses (the rotation
// kernel writes every element, rotated or copied, so nothing needs clearing
// first), and two calls whose work overlaps on the GPU (different streams, no
// ordering between them) race on it.
#include <cstdint>
#include <mutex>

#include <cuda_runtime.h>

#include "rope.h"

namespace {

constexpr int64_t kKeyScratchBytes = 32ll << 20;
constexpr int kMaxDevices = 64;

// Device storage of the rotated keys.  In host code this name is only a
// host-side handle of the symbol, not a device address: the address kernels
// may use comes from cudaGetSymbolAddress, per device.
static __device__ __align__(256) uint8_t g_key_scratch[kKeyScratchBytes];

void *g_scratch_addr[kMaxDevices];
std::mutex g_scratch_mutex;

// Device address of g_key_scratch on the current device, looked up once per
// device (with that device current) and then cached.  The cache is never
// invalidated: a process that resets a device must restart before calling
// rope_attention_fwd_noalloc again.
cudaError_t scratch_address(void **out)
{
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess)
        return e;
    if (dev < 0 || dev >= kMaxDevices)
        return cudaErrorInvalidDevice;
    std::lock_guard<std::mutex> lock(g_scratch_mutex);
    if (g_scratch_addr[dev] == nullptr) {
        void *p = nullptr;
        e = cudaGetSymbolAddress(&p, g_key_scratch);
        if (e != cudaSuccess)
            return e;
        g_scratch_addr[dev] = p;
    }
    *out = g_scratch_addr[dev];
    return cudaSuccess;
}

}  // namespace

namespace rope {
// rope_attention_fwd's host checks (rope_api.cu), without a workspace.
rope_status attention_args_status(const void *q, const void *k, const void *v, void *o,
                                  const float *cos, const float *sin, const int32_t *pos_q,
                                  const int32_t *pos_k, int64_t B, int32_t Hq, int32_t Hk,
                                  int64_t Sq, int64_t Sk, int32_t D, int32_t rotary_dim,
                                  int32_t layout, int32_t causal, float softmax_scale,
                                  int32_t dtype, int64_t table_rows);
}  // namespace rope

extern "C" rope_status rope_attention_fwd_noalloc(
    const void *q, const void *k, const void *v, void *o, const float *cos, const float *sin,
    const int32_t *pos_q, const int32_t *pos_k, int64_t B, int32_t Hq, int32_t Hk, int64_t Sq,
    int64_t Sk, int32_t D, int32_t rotary_dim, int32_t layout, int32_t causal,
    float softmax_scale, int32_t dtype, int64_t table_rows, void *stream)
{
    // the arguments first, as rope_attention_fwd checks them (an empty call
    // is accepted there and needs nothing of the array)
    const rope_status st =
        rope::attention_args_status(q, k, v, o, cos, sin, pos_q, pos_k, B, Hq, Hk, Sq, Sk, D,
                                    rotary_dim, layout, causal, softmax_scale, dtype, table_rows);
    if (st != ROPE_OK)
        return st;
    // rot(K) needs B * Hk * Sk * D elements of 2 bytes; larger calls do not
    // fit the array (checked before anything touches the device)
    int64_t n = 0, bytes = 0;
    if (__builtin_mul_overflow(B, (int64_t)Hk, &n) || __builtin_mul_overflow(n, Sk, &n) ||
        __builtin_mul_overflow(n, (int64_t)D * 2, &bytes))
        return ROPE_ERR_INVALID_ARG;
    if (bytes > kKeyScratchBytes)
        return ROPE_ERR_UNSUPPORTED;
    void *scratch = nullptr;
    if (bytes > 0 && scratch_address(&scratch) != cudaSuccess)
        return ROPE_ERR_CUDA;
    return rope_attention_fwd(q, k, v, o, cos, sin, pos_q, pos_k, B, Hq, Hk, Sq, Sk, D,
                              rotary_dim, layout, causal, softmax_scale, dtype, table_rows, scratch,
                              scratch != nullptr ? kKeyScratchBytes : 0, stream);
}
