// rope_attention.cu -- the attention entry point of librope without an
// attn_mask (the kernels of rope_attention.cuh instantiated with MASK = false;
// rope_attention_masked.cu holds the masked ones, compiled in parallel), and
// the probe of the bounded-wait expiry path.
#include "rope_attention.cuh"

namespace rope {

cudaError_t launch_attention(const AttnArgs &a, int32_t D, int32_t layout, int32_t dtype,
                             cudaStream_t st)
{
    if (a.mask_kind != 0)
        return launch_attention_masked(a, D, layout, dtype, st);
    return launch_attention_t<false>(a, D, layout, dtype, st);
}

// Probe of the expiry path: one thread waits, with the attention kernels'
// bounded wait, on a barrier that nothing arrives at; after `cycles` clock
// cycles the wait gives up and the thread records the expiry as those kernels
// do (bit 1 of the device flag).  Nothing else runs, so nothing stalls.
__global__ void rope_wait_probe_kernel(int32_t *flag, long long cycles)
{
    __shared__ __align__(8) uint64_t bar;
    if (threadIdx.x == 0)
        mbar_init(&bar, 1);
    __syncthreads();
    if (threadIdx.x == 0 && !attn_wait(&bar, 0u, nullptr, cycles))
        atomicOr(flag, 2);
}

cudaError_t launch_wait_probe(int32_t *flag, long long cycles, cudaStream_t st)
{
    rope_wait_probe_kernel<<<1, 32, 0, st>>>(flag, cycles);
    return cudaGetLastError();
}


}  // namespace rope
