// rope_apply_bf16.cu -- instantiates the rotation kernels for __nv_bfloat16 elements.
// One translation unit per element type so the library builds in parallel.
#include "rope_kernels.cuh"

namespace rope {

cudaError_t launch_apply_bf16(const ApplyArgs &a, int32_t layout, Variant v, cudaStream_t st)
{
    return launch_apply<__nv_bfloat16>(a, layout, v, st);
}

}  // namespace rope
