// rope_apply_f16.cu -- instantiates the rotation kernels for __half elements.
// One translation unit per element type so the library builds in parallel.
#include "rope_kernels.cuh"

namespace rope {

cudaError_t launch_apply_f16(const ApplyArgs &a, int32_t layout, Variant v, cudaStream_t st)
{
    return launch_apply<__half>(a, layout, v, st);
}

}  // namespace rope
