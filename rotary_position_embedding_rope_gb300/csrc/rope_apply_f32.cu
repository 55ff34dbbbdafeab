// rope_apply_f32.cu -- instantiates the rotation kernels for float elements.
// One translation unit per element type so the library builds in parallel.
#include "rope_kernels.cuh"

namespace rope {

cudaError_t launch_apply_f32(const ApplyArgs &a, int32_t layout, Variant v, cudaStream_t st)
{
    return launch_apply<float>(a, layout, v, st);
}

}  // namespace rope
