// rope_attention_masked.cu -- the attention kernels of rope_attention.cuh
// instantiated with MASK = true: the softmax step reads the attn_mask bits of
// each key tile.  Calls without a mask never run these instances, so the mask
// costs them nothing (kept apart, the unmasked softmax keeps its registers).
#include "rope_attention.cuh"

namespace rope {

cudaError_t launch_attention_masked(const AttnArgs &a, int32_t D, int32_t layout, int32_t dtype,
                                    cudaStream_t st)
{
    return launch_attention_t<true>(a, D, layout, dtype, st);
}

}  // namespace rope
