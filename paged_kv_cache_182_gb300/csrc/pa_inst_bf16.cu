// Kernel instantiations for bfloat16 inputs (bfloat16 or float32 output):
// tensor-core path.
#include "pa_kernels.cuh"

namespace pa {
SplitFn pick_split_bf16(bool f32_out, int D, int MT)
{
    return f32_out ? pick_split_mma<__nv_bfloat16, float>(D, MT)
                   : pick_split_mma<__nv_bfloat16, __nv_bfloat16>(D, MT);
}
CombineFn pick_combine_bf16(int D) { return pick_combine_typed<__nv_bfloat16>(D); }
}  // namespace pa
