// Kernel instantiations for bfloat16 inputs (bfloat16 or float32 output).
#include "pa_kernels.cuh"

namespace pa {
SplitFn pick_split_bf16(bool f32_out, int D, int RG)
{
    return f32_out ? pick_split_typed<__nv_bfloat16, float>(D, RG)
                   : pick_split_typed<__nv_bfloat16, __nv_bfloat16>(D, RG);
}
CombineFn pick_combine_bf16(int D) { return pick_combine_typed<__nv_bfloat16>(D); }
}  // namespace pa
