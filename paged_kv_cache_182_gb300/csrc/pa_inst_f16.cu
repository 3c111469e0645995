// Kernel instantiations for float16 inputs (float16 or float32 output).
#include "pa_kernels.cuh"

namespace pa {
SplitFn pick_split_f16(bool f32_out, int D, int RG)
{
    return f32_out ? pick_split_typed<__half, float>(D, RG) : pick_split_typed<__half, __half>(D, RG);
}
CombineFn pick_combine_f16(int D) { return pick_combine_typed<__half>(D); }
}  // namespace pa
