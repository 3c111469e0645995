// Kernel instantiations for float16 inputs (float16 or float32 output):
// tensor-core path.
#include "pa_kernels.cuh"

namespace pa {
SplitFn pick_split_f16(bool f32_out, int D, int MT)
{
    return f32_out ? pick_split_mma<__half, float>(D, MT) : pick_split_mma<__half, __half>(D, MT);
}
CombineFn pick_combine_f16(int D) { return pick_combine_typed<__half>(D); }
}  // namespace pa
