// Kernel instantiations for float32 inputs (float32 output): CUDA-core path.
#include "pa_kernels.cuh"

namespace pa {
SplitFn pick_split_f32(int D, int RG) { return pick_split_simt<float, float>(D, RG); }
CombineFn pick_combine_f32(int D) { return pick_combine_typed<float>(D); }
}  // namespace pa
