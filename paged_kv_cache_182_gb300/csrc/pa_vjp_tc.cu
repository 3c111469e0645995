// pa_vjp_tc.cu -- tcgen05 kernels of the attention backward (placeholder
// until they land: every size takes the CUDA-core kernels).
#include "pa_decode.h"
#include "pa_vjp.cuh"

namespace pa {

bool vjp_tc_supported(int, int, int) { return false; }

int launch_vjp_tc(const VjpParams&, int, bool, cudaStream_t, uint64_t*) { return PA_ERR_UNSUPPORTED; }

}  // namespace pa
