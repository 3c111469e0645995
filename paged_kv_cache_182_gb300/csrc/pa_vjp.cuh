// pa_vjp.cuh -- shared declarations of the attention backward kernels
// (pa_vjp.cu: checks, CUDA-core kernels, dispatch; pa_vjp_tc.cu: tcgen05
// kernels).
#pragma once

#include <cuda_runtime.h>

#include <cstdint>

namespace pa {

constexpr float kVjpLog2e = 1.4426950408889634f;
// Row statistics (lse2, delta) of each (batch, query head) start at a
// multiple of this many rows, so a 128-row tile of them is one aligned copy.
constexpr int kVjpRowPad = 128;

struct VjpParams {
    const void* q;
    const void* k;
    const void* v;
    const void* y;
    const void* g;
    const void* mask;
    void* dq;
    void* dk;
    void* dv;
    float* lse;     // [B][HQ][sqp] log2 of the softmax denominator, +inf on empty rows
    float* delta;   // [B][HQ][sqp] rowsum(y * g)
    float* dq_acc;  // [B][HQ][SQ][D] float32 dq accumulator; NULL when dq itself is float32
    float* dq_sum;  // where dq is accumulated: dq_acc, or dq when it is float32
    int* status;
    unsigned long long wait_ns;
    int B, HQ, HK, SQ, SK, D, groups, sqp, causal, mask_kind;
    int md[4];  // mask dims MB, MH, MQ, W
    float scale, scale_log2;
};

// Additive bias of score (b, h, i, j) in natural-log units: the causal rule
// (key j hidden from row i when j > i), then the mask (boolean: 0 or -inf;
// additive: the value; keys at or past a width W > 1 hidden).
__device__ __forceinline__ float vjp_bias(const VjpParams& p, int b, int h, int i, int j)
{
    if (p.causal && j > i)
        return -INFINITY;
    if (p.mask_kind == 0)
        return 0.f;
    int jj = 0;
    if (p.md[3] != 1) {
        if (j >= p.md[3])
            return -INFINITY;
        jj = j;
    }
    const int64_t idx =
        ((static_cast<int64_t>(p.md[0] == 1 ? 0 : b) * p.md[1] + (p.md[1] == 1 ? 0 : h)) * p.md[2] +
         (p.md[2] == 1 ? 0 : i)) * p.md[3] + jj;
    if (p.mask_kind == 1)
        return static_cast<const uint8_t*>(p.mask)[idx] ? 0.f : -INFINITY;
    return static_cast<const float*>(p.mask)[idx];
}

// Tensor-core path (pa_vjp_tc.cu): whether these sizes take it, and its
// launches (row statistics and the backward; dq rounding is left to the
// caller).  Returns PA_OK or a PA_ERR_* code.
bool vjp_tc_supported(int dtype, int D, int groups, int mask_kind);
int launch_vjp_tc(const VjpParams& p, int dtype, bool f32_out, cudaStream_t st, uint64_t* launches);

// Adds to the library's count of kernel launches (pa_kernel_launches).
void count_launches(uint64_t n);

}  // namespace pa
