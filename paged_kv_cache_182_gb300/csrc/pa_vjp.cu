// pa_vjp.cu -- dense attention backward (VJP): argument checks, workspace,
// the CUDA-core kernels, and the dispatch to the tensor-core kernels
// (pa_vjp_tc.cu).
//
// Operation: onnxruntime-ep-mlx 0.31.1, src/ops/attention_vjp/dense.rs,
// fn execute.  The page forms the whole score matrix; here it is never
// stored.  Three steps instead:
//
//   1. row statistics: for every query row, lse2 = log2 of the softmax
//      denominator in base-2 units (max + log2 sum, +inf for a row with no
//      visible key, so that every recomputed probability of it is 0), and
//      delta = rowsum(y * g).  It also zeroes the float32 dq accumulator.
//   2. one CTA per (batch, key/value head, tile of keys) walks every query
//      row of the group's query heads, recomputes p = exp2(s2 - lse2) and
//      ds = p (g.v - delta), keeps dk and dv of its keys on chip, and adds
//      its share of dq into the accumulator with atomics.
//   3. (16-bit dq only) the accumulator is rounded into dq.
//
// The CUDA-core kernels below take float32 inputs (and any input when asked
// for); they favour plainness over speed.

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <climits>
#include <cmath>
#include <cstdint>

#include "pa_attention_vjp.h"
#include "pa_common.cuh"
#include "pa_vjp.cuh"

namespace pa {
namespace {

constexpr int kStatRows = 8;   // query rows per CTA of the statistics kernel (one per warp)
constexpr int kStatKeys = 32;  // keys per staged tile of the statistics kernel
constexpr int kMainKeys = 16;  // keys per CTA of the CUDA-core backward
constexpr int kMainRows = 16;  // query rows per step of the CUDA-core backward
constexpr int kMaxD = 256;

template <typename T>
__device__ __forceinline__ float ldf(const T* p, int64_t i);
template <>
__device__ __forceinline__ float ldf<float>(const float* p, int64_t i) { return p[i]; }
template <>
__device__ __forceinline__ float ldf<__half>(const __half* p, int64_t i) { return __half2float(p[i]); }
template <>
__device__ __forceinline__ float ldf<__nv_bfloat16>(const __nv_bfloat16* p, int64_t i)
{
    return __bfloat162float(p[i]);
}

template <typename T>
__device__ __forceinline__ void stf(T* p, int64_t i, float x);
template <>
__device__ __forceinline__ void stf<float>(float* p, int64_t i, float x) { p[i] = x; }
template <>
__device__ __forceinline__ void stf<__half>(__half* p, int64_t i, float x) { p[i] = __float2half_rn(x); }
template <>
__device__ __forceinline__ void stf<__nv_bfloat16>(__nv_bfloat16* p, int64_t i, float x)
{
    p[i] = __float2bfloat16_rn(x);
}

__device__ __forceinline__ float warp_max(float x)
{
#pragma unroll
    for (int o = 16; o; o >>= 1)
        x = fmaxf(x, __shfl_xor_sync(0xffffffffu, x, o));
    return x;
}

__device__ __forceinline__ float warp_sum(float x)
{
#pragma unroll
    for (int o = 16; o; o >>= 1)
        x += __shfl_xor_sync(0xffffffffu, x, o);
    return x;
}

// Step 1.  grid (ceil(SQ / 8), HQ, B), 256 threads: warp w owns query row
// blockIdx.x * 8 + w; the CTA stages 32 keys at a time (float, rows padded
// to D + 1 so that 32 lanes reading 32 different keys hit 32 banks).
template <typename T>
__global__ void __launch_bounds__(256) vjp_stats_simt(VjpParams p)
{
    extern __shared__ float sm[];
    const int D = p.D, DP = D + 1;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int b = blockIdx.z, h = blockIdx.y, kh = h / p.groups;
    const int i = blockIdx.x * kStatRows + warp;
    const bool live = i < p.SQ;
    float* qrow = sm + warp * D;
    float* kt = sm + kStatRows * D;
    const int64_t row = (static_cast<int64_t>(b) * p.HQ + h) * p.SQ + (live ? i : 0);
    const T* q = static_cast<const T*>(p.q) + row * D;
    for (int d = lane; d < D; d += 32)
        qrow[d] = live ? ldf(q, d) * p.scale_log2 : 0.f;
    if (live) {
        const T* y = static_cast<const T*>(p.y) + row * D;
        const T* g = static_cast<const T*>(p.g) + row * D;
        float acc = 0.f;
        for (int d = lane; d < D; d += 32)
            acc = fmaf(ldf(y, d), ldf(g, d), acc);
        acc = warp_sum(acc);
        const int64_t srow = (static_cast<int64_t>(b) * p.HQ + h) * p.sqp + i;
        if (lane == 0)
            p.delta[srow] = acc;
        for (int d = lane; d < D; d += 32)
            p.dq_sum[row * D + d] = 0.f;
    }
    const T* kb = static_cast<const T*>(p.k) + (static_cast<int64_t>(b) * p.HK + kh) * p.SK * D;
    int kend = p.SK;
    if (p.causal)
        kend = min(kend, static_cast<int>(blockIdx.x) * kStatRows + kStatRows);
    float m = -INFINITY, l = 0.f;
    for (int j0 = 0; j0 < kend; j0 += kStatKeys) {
        __syncthreads();
        for (int e = threadIdx.x; e < kStatKeys * D; e += blockDim.x) {
            const int jj = e / D, d = e - jj * D;
            kt[jj * DP + d] = j0 + jj < p.SK ? ldf(kb, static_cast<int64_t>(j0 + jj) * D + d) : 0.f;
        }
        __syncthreads();
        const int j = j0 + lane;
        float s = -INFINITY;
        if (live && j < p.SK) {
            float dot = 0.f;
            for (int d = 0; d < D; ++d)
                dot = fmaf(qrow[d], kt[lane * DP + d], dot);
            s = dot + vjp_bias(p, b, h, i, j) * kVjpLog2e;
        }
        const float mn = fmaxf(m, warp_max(s));
        if (mn != -INFINITY) {
            const float e = s == -INFINITY ? 0.f : exp2f(s - mn);
            l = l * exp2f(m - mn) + warp_sum(e);
            m = mn;
        }
    }
    if (live && lane == 0)
        p.lse[(static_cast<int64_t>(b) * p.HQ + h) * p.sqp + i] = m == -INFINITY ? INFINITY : m + log2f(l);
}

// Step 2.  grid (ceil(SK / 16), HK, B), 256 threads.  Per step of 16 query
// rows of one head of the group: thread t computes the (key t / 16, row
// t % 16) entries of p and ds, then owns key t / 16 and columns t % 16 +
// 16 m of dk and dv (registers), then row t / 16 and the same columns of
// the step's dq (atomics into the accumulator).
template <typename T, typename TO>
__global__ void __launch_bounds__(256) vjp_main_simt(VjpParams p)
{
    extern __shared__ float sm[];
    const int D = p.D, DP = D + 1;
    float* Ks = sm;                       // [16][DP] keys (raw)
    float* Vs = Ks + kMainKeys * DP;      // [16][DP]
    float* Qs = Vs + kMainKeys * DP;      // [16][DP] rows of q (raw)
    float* Gs = Qs + kMainRows * DP;      // [16][DP] rows of g
    float* Ps = Gs + kMainRows * DP;      // [key][row], stride 17
    float* Ss = Ps + kMainKeys * 17;      // [key][row] scale * ds
    float* rl = Ss + kMainKeys * 17;      // [16] lse2 of the step's rows
    float* rd = rl + kMainRows;           // [16] delta
    const int t = threadIdx.x;
    const int b = blockIdx.z, kh = blockIdx.y, k0 = blockIdx.x * kMainKeys;
    const int64_t kvbase = (static_cast<int64_t>(b) * p.HK + kh) * p.SK;
    for (int e = t; e < kMainKeys * D; e += blockDim.x) {
        const int jj = e / D, d = e - jj * D;
        const bool in = k0 + jj < p.SK;
        Ks[jj * DP + d] = in ? ldf(static_cast<const T*>(p.k), (kvbase + k0 + jj) * D + d) : 0.f;
        Vs[jj * DP + d] = in ? ldf(static_cast<const T*>(p.v), (kvbase + k0 + jj) * D + d) : 0.f;
    }
    constexpr int kM = kMaxD / 16;
    float dk[kM], dv[kM];
#pragma unroll
    for (int m = 0; m < kM; ++m)
        dk[m] = dv[m] = 0.f;
    const int pj = t >> 4, pr = t & 15;  // phase 1: key, row
    const int i_start = p.causal ? min(k0, p.SQ) : 0;
    for (int gi = 0; gi < p.groups; ++gi) {
        const int h = kh * p.groups + gi;
        const int64_t qbase = (static_cast<int64_t>(b) * p.HQ + h) * p.SQ;
        const int64_t sbase = (static_cast<int64_t>(b) * p.HQ + h) * p.sqp;
        for (int i0 = i_start; i0 < p.SQ; i0 += kMainRows) {
            __syncthreads();  // the previous step is done with Qs, Gs, Ps, Ss
            for (int e = t; e < kMainRows * D; e += blockDim.x) {
                const int rr = e / D, d = e - rr * D;
                const bool in = i0 + rr < p.SQ;
                Qs[rr * DP + d] = in ? ldf(static_cast<const T*>(p.q), (qbase + i0 + rr) * D + d) : 0.f;
                Gs[rr * DP + d] = in ? ldf(static_cast<const T*>(p.g), (qbase + i0 + rr) * D + d) : 0.f;
            }
            if (t < kMainRows) {
                const bool in = i0 + t < p.SQ;
                rl[t] = in ? p.lse[sbase + i0 + t] : INFINITY;
                rd[t] = in ? p.delta[sbase + i0 + t] : 0.f;
            }
            __syncthreads();
            {
                const int key = k0 + pj, i = i0 + pr;
                float pv = 0.f, dsv = 0.f;
                if (key < p.SK && i < p.SQ) {
                    float s = 0.f, dp = 0.f;
                    for (int d = 0; d < D; ++d) {
                        s = fmaf(Qs[pr * DP + d], Ks[pj * DP + d], s);
                        dp = fmaf(Gs[pr * DP + d], Vs[pj * DP + d], dp);
                    }
                    const float s2 = s * p.scale_log2 + vjp_bias(p, b, h, i, key) * kVjpLog2e;
                    pv = exp2f(s2 - rl[pr]);
                    dsv = pv * (dp - rd[pr]) * p.scale;
                }
                Ps[pj * 17 + pr] = pv;
                Ss[pj * 17 + pr] = dsv;
            }
            __syncthreads();
            {
                const int key = t >> 4, c = t & 15;
                for (int rr = 0; rr < kMainRows; ++rr) {
                    const float pk = Ps[key * 17 + rr], sk = Ss[key * 17 + rr];
#pragma unroll
                    for (int m = 0; m < kM; ++m) {
                        const int d = c + 16 * m;
                        if (d < D) {
                            dv[m] = fmaf(pk, Gs[rr * DP + d], dv[m]);
                            dk[m] = fmaf(sk, Qs[rr * DP + d], dk[m]);
                        }
                    }
                }
            }
            {
                const int rr = t >> 4, c = t & 15, i = i0 + rr;
                if (i < p.SQ) {
                    float* acc = p.dq_sum;
#pragma unroll
                    for (int m = 0; m < kM; ++m) {
                        const int d = c + 16 * m;
                        if (d < D) {
                            float x = 0.f;
                            for (int jj = 0; jj < kMainKeys; ++jj)
                                x = fmaf(Ss[jj * 17 + rr], Ks[jj * DP + d], x);
                            if (x != 0.f)
                                atomicAdd(acc + (qbase + i) * D + d, x);
                        }
                    }
                }
            }
        }
    }
    const int key = k0 + (t >> 4), c = t & 15;
    if (key < p.SK) {
#pragma unroll
        for (int m = 0; m < kM; ++m) {
            const int d = c + 16 * m;
            if (d < D) {
                stf(static_cast<TO*>(p.dk), (kvbase + key) * D + d, dk[m]);
                stf(static_cast<TO*>(p.dv), (kvbase + key) * D + d, dv[m]);
            }
        }
    }
}

}  // namespace

// Step 3 (shared with the tensor-core path): dq = round(accumulator).
template <typename TO>
__global__ void __launch_bounds__(256) vjp_dq_round(const float* __restrict__ acc, TO* __restrict__ dq,
                                                     int64_t n)
{
    for (int64_t e = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; e < n;
         e += static_cast<int64_t>(gridDim.x) * blockDim.x)
        stf(dq, e, acc[e]);
}

namespace {

size_t round256(size_t x) { return (x + 255) & ~static_cast<size_t>(255); }

int out_type(int dtype, int out_dtype) { return out_dtype < 0 ? dtype : out_dtype; }

struct VjpLayout {
    size_t lse, delta, acc, total;
};

bool layout(int B, int HQ, int SQ, int D, int dtype, int out_dtype, VjpLayout* L)
{
    if (B < 0 || HQ < 1 || SQ < 0 || D < 1)
        return false;
    const size_t sqp = (static_cast<size_t>(SQ) + kVjpRowPad - 1) / kVjpRowPad * kVjpRowPad;
    const size_t rows = static_cast<size_t>(B) * HQ * sqp;
    L->lse = 0;
    L->delta = round256(rows * 4);
    L->acc = L->delta + round256(rows * 4);
    const bool need_acc = out_type(dtype, out_dtype) != PA_F32;
    L->total = L->acc + (need_acc ? round256(static_cast<size_t>(B) * HQ * SQ * D * 4) : 0);
    return true;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15) == 0; }

template <typename T, typename TO>
int launch_simt(const VjpParams& p, cudaStream_t st, uint64_t* launches)
{
    if (p.SQ > 0) {
        const size_t smem = (kStatRows * p.D + kStatKeys * (p.D + 1)) * sizeof(float);
        auto fn = vjp_stats_simt<T>;
        if (cudaFuncSetAttribute(reinterpret_cast<const void*>(fn),
                                 cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem)) !=
            cudaSuccess)
            return PA_ERR_CUDA;
        const dim3 grid((p.SQ + kStatRows - 1) / kStatRows, p.HQ, p.B);
        fn<<<grid, 256, smem, st>>>(p);
        if (cudaGetLastError() != cudaSuccess)
            return PA_ERR_CUDA;
        ++*launches;
    }
    if (p.SK > 0) {
        const size_t smem = ((kMainKeys + kMainKeys + kMainRows + kMainRows) * (p.D + 1) +
                             2 * kMainKeys * 17 + 2 * kMainRows) *
                            sizeof(float);
        auto fn = vjp_main_simt<T, TO>;
        if (cudaFuncSetAttribute(reinterpret_cast<const void*>(fn),
                                 cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem)) !=
            cudaSuccess)
            return PA_ERR_CUDA;
        const dim3 grid((p.SK + kMainKeys - 1) / kMainKeys, p.HK, p.B);
        fn<<<grid, 256, smem, st>>>(p);
        if (cudaGetLastError() != cudaSuccess)
            return PA_ERR_CUDA;
        ++*launches;
    }
    return PA_OK;
}

using SimtFn = int (*)(const VjpParams&, cudaStream_t, uint64_t*);

SimtFn pick_simt(int dtype, bool f32_out)
{
    if (dtype == PA_F32)
        return launch_simt<float, float>;
    if (dtype == PA_F16)
        return f32_out ? launch_simt<__half, float> : launch_simt<__half, __half>;
    return f32_out ? launch_simt<__nv_bfloat16, float> : launch_simt<__nv_bfloat16, __nv_bfloat16>;
}

}  // namespace
}  // namespace pa

using namespace pa;

extern "C" size_t pa_attention_vjp_workspace_bytes(int B, int HQ, int SQ, int D, int dtype, int out_dtype)
{
    VjpLayout L;
    if (dtype != PA_F32 && dtype != PA_F16 && dtype != PA_BF16)
        return 0;
    if (out_dtype != -1 && out_dtype != PA_F32 && out_dtype != dtype)
        return 0;
    if (!layout(B, HQ, SQ, D, dtype, out_dtype, &L))
        return 0;
    return L.total;
}

extern "C" int pa_attention_vjp(const void* q, const void* k, const void* v, const void* y, const void* g,
                                const void* mask, void* dq, void* dk, void* dv, float scale, int B, int HQ,
                                int HK, int SQ, int SK, int D, const pa_vjp_opts* opts, void* stream)
{
    if (!opts)
        return PA_ERR_NULL_POINTER;
    const pa_vjp_opts& o = *opts;
    if (B < 0 || HQ < 1 || HK < 1 || SQ < 0 || SK < 0 || D < 1 || HQ % HK != 0)
        return PA_ERR_BAD_DIMS;
    // a tensor with no elements may be NULL
    const bool rows = B > 0 && SQ > 0, keys = B > 0 && SK > 0;
    if ((rows && (!q || !y || !g || !dq)) || (keys && (!k || !v || !dk || !dv)))
        return PA_ERR_NULL_POINTER;
    if (!(scale > 0.f) || !std::isfinite(scale))
        return PA_ERR_BAD_DIMS;
    if (o.mask_kind < 0 || o.mask_kind > 2)
        return PA_ERR_BAD_DIMS;
    const int64_t qn = static_cast<int64_t>(B) * HQ * SQ * D, kn = static_cast<int64_t>(B) * HK * SK * D;
    if (qn >= (1ll << 31) || kn >= (1ll << 31))
        return PA_ERR_BAD_DIMS;
    if (o.mask_kind != 0) {
        if (!mask && rows && keys)
            return PA_ERR_NULL_POINTER;
        const int* md = o.mask_dims;
        if ((md[0] != 1 && md[0] != B) || (md[1] != 1 && md[1] != HQ) || (md[2] != 1 && md[2] != SQ) ||
            md[3] < 1 || md[3] > (SK > 0 ? SK : 1))
            return PA_ERR_BAD_DIMS;
        if (static_cast<int64_t>(md[0]) * md[1] * md[2] * md[3] >= (1ll << 31))
            return PA_ERR_BAD_DIMS;
    }
    if (o.dtype != PA_F32 && o.dtype != PA_F16 && o.dtype != PA_BF16)
        return PA_ERR_UNSUPPORTED;
    if (o.out_dtype != -1 && o.out_dtype != PA_F32 && o.out_dtype != o.dtype)
        return PA_ERR_UNSUPPORTED;
    if (D > kMaxD || B > 65535 || HQ > 65535)
        return PA_ERR_UNSUPPORTED;
    for (const void* t : {q, k, v, y, g, static_cast<const void*>(dq), static_cast<const void*>(dk),
                          static_cast<const void*>(dv)})
        if (!aligned16(t))
            return PA_ERR_ALIGNMENT;
    if (!rows && !keys)
        return PA_OK;
    VjpLayout L;
    layout(B, HQ, SQ, D, o.dtype, o.out_dtype, &L);
    if (!o.workspace)
        return PA_ERR_NULL_POINTER;
    if ((reinterpret_cast<uintptr_t>(o.workspace) & 255) != 0)
        return PA_ERR_ALIGNMENT;
    if (o.workspace_bytes < L.total)
        return PA_ERR_WORKSPACE;
    const int odt = out_type(o.dtype, o.out_dtype);
    unsigned char* ws = static_cast<unsigned char*>(o.workspace);
    VjpParams p{};
    p.q = q;
    p.k = k;
    p.v = v;
    p.y = y;
    p.g = g;
    p.mask = mask;
    p.dq = dq;
    p.dk = dk;
    p.dv = dv;
    p.lse = reinterpret_cast<float*>(ws + L.lse);
    p.delta = reinterpret_cast<float*>(ws + L.delta);
    p.dq_acc = odt == PA_F32 ? nullptr : reinterpret_cast<float*>(ws + L.acc);
    p.dq_sum = p.dq_acc ? p.dq_acc : static_cast<float*>(dq);
    p.status = o.status;
    p.wait_ns = o.wait_limit_ns ? o.wait_limit_ns : 1000000000ull;
    p.B = B;
    p.HQ = HQ;
    p.HK = HK;
    p.SQ = SQ;
    p.SK = SK;
    p.D = D;
    p.groups = HQ / HK;
    p.sqp = (SQ + kVjpRowPad - 1) / kVjpRowPad * kVjpRowPad;
    p.causal = o.causal ? 1 : 0;
    p.mask_kind = o.mask_kind;
    for (int e = 0; e < 4; ++e)
        p.md[e] = o.mask_kind ? o.mask_dims[e] : 1;
    p.scale = scale;
    p.scale_log2 = scale * kVjpLog2e;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    uint64_t launches = 0;
    int rc;
    if (o.kernel != 1 && vjp_tc_supported(o.dtype, D, HQ / HK, o.mask_kind))
        rc = launch_vjp_tc(p, o.dtype, odt == PA_F32, st, &launches);
    else
        rc = pick_simt(o.dtype, odt == PA_F32)(p, st, &launches);
    if (rc == PA_OK && p.dq_acc && SQ > 0) {
        const int64_t n = qn;
        const int blocks = static_cast<int>(std::min<int64_t>((n + 255) / 256, 152 * 16));
        if (odt == PA_F16)
            vjp_dq_round<__half><<<blocks, 256, 0, st>>>(p.dq_acc, static_cast<__half*>(dq), n);
        else
            vjp_dq_round<__nv_bfloat16><<<blocks, 256, 0, st>>>(p.dq_acc, static_cast<__nv_bfloat16*>(dq), n);
        rc = cudaGetLastError() == cudaSuccess ? PA_OK : PA_ERR_CUDA;
        ++launches;
    }
    count_launches(launches);
    return rc;
}
