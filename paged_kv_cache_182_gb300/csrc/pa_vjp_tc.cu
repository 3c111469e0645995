// pa_vjp_tc.cu -- the attention backward on the sm_103a tensor cores
// (tcgen05 MMAs from shared-memory descriptors, accumulators in tensor
// memory, operands staged by TMA), for 16-bit inputs with D = 128 and no
// mask beyond the causal rule.
//
// Operation: onnxruntime-ep-mlx 0.31.1, src/ops/attention_vjp/dense.rs,
// fn execute (p, dv = p^T g, dp = g v^T, delta = rowsum(y g),
// ds = p (dp - delta), dq = scale ds k, dk = scale ds^T q, the group sums of
// dk and dv, causal ki <= qi, p = 0 on rows with no visible key).
//
// Two kernels:
//
// vjp_stats_tc -- persistent (one CTA per SM), over items of (batch, query
//   head, 128 query rows) dealt longest first in a snake order:
//   S = Q K^T per 128-key tile (M 128 rows, N 128 keys, K = D; both operands
//   K-major), double-buffered in tensor memory; two threads a row (64 key
//   columns each) keep a running maximum and sum in base 2 over all tiles
//   and merge them at the end: lse2 = max + log2(sum), +inf for a row that
//   sees no key.  Warp 8 loads Q (two buffers: the next item's tile lands
//   while the current one is in use) and K tiles into a four-stage ring
//   that runs on across items; warp 9 issues the MMAs.  Warps 10-13 compute
//   delta = rowsum(y g) and zero the float32 dq accumulator rows of the same
//   items, with no wait on the others (plain coalesced loads and stores).
//
// vjp_main_tc -- one CTA per (batch, key/value head, 128 keys): K and V of
//   the tile stay in shared memory; dK and dV accumulate in tensor memory
//   over every 128-row step of every query head of the group.  Per step:
//     S^T  = K Q^T          M 128 keys, N 128 rows, K = D     (both K-major)
//     dP^T = V dO^T         same shapes
//     softmax threads: P = exp2(s2 - lse2), written back over S^T in tensor
//                      memory as 16-bit pairs; dS^T = P (dP^T - delta) scale,
//                      written to shared memory as a 16-bit operand
//     dV  += P dO           M 128 keys, N = D, K 128 rows     (P from tensor
//                                                              memory, dO MN-major)
//     dK  += dS^T Q         same, dS^T K-major, Q MN-major
//     dQ^T = K^T dS^T       M = D, N 128 rows, K 128 keys     (both MN-major),
//                           into the dP^T columns the softmax has read
//   and the same threads read dQ^T back and add it into the float32
//   accumulator (one reduction per element, coalesced over D; half of a
//   thread's rows at once, the other half in the next step, under its dK
//   and dQ^T products).  Every MMA
//   has N = 128: a tcgen05 MMA of M = 128 costs at least as much as N = 64
//   does.  Warp 16 loads K, V once and Q, dO, lse2, delta per step into a
//   two-stage ring; warp 17 issues the MMAs (one thread).  Tensor memory
//   (512 columns): dK | dV | S^T (then P) | dP^T (then dQ^T).
//
// Every wait is bounded (p.wait_ns); a wait that gives up ORs
// PA_STATUS_TIMEOUT into p.status, and every path frees the tensor memory.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include <cstdint>
#include <type_traits>

#include "pa_decode.h"
#include "pa_ptx.cuh"
#include "pa_tc.cuh"
#include "pa_tmem.cuh"
#include "pa_vjp.cuh"

namespace pa {
namespace {

using namespace tc;

constexpr unsigned kAll = 0xffffffffu;
constexpr int kD = 128;         // head size of this path
constexpr int kKeys = 128;      // keys per tile (both kernels)
constexpr int kSRows = 128;     // query rows per CTA of the statistics kernel
constexpr int kSoftmax = 256;   // statistics kernel: warps 0-7 softmax, 8 TMA, 9 MMA,
constexpr int kDeltaWarps = 4;  // 10-13 delta and dq zeroing
constexpr int kStatsThreads = kSoftmax + 64 + kDeltaWarps * 32;
constexpr int kKStages = 4;     // statistics kernel: K ring depth
constexpr int kHalf128 = 16384;  // one 64-column half of a 128-row tile, bytes

struct StatsBars {
    uint64_t q_full[2], q_empty[2], k_full[kKStages], k_empty[kKStages], s_full[2], s_free[2], fin;
    uint32_t tmem;
    int abort;
    float xm[2][kSRows], xl[2][kSRows];  // the high-half thread's max and sum, by item parity
};
// Q (2 buffers x 2 halves), K ring (kKStages stages x 2 halves), then the barriers
constexpr int kStatsBarBytes = 4096;
constexpr int kStatsSmem = (4 + 2 * kKStages) * kHalf128 + kStatsBarBytes;
static_assert(sizeof(StatsBars) <= kStatsBarBytes, "statistics barrier area");
static_assert(kStatsSmem <= 232448, "statistics shared memory");

// Item k of CTA c among G: longest first, the direction reversed every round
// (snake), so that every CTA's share of the tiles is about the same.
__device__ __forceinline__ int stats_item(int k, int c, int G) { return (k & 1) ? (k + 1) * G - 1 - c : k * G + c; }

struct StatsItem {
    int b, h, i0, nk, ntiles;
};

__device__ __forceinline__ StatsItem stats_item_at(const VjpParams& p, int n, int tiles)
{
    StatsItem it;
    const int bh = n % (p.B * p.HQ);
    it.b = bh / p.HQ;
    it.h = bh % p.HQ;
    it.i0 = (tiles - 1 - n / (p.B * p.HQ)) * kSRows;
    it.nk = p.causal ? min(p.SK, it.i0 + kSRows) : p.SK;
    it.ntiles = (it.nk + kKeys - 1) / kKeys;
    return it;
}

struct MainBars {
    uint64_t kv_full, qd_full[2], qd_empty[2], s_full, dp_full, p_ready, ds_ready, dq_full, dq_free, mma_done;
    uint32_t tmem;
    int abort;
};
constexpr int kBRows = 128;                            // query rows per step of the backward kernel
constexpr int kMSoftmax = 512;                         // warps 0-15: softmax and dQ^T, 32 rows a thread
constexpr int kMainThreads = kMSoftmax + 64;           // + warp 16 TMA, warp 17 MMA: 576
// K, V (2 halves of 16 KB each), the Q and dO rings (2 stages x 2 halves of
// 16 KB), dS^T (2 halves of 16 KB: rows 0-63 and 64-127), row statistics
// (2 stages x 1 KB), barriers
constexpr int kMainSmem = 4 * kHalf128 + 8 * kHalf128 + 2 * kHalf128 + 2 * 1024 + 512;
static_assert(sizeof(MainBars) <= 512, "backward barrier area");
static_assert(kMainSmem <= 232448, "backward shared memory");

__device__ __forceinline__ void red_add(float* addr, float v)
{
    asm volatile("red.global.add.f32 [%0], %1;" ::"l"(addr), "f"(v) : "memory");
}

template <typename T>
__device__ __forceinline__ uint32_t pack2(float a, float b)
{
    if constexpr (std::is_same<T, __nv_bfloat16>::value) {
        const __nv_bfloat162 h = __floats2bfloat162_rn(a, b);
        return *reinterpret_cast<const uint32_t*>(&h);
    } else {
        const __half2 h = __floats2half2_rn(a, b);
        return *reinterpret_cast<const uint32_t*>(&h);
    }
}

template <typename T>
__device__ __forceinline__ float2 unpack2(uint32_t w)
{
    if constexpr (std::is_same<T, __nv_bfloat16>::value)
        return __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&w));
    else
        return __half22float2(*reinterpret_cast<const __half2*>(&w));
}

// ---------------------------------------------------------------------------
// Row statistics.  grid = min(items, SMs); items = B * HQ * ceil(SQ / 128),
// numbered row tile slowest, the row tiles that see the most keys (causal)
// first.
template <typename T>
__global__ void __launch_bounds__(kStatsThreads, 1)
    vjp_stats_tc(const __grid_constant__ VjpParams p, const __grid_constant__ CUtensorMap qmap,
                 const __grid_constant__ CUtensorMap kmap)
{
    constexpr bool kBf = std::is_same<T, __nv_bfloat16>::value;
    extern __shared__ __align__(1024) unsigned char smem_raw[];
    if ((smem_u32(smem_raw) & 1023u) != 0) {
        if (threadIdx.x == 0 && p.status)
            atomicOr(p.status, PA_STATUS_TIMEOUT);
        return;
    }
    unsigned char* sQ = smem_raw;                  // buffer u at u * 2 * kHalf128
    unsigned char* sK = smem_raw + 4 * kHalf128;   // stage s at s * 2 * kHalf128
    StatsBars& bars = *reinterpret_cast<StatsBars*>(smem_raw + (4 + 2 * kKStages) * kHalf128);

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int tiles = (p.SQ + kSRows - 1) / kSRows;
    const int total = p.B * p.HQ * tiles;
    const int C = static_cast<int>(blockIdx.x), G = static_cast<int>(gridDim.x);
    const uint64_t wait_ns = p.wait_ns;

    if (tid == 0) {
        for (int u = 0; u < 2; ++u) {
            mbar_init(&bars.q_full[u], 1);
            mbar_init(&bars.q_empty[u], 1);
            mbar_init(&bars.s_full[u], 1);
            mbar_init(&bars.s_free[u], kSoftmax / 32);  // one arrival per softmax warp
        }
        for (int s = 0; s < kKStages; ++s) {
            mbar_init(&bars.k_full[s], 1);
            mbar_init(&bars.k_empty[s], 1);
        }
        mbar_init(&bars.fin, 1);
        bars.abort = 0;
        fence_mbar_init();
    }
    if (warp == 0) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                         smem_u32(&bars.tmem)),
                     "r"(256)
                     : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tS = bars.tmem;  // S of key tile g (counted over the CTA's items) at tS + 128 (g & 1)
    volatile int* abort_flag = &bars.abort;
    auto fail = [&]() {
        *abort_flag = 1;
        if (p.status)
            atomicOr(p.status, PA_STATUS_TIMEOUT);
    };

    if (warp == 8) {
        // --------------------------------------------------------------- TMA
        if (lane == 0) {
            tma_prefetch_desc(&qmap);
            tma_prefetch_desc(&kmap);
            int qn = 0, g = 0;  // Q tiles and K tiles issued
            bool ok = true;
            for (int k = 0; ok; ++k) {
                const int n = stats_item(k, C, G);
                if (n >= total)
                    break;
                const StatsItem it = stats_item_at(p, n, tiles);
                if (it.ntiles == 0)
                    continue;
                const int u = qn & 1;
                if (qn >= 2 && (*abort_flag || !mbar_wait_bounded(&bars.q_empty[u], ((qn >> 1) - 1) & 1, wait_ns))) {
                    ok = false;
                    break;
                }
                mbar_arrive_expect_tx(&bars.q_full[u], 2 * kHalf128);
                for (int hh = 0; hh < 2; ++hh)
                    tma_load_4d(sQ + u * 2 * kHalf128 + hh * kHalf128, &qmap, 0, hh, it.i0, it.b * p.HQ + it.h,
                                &bars.q_full[u]);
                ++qn;
                const int kh = it.h / p.groups;
                for (int t = 0; t < it.ntiles; ++t, ++g) {
                    const int s = g % kKStages;
                    if (g >= kKStages &&
                        (*abort_flag || !mbar_wait_bounded(&bars.k_empty[s], ((g / kKStages) - 1) & 1, wait_ns))) {
                        ok = false;
                        break;
                    }
                    mbar_arrive_expect_tx(&bars.k_full[s], 2 * kHalf128);
                    for (int hh = 0; hh < 2; ++hh)
                        tma_load_4d(sK + s * 2 * kHalf128 + hh * kHalf128, &kmap, 0, hh, t * kKeys, it.b * p.HK + kh,
                                    &bars.k_full[s]);
                }
            }
            if (!ok)
                fail();
            // no copy may land after the CTA's memory is released
            for (int t = g > kKStages ? g - kKStages : 0; t < g; ++t)
                mbar_wait_bounded(&bars.k_full[t % kKStages], (t / kKStages) & 1, wait_ns);
            for (int q = qn > 2 ? qn - 2 : 0; q < qn; ++q)
                mbar_wait_bounded(&bars.q_full[q & 1], (q >> 1) & 1, wait_ns);
        }
        __syncwarp();
    } else if (warp == 9) {
        // --------------------------------------------------------------- MMA
        if (lane == 0) {
            const uint32_t ka = smem_u32(sK);
            const uint32_t id = idesc<kBf>(kKeys, false);
            int qn = 0, g = 0;
            bool ok = true, issued = false;
            for (int k = 0; ok; ++k) {
                const int n = stats_item(k, C, G);
                if (n >= total)
                    break;
                const StatsItem it = stats_item_at(p, n, tiles);
                if (it.ntiles == 0)
                    continue;
                const int u = qn & 1;
                const uint32_t qa = smem_u32(sQ + u * 2 * kHalf128);
                ok = !*abort_flag && mbar_wait_bounded(&bars.q_full[u], (qn >> 1) & 1, wait_ns);
                for (int t = 0; t < it.ntiles && ok; ++t, ++g) {
                    const int s = g & 1, ks = g % kKStages;
                    ok = !*abort_flag && mbar_wait_bounded(&bars.k_full[ks], (g / kKStages) & 1, wait_ns);
                    if (ok && g >= 2)
                        ok = mbar_wait_bounded(&bars.s_free[s], ((g >> 1) - 1) & 1, wait_ns);
                    if (!ok)
                        break;
                    tc_fence_after();
                    const uint32_t kb = ka + ks * 2 * kHalf128;
                    for (int kk = 0; kk < kD / 16; ++kk) {
                        const uint32_t o = (kk >> 2) * kHalf128 + (kk & 3) * 32;
                        umma(tS + s * kKeys, smem_desc(qa + o, 16, 1024), smem_desc(kb + o, 16, 1024), id, kk > 0);
                    }
                    issued = true;
                    umma_commit(&bars.s_full[s]);
                    umma_commit(&bars.k_empty[ks]);
                }
                if (!ok)
                    break;
                umma_commit(&bars.q_empty[u]);  // this Q buffer is free once the item's MMAs complete
                ++qn;
            }
            if (!ok)
                fail();
            // every MMA completes before the tensor memory is released
            if (issued) {
                umma_commit(&bars.fin);
                mbar_wait_bounded(&bars.fin, 0, wait_ns);
            }
        }
        __syncwarp();
    } else if (warp < kSoftmax / 32) {
        // ------------------------------------------ statistics (two threads a row)
        const int row = (warp & 3) * 32 + lane;
        const int part = warp >> 2;  // key columns [64 part, 64 part + 64)
        const uint32_t lane_off = static_cast<uint32_t>((warp & 3) * 32) << 16;
        bool fault = false;
        int g = 0;
        for (int k = 0;; ++k) {
            const int n = stats_item(k, C, G);
            if (n >= total)
                break;
            const StatsItem it = stats_item_at(p, n, tiles);
            const int i = it.i0 + row;
            float m = -INFINITY, l = 0.f;
            for (int t = 0; t < it.ntiles && !fault; ++t, ++g) {
                const int s = g & 1;
                const bool got = __all_sync(
                    kAll, !*abort_flag && mbar_wait_bounded(&bars.s_full[s], (g >> 1) & 1, wait_ns));
                if (!got) {
                    fault = true;
                    if (lane == 0)
                        fail();  // the other roles stop at their next wait
                    break;
                }
                tc_fence_after();
                // raw scores (scale > 0 commutes with the maximum); eight
                // independent partial maxima and sums keep the dependency chains short
                float sc[64];
                float pm8[8];
#pragma unroll
                for (int e = 0; e < 8; ++e)
                    pm8[e] = -INFINITY;
                const int kbase = t * kKeys + part * 64;
                Cols32 xs[2];
                tmem_ld32_issue(xs[0], tS + s * kKeys + lane_off + part * 64);
                tmem_ld32_issue(xs[1], tS + s * kKeys + lane_off + part * 64 + 32);
                tmem_ld_wait(xs[1]);
                tmem_ld_wait(xs[0]);
                // the mask test is taken once per tile (warp-uniform), never per
                // score: a branch per score cost more than the rest of the tile
                if (kbase + 63 >= it.nk || (p.causal && kbase + 63 > it.i0)) {
                    // keys kbase + jj with jj < lim are visible to row i
                    const int lim = min(p.SK, p.causal ? i + 1 : p.SK) - kbase;
#pragma unroll
                    for (int c = 0; c < 2; ++c)
#pragma unroll
                        for (int j = 0; j < 32; ++j) {
                            const float v = c * 32 + j < lim ? __uint_as_float(xs[c].r[j]) : -INFINITY;
                            sc[c * 32 + j] = v;
                            pm8[j & 7] = fmaxf(pm8[j & 7], v);
                        }
                } else {
#pragma unroll
                    for (int c = 0; c < 2; ++c)
#pragma unroll
                        for (int j = 0; j < 32; ++j) {
                            const float v = __uint_as_float(xs[c].r[j]);
                            sc[c * 32 + j] = v;
                            pm8[j & 7] = fmaxf(pm8[j & 7], v);
                        }
                }
                tc_fence_before();
                __syncwarp();
                if (lane == 0)
                    mbar_arrive(&bars.s_free[s]);
                const float pm = fmaxf(fmaxf(fmaxf(pm8[0], pm8[1]), fmaxf(pm8[2], pm8[3])),
                                       fmaxf(fmaxf(pm8[4], pm8[5]), fmaxf(pm8[6], pm8[7])));
                const float mt = fmaxf(m, pm * p.scale_log2);  // base-2 units
                if (mt != -INFINITY) {
                    const float c2 = p.scale_log2;
                    float s8[8];
#pragma unroll
                    for (int e = 0; e < 8; ++e)
                        s8[e] = 0.f;
#pragma unroll
                    for (int j = 0; j < 64; ++j)
                        s8[j & 7] += fast_exp2(fmaf(sc[j], c2, -mt));
                    const float sum = ((s8[0] + s8[1]) + (s8[2] + s8[3])) + ((s8[4] + s8[5]) + (s8[6] + s8[7]));
                    l = l * fast_exp2(m - mt) + sum;
                    m = mt;
                }
            }
            // merge the two halves of every row (both warps of a pair pass
            // this barrier once per item, faulted or not)
            if (part == 1) {
                bars.xm[k & 1][row] = m;
                bars.xl[k & 1][row] = l;
            }
            asm volatile("bar.sync %0, 64;" ::"r"(1 + (warp & 3)) : "memory");
            if (part == 0 && !fault) {
                const float m1 = bars.xm[k & 1][row], l1 = bars.xl[k & 1][row];
                const float mt = fmaxf(m, m1);
                const int64_t srow = (static_cast<int64_t>(it.b) * p.HQ + it.h) * p.sqp + i;
                if (i >= p.SQ || mt == -INFINITY) {  // padding rows up to sqp, rows that see no key
                    p.lse[srow] = INFINITY;
                } else {
                    const float lt = l * exp2f(m - mt) + l1 * exp2f(m1 - mt);
                    p.lse[srow] = mt + log2f(lt);
                }
            }
        }
    } else {
        // ------------------------------- delta = rowsum(y g), dq accumulator rows zeroed
        // warp dw takes rows 32 dw .. 32 dw + 31 of each item, two rows per
        // load (16 lanes x 16 bytes a row), eight row pairs in flight
        const int dw = warp - (kSoftmax / 32 + 2);
        const int half = lane >> 4, c16 = lane & 15;
        for (int k = 0;; ++k) {
            const int n = stats_item(k, C, G);
            if (n >= total)
                break;
            const StatsItem it = stats_item_at(p, n, tiles);
            const int64_t r0 = (static_cast<int64_t>(it.b) * p.HQ + it.h) * p.SQ;
            const int64_t s0 = (static_cast<int64_t>(it.b) * p.HQ + it.h) * p.sqp;
#pragma unroll 1
            for (int rb = 0; rb < 32; rb += 16) {
                uint4 yv[8], gv[8];
#pragma unroll
                for (int e = 0; e < 8; ++e) {
                    const int i = it.i0 + dw * 32 + rb + 2 * e + half;
                    if (i < p.SQ) {
                        const int64_t off = (r0 + i) * kD + c16 * 8;
                        yv[e] = __ldg(reinterpret_cast<const uint4*>(static_cast<const T*>(p.y) + off));
                        gv[e] = __ldg(reinterpret_cast<const uint4*>(static_cast<const T*>(p.g) + off));
                    } else {
                        yv[e] = make_uint4(0u, 0u, 0u, 0u);
                        gv[e] = make_uint4(0u, 0u, 0u, 0u);
                    }
                }
#pragma unroll
                for (int e = 0; e < 8; ++e) {
                    const uint32_t ya[4] = {yv[e].x, yv[e].y, yv[e].z, yv[e].w};
                    const uint32_t ga[4] = {gv[e].x, gv[e].y, gv[e].z, gv[e].w};
                    float acc[4];
#pragma unroll
                    for (int w = 0; w < 4; ++w) {
                        const float2 a = unpack2<T>(ya[w]), bb = unpack2<T>(ga[w]);
                        acc[w] = fmaf(a.y, bb.y, a.x * bb.x);
                    }
                    float d = (acc[0] + acc[1]) + (acc[2] + acc[3]);
#pragma unroll
                    for (int sh = 8; sh >= 1; sh >>= 1)
                        d += __shfl_xor_sync(kAll, d, sh);
                    const int i = it.i0 + dw * 32 + rb + 2 * e + half;
                    if (c16 == 0)
                        p.delta[s0 + i] = i < p.SQ ? d : 0.f;  // padding rows up to sqp: no gradient
                }
            }
            // the item's real rows of the accumulator: contiguous, 512 bytes a row
            const int nreal = min(kSRows, p.SQ - it.i0);
            float4* acc = reinterpret_cast<float4*>(p.dq_sum + (r0 + it.i0) * kD);
            const int nvec = nreal * (kD / 4);
            for (int v = dw * 32 + lane; v < nvec; v += kDeltaWarps * 32)
                acc[v] = make_float4(0.f, 0.f, 0.f, 0.f);
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 0)
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(bars.tmem), "r"(256) : "memory");
}

// ---------------------------------------------------------------------------
// Backward.  grid = ceil(SK / 128) * B * HK, (batch, key/value head) fastest:
// the key tiles that the most (causal) rows see are launched first.
template <typename T, typename TO>
__global__ void __launch_bounds__(kMainThreads, 1)
    vjp_main_tc(const __grid_constant__ VjpParams p, const __grid_constant__ CUtensorMap qmap,
                const __grid_constant__ CUtensorMap gmap, const __grid_constant__ CUtensorMap kmap,
                const __grid_constant__ CUtensorMap vmap)
{
    constexpr bool kBf = std::is_same<T, __nv_bfloat16>::value;
    extern __shared__ __align__(1024) unsigned char smem_raw[];
    if ((smem_u32(smem_raw) & 1023u) != 0) {
        if (threadIdx.x == 0 && p.status)
            atomicOr(p.status, PA_STATUS_TIMEOUT);
        return;
    }
    unsigned char* sK = smem_raw;                  // 2 halves of 16 KB
    unsigned char* sV = sK + 2 * kHalf128;         // 2 halves
    unsigned char* sQ = sV + 2 * kHalf128;         // 2 stages x 2 halves of 16 KB
    unsigned char* sG = sQ + 4 * kHalf128;         // 2 stages x 2 halves
    unsigned char* sS = sG + 4 * kHalf128;         // dS^T: rows 0-63 | rows 64-127
    float* sStat = reinterpret_cast<float*>(sS + 2 * kHalf128);  // 2 stages x (128 lse2, 128 delta)
    MainBars& bars = *reinterpret_cast<MainBars*>(sS + 2 * kHalf128 + 2048);

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int BH = p.B * p.HK;
    const int kt = blockIdx.x / BH;
    const int b = (blockIdx.x % BH) / p.HK;
    const int kh = blockIdx.x % p.HK;
    const int k0 = kt * kKeys;
    const int nrt = (p.SQ + kBRows - 1) / kBRows;
    const int r_first = p.causal ? min(k0 / kBRows, nrt) : 0;
    const int per_head = nrt - r_first;
    const int n = per_head * p.groups;
    const uint64_t wait_ns = p.wait_ns;

    if (tid == 0) {
        mbar_init(&bars.kv_full, 1);
        for (int s = 0; s < 2; ++s) {
            mbar_init(&bars.qd_full[s], 1);
            mbar_init(&bars.qd_empty[s], 1);
        }
        mbar_init(&bars.s_full, 1);
        mbar_init(&bars.dp_full, 1);
        // the softmax warps arrive once each (lane 0, after the warp's fences and a __syncwarp)
        mbar_init(&bars.p_ready, kMSoftmax / 32);
        mbar_init(&bars.ds_ready, kMSoftmax / 32);
        mbar_init(&bars.dq_full, 1);
        mbar_init(&bars.dq_free, kMSoftmax / 32);
        mbar_init(&bars.mma_done, 1);
        bars.abort = 0;
        fence_mbar_init();
    }
    if (warp == 0) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                         smem_u32(&bars.tmem)),
                     "r"(512)
                     : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    // tensor memory: dK | dV | S^T (P overwrites it, packed 16-bit) | dP^T (dQ^T
    // overwrites it once the softmax has read dP^T)
    const uint32_t tdK = bars.tmem, tdV = bars.tmem + 128, tS = bars.tmem + 256, tP = bars.tmem + 384;
    volatile int* abort_flag = &bars.abort;
    auto fail = [&]() {
        *abort_flag = 1;
        if (p.status)
            atomicOr(p.status, PA_STATUS_TIMEOUT);
    };
    auto step_head = [&](int it, int& h, int& i0) {
        const int gi = it / per_head;
        h = kh * p.groups + gi;
        i0 = (r_first + it - gi * per_head) * kBRows;
    };
    const uint32_t lane_off = static_cast<uint32_t>((warp & 3) * 32) << 16;  // this warp's TMEM lanes
    const int ln = (warp & 3) * 32 + lane;                                   // key, or d for dQ^T

    if (warp == 16) {
        // --------------------------------------------------------------- TMA
        if (lane == 0 && n > 0) {
            tma_prefetch_desc(&qmap);
            tma_prefetch_desc(&gmap);
            tma_prefetch_desc(&kmap);
            tma_prefetch_desc(&vmap);
            mbar_arrive_expect_tx(&bars.kv_full, 4 * kHalf128);
            for (int hh = 0; hh < 2; ++hh) {
                tma_load_4d(sK + hh * kHalf128, &kmap, 0, hh, k0, b * p.HK + kh, &bars.kv_full);
                tma_load_4d(sV + hh * kHalf128, &vmap, 0, hh, k0, b * p.HK + kh, &bars.kv_full);
            }
            int issued = 0;
            for (int it = 0; it < n; ++it) {
                const int st = it & 1;
                if (it >= 2 &&
                    (*abort_flag || !mbar_wait_bounded(&bars.qd_empty[st], ((it >> 1) - 1) & 1, wait_ns))) {
                    fail();
                    break;
                }
                int h, i0;
                step_head(it, h, i0);
                mbar_arrive_expect_tx(&bars.qd_full[st], 4 * kHalf128 + 1024);
                for (int hh = 0; hh < 2; ++hh) {
                    tma_load_4d(sQ + st * 2 * kHalf128 + hh * kHalf128, &qmap, 0, hh, i0, b * p.HQ + h,
                                &bars.qd_full[st]);
                    tma_load_4d(sG + st * 2 * kHalf128 + hh * kHalf128, &gmap, 0, hh, i0, b * p.HQ + h,
                                &bars.qd_full[st]);
                }
                const int64_t srow = (static_cast<int64_t>(b) * p.HQ + h) * p.sqp + i0;
                bulk_load(sStat + st * 256, p.lse + srow, 512, &bars.qd_full[st]);
                bulk_load(sStat + st * 256 + 128, p.delta + srow, 512, &bars.qd_full[st]);
                issued = it + 1;
            }
            // no copy may land after the CTA's memory is released
            for (int it = issued > 2 ? issued - 2 : 0; it < issued; ++it)
                mbar_wait_bounded(&bars.qd_full[it & 1], (it >> 1) & 1, wait_ns);
            mbar_wait_bounded(&bars.kv_full, 0, wait_ns);
        }
        __syncwarp();
    } else if (warp == 17) {
        // --------------------------------------------------------------- MMA
        // Per step it: dV += P dO (P from tensor memory) once the softmax has
        // written P; dK += dS^T Q and dQ^T = K^T dS^T once it has written dS^T;
        // then S^T of step it + 1 (into the P columns, after dV in the pipe)
        // and, once the dQ warps have read dQ^T, dP^T of step it + 1.
        if (lane == 0 && n > 0) {
            const uint32_t id_s = idesc<kBf>(kBRows, false);       // S^T, dP^T: N 128 rows, both K-major
            const uint32_t id_o = idesc<kBf>(kD, true);            // dV, dK: N 128 (D), B MN-major
            const uint32_t id_q = idesc<kBf>(kBRows, true, true);  // dQ^T: N 128 rows, A and B MN-major
            // descriptors of the operand bases; a byte offset o adds o >> 4
            const uint64_t dK_k = smem_desc(smem_u32(sK), 16, 1024);          // K, K-major A
            const uint64_t dK_mn = smem_desc(smem_u32(sK), kHalf128, 1024);   // K, MN-major A
            const uint64_t dV_k = smem_desc(smem_u32(sV), 16, 1024);
            const uint64_t dQ_k = smem_desc(smem_u32(sQ), 16, 1024);          // Q, dO: K-major B
            const uint64_t dG_k = smem_desc(smem_u32(sG), 16, 1024);
            const uint64_t dQ_mn = smem_desc(smem_u32(sQ), kHalf128, 1024);   // Q, dO: MN-major B
            const uint64_t dG_mn = smem_desc(smem_u32(sG), kHalf128, 1024);
            const uint64_t dS_k = smem_desc(smem_u32(sS), 16, 1024);          // dS^T: K-major A
            const uint64_t dS_mn = smem_desc(smem_u32(sS), kHalf128, 1024);   // dS^T: MN-major B
            auto at = [](uint64_t d, uint32_t off) { return d + (off >> 4); };
            // K-major k-step ks of a 128-column operand: 64-column halves 16 KB apart
            auto kmaj = [](int ks) { return static_cast<uint32_t>((ks >> 2) * kHalf128 + (ks & 3) * 32); };
            auto issue_s = [&](int u) {  // S^T = K Q^T of step u
                const int su = u & 1;
                if (*abort_flag || !mbar_wait_bounded(&bars.qd_full[su], (u >> 1) & 1, wait_ns))
                    return false;
                tc_fence_after();
#pragma unroll
                for (int ks = 0; ks < kD / 16; ++ks)
                    umma(tS, at(dK_k, kmaj(ks)), at(dQ_k, su * 2 * kHalf128 + kmaj(ks)), id_s, ks > 0);
                umma_commit(&bars.s_full);
                return true;
            };
            auto issue_dp = [&](int u) {  // dP^T = V dO^T of step u (its stage has landed)
                const int su = u & 1;
#pragma unroll
                for (int ks = 0; ks < kD / 16; ++ks)
                    umma(tP, at(dV_k, kmaj(ks)), at(dG_k, su * 2 * kHalf128 + kmaj(ks)), id_s, ks > 0);
                umma_commit(&bars.dp_full);
            };
            bool ok = mbar_wait_bounded(&bars.kv_full, 0, wait_ns) && issue_s(0);
            if (ok)
                issue_dp(0);
            for (int it = 0; it < n && ok; ++it) {
                const int st = it & 1;
                const uint32_t qo = st * 2 * kHalf128;
                ok = mbar_wait_bounded(&bars.p_ready, it & 1, wait_ns);
                if (!ok)
                    break;
                tc_fence_after();
                // dV += P dO: P (keys x rows) from tensor memory, rows 32 k .. 32 k + 31
                // packed in columns 32 k .. 32 k + 15 of the S^T block; dO MN-major
#pragma unroll
                for (int ks = 0; ks < kBRows / 16; ++ks)
                    umma_ts(tdV, tS + (ks >> 1) * 32 + (ks & 1) * 8, at(dG_mn, qo + ks * 2048), id_o,
                            it > 0 || ks > 0);
                ok = mbar_wait_bounded(&bars.ds_ready, it & 1, wait_ns);
                if (!ok)
                    break;
                tc_fence_after();
                // dK += dS^T Q (dS^T K-major over rows, Q MN-major)
#pragma unroll
                for (int ks = 0; ks < kBRows / 16; ++ks)
                    umma(tdK, at(dS_k, kmaj(ks)), at(dQ_mn, qo + ks * 2048), id_o, it > 0 || ks > 0);
                // dQ^T = K^T dS^T over the tile's 128 keys (both MN-major: K's rows
                // and dS^T's rows are keys) into the dP^T columns, which the
                // softmax has read
#pragma unroll
                for (int ks = 0; ks < kKeys / 16; ++ks)
                    umma(tP, at(dK_mn, ks * 2048), at(dS_mn, ks * 2048), id_q, ks > 0);
                umma_commit(&bars.dq_full);
                umma_commit(&bars.qd_empty[st]);
                if (it + 1 < n) {
                    if (!(ok = issue_s(it + 1)))
                        break;
                    ok = mbar_wait_bounded(&bars.dq_free, it & 1, wait_ns);
                    if (!ok)
                        break;
                    tc_fence_after();
                    issue_dp(it + 1);
                }
            }
            if (ok)
                umma_commit(&bars.mma_done);
            else
                fail();
        }
        __syncwarp();
    } else {
        // ------------------------------------------- softmax and dQ^T reduction
        // tensor-memory lane = key (S^T, dP^T, dK, dV) or d (dQ^T); this thread
        // takes rows [32 part, 32 part + 32)
        const int part = warp >> 2;
        const int key = k0 + ln;
        const bool key_ok = key < p.SK;
        const bool keys_all = k0 + kKeys <= p.SK;  // every key of the tile is real
        bool fault = false;
        // the dQ^T reductions of a step are issued in two halves: rows 0-15 of
        // this thread's 32 as soon as they are read, rows 16-31 held in
        // registers and issued in the next step once its dS^T is handed over,
        // while the MMA warp computes dK and dQ^T (the softmax warps would
        // otherwise wait for dQ^T), so that the reductions drain under the MMAs
        float held[16];
        float* held_dst = nullptr;
        int held_rows = 0;
        auto reduce_half = [&](float* dst, const float* v, int rows) {  // rows of this half present
            if (rows >= 16) {
#pragma unroll
                for (int j = 0; j < 16; ++j)
                    red_add(dst + static_cast<int64_t>(j) * kD, v[j]);
            } else {
#pragma unroll
                for (int j = 0; j < 16; ++j)
                    if (j < rows)
                        red_add(dst + static_cast<int64_t>(j) * kD, v[j]);
            }
        };
        for (int it = 0; it < n; ++it) {
            const int st = it & 1;
            int h, i0;
            step_head(it, h, i0);
            bool got = !fault && !*abort_flag && mbar_wait_bounded(&bars.s_full, it & 1, wait_ns);
            got = got && mbar_wait_bounded(&bars.qd_full[st], (it >> 1) & 1, wait_ns);
            if (!__all_sync(kAll, got)) {
                fault = true;
                break;
            }
            tc_fence_after();
            const int rb = i0 + part * 32;  // first row of this thread's columns
            // no mask on this thread's block: every key real, every row real,
            // and (causal) the last key at or before the first row (warp-uniform)
            const bool plain = keys_all && rb + 32 <= p.SQ && (!p.causal || k0 + kKeys - 1 <= rb);
            const float4* l4 = reinterpret_cast<const float4*>(sStat + st * 256 + part * 32);
            const float4* d4 = reinterpret_cast<const float4*>(sStat + st * 256 + 128 + part * 32);
            float pv[32];
#pragma unroll
            for (int hf = 0; hf < 2; ++hf) {
                Cols16 x;
                tmem_ld16(x, tS + lane_off + part * 32 + hf * 16);
                const float c = p.scale_log2;
#pragma unroll
                for (int q4 = 0; q4 < 4; ++q4) {
                    const float4 l = l4[hf * 4 + q4];
                    const float lv[4] = {l.x, l.y, l.z, l.w};
#pragma unroll
                    for (int e = 0; e < 4; ++e)
                        pv[hf * 16 + 4 * q4 + e] = fast_exp2(fmaf(__uint_as_float(x.r[4 * q4 + e]), c, -lv[e]));
                }
            }
            if (!plain) {
#pragma unroll
                for (int j = 0; j < 32; ++j) {
                    const int row = rb + j;
                    if (!(key_ok && row < p.SQ && (!p.causal || key <= row)))
                        pv[j] = 0.f;
                }
            }
            // P (16-bit pairs) into the first 16 of this thread's 32 S^T columns
            {
                uint32_t w[16];
#pragma unroll
                for (int e = 0; e < 16; ++e)
                    w[e] = pack2<T>(pv[2 * e], pv[2 * e + 1]);
                tmem_st16(w, tS + lane_off + part * 32);
                asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0)
                mbar_arrive(&bars.p_ready);
            got = __all_sync(kAll, mbar_wait_bounded(&bars.dp_full, it & 1, wait_ns));
            if (!got) {
                fault = true;
                break;
            }
            tc_fence_after();
#pragma unroll
            for (int hf = 0; hf < 2; ++hf) {
                Cols16 x;
                tmem_ld16(x, tP + lane_off + part * 32 + hf * 16);
                const float sc = p.scale;
#pragma unroll
                for (int q4 = 0; q4 < 4; ++q4) {
                    const float4 d = d4[hf * 4 + q4];
                    const float dv[4] = {d.x, d.y, d.z, d.w};
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        const int j = hf * 16 + 4 * q4 + e;
                        const float ds = pv[j] * sc * (__uint_as_float(x.r[4 * q4 + e]) - dv[e]);
                        // rows past SQ: p = 0, and their delta is not defined
                        pv[j] = plain || pv[j] != 0.f ? ds : 0.f;
                    }
                }
            }
            // dS^T (K-major over rows): rows 32 part .. + 31 are chunks 4 (part & 1) ..
            // + 3 of the 128-byte row of this key in row half part >> 1
            unsigned char* sb = sS + (part >> 1) * kHalf128;
#pragma unroll
            for (int c = 0; c < 4; ++c) {
                uint32_t w[4];
#pragma unroll
                for (int e = 0; e < 4; ++e)
                    w[e] = pack2<T>(pv[8 * c + 2 * e], pv[8 * c + 2 * e + 1]);
                *reinterpret_cast<uint4*>(sb + sw128(ln, (part & 1) * 4 + c)) = make_uint4(w[0], w[1], w[2], w[3]);
            }
            fence_proxy_async_smem();
            tc_fence_before();
            __syncwarp();
            if (lane == 0)
                mbar_arrive(&bars.ds_ready);
            if (held_dst) {
                reduce_half(held_dst, held, held_rows);
                held_dst = nullptr;
            }
            // dQ^T of the step (lane = d, columns = rows): read, hand the columns
            // back for the next dP^T, then add into the float32 accumulator
            got = __all_sync(kAll, mbar_wait_bounded(&bars.dq_full, it & 1, wait_ns));
            if (!got) {
                fault = true;
                break;
            }
            tc_fence_after();
            {
                Cols32 x;
                tmem_ld32(x, tP + lane_off + part * 32);
                tc_fence_before();
                __syncwarp();
                if (lane == 0)
                    mbar_arrive(&bars.dq_free);
                float* dst = p.dq_sum + ((static_cast<int64_t>(b) * p.HQ + h) * p.SQ + rb) * kD + ln;
                const int rows = min(32, p.SQ - rb);
                float v[16];
#pragma unroll
                for (int j = 0; j < 16; ++j) {
                    v[j] = __uint_as_float(x.r[j]);
                    held[j] = __uint_as_float(x.r[16 + j]);
                }
                reduce_half(dst, v, rows);
                if (rows > 16) {
                    held_dst = dst + static_cast<int64_t>(16) * kD;
                    held_rows = rows - 16;
                }
            }
        }
        if (held_dst)  // the last step's held rows
            reduce_half(held_dst, held, held_rows);
        if (!fault && n > 0)
            fault = !__all_sync(kAll, !*abort_flag && mbar_wait_bounded(&bars.mma_done, 0, wait_ns));
        if (fault) {
            if (lane == 0)
                fail();
        } else {
            // dK and dV of this thread's key: columns [32 part, 32 part + 32)
            // (the tensor-memory loads are warp-wide; only the stores depend on the key)
            tc_fence_after();
            const int64_t o = ((static_cast<int64_t>(b) * p.HK + kh) * p.SK + key) * kD + part * 32;
            float v[32];
            if (n > 0) {
                Cols32 x;
                tmem_ld32(x, tdK + lane_off + part * 32);
#pragma unroll
                for (int j = 0; j < 32; ++j)
                    v[j] = __uint_as_float(x.r[j]);
            } else {
#pragma unroll
                for (int j = 0; j < 32; ++j)
                    v[j] = 0.f;
            }
            if (key_ok)
                store_row<TO>(static_cast<TO*>(p.dk) + o, v);
            if (n > 0) {
                Cols32 x;
                tmem_ld32(x, tdV + lane_off + part * 32);
#pragma unroll
                for (int j = 0; j < 32; ++j)
                    v[j] = __uint_as_float(x.r[j]);
            }
            if (key_ok)
                store_row<TO>(static_cast<TO*>(p.dv) + o, v);
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 0)
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(bars.tmem), "r"(512) : "memory");
}

using StatsFn = void (*)(VjpParams, CUtensorMap, CUtensorMap);
using MainFn = void (*)(VjpParams, CUtensorMap, CUtensorMap, CUtensorMap, CUtensorMap);

// [B * heads][rows][128] 16-bit as {64, 2, rows, B * heads}; box {64, 1, box_rows, 1}:
// one 64-column half of box_rows rows of one head
int encode_rows(CUtensorMap* map, const void* base, CUtensorMapDataType dt, int rows, int heads, int box_rows)
{
    auto enc = tc_encoder();
    if (!enc)
        return PA_ERR_DRIVER;
    cuuint64_t dims[4] = {64u, 2u, static_cast<cuuint64_t>(rows), static_cast<cuuint64_t>(heads)};
    cuuint64_t str[3] = {128u, kD * 2u, static_cast<cuuint64_t>(rows) * kD * 2};
    cuuint32_t box[4] = {64u, 1u, static_cast<cuuint32_t>(box_rows), 1u};
    cuuint32_t es[4] = {1u, 1u, 1u, 1u};
    return enc(map, dt, 4, const_cast<void*>(base), dims, str, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE,
               CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) ==
                   CUDA_SUCCESS
               ? PA_OK
               : PA_ERR_CUDA;
}

}  // namespace

bool vjp_tc_supported(int dtype, int D, int groups, int mask_kind)
{
    return (dtype == PA_F16 || dtype == PA_BF16) && D == kD && groups >= 1 && mask_kind == 0;
}

int launch_vjp_tc(const VjpParams& p, int dtype, bool f32_out, cudaStream_t st, uint64_t* launches)
{
    const CUtensorMapDataType dt =
        dtype == PA_BF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16;
    const bool bf = dtype == PA_BF16;
    if (p.SQ > 0) {
        CUtensorMap qmap, kmap;
        int rc = encode_rows(&qmap, p.q, dt, p.SQ, p.B * p.HQ, kSRows);
        if (rc == PA_OK && p.SK > 0)
            rc = encode_rows(&kmap, p.k, dt, p.SK, p.B * p.HK, kKeys);
        else
            kmap = qmap;  // no key tile is ever loaded
        if (rc != PA_OK)
            return rc;
        const StatsFn fn = bf ? vjp_stats_tc<__nv_bfloat16> : vjp_stats_tc<__half>;
        if (cudaFuncSetAttribute(reinterpret_cast<const void*>(fn), cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 kStatsSmem) != cudaSuccess)
            return PA_ERR_CUDA;
        const long long items = static_cast<long long>(p.B) * p.HQ * ((p.SQ + kSRows - 1) / kSRows);
        if (items >= (1ll << 31) / 4)
            return PA_ERR_BAD_DIMS;
        // persistent: one CTA per SM (its shared memory allows no more)
        int dev = 0, sms = 0;
        if (cudaGetDevice(&dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || sms < 1)
            return PA_ERR_CUDA;
        const long long grid = items < sms ? items : sms;
        fn<<<static_cast<unsigned>(grid), kStatsThreads, kStatsSmem, st>>>(p, qmap, kmap);
        if (cudaGetLastError() != cudaSuccess)
            return PA_ERR_CUDA;
        ++*launches;
    }
    if (p.SK > 0) {
        CUtensorMap qmap, gmap, kmap, vmap;
        int rc = encode_rows(&kmap, p.k, dt, p.SK, p.B * p.HK, kKeys);
        if (rc == PA_OK)
            rc = encode_rows(&vmap, p.v, dt, p.SK, p.B * p.HK, kKeys);
        if (rc == PA_OK && p.SQ > 0) {
            rc = encode_rows(&qmap, p.q, dt, p.SQ, p.B * p.HQ, kBRows);
            if (rc == PA_OK)
                rc = encode_rows(&gmap, p.g, dt, p.SQ, p.B * p.HQ, kBRows);
        } else {
            qmap = gmap = kmap;  // no row tile is ever loaded
        }
        if (rc != PA_OK)
            return rc;
        MainFn fn;
        if (bf)
            fn = f32_out ? vjp_main_tc<__nv_bfloat16, float> : vjp_main_tc<__nv_bfloat16, __nv_bfloat16>;
        else
            fn = f32_out ? vjp_main_tc<__half, float> : vjp_main_tc<__half, __half>;
        if (cudaFuncSetAttribute(reinterpret_cast<const void*>(fn), cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 kMainSmem) != cudaSuccess)
            return PA_ERR_CUDA;
        const long long grid = static_cast<long long>(p.B) * p.HK * ((p.SK + kKeys - 1) / kKeys);
        if (grid >= (1ll << 31))
            return PA_ERR_BAD_DIMS;
        fn<<<static_cast<unsigned>(grid), kMainThreads, kMainSmem, st>>>(p, qmap, gmap, kmap, vmap);
        if (cudaGetLastError() != cudaSuccess)
            return PA_ERR_CUDA;
        ++*launches;
    }
    return PA_OK;
}

}  // namespace pa
