// pa_kernels.cuh -- the sm_103a kernels of decode attention over a paged KV
// cache: the partition kernel and the log-sum-exp merge kernel.
//
// What is computed follows onnxruntime-ep-mlx 0.31.1,
// src/ops/paged_attention.rs:
//   VECTOR_BODY      block-table gather of K/V rows, grouped-query map
//                    kh = h / (H / KV), new rows for keys i >= past, causal
//                    bound past + row + 1, online softmax (running max,
//                    rescaled sum and accumulator);
//   VECTOR_PARTIALS  unnormalised accumulator, sum and max of one partition;
//   PARTIALS_REDUCE  max over partitions, rescaled sums, out = sum == 0 ? o : o / sum.
//
// How it is computed here (GB300 design, not the page's Metal layout):
//   * one CTA per work item = (sequence, contiguous key range, row group,
//     KV head); the CTA serves every query head of its KV head, so each K/V
//     row is read from HBM once (the page runs one threadgroup per query
//     head and re-reads K/V H/KV times);
//   * key ranges are whole cache blocks, sized on the device from the
//     sequence lengths so that the item count fills the GPU (or P ranges per
//     sequence when the caller fixes the partition count);
//   * a producer warp streams cache blocks into a 3-stage shared-memory ring
//     with TMA tensor copies (one box = one block of one KV head) completing
//     on mbarriers; four consumer warps compute in float32 with 16-byte
//     shared-memory vector reads, warp-shuffle dot reductions and an online
//     base-2 softmax updated once per four token steps;
//   * a sequence covered by one item is normalised and written directly;
//     otherwise partial states go to the workspace and the merge kernel,
//     launched with programmatic dependent launch, combines them.
//
// Every wait is bounded (PA_STATUS_TIMEOUT); no kernel traps.
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include <cfloat>
#include <cstring>

#include "pa_common.cuh"
#include "pa_decode.h"
#include "pa_ptx.cuh"

namespace pa {

constexpr unsigned kFull = 0xffffffffu;

// ----------------------------------------------------------- element types
template <typename T>
struct Elem;

template <>
struct Elem<float> {
    static constexpr int kVec = 4;
    __device__ static void load(const float* p, float* f)
    {
        const float4 v = *reinterpret_cast<const float4*>(p);
        f[0] = v.x;
        f[1] = v.y;
        f[2] = v.z;
        f[3] = v.w;
    }
};

template <>
struct Elem<__half> {
    static constexpr int kVec = 8;
    __device__ static void load(const __half* p, float* f)
    {
        const uint4 u = *reinterpret_cast<const uint4*>(p);
        const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            __half2 h;
            memcpy(&h, &w[i], 4);
            const float2 t = __half22float2(h);
            f[2 * i] = t.x;
            f[2 * i + 1] = t.y;
        }
    }
};

template <>
struct Elem<__nv_bfloat16> {
    static constexpr int kVec = 8;
    __device__ static void load(const __nv_bfloat16* p, float* f)
    {
        const uint4 u = *reinterpret_cast<const uint4*>(p);
        const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            f[2 * i] = __uint_as_float(w[i] << 16);
            f[2 * i + 1] = __uint_as_float(w[i] & 0xffff0000u);
        }
    }
};

template <typename TO>
__device__ __forceinline__ TO from_float(float x);
template <>
__device__ __forceinline__ float from_float<float>(float x) { return x; }
template <>
__device__ __forceinline__ __half from_float<__half>(float x) { return __float2half_rn(x); }
template <>
__device__ __forceinline__ __nv_bfloat16 from_float<__nv_bfloat16>(float x)
{
    return __float2bfloat16_rn(x);
}

// ---------------------------------------------------------------- schedule
struct Item {
    int b, c, kh, rsg, n, chunk, past;
};

__device__ __forceinline__ int clamped_past(const SplitParams& p, int b, bool report)
{
    int s = p.seq_lens[b];
    const int cap = p.maxb * p.BLOCK;
    if (s < 0 || s > cap) {
        if (report && p.status)
            atomicOr(p.status, PA_STATUS_BAD_LENGTH);
        s = s < 0 ? 0 : cap;
    }
    return s;
}

__device__ __forceinline__ int chunk_of(const SplitParams& p, int total, int auto_chunk)
{
    if (p.partitions == 0)
        return auto_chunk;
    const int per = p.partitions == 1 ? total : (total + p.partitions - 1) / p.partitions;
    return ((per + p.BLOCK - 1) / p.BLOCK) * p.BLOCK;
}

// Automatic key-range length (identical in every CTA of a launch): the
// smallest multiple of BLOCK, at least min_chunk, that splits all keys of all
// sequences, row groups and KV heads into about target_items items.
__device__ __forceinline__ int auto_chunk(const SplitParams& p, int lane)
{
    if (p.partitions != 0)
        return 0;
    long long sum = 0;
    for (int b = lane; b < p.B; b += 32)
        sum += clamped_past(p, b, false) + p.NQ;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1)
        sum += __shfl_xor_sync(kFull, sum, o);
    const long long units = sum * p.KV * p.NRS;
    long long per = (units + p.target_items - 1) / p.target_items;
    per = ((per + p.BLOCK - 1) / p.BLOCK) * p.BLOCK;
    if (per < p.min_chunk)
        per = p.min_chunk;
    if (per > (1 << 30))
        per = 1 << 30;
    return static_cast<int>(per);
}

// Executed by one full warp.  Finds work item `item`: items are ordered by
// sequence, then key range, then row group, then KV head (adjacent KV heads
// read interleaved rows of the same cache blocks).  With `write_sched`, also
// records every sequence's (first chunk, chunk count) for the merge kernel
// and reports out-of-range lengths.
__device__ __forceinline__ bool locate_item(const SplitParams& p, int item, int lane,
                                            bool write_sched, Item& it)
{
    const int C = auto_chunk(p, lane);
    const int U = p.NRS * p.KV;
    long long run = 0;
    bool found = false;
    for (int base = 0; base < p.B; base += 32) {
        const int b = base + lane;
        int past = 0, chunk = 1, n = 0;
        if (b < p.B) {
            past = clamped_past(p, b, write_sched);
            const int total = past + p.NQ;
            chunk = chunk_of(p, total, C);
            n = (total + chunk - 1) / chunk;
        }
        int incl = n;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int y = __shfl_up_sync(kFull, incl, o);
            if (lane >= o)
                incl += y;
        }
        const long long first = (run + incl - n) * U;
        const long long last = (run + incl) * U;
        if (write_sched && p.sched && b < p.B)
            p.sched[b] = make_int2(static_cast<int>(run + incl - n), n);
        const unsigned hit = __ballot_sync(kFull, b < p.B && item >= first && item < last);
        if (hit && !found) {
            const int src = __ffs(hit) - 1;
            const long long rem = item - first;
            const int mc = static_cast<int>(rem / U);
            const int mrsg = static_cast<int>((rem % U) / p.KV);
            const int mkh = static_cast<int>(rem % p.KV);
            it.b = __shfl_sync(kFull, b, src);
            it.c = __shfl_sync(kFull, mc, src);
            it.rsg = __shfl_sync(kFull, mrsg, src);
            it.kh = __shfl_sync(kFull, mkh, src);
            it.n = __shfl_sync(kFull, n, src);
            it.chunk = __shfl_sync(kFull, chunk, src);
            it.past = __shfl_sync(kFull, past, src);
            found = true;
            if (!write_sched)
                break;
        }
        run += __shfl_sync(kFull, incl, 31);
    }
    return found;
}

__device__ __forceinline__ void consumer_bar_sync()
{
    asm volatile("bar.sync 1, %0;" ::"n"(kConsumerWarps * 32) : "memory");
}

// ---------------------------------------------------------- partition kernel
// T: element type of q/K/V; D: head size; RG: query rows per consumer warp;
// TO: output element type.
template <typename T, int D, int RG, typename TO>
__global__ void __launch_bounds__(kThreads, 2)
    pa_split_kernel(const __grid_constant__ SplitParams p, const __grid_constant__ CUtensorMap kmap,
                    const __grid_constant__ CUtensorMap vmap)
{
    using E = Elem<T>;
    constexpr int VEC = E::kVec;
    constexpr int LPT = D / VEC;   // lanes sharing one token row
    constexpr int TPW = 32 / LPT;  // tokens per warp step
    static_assert(LPT <= 32 && 32 % LPT == 0, "a row must split evenly over lanes");

    extern __shared__ __align__(1024) unsigned char smem_raw[];
    // TMA destinations want 128-byte alignment; align the carve-up to 1024.
    unsigned char* smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
    uint64_t* full = reinterpret_cast<uint64_t*>(smem);
    uint64_t* empty = full + kStages;
    uint64_t* newbar = empty + kStages;
    int* info = reinterpret_cast<int*>(newbar + 1);  // 16 ints
    volatile int* abort_flag = info + 15;
    T* stages = reinterpret_cast<T*>(smem + kHeaderBytes);
    const int stage_elems = p.TT * D;  // per K (or V) per stage
    T* knew = stages + 2 * kStages * stage_elems;
    T* vnew = knew + p.NQ * D;

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;

    // Inputs may be produced by the previous kernel on the stream.
    grid_dependency_wait();
    grid_dependents_launch();

    if (warp == kConsumerWarps) {
        Item it{};
        const bool ok = locate_item(p, blockIdx.x, lane, blockIdx.x == 0, it);
        if (lane == 0) {
            info[0] = ok;
            info[1] = it.b;
            info[2] = it.c;
            info[3] = it.kh;
            info[4] = it.rsg;
            info[5] = it.n;
            info[6] = it.chunk;
            info[7] = it.past;
            info[15] = 0;
            for (int s = 0; s < kStages; ++s) {
                mbar_init(&full[s], 1);
                mbar_init(&empty[s], kConsumerWarps);
            }
            mbar_init(newbar, 1);
            fence_mbar_init();
        }
    }
    __syncthreads();
    if (!info[0])
        return;  // beyond the last work item
    const int b = info[1], c = info[2], kh = info[3], rsg = info[4], n_b = info[5];
    const int chunk = info[6], past = info[7];
    const int total_max = past + p.NQ;
    const int chunk_start = c * chunk;
    const int chunk_end = min(chunk_start + chunk, total_max);
    const int TT = p.TT;
    const int ntiles = (chunk_end - chunk_start + TT - 1) / TT;
    const bool need_new = chunk_end > past;
    const int R_cta = min(p.rows_per_cta, p.R - rsg * p.rows_per_cta);

    if (warp == kConsumerWarps) {
        // ------------------------------------------------------ producer
        if (lane == 0) {
            tma_prefetch_desc(&kmap);
            tma_prefetch_desc(&vmap);
        }
        if (need_new && lane == 0) {
            const size_t off = (static_cast<size_t>(b) * p.KV + kh) * p.NQ * D;
            const uint32_t bytes = static_cast<uint32_t>(p.NQ * D * sizeof(T));
            mbar_arrive_expect_tx(newbar, 2 * bytes);
            bulk_load(knew, static_cast<const T*>(p.k_new) + off, bytes, newbar);
            bulk_load(vnew, static_cast<const T*>(p.v_new) + off, bytes, newbar);
        }
        const uint32_t block_bytes = static_cast<uint32_t>(p.BLOCK * D * sizeof(T));
        int issued = 0;
        for (int j = 0; j < ntiles; ++j) {
            const int s = j % kStages;
            if (j >= kStages) {
                bool ok = !*abort_flag &&
                          mbar_wait_bounded(&empty[s], ((j / kStages) - 1) & 1, kWaitLimitNs);
                ok = __all_sync(kFull, ok);
                if (!ok) {
                    if (lane == 0) {
                        *abort_flag = 1;
                        if (p.status)
                            atomicOr(p.status, PA_STATUS_TIMEOUT);
                    }
                    break;
                }
            }
            const int t0 = chunk_start + j * TT;
            const int cache_end = min(min(t0 + TT, chunk_end), past);
            const int nb = cache_end > t0 ? (cache_end - t0 + p.BLOCK - 1) / p.BLOCK : 0;
            int phys = 0;
            if (lane < nb) {
                phys = p.table[static_cast<size_t>(b) * p.maxb + t0 / p.BLOCK + lane];
                if (p.checked && (phys < 0 || phys >= p.num_blocks) && p.status)
                    atomicOr(p.status, PA_STATUS_BAD_BLOCK);
            }
            if (lane == 0)
                mbar_arrive_expect_tx(&full[s], 2u * nb * block_bytes);
            __syncwarp();
            if (lane < nb) {
                // Out-of-pool coordinates read as zeros: the copy never faults.
                T* kdst = stages + (2 * s) * stage_elems + lane * p.BLOCK * D;
                T* vdst = stages + (2 * s + 1) * stage_elems + lane * p.BLOCK * D;
                tma_load_3d(kdst, &kmap, 0, kh, phys * p.BLOCK, &full[s]);
                tma_load_3d(vdst, &vmap, 0, kh, phys * p.BLOCK, &full[s]);
            }
            issued = j + 1;
        }
        // Leave no copy in flight if the pipeline was abandoned.
        __syncwarp();
        if (*abort_flag && lane == 0) {
            for (int j = max(0, issued - kStages); j < issued; ++j)
                mbar_wait_bounded(&full[j % kStages], (j / kStages) & 1, kWaitLimitNs);
            if (need_new)
                mbar_wait_bounded(newbar, 0, kWaitLimitNs);
        }
        return;
    }

    // ---------------------------------------------------------- consumers
    const int nrg_raw = (R_cta + RG - 1) / RG;
    const int nrg = nrg_raw <= 1 ? 1 : (nrg_raw <= 2 ? 2 : 4);  // row groups in the CTA
    const int TS = kConsumerWarps / nrg;                         // token subsets
    const int rg = warp % nrg;
    const int ts = warp / nrg;
    const int lg = lane / LPT;
    const int li = lane % LPT;

    float q[RG][VEC];
    int limit[RG];
    {
        const T* qbase =
            static_cast<const T*>(p.q) + (static_cast<size_t>(b) * p.KV + kh) * p.R * D;
#pragma unroll
        for (int r = 0; r < RG; ++r) {
            const int rl = rg * RG + r;
            const int rho = rsg * p.rows_per_cta + rl;
            if (rl < R_cta) {
                E::load(qbase + static_cast<size_t>(rho) * D + li * VEC, q[r]);
#pragma unroll
                for (int v = 0; v < VEC; ++v)
                    q[r][v] *= p.qscale;
                limit[r] = past + (p.causal ? (rho % p.NQ) + 1 : p.NQ);
            } else {
#pragma unroll
                for (int v = 0; v < VEC; ++v)
                    q[r][v] = 0.f;
                limit[r] = 0;
            }
        }
    }

    float m[RG], l[RG], o[RG][VEC];
#pragma unroll
    for (int r = 0; r < RG; ++r) {
        m[r] = -FLT_MAX;
        l[r] = 0.f;
#pragma unroll
        for (int v = 0; v < VEC; ++v)
            o[r][v] = 0.f;
    }

    bool alive = true;
    if (need_new) {
        alive = __all_sync(kFull, mbar_wait_bounded(newbar, 0, kWaitLimitNs));
        if (!alive && lane == 0) {
            *abort_flag = 1;
            if (p.status)
                atomicOr(p.status, PA_STATUS_TIMEOUT);
        }
    }
    const int step = TS * TPW;  // tokens per warp step across the CTA
    for (int j = 0; j < ntiles && alive; ++j) {
        const int s = j % kStages;
        alive = !*abort_flag && mbar_wait_bounded(&full[s], (j / kStages) & 1, kWaitLimitNs);
        alive = __all_sync(kFull, alive);
        if (!alive) {
            if (lane == 0) {
                *abort_flag = 1;
                if (p.status)
                    atomicOr(p.status, PA_STATUS_TIMEOUT);
            }
            break;
        }
        const T* ks = stages + (2 * s) * stage_elems;
        const T* vs = stages + (2 * s + 1) * stage_elems;
        const int t0 = chunk_start + j * TT;
        const int n_tile = min(TT, chunk_end - t0);

        for (int base = 0; base < n_tile; base += kSubBatch * step) {
            float sc[kSubBatch][RG];
#pragma unroll
            for (int i = 0; i < kSubBatch; ++i) {
                const int t_rel = base + (i * TS + ts) * TPW + lg;
                const int t_abs = t0 + t_rel;
                const bool live = t_rel < n_tile;
                float kf[VEC];
                if (live) {
                    const T* row = t_abs < past ? ks + t_rel * D : knew + (t_abs - past) * D;
                    E::load(row + li * VEC, kf);
                } else {
#pragma unroll
                    for (int v = 0; v < VEC; ++v)
                        kf[v] = 0.f;
                }
#pragma unroll
                for (int r = 0; r < RG; ++r) {
                    float acc = 0.f;
#pragma unroll
                    for (int v = 0; v < VEC; ++v)
                        acc = fmaf(q[r][v], kf[v], acc);
#pragma unroll
                    for (int off = LPT / 2; off > 0; off >>= 1)
                        acc += __shfl_xor_sync(kFull, acc, off);
                    sc[i][r] = (live && t_abs < limit[r]) ? acc : -INFINITY;
                }
            }
#pragma unroll
            for (int r = 0; r < RG; ++r) {
                float mx = sc[0][r];
#pragma unroll
                for (int i = 1; i < kSubBatch; ++i)
                    mx = fmaxf(mx, sc[i][r]);
                const float mn = fmaxf(m[r], mx);
                const float f = fast_exp2(m[r] - mn);
                m[r] = mn;
                l[r] *= f;
#pragma unroll
                for (int v = 0; v < VEC; ++v)
                    o[r][v] *= f;
            }
#pragma unroll
            for (int i = 0; i < kSubBatch; ++i) {
                const int t_rel = base + (i * TS + ts) * TPW + lg;
                if (t_rel >= n_tile)
                    continue;
                const int t_abs = t0 + t_rel;
                const T* row = t_abs < past ? vs + t_rel * D : vnew + (t_abs - past) * D;
                float vf[VEC];
                E::load(row + li * VEC, vf);
#pragma unroll
                for (int r = 0; r < RG; ++r) {
                    const float pr = fast_exp2(sc[i][r] - m[r]);
                    l[r] += pr;
#pragma unroll
                    for (int v = 0; v < VEC; ++v)
                        o[r][v] = fmaf(pr, vf[v], o[r][v]);
                }
            }
        }
        __syncwarp();
        if (lane == 0)
            mbar_arrive(&empty[s]);
    }

    // Merge the lane groups of this warp (they saw different tokens).
#pragma unroll
    for (int off = LPT; off < 32; off <<= 1) {
#pragma unroll
        for (int r = 0; r < RG; ++r) {
            const float mo = __shfl_xor_sync(kFull, m[r], off);
            const float lo = __shfl_xor_sync(kFull, l[r], off);
            const float mn = fmaxf(m[r], mo);
            const float fa = fast_exp2(m[r] - mn), fb = fast_exp2(mo - mn);
            l[r] = l[r] * fa + lo * fb;
#pragma unroll
            for (int v = 0; v < VEC; ++v) {
                const float oo = __shfl_xor_sync(kFull, o[r][v], off);
                o[r][v] = o[r][v] * fa + oo * fb;
            }
            m[r] = mn;
        }
    }

    // All consumers are done with the stages: reuse them as the merge buffer.
    consumer_bar_sync();
    if (*abort_flag)
        return;
    // State slot of (token subset ts, local row rl): ts * span + rl.
    const int span = nrg * RG;
    float* mb_o = reinterpret_cast<float*>(stages);  // [TS * span][D]
    float* mb_m = mb_o + kConsumerWarps * RG * D;    // [TS * span]
    float* mb_l = mb_m + kConsumerWarps * RG;
    if (lane < LPT) {
#pragma unroll
        for (int r = 0; r < RG; ++r) {
            const int slot = ts * span + rg * RG + r;
#pragma unroll
            for (int v = 0; v < VEC; ++v)
                mb_o[slot * D + li * VEC + v] = o[r][v];
            if (li == 0) {
                mb_m[slot] = m[r];
                mb_l[slot] = l[r];
            }
        }
    }
    consumer_bar_sync();

    const int tid = threadIdx.x;  // 0 .. 127 (consumers only reach here)
    const size_t out_row0 = (static_cast<size_t>(b) * p.KV + kh) * p.R + rsg * p.rows_per_cta;
    for (int idx = tid; idx < R_cta * D; idx += kConsumerWarps * 32) {
        const int rl = idx / D, d = idx % D;
        float M = -FLT_MAX;
        for (int t = 0; t < TS; ++t)
            M = fmaxf(M, mb_m[t * span + rl]);
        float L = 0.f, O = 0.f;
        for (int t = 0; t < TS; ++t) {
            const int slot = t * span + rl;
            const float f = fast_exp2(mb_m[slot] - M);
            L = fmaf(mb_l[slot], f, L);
            O = fmaf(mb_o[slot * D + d], f, O);
        }
        if (n_b == 1) {
            const float val = L == 0.f ? O : O / L;
            static_cast<TO*>(p.out)[(out_row0 + rl) * D + d] = from_float<TO>(val);
        } else {
            const size_t wrow = static_cast<size_t>(blockIdx.x) * p.row_stride + rl;
            p.ws_o[wrow * D + d] = O;
            if (d == 0)
                p.ws_ml[wrow] = make_float2(M, L);
        }
    }
}

// -------------------------------------------------------------- merge kernel
// One CTA per (sequence, row group, KV head); one warp per query row; lanes
// split D.  Sequences covered by a single item were finished by the
// partition kernel and are skipped.
template <int D, typename TO>
__global__ void __launch_bounds__(128) pa_combine_kernel(const __grid_constant__ CombineParams p)
{
    grid_dependency_wait();
    grid_dependents_launch();
    const int idx = blockIdx.x;
    const int kh = idx % p.KV;
    const int rsg = (idx / p.KV) % p.NRS;
    const int b = idx / (p.KV * p.NRS);
    const int2 sc = p.sched[b];
    const int n = sc.y;
    if (n <= 1)
        return;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int R_cta = min(p.rows_per_cta, p.R - rsg * p.rows_per_cta);
    constexpr int PER = D / 32;
    for (int rl = warp; rl < R_cta; rl += 4) {
        float M = -FLT_MAX;
        for (int c = lane; c < n; c += 32) {
            const size_t item = (static_cast<size_t>(sc.x + c) * p.NRS + rsg) * p.KV + kh;
            M = fmaxf(M, p.ws_ml[item * p.row_stride + rl].x);
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1)
            M = fmaxf(M, __shfl_xor_sync(kFull, M, o));
        float L = 0.f;
        for (int c = lane; c < n; c += 32) {
            const size_t item = (static_cast<size_t>(sc.x + c) * p.NRS + rsg) * p.KV + kh;
            const float2 ml = p.ws_ml[item * p.row_stride + rl];
            L = fmaf(ml.y, fast_exp2(ml.x - M), L);
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1)
            L += __shfl_xor_sync(kFull, L, o);
        float O[PER];
#pragma unroll
        for (int k = 0; k < PER; ++k)
            O[k] = 0.f;
        for (int c = 0; c < n; ++c) {
            const size_t item = (static_cast<size_t>(sc.x + c) * p.NRS + rsg) * p.KV + kh;
            const size_t wrow = item * p.row_stride + rl;
            const float f = fast_exp2(p.ws_ml[wrow].x - M);
#pragma unroll
            for (int k = 0; k < PER; ++k)
                O[k] = fmaf(f, p.ws_o[wrow * D + lane + 32 * k], O[k]);
        }
        const size_t orow =
            (static_cast<size_t>(b) * p.KV + kh) * p.R + rsg * p.rows_per_cta + rl;
#pragma unroll
        for (int k = 0; k < PER; ++k) {
            const float val = L == 0.f ? O[k] : O[k] / L;
            static_cast<TO*>(p.out)[orow * D + lane + 32 * k] = from_float<TO>(val);
        }
    }
}

template <typename T, typename TO>
SplitFn pick_split_typed(int D, int RG)
{
    if (D == 64)
        return RG == 4 ? pa_split_kernel<T, 64, 4, TO> : pa_split_kernel<T, 64, 8, TO>;
    return RG == 4 ? pa_split_kernel<T, 128, 4, TO> : pa_split_kernel<T, 128, 8, TO>;
}

template <typename TO>
CombineFn pick_combine_typed(int D)
{
    return D == 64 ? pa_combine_kernel<64, TO> : pa_combine_kernel<128, TO>;
}

}  // namespace pa
