// pa_kernels.cuh -- the sm_103a kernels of decode attention over a paged KV
// cache: the persistent partition kernel and the log-sum-exp merge kernel.
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
//   * work item = (sequence, contiguous key range of whole blocks, row group,
//     KV head); the item's CTA serves every query row of its KV head, so each
//     K/V row is read from HBM once (the page runs one threadgroup per query
//     head and re-reads K/V H/KV times);
//   * the kernel is persistent: one CTA per SM walks items blockIdx.x,
//     blockIdx.x + gridDim.x, ...; key ranges are sized on the device from the
//     lengths so that the item count is a few times the CTA count (or P ranges
//     per sequence when the caller fixes the partition count);
//   * a producer warp streams cache blocks into a shared-memory ring with TMA
//     tensor copies (one box = one block of one KV head) and the new rows with
//     bulk copies, completing on mbarriers; it runs ahead across item
//     boundaries, so HBM keeps streaming while the consumers merge an item;
//   * eight consumer warps compute in float32: 16-byte shared-memory vector
//     reads, packed f32x2 FMAs, warp-shuffle dot reductions and an online
//     base-2 softmax updated once per four token steps;
//   * an item that covers a whole sequence writes the normalised output;
//     otherwise its partial state goes to the workspace and the merge kernel,
//     launched with programmatic dependent launch, combines the partials.
//
// Every wait is bounded (PA_STATUS_TIMEOUT); no kernel traps.
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include <cfloat>
#include <cstring>
#include <type_traits>

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
    static constexpr int kVec = 4;  // elements per 16-byte vector
    __device__ static void load2(const float* p, float2* f)
    {
        const float4 v = *reinterpret_cast<const float4*>(p);
        f[0] = make_float2(v.x, v.y);
        f[1] = make_float2(v.z, v.w);
    }
};

template <>
struct Elem<__half> {
    static constexpr int kVec = 8;
    __device__ static void load2(const __half* p, float2* f)
    {
        const uint4 u = *reinterpret_cast<const uint4*>(p);
        const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            __half2 h;
            memcpy(&h, &w[i], 4);
            f[i] = __half22float2(h);
        }
    }
};

template <>
struct Elem<__nv_bfloat16> {
    static constexpr int kVec = 8;
    __device__ static void load2(const __nv_bfloat16* p, float2* f)
    {
        const uint4 u = *reinterpret_cast<const uint4*>(p);
        const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
        for (int i = 0; i < 4; ++i)
            f[i] = make_float2(__uint_as_float(w[i] << 16), __uint_as_float(w[i] & 0xffff0000u));
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
    int b, c, kh, rsg, n, past, start, end;  // key range [start, end)
};

__device__ __forceinline__ int chunk_of(const SplitParams& p, int total, int auto_chunk)
{
    if (p.partitions == 0)
        return auto_chunk;
    const int per = p.partitions == 1 ? total : (total + p.partitions - 1) / p.partitions;
    return ((per + p.BLOCK - 1) / p.BLOCK) * p.BLOCK;
}

// Shared-memory schedule built once per CTA: clamped lengths, the automatic
// key-range length, and the prefix sum of key ranges per sequence.
struct Sched {
    const int* lens;    // [B]
    const int* prefix;  // [B + 1] key ranges before sequence b
    int auto_chunk;
    int total_items;
};

// Executed by one full warp after `lens` is in shared memory.  CTA 0 also
// records every sequence's (first range, range count) for the merge kernel.
__device__ __forceinline__ void build_schedule(const SplitParams& p, const int* lens, int* prefix, int* info,
                               int lane)
{
    int C = 0;
    if (p.partitions == 0) {
        long long sum = 0;
        for (int b = lane; b < p.B; b += 32)
            sum += lens[b] + p.NQ;
#pragma unroll
        for (int o = 16; o > 0; o >>= 1)
            sum += __shfl_xor_sync(kFull, sum, o);
        const long long units = sum * p.KV * p.NRS;
        long long per = (units + p.target_items - 1) / p.target_items;
        per = ((per + p.chunk_align - 1) / p.chunk_align) * p.chunk_align;
        if (per < p.min_chunk)
            per = p.min_chunk;
        if (per > (1 << 30))
            per = 1 << 30;
        C = static_cast<int>(per);
    }
    int run = 0;
    for (int base = 0; base < p.B; base += 32) {
        const int b = base + lane;
        int n = 0;
        if (b < p.B) {
            const int total = lens[b] + p.NQ;
            const int chunk = chunk_of(p, total, C);
            n = (total + chunk - 1) / chunk;
        }
        int incl = n;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int y = __shfl_up_sync(kFull, incl, o);
            if (lane >= o)
                incl += y;
        }
        if (b < p.B) {
            prefix[b] = run + incl - n;
            if (blockIdx.x == 0 && p.sched)
                p.sched[b] = make_int2(run + incl - n, n);
        }
        run += __shfl_sync(kFull, incl, 31);
    }
    if (lane == 0) {
        prefix[p.B] = run;
        info[0] = C;
        info[1] = run * p.NRS * p.KV;
    }
}

// Work item `item`: items are ordered by sequence, key range, row group, KV
// head (adjacent KV heads read interleaved rows of the same cache blocks).
__device__ __forceinline__ Item decode_item(const SplitParams& p, const Sched& s, int item)
{
    const int U = p.NRS * p.KV;
    const int g = item / U;
    const int rem = item - g * U;
    Item it;
    it.rsg = rem / p.KV;
    it.kh = rem - it.rsg * p.KV;
    int lo = 0, hi = p.B - 1;  // last b with prefix[b] <= g
    while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (s.prefix[mid] <= g)
            lo = mid;
        else
            hi = mid - 1;
    }
    it.b = lo;
    it.c = g - s.prefix[lo];
    it.n = s.prefix[lo + 1] - s.prefix[lo];
    it.past = s.lens[lo];
    const int total = it.past + p.NQ;
    const int chunk = chunk_of(p, total, s.auto_chunk);
    it.start = it.c * chunk;
    it.end = min(it.start + chunk, total);
    return it;
}

__device__ __forceinline__ void consumer_bar_sync()
{
    asm volatile("bar.sync 1, %0;" ::"n"(kConsumerWarps * 32) : "memory");
}

// Consumer barrier that also returns the OR of `v` over all consumer threads,
// so that every consumer warp takes the same decision after it.
__device__ __forceinline__ bool consumer_bar_or(bool v)
{
    uint32_t r;
    asm volatile(
        "{\n\t.reg .pred pi, po;\n\t"
        "setp.ne.u32 pi, %1, 0;\n\t"
        "bar.red.or.pred po, 1, %2, pi;\n\t"
        "selp.u32 %0, 1, 0, po;\n\t}"
        : "=r"(r)
        : "r"(static_cast<uint32_t>(v)), "n"(kConsumerWarps * 32)
        : "memory");
    return r != 0;
}

__device__ __forceinline__ void flag_timeout(const SplitParams& p, volatile int* abort_flag)
{
    *abort_flag = 1;
    if (p.status)
        atomicOr(p.status, PA_STATUS_TIMEOUT);
}

// ------------------------------------------------------- float32 CUDA-core math
// One warp: RG query rows, a subset of the tokens of each tile.  A token row
// of D elements is split over LPT lanes (16 bytes each); TPW tokens per warp
// step.  State per lane: running max m and sum l per row (replicated over the
// lanes of a token) and the accumulator slice o[row][VEC].
template <typename T, int D, int RG>
struct SimtMath {
    using E = Elem<T>;
    static constexpr int VEC = E::kVec;
    static constexpr int V2 = VEC / 2;
    static constexpr int LPT = D / VEC;
    static constexpr int TPW = 32 / LPT;
    static_assert(LPT <= 32 && 32 % LPT == 0, "a row must split evenly over lanes");

    float2 q[RG][V2];
    float2 o[RG][V2];
    float m[RG], l[RG];
    int limit[RG];
    int lg, li, ts, TS;

    __device__ void begin(const SplitParams& p, const Item& it, int row0, int R_cta, int lane,
                          int ts_, int TS_)
    {
        lg = lane / LPT;
        li = lane % LPT;
        ts = ts_;
        TS = TS_;
        const T* qbase =
            static_cast<const T*>(p.q) + (static_cast<size_t>(it.b) * p.KV + it.kh) * p.R * D;
        const float2 sc2 = make_float2(p.qscale, p.qscale);
#pragma unroll
        for (int r = 0; r < RG; ++r) {
            const int rl = row0 + r;
            const int rho = it.rsg * p.rows_per_cta + rl;
            if (rl < R_cta) {
                E::load2(qbase + static_cast<size_t>(rho) * D + li * VEC, q[r]);
#pragma unroll
                for (int v = 0; v < V2; ++v)
                    q[r][v] = __fmul2_rn(q[r][v], sc2);
                limit[r] = it.past + (p.causal ? (rho % p.NQ) + 1 : p.NQ);
            } else {
#pragma unroll
                for (int v = 0; v < V2; ++v)
                    q[r][v] = make_float2(0.f, 0.f);
                limit[r] = 0;
            }
            m[r] = -FLT_MAX;
            l[r] = 0.f;
#pragma unroll
            for (int v = 0; v < V2; ++v)
                o[r][v] = make_float2(0.f, 0.f);
        }
    }

    // Tile of n_tile tokens starting at absolute key t0: rows < past come from
    // the cache tile (ks / vs), rows >= past from the new rows (kn / vn).
    __device__ void tile(const T* ks, const T* kn, const T* vs, const T* vn, int t0, int n_tile,
                         int past)
    {
        const int step = TS * TPW;
        for (int base = 0; base < n_tile; base += kSubBatch * step) {
            float sc[kSubBatch][RG];
#pragma unroll
            for (int i = 0; i < kSubBatch; ++i) {
                const int t_rel = base + (i * TS + ts) * TPW + lg;
                const int t_abs = t0 + t_rel;
                const bool live = t_rel < n_tile;
                float2 k2[V2];
                if (live) {
                    const T* row = t_abs < past ? ks + t_rel * D : kn + (t_abs - past) * D;
                    E::load2(row + li * VEC, k2);
                } else {
#pragma unroll
                    for (int v = 0; v < V2; ++v)
                        k2[v] = make_float2(0.f, 0.f);
                }
#pragma unroll
                for (int r = 0; r < RG; ++r) {
                    float2 a = make_float2(0.f, 0.f);
#pragma unroll
                    for (int v = 0; v < V2; ++v)
                        a = __ffma2_rn(q[r][v], k2[v], a);
                    float acc = a.x + a.y;
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
                const float2 f2 = make_float2(f, f);
                m[r] = mn;
                l[r] *= f;
#pragma unroll
                for (int v = 0; v < V2; ++v)
                    o[r][v] = __fmul2_rn(o[r][v], f2);
            }
#pragma unroll
            for (int i = 0; i < kSubBatch; ++i) {
                const int t_rel = base + (i * TS + ts) * TPW + lg;
                if (t_rel >= n_tile)
                    continue;
                const int t_abs = t0 + t_rel;
                const T* row = t_abs < past ? vs + t_rel * D : vn + (t_abs - past) * D;
                float2 v2[V2];
                E::load2(row + li * VEC, v2);
#pragma unroll
                for (int r = 0; r < RG; ++r) {
                    const float pr = fast_exp2(sc[i][r] - m[r]);
                    const float2 p2 = make_float2(pr, pr);
                    l[r] += pr;
#pragma unroll
                    for (int v = 0; v < V2; ++v)
                        o[r][v] = __ffma2_rn(p2, v2[v], o[r][v]);
                }
            }
        }
    }

    // Merge the lane groups of the warp (they saw different tokens), then
    // write the warp's per-row state into the merge buffer slots row0.. .
    __device__ void store(float* mb_o, float* mb_m, float* mb_l, int slot0)
    {
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
                for (int v = 0; v < V2; ++v) {
                    const float ox = __shfl_xor_sync(kFull, o[r][v].x, off);
                    const float oy = __shfl_xor_sync(kFull, o[r][v].y, off);
                    o[r][v].x = o[r][v].x * fa + ox * fb;
                    o[r][v].y = o[r][v].y * fa + oy * fb;
                }
                m[r] = mn;
            }
        }
        if (lg == 0) {
#pragma unroll
            for (int r = 0; r < RG; ++r) {
                const int slot = slot0 + r;
#pragma unroll
                for (int v = 0; v < V2; ++v)
                    *reinterpret_cast<float2*>(&mb_o[slot * D + li * VEC + 2 * v]) = o[r][v];
                if (li == 0) {
                    mb_m[slot] = m[r];
                    mb_l[slot] = l[r];
                }
            }
        }
    }
};

// ------------------------------------------------------- CTA set-up, producer
// Shared memory of the partition kernels, carved from a 1024-aligned base:
//   [0, 64)      full barriers     [64, 128)  empty barriers
//   [128, 192)   broadcast scalars [256, 272) a zeroed 16-byte row (mma path)
//   lens[B] | prefix[B+1] | consumer scratch | ring of `stages` stages.
struct Smem {
    uint64_t* full;
    uint64_t* empty;
    int* info;
    volatile int* abort_flag;
    const void* zero16;
    int* lens;
    int* prefix;
    unsigned char* scratch;
    unsigned char* ring;
};

__device__ __forceinline__ Smem carve(const SplitParams& p, unsigned char* raw)
{
    unsigned char* base = raw + ((1024u - (smem_u32(raw) & 1023u)) & 1023u);
    Smem sm;
    sm.full = reinterpret_cast<uint64_t*>(base);
    sm.empty = sm.full + kMaxStages;
    sm.info = reinterpret_cast<int*>(base + 128);
    sm.abort_flag = sm.info + 15;
    sm.zero16 = base + 256;
    sm.lens = reinterpret_cast<int*>(base + p.lens_off);
    sm.prefix = reinterpret_cast<int*>(base + p.prefix_off);
    sm.scratch = base + p.merge_off;
    sm.ring = base + p.stage_off;
    return sm;
}

// All threads: barriers, clamped lengths, the schedule.
__device__ __forceinline__ Sched setup_cta(const SplitParams& p, const Smem& sm)
{
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (threadIdx.x == 0) {
        for (int s = 0; s < p.stages; ++s) {
            mbar_init(&sm.full[s], 1);
            mbar_init(&sm.empty[s], kConsumerWarps);
        }
        sm.info[15] = 0;
        *reinterpret_cast<uint4*>(const_cast<void*>(sm.zero16)) = make_uint4(0, 0, 0, 0);
        fence_mbar_init();
    }
    const int cap = p.maxb * p.BLOCK;
    for (int b = threadIdx.x; b < p.B; b += kThreads) {
        int s = p.seq_lens[b];
        if (s < 0 || s > cap) {
            if (blockIdx.x == 0 && p.status)
                atomicOr(p.status, PA_STATUS_BAD_LENGTH);
            s = s < 0 ? 0 : cap;
        }
        sm.lens[b] = s;
    }
    __syncthreads();
    if (warp == 0)
        build_schedule(p, sm.lens, sm.prefix, sm.info, lane);
    __syncthreads();
    Sched sc;
    sc.lens = sm.lens;
    sc.prefix = sm.prefix;
    sc.auto_chunk = sm.info[0];
    sc.total_items = sm.info[1];
    return sc;
}

// The producer warp: for every tile of every item of this CTA, wait for a
// free stage, read the table entries of the tile (one per lane), and issue
// one TMA box per cache block for K and for V (two 64-column boxes per block
// with the 128-byte swizzle when kSwizzled), plus a bulk copy of the new rows
// when the tile reaches them.  Completion is counted on the stage's full
// barrier.
template <typename T, int D, bool kSwizzled>
__device__ void produce(const SplitParams& p, const Sched& sc, const Smem& sm, const CUtensorMap* kmap,
                        const CUtensorMap* vmap, int lane)
{
    if (lane == 0) {
        tma_prefetch_desc(kmap);
        tma_prefetch_desc(vmap);
    }
    const int S = p.stages, TT = p.TT;
    const uint32_t block_bytes = static_cast<uint32_t>(p.BLOCK * D * sizeof(T));
    const uint32_t new_bytes = static_cast<uint32_t>(p.NQ * D * sizeof(T));
    uint32_t gt = 0;  // tiles issued by this CTA
    bool ok = true;
    for (int item = blockIdx.x; item < sc.total_items && ok; item += gridDim.x) {
        const Item it = decode_item(p, sc, item);
        const int ntiles = (it.end - it.start + TT - 1) / TT;
        for (int j = 0; j < ntiles; ++j, ++gt) {
            const int s = gt % S;
            if (gt >= static_cast<uint32_t>(S)) {
                ok = !*sm.abort_flag &&
                     mbar_wait_bounded(&sm.empty[s], ((gt / S) - 1) & 1, kWaitLimitNs);
                ok = __all_sync(kFull, ok);
                if (!ok) {
                    if (lane == 0)
                        flag_timeout(p, sm.abort_flag);
                    break;
                }
            }
            const int t0 = it.start + j * TT;
            const int t1 = min(t0 + TT, it.end);
            const int cache_end = min(t1, it.past);
            const int nb = cache_end > t0 ? (cache_end - t0 + p.BLOCK - 1) / p.BLOCK : 0;
            const bool has_new = t1 > it.past;
            int phys = 0;
            if (lane < nb) {
                phys = p.table[static_cast<size_t>(it.b) * p.maxb + t0 / p.BLOCK + lane];
                if (p.checked && (phys < 0 || phys >= p.num_blocks) && p.status)
                    atomicOr(p.status, PA_STATUS_BAD_BLOCK);
            }
            unsigned char* st = sm.ring + static_cast<size_t>(s) * p.stage_bytes;
            unsigned char* ks = st;
            unsigned char* vs = st + p.v_off;
            if (lane == 0)
                mbar_arrive_expect_tx(&sm.full[s],
                                      2u * nb * block_bytes + (has_new ? 2u * new_bytes : 0u));
            __syncwarp();
            if (lane < nb) {
                // Out-of-pool coordinates read as zeros: the copy never faults.
                const int z = phys * p.BLOCK;
                if constexpr (kSwizzled) {
                    // [D/64 halves][TT rows][64 columns], 128-byte swizzle
#pragma unroll
                    for (int h = 0; h < D / 64; ++h) {
                        const size_t off = static_cast<size_t>(h) * TT * 128 + lane * p.BLOCK * 128;
                        tma_load_3d(ks + off, kmap, 64 * h, it.kh, z, &sm.full[s]);
                        tma_load_3d(vs + off, vmap, 64 * h, it.kh, z, &sm.full[s]);
                    }
                } else {
                    const size_t off = static_cast<size_t>(lane) * p.BLOCK * D * sizeof(T);
                    tma_load_3d(ks + off, kmap, 0, it.kh, z, &sm.full[s]);
                    tma_load_3d(vs + off, vmap, 0, it.kh, z, &sm.full[s]);
                }
            }
            if (has_new && lane == 0) {
                const size_t off = (static_cast<size_t>(it.b) * p.KV + it.kh) * p.NQ * D;
                bulk_load(st + p.knew_off, static_cast<const T*>(p.k_new) + off, new_bytes,
                          &sm.full[s]);
                bulk_load(st + p.vnew_off, static_cast<const T*>(p.v_new) + off, new_bytes,
                          &sm.full[s]);
            }
        }
    }
    // Leave no copy in flight if the pipeline was abandoned.
    __syncwarp();
    if (*sm.abort_flag && lane == 0) {
        const uint32_t first = gt > static_cast<uint32_t>(S) ? gt - S : 0u;
        for (uint32_t g = first; g < gt; ++g)
            mbar_wait_bounded(&sm.full[g % S], (g / S) & 1, kWaitLimitNs);
    }
}

// ------------------------------------------- float32 CUDA-core partition kernel
// T: element type of q/K/V; D: head size; RG: query rows per consumer warp;
// TO: output element type.  One CTA per SM (persistent).
template <typename T, int D, int RG, typename TO>
__global__ void __launch_bounds__(kThreads, 1)
    pa_split_kernel(const __grid_constant__ SplitParams p, const __grid_constant__ CUtensorMap kmap,
                    const __grid_constant__ CUtensorMap vmap)
{
    extern __shared__ __align__(1024) unsigned char smem_raw[];
    const Smem sm = carve(p, smem_raw);
    float* mb_o = reinterpret_cast<float*>(sm.scratch);  // [kConsumerWarps*RG][D]
    float* mb_m = mb_o + kConsumerWarps * RG * D;
    float* mb_l = mb_m + kConsumerWarps * RG;

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int S = p.stages;
    const int TT = p.TT;

    // Inputs may be produced by the previous kernel on the stream.
    grid_dependency_wait();
    grid_dependents_launch();
    const Sched sc = setup_cta(p, sm);

    if (warp == kConsumerWarps) {
        produce<T, D, false>(p, sc, sm, &kmap, &vmap, lane);
        return;
    }

    using Math = SimtMath<T, D, RG>;
    uint32_t gt = 0;
    const int tid = threadIdx.x;  // 0 .. kConsumerWarps*32-1
    for (int item = blockIdx.x; item < sc.total_items; item += gridDim.x) {
        const Item it = decode_item(p, sc, item);
        const int ntiles = (it.end - it.start + TT - 1) / TT;
        const int R_cta = min(p.rows_per_cta, p.R - it.rsg * p.rows_per_cta);
        const int nrg_raw = (R_cta + RG - 1) / RG;
        const int nrg = nrg_raw <= 1 ? 1 : nrg_raw <= 2 ? 2 : nrg_raw <= 4 ? 4 : 8;
        const int TS = kConsumerWarps / nrg;
        const int rg = warp % nrg;
        const int ts = warp / nrg;

        Math mt;
        mt.begin(p, it, rg * RG, R_cta, lane, ts, TS);
        bool alive = true;
        for (int j = 0; j < ntiles; ++j, ++gt) {
            const int s = gt % S;
            if (alive) {
                alive = !*sm.abort_flag &&
                        mbar_wait_bounded(&sm.full[s], (gt / S) & 1, kWaitLimitNs);
                alive = __all_sync(kFull, alive);
                if (!alive && lane == 0)
                    flag_timeout(p, sm.abort_flag);
            }
            if (!alive)
                continue;
            const unsigned char* st = sm.ring + static_cast<size_t>(s) * p.stage_bytes;
            const int t0 = it.start + j * TT;
            mt.tile(reinterpret_cast<const T*>(st), reinterpret_cast<const T*>(st + p.knew_off),
                    reinterpret_cast<const T*>(st + p.v_off),
                    reinterpret_cast<const T*>(st + p.vnew_off), t0, min(TT, it.end - t0),
                    it.past);
            __syncwarp();
            if (lane == 0)
                mbar_arrive(&sm.empty[s]);
        }

        // Merge the token subsets of each row and finish the item.
        const int span = nrg * RG;
        consumer_bar_sync();  // the previous item's readers are done with the buffer
        mt.store(mb_o, mb_m, mb_l, ts * span + rg * RG);
        // Uniform decision: a flag set by any warp (or the producer) stops all.
        if (consumer_bar_or(*sm.abort_flag != 0))
            break;
        const size_t out_row0 =
            (static_cast<size_t>(it.b) * p.KV + it.kh) * p.R + it.rsg * p.rows_per_cta;
        for (int idx = tid; idx < R_cta * D; idx += kConsumerWarps * 32) {
            const int rl = idx / D, d = idx - rl * D;
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
            if (it.n == 1) {
                const float val = L == 0.f ? O : O / L;
                static_cast<TO*>(p.out)[(out_row0 + rl) * D + d] = from_float<TO>(val);
            } else {
                const size_t wrow = static_cast<size_t>(item) * p.row_stride + rl;
                p.ws_o[wrow * D + d] = O;
                if (d == 0)
                    p.ws_ml[wrow] = make_float2(M, L);
            }
        }
    }
}

// ------------------------------------------- 16-bit tensor-core partition kernel
template <typename T>
struct Pack;
template <>
struct Pack<__half> {
    // (hi, lo) with hi + lo = (x, y) to about 22 bits
    __device__ static void split(float x, float y, uint32_t& hi, uint32_t& lo)
    {
        const __half2 h = __floats2half2_rn(x, y);
        const float2 hf = __half22float2(h);
        const __half2 l = __floats2half2_rn(x - hf.x, y - hf.y);
        memcpy(&hi, &h, 4);
        memcpy(&lo, &l, 4);
    }
};
template <>
struct Pack<__nv_bfloat16> {
    __device__ static void split(float x, float y, uint32_t& hi, uint32_t& lo)
    {
        const __nv_bfloat162 h = __floats2bfloat162_rn(x, y);
        const float2 hf = __bfloat1622float2(h);
        const __nv_bfloat162 l = __floats2bfloat162_rn(x - hf.x, y - hf.y);
        memcpy(&hi, &h, 4);
        memcpy(&lo, &l, 4);
    }
};

// Stage of the tensor-core kernel: K and V tiles of kMmaTokens tokens stored
// [D/64 halves][tokens][64 columns] with the TMA 128-byte swizzle (16-byte
// chunk c of token row t sits at chunk c ^ (t % 8)); the new rows unswizzled.
template <int D>
__device__ __forceinline__ uint32_t tile_chunk_addr(uint32_t tile, int tok, int chunk)
{
    const int h = chunk >> 3, c = chunk & 7;
    return tile + h * (kMmaTokens * 128) + tok * 128 + ((c ^ (tok & 7)) << 4);
}

// Shared-memory address of 16-byte chunk `chunk` of token `tok` of the tile
// starting at key t0: a cache row, a new row, or the zero row past the tile.
template <int D>
__device__ __forceinline__ uint32_t row_chunk(uint32_t tile, uint32_t fresh, uint32_t zero, int tok,
                                              int n_tile, int t0, int past, int chunk)
{
    if (tok >= n_tile)
        return zero;
    const int ta = t0 + tok;
    if (ta < past)
        return tile_chunk_addr<D>(tile, tok, chunk);
    return fresh + (ta - past) * (D * 2) + chunk * 16;
}

// T: __half or __nv_bfloat16; D: head size; MT: 16-row tiles per CTA pass;
// TO: output element type.  One CTA per SM (persistent).
//
// Per stage of kMmaTokens tokens: warp w computes S = Q K^T for tokens
// [16w, 16w+16) with m16n8k16 MMAs (float32 accumulators), scales and masks
// them, and publishes its row maxima; after a barrier every warp forms the
// common running maximum, writes its probabilities P (split into a 16-bit
// high part and a 16-bit remainder so that P V keeps about 22 bits) to shared
// memory; after a second barrier warp w accumulates O[:, its D/8 columns] +=
// P V over all tokens of the stage.  Every warp therefore owns distinct output
// columns and no cross-warp merge of O is needed; the row sums are added at
// the end of the item.
template <typename T, int D, int MT, typename TO>
__global__ void __launch_bounds__(kThreads, 1)
    pa_mma_kernel(const __grid_constant__ SplitParams p, const __grid_constant__ CUtensorMap kmap,
                  const __grid_constant__ CUtensorMap vmap)
{
    constexpr bool kBf = std::is_same<T, __nv_bfloat16>::value;
    constexpr int KS = D / 16;                     // k-steps of Q K^T
    constexpr int NTW = D / 8 / kConsumerWarps;    // 8-column tiles of O per warp
    constexpr int ROWS = 16 * MT;
    constexpr int PP = kMmaTokens + 8;             // P row pitch (halves), breaks bank conflicts
    static_assert(NTW == 1 || NTW == 2, "D must be 64 or 128");

    extern __shared__ __align__(1024) unsigned char smem_raw[];
    const Smem sm = carve(p, smem_raw);
    uint16_t* Phi = reinterpret_cast<uint16_t*>(sm.scratch);  // [ROWS][PP]
    uint16_t* Plo = Phi + ROWS * PP;
    float* red_max = reinterpret_cast<float*>(Plo + ROWS * PP);  // [warps][ROWS]
    float* red_l = red_max + kConsumerWarps * ROWS;

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int S = p.stages;
    const int TT = kMmaTokens;

    grid_dependency_wait();
    grid_dependents_launch();
    const Sched sc = setup_cta(p, sm);

    if (warp == kConsumerWarps) {
        produce<T, D, true>(p, sc, sm, &kmap, &vmap, lane);
        return;
    }

    const int g = lane >> 2, qd = lane & 3;
    const uint32_t zero = smem_u32(sm.zero16);
    const uint32_t phi_base = smem_u32(Phi), plo_base = smem_u32(Plo);
    const int tb = 16 * warp;  // this warp's tokens of every stage
    uint32_t gt = 0;

    for (int item = blockIdx.x; item < sc.total_items; item += gridDim.x) {
        const Item it = decode_item(p, sc, item);
        const int ntiles = (it.end - it.start + TT - 1) / TT;
        const int R_cta = min(ROWS, p.R - it.rsg * ROWS);
        const T* qbase = static_cast<const T*>(p.q) +
                         ((static_cast<size_t>(it.b) * p.KV + it.kh) * p.R + it.rsg * ROWS) * D;

        // Q fragments (row-major A of m16n8k16), zero for padding rows.
        uint32_t qa[MT][KS][4];
        int lim[MT][2];
#pragma unroll
        for (int mt = 0; mt < MT; ++mt) {
            const int r0 = mt * 16 + g, r1 = r0 + 8;
#pragma unroll
            for (int ks = 0; ks < KS; ++ks) {
                const int d0 = ks * 16 + 2 * qd;
                qa[mt][ks][0] = r0 < R_cta ? *reinterpret_cast<const uint32_t*>(qbase + r0 * D + d0) : 0u;
                qa[mt][ks][1] = r1 < R_cta ? *reinterpret_cast<const uint32_t*>(qbase + r1 * D + d0) : 0u;
                qa[mt][ks][2] = r0 < R_cta ? *reinterpret_cast<const uint32_t*>(qbase + r0 * D + d0 + 8) : 0u;
                qa[mt][ks][3] = r1 < R_cta ? *reinterpret_cast<const uint32_t*>(qbase + r1 * D + d0 + 8) : 0u;
            }
#pragma unroll
            for (int h = 0; h < 2; ++h) {
                const int rl = mt * 16 + g + 8 * h;
                const int rho = it.rsg * ROWS + rl;
                lim[mt][h] = rl < R_cta ? it.past + (p.causal ? (rho % p.NQ) + 1 : p.NQ) : 0;
            }
        }

        float m[MT][2], lp[MT][2], o[MT][NTW][4];
#pragma unroll
        for (int mt = 0; mt < MT; ++mt) {
#pragma unroll
            for (int h = 0; h < 2; ++h) {
                m[mt][h] = -FLT_MAX;
                lp[mt][h] = 0.f;
            }
#pragma unroll
            for (int i = 0; i < NTW; ++i)
#pragma unroll
                for (int e = 0; e < 4; ++e)
                    o[mt][i][e] = 0.f;
        }

        bool failed = false;
        for (int j = 0; j < ntiles; ++j, ++gt) {
            const int s = gt % S;
            bool ok = !*sm.abort_flag && mbar_wait_bounded(&sm.full[s], (gt / S) & 1, kWaitLimitNs);
            ok = __all_sync(kFull, ok);
            const uint32_t st = smem_u32(sm.ring) + s * p.stage_bytes;
            const uint32_t k_tile = st, k_new = st + p.knew_off;
            const uint32_t v_tile = st + p.v_off, v_new = st + p.vnew_off;
            const int t0 = it.start + j * TT;
            const int n_tile = min(TT, it.end - t0);

            // ---- S = Q K^T for tokens [tb, tb + 16)
            float sa[MT][2][4];
#pragma unroll
            for (int mt = 0; mt < MT; ++mt)
#pragma unroll
                for (int nt = 0; nt < 2; ++nt)
#pragma unroll
                    for (int e = 0; e < 4; ++e)
                        sa[mt][nt][e] = 0.f;
            if (ok) {
                const int tok = tb + (lane & 7) + ((lane >> 4) << 3);
#pragma unroll
                for (int ks = 0; ks < KS; ++ks) {
                    const int chunk = 2 * ks + ((lane >> 3) & 1);
                    uint32_t b00, b01, b10, b11;
                    ldsm_x4(row_chunk<D>(k_tile, k_new, zero, tok, n_tile, t0, it.past, chunk), b00,
                            b01, b10, b11);
#pragma unroll
                    for (int mt = 0; mt < MT; ++mt) {
                        mma_16816<kBf>(sa[mt][0], qa[mt][ks], b00, b01);
                        mma_16816<kBf>(sa[mt][1], qa[mt][ks], b10, b11);
                    }
                }
            }
            // scale, mask, partial row maxima over this warp's 16 tokens
#pragma unroll
            for (int mt = 0; mt < MT; ++mt) {
#pragma unroll
                for (int h = 0; h < 2; ++h) {
                    float mx = -INFINITY;
#pragma unroll
                    for (int nt = 0; nt < 2; ++nt)
#pragma unroll
                        for (int e = 0; e < 2; ++e) {
                            const int tk = tb + nt * 8 + 2 * qd + e;
                            const float v = sa[mt][nt][2 * h + e] * p.qscale;
                            const bool valid = tk < n_tile && t0 + tk < lim[mt][h];
                            sa[mt][nt][2 * h + e] = valid ? v : -INFINITY;
                            mx = fmaxf(mx, sa[mt][nt][2 * h + e]);
                        }
                    mx = fmaxf(mx, __shfl_xor_sync(kFull, mx, 1));
                    mx = fmaxf(mx, __shfl_xor_sync(kFull, mx, 2));
                    if (qd == 0)
                        red_max[warp * ROWS + mt * 16 + g + 8 * h] = mx;
                }
            }
            if (consumer_bar_or(!ok)) {  // (A) uniform stop if any wait failed
                if (threadIdx.x == 0)
                    flag_timeout(p, sm.abort_flag);
                failed = true;
                break;
            }
            // common running maximum, probabilities, row-sum partials
            float f[MT][2];
#pragma unroll
            for (int mt = 0; mt < MT; ++mt) {
#pragma unroll
                for (int h = 0; h < 2; ++h) {
                    const int row = mt * 16 + g + 8 * h;
                    float tmax = red_max[row];
#pragma unroll
                    for (int w = 1; w < kConsumerWarps; ++w)
                        tmax = fmaxf(tmax, red_max[w * ROWS + row]);
                    const float mn = fmaxf(m[mt][h], tmax);
                    f[mt][h] = fast_exp2(m[mt][h] - mn);
                    m[mt][h] = mn;
                    lp[mt][h] *= f[mt][h];
                }
#pragma unroll
                for (int nt = 0; nt < 2; ++nt) {
#pragma unroll
                    for (int h = 0; h < 2; ++h) {
                        const float p0 = fast_exp2(sa[mt][nt][2 * h] - m[mt][h]);
                        const float p1 = fast_exp2(sa[mt][nt][2 * h + 1] - m[mt][h]);
                        lp[mt][h] += p0 + p1;
                        uint32_t hi, lo;
                        Pack<T>::split(p0, p1, hi, lo);
                        const int row = mt * 16 + g + 8 * h;
                        const int col = tb + nt * 8 + 2 * qd;
                        *reinterpret_cast<uint32_t*>(&Phi[row * PP + col]) = hi;
                        *reinterpret_cast<uint32_t*>(&Plo[row * PP + col]) = lo;
                    }
                }
            }
            consumer_bar_sync();  // (B) P of all warps is in shared memory
#pragma unroll
            for (int mt = 0; mt < MT; ++mt)
#pragma unroll
                for (int i = 0; i < NTW; ++i)
#pragma unroll
                    for (int e = 0; e < 4; ++e)
                        o[mt][i][e] *= f[mt][e >> 1];

            // ---- O[:, this warp's columns] += P V over the tokens of the stage
            const int nk = (n_tile + 15) >> 4;
            for (int kk = 0; kk < nk; ++kk) {
                uint32_t ahi[MT][4], alo[MT][4];
#pragma unroll
                for (int mt = 0; mt < MT; ++mt) {
                    const int row = mt * 16 + (lane & 7) + (((lane >> 3) & 1) << 3);
                    const int col = kk * 16 + ((lane >> 4) << 3);
                    const uint32_t off = (row * PP + col) * 2;
                    ldsm_x4(phi_base + off, ahi[mt][0], ahi[mt][1], ahi[mt][2], ahi[mt][3]);
                    ldsm_x4(plo_base + off, alo[mt][0], alo[mt][1], alo[mt][2], alo[mt][3]);
                }
                const int tok = kk * 16 + (lane & 7) + (((lane >> 3) & 1) << 3);
                uint32_t vb[NTW][2];
                if constexpr (NTW == 2) {
                    const int chunk = warp * 2 + (lane >> 4);
                    ldsm_x4_t(row_chunk<D>(v_tile, v_new, zero, tok, n_tile, t0, it.past, chunk),
                              vb[0][0], vb[0][1], vb[1][0], vb[1][1]);
                } else {
                    ldsm_x2_t(row_chunk<D>(v_tile, v_new, zero, tok, n_tile, t0, it.past, warp),
                              vb[0][0], vb[0][1]);
                }
#pragma unroll
                for (int mt = 0; mt < MT; ++mt)
#pragma unroll
                    for (int i = 0; i < NTW; ++i) {
                        mma_16816<kBf>(o[mt][i], ahi[mt], vb[i][0], vb[i][1]);
                        mma_16816<kBf>(o[mt][i], alo[mt], vb[i][0], vb[i][1]);
                    }
            }
            __syncwarp();
            if (lane == 0)
                mbar_arrive(&sm.empty[s]);
        }
        if (failed)
            break;

        // ---- item end: row sums over all warps, then each warp writes its columns
#pragma unroll
        for (int mt = 0; mt < MT; ++mt)
#pragma unroll
            for (int h = 0; h < 2; ++h) {
                float l = lp[mt][h];
                l += __shfl_xor_sync(kFull, l, 1);
                l += __shfl_xor_sync(kFull, l, 2);
                if (qd == 0)
                    red_l[warp * ROWS + mt * 16 + g + 8 * h] = l;
            }
        if (consumer_bar_or(*sm.abort_flag != 0))
            break;
        const size_t out_row0 =
            (static_cast<size_t>(it.b) * p.KV + it.kh) * p.R + it.rsg * ROWS;
#pragma unroll
        for (int mt = 0; mt < MT; ++mt)
#pragma unroll
            for (int h = 0; h < 2; ++h) {
                const int rl = mt * 16 + g + 8 * h;
                if (rl >= R_cta)
                    continue;
                float L = 0.f;
#pragma unroll
                for (int w = 0; w < kConsumerWarps; ++w)
                    L += red_l[w * ROWS + rl];
#pragma unroll
                for (int i = 0; i < NTW; ++i) {
                    const int d = (warp * NTW + i) * 8 + 2 * qd;
                    const float ox = o[mt][i][2 * h], oy = o[mt][i][2 * h + 1];
                    if (it.n == 1) {
                        const float sx = L == 0.f ? ox : ox / L;
                        const float sy = L == 0.f ? oy : oy / L;
                        TO* dst = static_cast<TO*>(p.out) + (out_row0 + rl) * D + d;
                        dst[0] = from_float<TO>(sx);
                        dst[1] = from_float<TO>(sy);
                    } else {
                        const size_t wrow = static_cast<size_t>(item) * p.row_stride + rl;
                        *reinterpret_cast<float2*>(&p.ws_o[wrow * D + d]) = make_float2(ox, oy);
                        if (warp == 0 && i == 0 && qd == 0)
                            p.ws_ml[wrow] = make_float2(m[mt][h], L);
                    }
                }
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
#pragma unroll 4
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
SplitFn pick_split_simt(int D, int RG)
{
    if (D == 64)
        return RG == 4 ? pa_split_kernel<T, 64, 4, TO> : pa_split_kernel<T, 64, 8, TO>;
    return RG == 4 ? pa_split_kernel<T, 128, 4, TO> : pa_split_kernel<T, 128, 8, TO>;
}

template <typename T, typename TO>
SplitFn pick_split_mma(int D, int MT)
{
    if (D == 64)
        return MT == 1 ? pa_mma_kernel<T, 64, 1, TO> : pa_mma_kernel<T, 64, 2, TO>;
    return MT == 1 ? pa_mma_kernel<T, 128, 1, TO> : pa_mma_kernel<T, 128, 2, TO>;
}

template <typename TO>
CombineFn pick_combine_typed(int D)
{
    return D == 64 ? pa_combine_kernel<64, TO> : pa_combine_kernel<128, TO>;
}

}  // namespace pa
