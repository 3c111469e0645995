// pa_kernels.cuh -- the sm_103a kernels of decode attention over a paged KV
// cache: the persistent partition kernels and the log-sum-exp merge kernel.
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
//   * a segment is (sequence, row group, KV head) over its keys; its CTA serves
//     every query row of the KV head, so each K/V row is read from HBM once
//     (the page runs one threadgroup per query head and re-reads K/V H/KV
//     times);
//   * the kernels are persistent, one CTA per SM.  Automatic split: the
//     segments, cut into stage-sized units, are laid end to end and each CTA
//     takes a cost-balanced contiguous range, computed on the device from the
//     lengths (schedule section below); fixed partitions: P ranges of whole
//     blocks per segment dealt round-robin;
//   * two producer warps stream cache blocks into a shared-memory ring with
//     TMA tensor copies (one box = one block of one KV head; K by one warp, V
//     by the other) and the query and new rows with bulk copies, completing on
//     mbarriers; they run ahead across piece boundaries;
//   * eight consumer warps: 16-bit caches on tensor cores (mma.sync
//     m16n8k16, float32 accumulators) -- pa_mmat_kernel with the tokens on the
//     MMA's 16-row side for at most 8 query rows per KV head, pa_mma_kernel
//     with the query rows there otherwise (more than 16 rows at D = 128 run
//     on tcgen05 instead: pa_umma32_kernel, pa_decode_tc.cu, on the same
//     schedule, pieces and merge); float32 caches on CUDA cores
//     (pa_split_kernel: 16-byte shared-memory reads, FMAs, warp-shuffle dot
//     reductions); an online base-2 softmax throughout;
//   * a piece that covers a whole segment writes the normalised output;
//     otherwise its partial state goes to the workspace, and the last CTA to
//     finish a split segment merges it in the kernel (automatic split) or the
//     merge kernel, launched with programmatic dependent launch, combines the
//     partials (fixed partitions).
//
// Every wait is bounded (PA_STATUS_TIMEOUT); no kernel traps.
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include <cfloat>
#include <climits>
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
// A segment is the key range [0, past + NQ) of one (sequence b, row group rsg,
// KV head kh).  A piece is a contiguous part [start, end) of one segment that
// one CTA processes; `whole` pieces write the normalised output, the others a
// partial (max, sum, accumulator) record `rec` of the workspace.
//
// Automatic mode (partitions == 0): the segments, cut into units of one
// pipeline stage (TT tokens), are laid end to end (sequence, then row group,
// then KV head) and each persistent CTA takes a contiguous range of units
// (cost-balanced, below).  A stage costs about the same whether full or not, so
// CTA boundaries fall on stage boundaries and only a segment's last stage is
// partial.  Only the pieces cut at CTA boundaries need merging (records 2k and
// 2k+1: the CTA's first and last piece).
// Fixed partitions (P >= 1): each segment is split into P ranges of whole
// blocks (P == 1: no split); the ranges are items dealt to CTAs round-robin;
// range c of segment (b, rsg, kh) writes record ((b P + c) NRS + rsg) KV + kh,
// so the merge kernel finds a segment's records without the schedule.
struct Item {
    int b, rsg, kh, past, start, end;
    int whole;  // the piece is its whole segment
    int rec;    // workspace record of a partial piece
    int units;  // automatic mode: units of the piece
};

__device__ __forceinline__ int chunk_of(const SplitParams& p, int total)
{
    const int per = p.partitions == 1 ? total : (total + p.partitions - 1) / p.partitions;
    return ((per + p.BLOCK - 1) >> p.lg_block) << p.lg_block;
}

// Shared-memory schedule built once per CTA.
struct Sched {
    const int* lens;    // [B] clamped cached lengths
    const int* prefix;  // [B + 1] automatic: units before sequence b (all its segments);
                        //         fixed: ranges before sequence b (one segment's worth)
    int total;          // automatic: W units; fixed: number of items
    long long cost;     // automatic: C = W + vunits * (number of segments)
    int pos0, stop0;    // automatic: this CTA's units [pos0, stop0)
    int b0, seg0, uu0;  // automatic: where unit pos0 lies (sequence, segment, unit)
};

// Automatic mode deals cost, not units: segment g (in stream order) costs
// vunits + its units, the virtual units charged ahead of its first real unit,
// so that a CTA holding many short pieces (each with a fixed overhead) gets
// fewer units.  Real unit x of segment g sits at cost position
// c(x) = x + vunits * (g + 1); CTA k of G owns the units whose c * G / C
// rounds down to k, a contiguous and, for the CTAs inside a segment, non-empty
// range (G <= C).

// CTA of G owning cost position c: the k with T(k) <= c < T(k + 1), where
// T(k) = ceil(k C / G) (all in int32: C < 2^31, G <= kMaxGrid).
__device__ __forceinline__ int cost_owner(int c, int C, int G)
{
    const int q = C / G, r = C - q * G;
    auto T = [&](int k) { return k * q + (k * r + G - 1) / G; };
    int k = min(static_cast<int>(static_cast<float>(c) * static_cast<float>(G) / static_cast<float>(C)),
                G - 1);
    while (k + 1 < G && T(k + 1) <= c)
        ++k;
    while (k > 0 && T(k) > c)
        --k;
    return k;
}

// CTAs holding segment g = its units [x0, x0 + nu): the first (k0), how many,
// and the workspace record of the segment's piece in CTA k0 (2 k0 when the
// segment starts that CTA's range, else 2 k0 + 1).
struct SegSpan {
    int k0, n, rec_first;
};
__device__ __forceinline__ SegSpan seg_span(int x0, int nu, int g, int V, int C, int G)
{
    const int c0 = x0 + V * (g + 1);
    SegSpan r;
    r.k0 = cost_owner(c0, C, G);
    r.n = cost_owner(c0 + nu - 1, C, G) - r.k0 + 1;
    const bool cont = x0 > 0 && cost_owner(x0 - 1 + V * g, C, G) == r.k0;
    r.rec_first = 2 * r.k0 + (cont ? 1 : 0);
    return r;
}

// Warp 0 alone: loads and clamps the lengths into `lens` (a length beyond the
// table sets PA_STATUS_BAD_LENGTH) and writes the exclusive prefix of the
// per-sequence counts into `prefix` (automatic mode: the units of all NRS * KV
// segments of a sequence; fixed partitions: its key ranges), up to four
// 32-sequence chunks of loads in flight at once.  CTA 0 also records every
// sequence's (prefix, count) for the merge kernel.  Returns the prefix total.
__device__ __forceinline__ int scan_lengths(const SplitParams& p, int* lens, int* prefix, int lane)
{
    const int U = p.NRS * p.KV;
    const bool stream = p.partitions == 0;
    const int cap = p.maxb << p.lg_block;
    int run = 0;
    for (int base = 0; base < p.B; base += 128) {
        int sv[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const int b = base + 32 * i + lane;
            sv[i] = b < p.B ? __ldg(p.seq_lens + b) : 0;
        }
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            if (base + 32 * i >= p.B)
                break;  // warp-uniform
            const int b = base + 32 * i + lane;
            int n = 0;
            if (b < p.B) {
                int v = sv[i];
                if (v < 0 || v > cap) {
                    if (blockIdx.x == 0 && p.status)
                        atomicOr(p.status, PA_STATUS_BAD_LENGTH);
                    v = v < 0 ? 0 : cap;
                }
                lens[b] = v;
                const int total = v + p.NQ;
                if (stream) {
                    n = (total + p.TT - 1) >> p.lg_tt;
                } else {
                    const int chunk = chunk_of(p, total);
                    n = (total + chunk - 1) / chunk;
                }
            }
            const int w = stream ? n * U : n;
            int incl = w;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const int y = __shfl_up_sync(kFull, incl, o);
                if (lane >= o)
                    incl += y;
            }
            if (b < p.B) {
                prefix[b] = run + incl - w;
                if (blockIdx.x == 0 && p.sched)
                    p.sched[b] = make_int2(run + incl - w, n);
            }
            run += __shfl_sync(kFull, incl, 31);
        }
    }
    if (lane == 0)
        prefix[p.B] = run;
    return run;
}

__device__ __forceinline__ int last_le(const int* prefix, int B, long long x)
{
    int lo = 0, hi = B - 1;  // last b with prefix[b] <= x
    while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (prefix[mid] <= x)
            lo = mid;
        else
            hi = mid - 1;
    }
    return lo;
}

// Last b in [0, B) whose cost prefix prefix[b] + VU * b is <= T (warp-
// collective; the cost prefix is non-decreasing and 0 at b = 0): a ballot over
// every 32nd sequence, then one within the chunk found.
__device__ __forceinline__ int last_cost_le(const int* prefix, int B, int VU, int T, int lane)
{
    int lo = 0;
    for (int base = 0; base < B; base += 32 * 32) {
        const int b = base + 32 * lane;
        const unsigned m = __ballot_sync(kFull, b < B && prefix[b] + VU * b <= T);
        if (m == 0)
            break;
        lo = base + 32 * (31 - __clz(m));
        if (m != kFull)
            break;
    }
    const int b = lo + lane;
    const unsigned m = __ballot_sync(kFull, b < B && prefix[b] + VU * b <= T);
    return lo + 31 - __clz(m);
}

// First real unit of CTA k of G (automatic mode): the smallest x with
// c(x) >= ceil(k C / G), or W when there is none, with its sequence, segment
// and unit within the segment (warp-collective, the same in every lane).
// C < 2^31 and G <= kMaxGrid keep it in int32.
struct CostPos {
    int x, b, seg, uu;
};
__device__ __forceinline__ CostPos cost_start(const SplitParams& p, const Sched& sc, int k, int G, int lane)
{
    const int C = static_cast<int>(sc.cost);
    const int q = C / G, r = C - q * G;
    const int T = k * q + (k * r + G - 1) / G;
    if (T >= C)
        return CostPos{sc.total, p.B, 0, 0};
    const int VU = p.vunits * p.NRS * p.KV;  // cost of one sequence's virtual units
    const int lo = last_cost_le(sc.prefix, p.B, VU, T, lane);
    const int nb = (sc.lens[lo] + p.NQ + p.TT - 1) >> p.lg_tt;
    const int local = T - (sc.prefix[lo] + VU * lo);
    const int per = nb + p.vunits;
    const int s = local / per;
    const int uu = max(local - s * per - p.vunits, 0);
    return CostPos{sc.prefix[lo] + s * nb + uu, lo, s, uu};
}

// Iterates this CTA's pieces in order (identically in every warp).  In the
// automatic mode only first() searches the schedule; next() steps to the
// following segment, since every piece but the CTA's last ends where its
// segment ends and every segment holds at least one unit.
struct PieceIter {
    long long pos, stop;
    bool ok;
    Item it;
    int seg_units;  // automatic mode: units of each segment of sequence it.b

    __device__ __forceinline__ void first(const SplitParams& p, const Sched& sc)
    {
        if (p.partitions == 0) {
            // the CTA's range and first piece, located once in setup_cta
            pos = sc.pos0;
            stop = sc.stop0;
            ok = pos < stop;
            if (!ok)
                return;
            const int b = sc.b0, seg = sc.seg0, uu = sc.uu0;
            seg_units = (sc.lens[b] + p.NQ + p.TT - 1) >> p.lg_tt;
            it.b = b;
            it.rsg = seg / p.KV;
            it.kh = seg - it.rsg * p.KV;
            it.past = sc.lens[b];
            it.start = uu << p.lg_tt;
            set_len(p, seg_units - uu, uu == 0);
            it.rec = 2 * blockIdx.x;
        } else {
            pos = blockIdx.x;
            stop = sc.total;
            load_fixed(p, sc);
        }
    }

    __device__ __forceinline__ void next(const SplitParams& p, const Sched& sc)
    {
        if (p.partitions == 0) {
            pos += it.units;
            ok = pos < stop;
            if (!ok)
                return;
            if (++it.kh == p.KV) {
                it.kh = 0;
                if (++it.rsg == p.NRS) {
                    it.rsg = 0;
                    ++it.b;
                    it.past = sc.lens[it.b];
                    seg_units = (it.past + p.NQ + p.TT - 1) >> p.lg_tt;
                }
            }
            it.start = 0;
            set_len(p, seg_units, true);
            it.rec = 2 * blockIdx.x + 1;
        } else {
            pos += gridDim.x;
            load_fixed(p, sc);
        }
    }

    // automatic mode: the piece takes min(left, stop - pos) units of its segment
    __device__ __forceinline__ void set_len(const SplitParams& p, int left, bool at_start)
    {
        const int len = static_cast<int>(min(static_cast<long long>(left), stop - pos));
        it.end = min(it.start + (len << p.lg_tt), it.past + p.NQ);
        it.whole = at_start && len == seg_units;
        it.units = len;
    }

    __device__ __forceinline__ void load_fixed(const SplitParams& p, const Sched& sc)
    {
        ok = pos < stop;
        if (!ok)
            return;
        const int U = p.NRS * p.KV;
        const int item = static_cast<int>(pos);
        const int g = item / U;
        const int rem = item - g * U;
        const int b = last_le(sc.prefix, p.B, g);
        const int c = g - sc.prefix[b];
        const int total = sc.lens[b] + p.NQ;
        const int chunk = chunk_of(p, total);
        it.b = b;
        it.rsg = rem / p.KV;
        it.kh = rem - it.rsg * p.KV;
        it.past = sc.lens[b];
        it.start = c * chunk;
        it.end = min(it.start + chunk, total);
        it.whole = sc.prefix[b + 1] - sc.prefix[b] == 1;
        it.rec = ((b * p.partitions + c) * p.NRS + it.rsg) * p.KV + it.kh;
        it.units = 0;
    }
};

// Pieces of segment (b, rsg, kh) and the workspace record of piece c, as the
// partition kernel laid them out (see the schedule comment above).
struct SegPieces {
    int n;          // pieces of the segment
    int k0;         // automatic mode: CTA of the first piece
    int rec_first;  // automatic mode: record of the first piece
    int item0;      // fixed partitions: first key range of the sequence
};

__device__ __forceinline__ SegPieces seg_pieces(const SplitParams& p, const Sched& sc, int b, int rsg,
                                                int kh)
{
    SegPieces sp;
    if (p.partitions == 0) {
        const int C = static_cast<int>(sc.cost);
        const int G = active_ctas(gridDim.x, C, static_cast<long long>(p.B) * p.NRS * p.KV);
        const int units = (sc.lens[b] + p.NQ + p.TT - 1) >> p.lg_tt;
        const int gl = rsg * p.KV + kh;
        const SegSpan ss = seg_span(sc.prefix[b] + gl * units, units, b * p.NRS * p.KV + gl, p.vunits, C, G);
        sp.k0 = ss.k0;
        sp.n = ss.n;
        sp.rec_first = ss.rec_first;
        sp.item0 = 0;
    } else {
        sp.n = sc.prefix[b + 1] - sc.prefix[b];
        sp.item0 = sc.prefix[b];
        sp.k0 = 0;
        sp.rec_first = 0;
    }
    return sp;
}

__device__ __forceinline__ size_t seg_record(const SplitParams& p, const SegPieces& sp, int c, int rsg,
                                             int kh)
{
    if (p.partitions == 0)
        return c == 0 ? static_cast<size_t>(sp.rec_first) : static_cast<size_t>(2 * (sp.k0 + c));
    return (static_cast<size_t>(sp.item0 + c) * p.NRS + rsg) * p.KV + kh;
}

// One word of every 32 bytes of a kernel parameter (0 past its end): the
// loads of all three parameters are issued together at entry, so that their
// constant-cache lines arrive in one round trip instead of one by one at
// their first use on the issue path.
template <typename Tp>
__device__ __forceinline__ int param_word(const Tp& x)
{
    constexpr int kWords = static_cast<int>(sizeof(Tp) / 4);
    const int i = static_cast<int>(threadIdx.x) * 8;
    return i < kWords ? reinterpret_cast<const int*>(&x)[i] : 0;
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
//   [0, 256)     full barriers      [256, 512)  empty barriers
//   [512, 576)   broadcast scalars  [576, 608)  query-buffer barriers (full, free)
//   [640, 896)   a zeroed 256-byte row (tensor-core path)
//   [1024, 3072) table-entry slots of the two producer warps
//   [3072, 3584) split pieces awaiting their counts
//   lens[B] | prefix[B+1] | consumer scratch | ring of `stages` stages.
struct Smem {
    uint64_t* full;
    uint64_t* empty;
    uint64_t* q_full;  // [2]
    uint64_t* q_free;  // [2]
    int* info;
    volatile int* abort_flag;
    const void* zero16;
    int* lens;
    int* prefix;
    unsigned char* scratch;
    unsigned char* ring;
    int* entries;  // producer warps' table-entry slots [2][kTableSlots][kSlotInts]
    int4* split_list;  // [kSplitList] split pieces awaiting their counts (b, rsg, kh, flag)
};

__device__ __forceinline__ Smem carve(const SplitParams& p, unsigned char* raw)
{
    unsigned char* base = raw + ((1024u - (smem_u32(raw) & 1023u)) & 1023u);
    Smem sm;
    sm.full = reinterpret_cast<uint64_t*>(base);
    sm.empty = sm.full + kMaxStages;
    sm.info = reinterpret_cast<int*>(base + 512);
    sm.abort_flag = sm.info + 15;
    sm.q_full = reinterpret_cast<uint64_t*>(base + 576);
    sm.q_free = sm.q_full + 2;
    sm.zero16 = base + 640;
    sm.entries = reinterpret_cast<int*>(base + 1024);
    sm.split_list = reinterpret_cast<int4*>(base + 3072);
    sm.lens = reinterpret_cast<int*>(base + p.lens_off);
    sm.prefix = reinterpret_cast<int*>(base + p.prefix_off);
    sm.scratch = base + p.merge_off;
    sm.ring = base + p.stage_off;
    return sm;
}

// Thread 0: the ring and query-buffer barriers, the abort flag and the zero
// row.  Touches no global memory, so it runs before the grid-dependency wait
// (made visible to the other threads by setup_cta's first CTA barrier).
__device__ __forceinline__ void init_cta(const SplitParams& p, const Smem& sm)
{
    if (threadIdx.x == 0) {
        for (int s = 0; s < p.stages; ++s) {
            mbar_init(&sm.full[s], kProducerWarps);
            mbar_init(&sm.empty[s], p.empty_count);
        }
        for (int i = 0; i < 2; ++i) {
            mbar_init(&sm.q_full[i], 1);
            mbar_init(&sm.q_free[i], kConsumerWarps);
        }
        sm.info[15] = 0;
        for (int i = 0; i < 16; ++i)
            reinterpret_cast<uint4*>(const_cast<void*>(sm.zero16))[i] = make_uint4(0, 0, 0, 0);
        fence_mbar_init();
    }
}

// Block-table bytes prefetched into L2 at entry, at most: a table this small
// is fetched whole (all CTAs together, one 128-byte line per thread), so that
// the producers' first table reads, which wait on the schedule, hit in L2.
constexpr long long kTablePrefetchBytes = 512 * 1024;

// Entry of the partition kernels, before anything that reads inputs the
// previous kernel on the stream may still write: the tensor maps are fetched
// (producer warps), the block table is prefetched into L2 (coherent: a later
// write by the previous kernel still wins), the parameters are warmed, the
// barriers initialised; then the grid-dependency wait.  With p.early (the
// caller guarantees that the previous kernel writes no input) the wait is
// left to the consumer warps, before their first write of the output or the
// workspace: the schedule, the table entries and the first stages are then
// read while the previous kernel finishes.
__device__ __forceinline__ void kernel_entry(const SplitParams& p, const CUtensorMap& kmap,
                                             const CUtensorMap& vmap, const Smem& sm)
{
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (warp >= kConsumerWarps && lane == 0)
        tma_prefetch_desc(warp == kConsumerWarps ? &kmap : &vmap);
    const long long tbytes = static_cast<long long>(p.B) * p.maxb * 4;
    if (tbytes <= kTablePrefetchBytes) {
        const long long line = static_cast<long long>(threadIdx.x) * gridDim.x + blockIdx.x;
        if (line * 128 < tbytes)
            asm volatile("prefetch.global.L2 [%0];" ::"l"(reinterpret_cast<const char*>(p.table) + line * 128));
    }
    const int w0 = param_word(p), w1 = param_word(kmap), w2 = param_word(vmap);
    asm volatile("" ::"r"(w0), "r"(w1), "r"(w2));
    init_cta(p, sm);
    if (!p.early)
        grid_dependency_wait();
    grid_dependents_launch();
}

// All threads, after kernel_entry: clamped lengths, the schedule.
__device__ __forceinline__ Sched setup_cta(const SplitParams& p, const Smem& sm)
{
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    Sched sc;
    sc.lens = sm.lens;
    sc.prefix = sm.prefix;
    // Warp 0 alone: lengths, schedule and (automatic mode) this CTA's range,
    // with warp barriers in between and one CTA barrier at the end.
    if (warp == 0) {
        const int run = scan_lengths(p, sm.lens, sm.prefix, lane);
        __syncwarp();
        sc.total = p.partitions == 0 ? run : run * p.NRS * p.KV;
        sc.cost = sc.total + static_cast<long long>(p.vunits) * p.B * p.NRS * p.KV;
        if (lane == 0)
            sm.info[1] = sc.total;
        if (p.partitions == 0) {
            // G <= C: every CTA inside a segment then holds a unit.  The starts
            // of this CTA's range and of the next CTA's.
            const long long S = static_cast<long long>(p.B) * p.NRS * p.KV;
            const int G = active_ctas(gridDim.x, sc.cost, S);
            CostPos c0{0, 0, 0, 0}, c1{0, 0, 0, 0};
            int max_units = 0;  // the longest segment, in stages
            for (int b = lane; b < p.B; b += 32)
                max_units = max(max_units, (sm.lens[b] + p.NQ + p.TT - 1) >> p.lg_tt);
            max_units = __reduce_max_sync(kFull, max_units);
            if (p.counters && whole_segments(S, G, sc.total, max_units)) {
                // segment k for CTA k (the range of its units), none for the rest
                const int k = blockIdx.x, U = p.NRS * p.KV;
                c0 = c1 = CostPos{sc.total, p.B, 0, 0};
                if (k < S) {
                    const int b = k / U, seg = k - b * U;
                    const int nb = (sm.lens[b] + p.NQ + p.TT - 1) >> p.lg_tt;
                    c0 = CostPos{sm.prefix[b] + seg * nb, b, seg, 0};
                    c1.x = c0.x + nb;
                }
            } else if (static_cast<int>(blockIdx.x) < G) {
                c0 = cost_start(p, sc, blockIdx.x, G, lane);
                c1 = cost_start(p, sc, blockIdx.x + 1, G, lane);
            }
            if (lane == 0) {
                sm.info[2] = c0.x;
                sm.info[3] = c0.b;
                sm.info[4] = c0.seg;
                sm.info[5] = c0.uu;
                sm.info[6] = c1.x;
                sm.info[7] = c1.b;
                sm.info[8] = c1.seg;
                sm.info[9] = c1.uu;
            }
        }
    }
    __syncthreads();
    sc.total = sm.info[1];
    sc.cost = sc.total + static_cast<long long>(p.vunits) * p.B * p.NRS * p.KV;
    if (p.partitions == 0) {
        sc.pos0 = sm.info[2];
        sc.b0 = sm.info[3];
        sc.seg0 = sm.info[4];
        sc.uu0 = sm.info[5];
        sc.stop0 = sm.info[6];
    }
    return sc;
}

// Walks the tiles of this CTA's pieces in order.
struct TileIter {
    PieceIter pc;
    int j, ntiles;
    __device__ __forceinline__ void start(const SplitParams& p, const Sched& sc)
    {
        pc.first(p, sc);
        j = 0;
        ntiles = pc.ok ? (pc.it.end - pc.it.start + p.TT - 1) >> p.lg_tt : 0;
    }
    __device__ __forceinline__ bool valid() const { return pc.ok; }
    __device__ __forceinline__ void next(const SplitParams& p, const Sched& sc)
    {
        if (++j == ntiles) {
            pc.next(p, sc);
            j = 0;
            ntiles = pc.ok ? (pc.it.end - pc.it.start + p.TT - 1) >> p.lg_tt : 0;
        }
    }
};

constexpr int kTableAhead = 8;   // tiles whose table entries are in flight ahead of use
constexpr int kTableSlots = 16;  // entry slots (> kTableAhead)
constexpr int kSlotInts = 16;    // entries per slot (boxes per tile at most)

// Starts a non-blocking copy of the table entries of the tile at `t` into
// entry slot `slot` (lane i copies entry i), as one cp.async group.
__device__ __forceinline__ void fetch_entries(const SplitParams& p, const TileIter& t, int* slot,
                                              int lane)
{
    if (t.valid()) {
        const Item& it = t.pc.it;
        const int t0 = it.start + (t.j << p.lg_tt);
        const int cache_end = min(min(t0 + p.TT, it.end), it.past);
        const int nb = cache_end > t0 ? (cache_end - t0 + p.box_rows - 1) >> p.lg_box : 0;
        if (lane < nb) {
            const int32_t* src = p.table + static_cast<size_t>(it.b) * p.maxb +
                                 ((t0 + (lane << p.lg_box)) >> p.lg_block);
            asm volatile("cp.async.ca.shared.global [%0], [%1], 4;" ::"r"(smem_u32(slot + lane)),
                         "l"(src)
                         : "memory");
        }
    }
    asm volatile("cp.async.commit_group;" ::: "memory");
}

// A producer warp: for every tile of every item of this CTA, wait for a free
// stage and issue one TMA box per cache block (or per tile when a block spans
// several tiles).  Role 0 issues the K boxes, the query rows of each piece
// (tensor-core path) and the new rows; role 1 the V boxes.  The issue cost of
// a box is paid serially by the issuing warp, so two warps halve it.  Each
// role counts its bytes on the stage's full barrier (two arrivals).  Table
// entries are fetched kTableAhead tiles ahead with cp.async, so no dependent
// global load sits on the issue path.
template <typename T, int D, bool kSwizzled>
__device__ void produce(const SplitParams& p, const Sched& sc, const Smem& sm, const CUtensorMap* kmap,
                        const CUtensorMap* vmap, int role, int lane)
{
    const CUtensorMap* map = role == 0 ? kmap : vmap;  // fetched at kernel entry
    const int S = p.stages;
    const uint32_t box_bytes = static_cast<uint32_t>(p.box_rows * D * sizeof(T));
    const uint32_t new_bytes = static_cast<uint32_t>(p.NQ * D * sizeof(T));
    int* entries = sm.entries + role * (kTableSlots * kSlotInts);  // this role's slots

    TileIter cur, ahead;
    cur.start(p, sc);
    ahead = cur;
    // tile 0's entries first: its boxes go out before the rest of the
    // look-ahead window is fetched (tiles 1 .. kTableAhead, after its issue)
    fetch_entries(p, ahead, entries, lane);
    if (ahead.valid())
        ahead.next(p, sc);
    const int HB = p.box_rows;
    uint32_t gt = 0;  // tiles issued by this CTA
    int s = 0;        // ring slot of tile gt
    uint32_t ph = 0;  // completed passes over the ring
    int piece = -1;   // pieces begun by this CTA
    for (; cur.valid(); cur.next(p, sc), ++gt) {
        if (gt == 0) {
            asm volatile("cp.async.wait_group 0;" ::: "memory");
        } else {
            // one group per tile: tile gt's group is the oldest of kTableAhead + 1
            fetch_entries(p, ahead, entries + ((gt + kTableAhead) % kTableSlots) * kSlotInts, lane);
            if (ahead.valid())
                ahead.next(p, sc);
            asm volatile("cp.async.wait_group %0;" ::"n"(kTableAhead) : "memory");
        }
        if (ph > 0) {
            bool ok = !*sm.abort_flag && mbar_wait_bounded(&sm.empty[s], (ph - 1) & 1, p.wait_ns);
            ok = __all_sync(kFull, ok);
            if (!ok) {
                if (lane == 0)
                    flag_timeout(p, sm.abort_flag);
                break;
            }
        }
        const Item& it = cur.pc.it;
        if (kSwizzled && cur.j == 0) {
            ++piece;
            // the piece's query rows go to buffer piece & 1 once every
            // consumer warp has finished the tiles of the piece two back
            const int par = piece & 1;
            if (role == 0 && piece >= 2) {
                bool ok = !*sm.abort_flag &&
                          mbar_wait_bounded(&sm.q_free[par], ((piece >> 1) - 1) & 1, p.wait_ns);
                ok = __all_sync(kFull, ok);
                if (!ok) {
                    if (lane == 0)
                        flag_timeout(p, sm.abort_flag);
                    break;
                }
            }
            if (role == 0) {
                // one bulk copy per row (lane r: row r) into rows padded to
                // q_row_bytes(D); the expected bytes are set first
                const int rows = min(p.rows_per_cta, p.R - it.rsg * p.rows_per_cta);
                const uint32_t rb = static_cast<uint32_t>(D * sizeof(T));
                if (lane == 0)
                    mbar_arrive_expect_tx(&sm.q_full[par], rows * rb);
                __syncwarp();
                if (lane < rows) {
                    const size_t off =
                        ((static_cast<size_t>(it.b) * p.KV + it.kh) * p.R + it.rsg * p.rows_per_cta + lane) *
                        D;
                    unsigned char* dst =
                        sm.scratch + p.qbuf_off + (par * p.rows_per_cta + lane) * q_row_bytes(D);
                    bulk_load(dst, static_cast<const T*>(p.q) + off, rb, &sm.q_full[par]);
                }
            }
        }
        const int t0 = it.start + (cur.j << p.lg_tt);
        const int t1 = min(t0 + p.TT, it.end);
        const int cache_end = min(t1, it.past);
        const int nb = cache_end > t0 ? (cache_end - t0 + HB - 1) >> p.lg_box : 0;
        const bool has_new = role == 0 && t1 > it.past;
        const int* ent = entries + (gt % kTableSlots) * kSlotInts;
        if (role == 0 && lane < nb && p.checked) {
            const int phys = ent[lane];  // own cp.async
            if ((phys < 0 || phys >= p.num_blocks) && p.status)
                atomicOr(p.status, PA_STATUS_BAD_BLOCK);
        }
        unsigned char* st = sm.ring + static_cast<size_t>(s) * p.stage_bytes;
        // test switch (pa_opts.debug_withhold_stage): every CTA's V producer
        // leaves one stage out, so that the consumers' wait for it runs out
        const bool withheld = p.withhold > 0 && role == 1 && gt + 1 == static_cast<uint32_t>(p.withhold);
        if (lane == 0 && !withheld)
            mbar_arrive_expect_tx(&sm.full[s], nb * box_bytes + (has_new ? 2u * new_bytes : 0u));
        __syncwarp();  // entries written by other lanes' cp.async are visible
        // One warp instruction issues every box of the stage (lane i: box i).
        if (lane < nb && !withheld) {
            const int phys = ent[lane];
            // Out-of-pool coordinates read as zeros: the copy never faults.
            const int z = (phys << p.lg_block) + ((t0 + (lane << p.lg_box)) & (p.BLOCK - 1));
            unsigned char* dst = st + (role == 0 ? 0 : p.v_off) + static_cast<size_t>(lane) * HB * D * sizeof(T);
            if constexpr (kSwizzled) {
                // box [HB rows][D/64 halves][64 columns], 128-byte swizzle
                tma_load_4d(dst, map, 0, 0, it.kh, z, &sm.full[s]);
            } else {
                tma_load_3d(dst, map, 0, it.kh, z, &sm.full[s]);
            }
        }
        if (has_new && lane == 0) {
            const size_t off = (static_cast<size_t>(it.b) * p.KV + it.kh) * p.NQ * D;
            bulk_load(st + p.knew_off, static_cast<const T*>(p.k_new) + off, new_bytes, &sm.full[s]);
            bulk_load(st + p.vnew_off, static_cast<const T*>(p.v_new) + off, new_bytes, &sm.full[s]);
        }
        if (++s == S) {
            s = 0;
            ++ph;
        }
        if (gt == 0)
            for (int k = 1; k <= kTableAhead; ++k) {
                fetch_entries(p, ahead, entries + (k % kTableSlots) * kSlotInts, lane);
                if (ahead.valid())
                    ahead.next(p, sc);
            }
    }
    asm volatile("cp.async.wait_all;" ::: "memory");
    // Leave no copy in flight if the pipeline was abandoned (a stage whose
    // other role never arrived gives up after the wait limit).
    __syncwarp();
    if (*sm.abort_flag && lane == 0) {
        const uint32_t first = gt > static_cast<uint32_t>(S) ? gt - S : 0u;
        for (uint32_t g = first; g < gt; ++g)
            mbar_wait_bounded(&sm.full[g % S], (g / S) & 1, p.wait_ns);
        if (role == 0)
            for (int pc = max(0, piece - 1); pc <= piece; ++pc)
                mbar_wait_bounded(&sm.q_full[pc & 1], (pc >> 1) & 1, p.wait_ns);
    }
}

// ---------------------------------------------------------- in-kernel merge
// Counter increment with acquire-release semantics at GPU scope: after a CTA
// barrier, the release publishes every record store of the CTA's threads
// (cumulativity through the barrier); the acquire makes the records of the
// CTAs that counted before visible to this CTA after its next barrier.
__device__ __forceinline__ int count_piece(int* counter)
{
    int old;
    asm volatile("atom.add.acq_rel.gpu.s32 %0, [%1], 1;" : "=r"(old) : "l"(counter) : "memory");
    return old;
}

// Merges every partial record of segment (it.b, it.rsg, it.kh) into the
// output: M = max m, L = sum l 2^(m - M), O = sum o 2^(m - M),
// out = L == 0 ? O : O / L.  Threads t0 .. t0 + kT - 1 of the consumer warps.
// Segments of at most 128 items (4 columns of one row) are merged in one pass
// by one thread per item; larger ones in two (the (max, sum) pairs first, into
// `tot` (rows_per_cta pairs) and `fac` (fac_cap floats) of shared scratch,
// then the accumulators).  Records written by other CTAs are read through L2
// (ld.global.cg).
template <int D, typename TO>
__device__ void merge_segment(const SplitParams& p, const Sched& sc, const int4 seg, float2* tot,
                              float* fac, int fac_cap, int t0, int kT, int bar_id)
{
    const int tid = threadIdx.x - t0, warp = tid >> 5, lane = tid & 31;
    const int nwarps = kT >> 5;
    struct {
        int b, rsg, kh;
    } it{seg.x, seg.y, seg.z};
    const int R_cta = min(p.rows_per_cta, p.R - it.rsg * p.rows_per_cta);
    const SegPieces sp = seg_pieces(p, sc, it.b, it.rsg, it.kh);
    const int n = sp.n;
    const bool fac_smem = n * R_cta <= fac_cap;
    // O is computed in items of 4 columns of one row (at most 4 per thread);
    // TPI adjacent lanes split the records of an item when the items are
    // few.  TPI depends on the item count only, so the sums are formed in the
    // same order whether a whole or a half CTA merges the segment.
    constexpr int D4 = D / 4;
    constexpr int LG4 = D4 == 16 ? 4 : 5;
    const int NI = R_cta * D4;
    const size_t out_row0 = (static_cast<size_t>(it.b) * p.KV + it.kh) * p.R + it.rsg * p.rows_per_cta;
    if (NI <= kConsumerWarps * 16) {
        // At most one item per thread of a half CTA: each thread merges every
        // record of its item online, eight records' (max, sum) and accumulator
        // loads in flight together -- one L2 round trip for up to eight
        // records, no shared memory and no barrier.  The order of the sums
        // depends on the record count only.
        if (tid < NI) {
            const int rl = tid >> LG4, d4 = tid & (D4 - 1);
            float M = -FLT_MAX, L = 0.f;
            float4 O = make_float4(0.f, 0.f, 0.f, 0.f);
            for (int c0 = 0; c0 < n; c0 += 8) {
                float2 ml[8];
                float4 v[8];
#pragma unroll
                for (int u = 0; u < 8; ++u) {
                    if (c0 + u < n) {
                        const size_t wrow = seg_record(p, sp, c0 + u, it.rsg, it.kh) * p.row_stride + rl;
                        ml[u] = __ldcg(&p.ws_ml[wrow]);
                        v[u] = __ldcg(reinterpret_cast<const float4*>(p.ws_o + wrow * D) + d4);
                    } else {
                        ml[u] = make_float2(-FLT_MAX, 0.f);
                        v[u] = make_float4(0.f, 0.f, 0.f, 0.f);
                    }
                }
                float Mb = M;
#pragma unroll
                for (int u = 0; u < 8; ++u)
                    Mb = fmaxf(Mb, ml[u].x);
                const float fs = fast_exp2(M - Mb);  // rescale of the records before this batch
                L *= fs;
                O.x *= fs;
                O.y *= fs;
                O.z *= fs;
                O.w *= fs;
#pragma unroll
                for (int u = 0; u < 8; ++u) {
                    const float f = fast_exp2(ml[u].x - Mb);
                    L = fmaf(ml[u].y, f, L);
                    O.x = fmaf(f, v[u].x, O.x);
                    O.y = fmaf(f, v[u].y, O.y);
                    O.z = fmaf(f, v[u].z, O.z);
                    O.w = fmaf(f, v[u].w, O.w);
                }
                M = Mb;
            }
            const float inv = L == 0.f ? 1.f : 1.f / L;
            TO* dst = static_cast<TO*>(p.out) + (out_row0 + rl) * D + 4 * d4;
            dst[0] = from_float<TO>(O.x * inv);
            dst[1] = from_float<TO>(O.y * inv);
            dst[2] = from_float<TO>(O.z * inv);
            dst[3] = from_float<TO>(O.w * inv);
        }
        return;
    }
    int TPI = (kConsumerWarps * 32) / NI;
    TPI = TPI >= 8 ? 8 : TPI >= 4 ? 4 : TPI >= 2 ? 2 : 1;
    const int per_pass = kT / TPI;
    const int sub = tid % TPI, i0 = tid / TPI;
    float4 O[4];
    int rl_of[4];
    bool act[4];
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        O[j] = make_float4(0.f, 0.f, 0.f, 0.f);
        const int item = i0 + j * per_pass;
        act[j] = item < NI;
        rl_of[j] = act[j] ? item >> LG4 : 0;
    }
    // (M, L) of each row: warp w takes rows w, w + nwarps, ...; lanes split
    // the records.  With at most 32 records, four rows' loads are in flight.
    if (n <= 32) {
        for (int rl0 = warp; rl0 < R_cta; rl0 += 4 * nwarps) {
            float2 ml[4];
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const int rl = rl0 + i * nwarps;
                ml[i] = rl < R_cta && lane < n
                            ? __ldcg(&p.ws_ml[seg_record(p, sp, lane, it.rsg, it.kh) * p.row_stride + rl])
                            : make_float2(-FLT_MAX, 0.f);
            }
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const int rl = rl0 + i * nwarps;
                float M = ml[i].x;
#pragma unroll
                for (int o = 16; o > 0; o >>= 1)
                    M = fmaxf(M, __shfl_xor_sync(kFull, M, o));
                const float f = lane < n ? fast_exp2(ml[i].x - M) : 0.f;
                float L = ml[i].y * f;
#pragma unroll
                for (int o = 16; o > 0; o >>= 1)
                    L += __shfl_xor_sync(kFull, L, o);
                if (rl < R_cta) {
                    if (fac_smem && lane < n)
                        fac[lane * R_cta + rl] = f;
                    if (lane == 0)
                        tot[rl] = make_float2(M, L);
                }
            }
        }
    } else {
        for (int rl = warp; rl < R_cta; rl += nwarps) {
            float M = -FLT_MAX;
            for (int c = lane; c < n; c += 32)
                M = fmaxf(M, __ldcg(&p.ws_ml[seg_record(p, sp, c, it.rsg, it.kh) * p.row_stride + rl]).x);
#pragma unroll
            for (int o = 16; o > 0; o >>= 1)
                M = fmaxf(M, __shfl_xor_sync(kFull, M, o));
            float L = 0.f;
            for (int c = lane; c < n; c += 32) {
                const float2 ml = __ldcg(&p.ws_ml[seg_record(p, sp, c, it.rsg, it.kh) * p.row_stride + rl]);
                const float f = fast_exp2(ml.x - M);
                L = fmaf(ml.y, f, L);
                if (fac_smem)
                    fac[c * R_cta + rl] = f;
            }
#pragma unroll
            for (int o = 16; o > 0; o >>= 1)
                L += __shfl_xor_sync(kFull, L, o);
            if (lane == 0)
                tot[rl] = make_float2(M, L);
        }
    }
    asm volatile("bar.sync %0, %1;" ::"r"(bar_id), "r"(kT) : "memory");
    auto fma4 = [](float4& a, float f, const float4& v) {
        a.x = fmaf(f, v.x, a.x);
        a.y = fmaf(f, v.y, a.y);
        a.z = fmaf(f, v.z, a.z);
        a.w = fmaf(f, v.w, a.w);
    };
    {
        auto add_record = [&](int c, float4* v, float* f) {
            const size_t rec = seg_record(p, sp, c, it.rsg, it.kh);
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                if (!act[j])
                    continue;
                const int item = i0 + j * per_pass;
                const size_t wrow = rec * p.row_stride + rl_of[j];
                v[j] = __ldcg(reinterpret_cast<const float4*>(p.ws_o + wrow * D) + (item & (D4 - 1)));
                f[j] = fac_smem ? fac[c * R_cta + rl_of[j]]
                                : fast_exp2(__ldcg(&p.ws_ml[wrow]).x - tot[rl_of[j]].x);
            }
        };
        int c = sub;
        if (NI <= per_pass) {
            // one item per thread: eight records in flight
            const int rl = rl_of[0];
            const int d4 = i0 & (D4 - 1);
            for (; c + 7 * TPI < n; c += 8 * TPI) {
                float4 v[8];
                float f[8];
#pragma unroll
                for (int u = 0; u < 8; ++u) {
                    const size_t wrow = seg_record(p, sp, c + u * TPI, it.rsg, it.kh) * p.row_stride + rl;
                    v[u] = act[0] ? __ldcg(reinterpret_cast<const float4*>(p.ws_o + wrow * D) + d4)
                                  : make_float4(0.f, 0.f, 0.f, 0.f);
                    f[u] = fac_smem ? fac[(c + u * TPI) * R_cta + rl]
                                    : fast_exp2(__ldcg(&p.ws_ml[wrow]).x - tot[rl].x);
                }
#pragma unroll
                for (int u = 0; u < 8; ++u)
                    fma4(O[0], f[u], v[u]);
            }
        }
        // items of up to four rows per thread: two records in flight per item
        for (; c + TPI < n; c += 2 * TPI) {
            float4 va[4], vb[4];
            float fa[4], fb[4];
            add_record(c, va, fa);
            add_record(c + TPI, vb, fb);
#pragma unroll
            for (int j = 0; j < 4; ++j)
                if (act[j]) {
                    fma4(O[j], fa[j], va[j]);
                    fma4(O[j], fb[j], vb[j]);
                }
        }
        if (c < n) {
            float4 va[4];
            float fa[4];
            add_record(c, va, fa);
#pragma unroll
            for (int j = 0; j < 4; ++j)
                if (act[j])
                    fma4(O[j], fa[j], va[j]);
        }
    }
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        for (int o = 1; o < TPI; o <<= 1) {
            O[j].x += __shfl_xor_sync(kFull, O[j].x, o);
            O[j].y += __shfl_xor_sync(kFull, O[j].y, o);
            O[j].z += __shfl_xor_sync(kFull, O[j].z, o);
            O[j].w += __shfl_xor_sync(kFull, O[j].w, o);
        }
        if (act[j] && sub == 0) {
            const float2 ml = tot[rl_of[j]];
            const float inv = ml.y == 0.f ? 1.f : 1.f / ml.y;
            const int item = i0 + j * per_pass;
            TO* dst = static_cast<TO*>(p.out) + (out_row0 + rl_of[j]) * D + 4 * (item & (D4 - 1));
            dst[0] = from_float<TO>(O[j].x * inv);
            dst[1] = from_float<TO>(O[j].y * inv);
            dst[2] = from_float<TO>(O[j].z * inv);
            dst[3] = from_float<TO>(O[j].w * inv);
        }
    }
}

constexpr int kSplitList = 32;  // list capacity (the automatic schedule needs two)

// Called by all consumer threads at the end of the CTA's stream, once the
// partial records of the `n` split pieces in `list` ((b, rsg, kh, -) each) are
// written (automatic schedule only: a CTA's first and last pieces).  Each
// piece is counted finished on its segment's counter (one lane each, the
// atomics in flight together); the CTA that finishes the last piece of a
// segment merges the segment's records and resets its counter for the next
// call.  Counting at the end keeps merges out of the CTA's stream.
template <int D, typename TO>
__device__ void flush_split_pieces(const SplitParams& p, const Sched& sc, int4* list, int n, float2* tot,
                                   int tot_cap, float* fac, int fac_cap)
{
    const int tid = threadIdx.x;
    consumer_bar_sync();  // every thread's record stores (and the list) precede the counts
    if (tid < n) {
        int4 e = list[tid];
        const int seg = (e.x * p.NRS + e.y) * p.KV + e.z;
        const SegPieces sp = seg_pieces(p, sc, e.x, e.y, e.z);
        const bool last = count_piece(&p.counters[seg]) == sp.n - 1;
        if (last)
            p.counters[seg] = 0;  // every piece has arrived: ready for the next call
        e.w = last;
        list[tid] = e;
    }
    consumer_bar_sync();
    // Segments to merge go two at a time, one per half of the consumer warps
    // (named barriers 2 and 3), when each fits four items per thread of a half.
    constexpr int kHalf = kConsumerWarps * 16;
    auto fits_half = [&](int4 e) {
        const int R_cta = min(p.rows_per_cta, p.R - e.y * p.rows_per_cta);
        return R_cta * (D / 4) <= 4 * kHalf && 2 * p.rows_per_cta <= tot_cap;
    };
    int i = 0;
    while (true) {
        while (i < n && !list[i].w)
            ++i;
        if (i == n)
            break;
        int j = i + 1;
        while (j < n && !list[j].w)
            ++j;
        const bool pair = j < n && fits_half(list[i]) && fits_half(list[j]);
        const bool upper = pair && tid >= kHalf;
        merge_segment<D, TO>(p, sc, list[upper ? j : i], tot + (upper ? p.rows_per_cta : 0),
                             fac + (upper ? fac_cap / 2 : 0), pair ? fac_cap / 2 : fac_cap,
                             upper ? kHalf : 0, pair ? kHalf : 2 * kHalf, pair ? (upper ? 3 : 2) : 1);
        i = pair ? j + 1 : i + 1;
        consumer_bar_sync();  // `tot` and `fac` are free again
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
    float2* merge_tot = reinterpret_cast<float2*>(mb_l + kConsumerWarps * RG);  // [rows per pass]

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int S = p.stages;
    const int TT = p.TT;

    // inputs may be produced by the previous kernel on the stream
    kernel_entry(p, kmap, vmap, sm);
    const Sched sc = setup_cta(p, sm);

    if (warp >= kConsumerWarps) {
        produce<T, D, false>(p, sc, sm, &kmap, &vmap, warp - kConsumerWarps, lane);
        return;
    }
    // consumers: with p.early (the inputs read before the previous kernel
    // completed), the grid-dependency wait comes at the first piece end,
    // before any write of the output or the workspace
    bool dep_ok = !p.early;

    using Math = SimtMath<T, D, RG>;
    uint32_t gt = 0;
    int nsplit = 0;  // split pieces listed since the last flush (uniform)
    const int tid = threadIdx.x;  // 0 .. kConsumerWarps*32-1
    PieceIter pi;
    for (pi.first(p, sc); pi.ok; pi.next(p, sc)) {
        const Item& it = pi.it;
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
                        mbar_wait_bounded(&sm.full[s], (gt / S) & 1, p.wait_ns);
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
        if (!dep_ok) {
            grid_dependency_wait();
            dep_ok = true;
        }
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
            if (it.whole) {
                const float val = L == 0.f ? O : O / L;
                static_cast<TO*>(p.out)[(out_row0 + rl) * D + d] = from_float<TO>(val);
            } else {
                const size_t wrow = static_cast<size_t>(it.rec) * p.row_stride + rl;
                p.ws_o[wrow * D + d] = O;
                if (d == 0)
                    p.ws_ml[wrow] = make_float2(M, L);
            }
        }
        // automatic schedule: the CTA's first and last pieces at most
        if (!it.whole && p.counters && nsplit < kSplitList) {
            if (tid == 0)
                sm.split_list[nsplit] = make_int4(it.b, it.rsg, it.kh, 0);
            ++nsplit;
        }
    }
    // uniform over the consumer warps (a late abort flag must not split them)
    if (nsplit > 0 && !consumer_bar_or(*sm.abort_flag != 0))
        flush_split_pieces<D, TO>(p, sc, sm.split_list, nsplit, merge_tot, p.rows_per_cta, mb_o,
                                  kConsumerWarps * RG * D);
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

// Stage of the tensor-core kernel: K and V tiles of kMmaTokens (16) tokens
// stored [16 tokens][D/64 halves][64 columns]: 128-byte lines, line
// L = token * (D/64) + half, with the TMA 128-byte swizzle (16-byte chunk c of
// line L sits at chunk c ^ (L % 8)); the new rows unswizzled [NQ][D]; a
// 256-byte zero row stands in for tokens past the tile.
struct RowAddr {
    uint32_t base;  // address of the row's first 128-byte line
    uint32_t swz;   // XOR of the first line (the second line's is swz ^ hx)
    uint32_t hx;    // 1 for swizzled rows of two lines, else 0
    __device__ __forceinline__ uint32_t at(int chunk) const
    {
        const uint32_t h = static_cast<uint32_t>(chunk) >> 3;
        return base + h * 128 + ((static_cast<uint32_t>(chunk & 7) ^ swz ^ (h * hx)) << 4);
    }
};

template <int D>
__device__ __forceinline__ RowAddr row_addr(uint32_t tile, uint32_t fresh, uint32_t zero, int tok,
                                            int n_tile, int t0, int past)
{
    constexpr int NH = D / 64;
    RowAddr r;
    const int ta = t0 + tok;
    if (tok >= n_tile) {
        r.base = zero;
        r.swz = 0;
        r.hx = 0;
    } else if (ta < past) {
        r.base = tile + tok * (D * 2);
        r.swz = (tok * NH) & 7;
        r.hx = NH - 1;
    } else {
        r.base = fresh + (ta - past) * (D * 2);
        r.swz = 0;
        r.hx = 0;
    }
    return r;
}

// ---- piece-end merge of the consumer warps (both tensor-core kernels).
// Each warp leaves its running (max, sum) per row in a [warp][16] table and
// its unscaled accumulators in obuf, [warp][RU rows][DRr columns] per round of
// DRr = 2^lg columns; columns are XOR-swizzled by row in groups of 8 floats so
// that the rows a warp stores at once fall in different banks.
__device__ __forceinline__ int obuf_swz(int row) { return ((row >> 1) & 3) << 3; }

// log2 of the round width: the widest power of two <= D whose round of RU
// rows from every consumer warp fits `cap` floats.
__device__ __forceinline__ int obuf_lg(int D, int RU, int cap = kObufFloats)
{
    int lg = 31 - __clz(D);
    while (lg > 3 && kConsumerWarps * RU * (1 << lg) > cap)
        --lg;
    return lg;
}

// Sums round r of the stashed states of the TS = kConsumerWarps / MT warps of
// every row: M = max m_t, L = sum l_t 2^(m_t - M), acc = sum o_t 2^(m_t - M);
// writes out = acc / L for a whole segment, else the partial record
// (acc, (M, L)).  Warp w holds rows of row group w % MT.  All consumer threads.
template <int D, int MT, typename TO>
__device__ __forceinline__ void sum_warps(const SplitParams& p, const Item& it, int R_cta, int RU, int lg,
                                          int r, const float2* ml_buf, const float* obuf)
{
    constexpr int TS = kConsumerWarps / MT;
    constexpr int NT = kConsumerWarps * 32;
    const int DRr = 1 << lg;
    const size_t out_row0 = (static_cast<size_t>(it.b) * p.KV + it.kh) * p.R +
                            static_cast<size_t>(it.rsg) * p.rows_per_cta;
    auto put = [&](int rl, int d, float M, float L, float acc) {
        if (it.whole) {
            const float val = L == 0.f ? acc : acc / L;
            static_cast<TO*>(p.out)[(out_row0 + rl) * D + d] = from_float<TO>(val);
        } else {
            const size_t wrow = static_cast<size_t>(it.rec) * p.row_stride + rl;
            p.ws_o[wrow * D + d] = acc;
            if (d == 0)
                p.ws_ml[wrow] = make_float2(M, L);
        }
    };
    if constexpr (MT >= 2) {
        // 32 rows: tpr threads per row (a power of two), each computes the
        // row's factors 2^(m_t - M) once and sums its columns of the round
        // with them (measured faster on 32 rows, slower on 4)
        int tpr = 1;
        while (tpr * 2 * R_cta <= NT && tpr * 2 <= DRr)
            tpr *= 2;
        for (int rl = static_cast<int>(threadIdx.x) / tpr; rl < R_cta; rl += NT / tpr) {
            const int grp = rl >> 4, rr = rl & 15;
            float M = -FLT_MAX;
#pragma unroll
            for (int t = 0; t < TS; ++t)
                M = fmaxf(M, ml_buf[(t * MT + grp) * 16 + rr].x);
            float f[TS];
            float L = 0.f;
#pragma unroll
            for (int t = 0; t < TS; ++t) {
                const float2 ml = ml_buf[(t * MT + grp) * 16 + rr];
                f[t] = fast_exp2(ml.x - M);
                L = fmaf(ml.y, f[t], L);
            }
            for (int dd = static_cast<int>(threadIdx.x) & (tpr - 1); dd < DRr; dd += tpr) {
                const int col = (dd ^ obuf_swz(rr)) & (DRr - 1);
                float acc = 0.f;
#pragma unroll
                for (int t = 0; t < TS; ++t)
                    acc = fmaf(f[t], obuf[(((t * MT + grp) * RU + rr) << lg) + col], acc);
                put(rl, (r << lg) + dd, M, L, acc);
            }
        }
    } else {
        // few rows: one output per thread and pass, factors per output
        for (int idx = threadIdx.x; idx < (R_cta << lg); idx += NT) {
            const int rl = idx >> lg, dd = idx & (DRr - 1);
            const int grp = rl >> 4, rr = rl & 15;
            float M = -FLT_MAX;
#pragma unroll
            for (int t = 0; t < TS; ++t)
                M = fmaxf(M, ml_buf[(t * MT + grp) * 16 + rr].x);
            float L = 0.f, acc = 0.f;
            const int col = (dd ^ obuf_swz(rr)) & (DRr - 1);
#pragma unroll
            for (int t = 0; t < TS; ++t) {
                const float2 ml = ml_buf[(t * MT + grp) * 16 + rr];
                const float f = fast_exp2(ml.x - M);
                L = fmaf(ml.y, f, L);
                acc = fmaf(f, obuf[(((t * MT + grp) * RU + rr) << lg) + col], acc);
            }
            put(rl, (r << lg) + dd, M, L, acc);
        }
    }
}

// T: __half or __nv_bfloat16; D: head size; MT: 16-row groups per CTA pass;
// TO: output element type.  One CTA per SM (persistent).
//
// The ring holds stages of TT tokens (up to 64 KB of K and V).  Stage g of the
// CTA belongs to warp set g % nsets: each warp of the set takes one 16-token
// group and one 16-row group and computes S = Q K^T with m16n8k16 MMAs
// (float32 accumulators), scales and masks S, updates its running row maxima
// (rescaling its accumulators only when a maximum grew), and accumulates
// O += P V with P kept in registers as a 16-bit high part plus a 16-bit
// remainder (P V keeps about 22 bits of P).  Warps never wait for one another
// inside a piece; at the end of a piece their (max, sum, O) states are merged
// through shared memory, in the piece's last stage, whose slot the warps keep
// until the merge is done.  The query rows of each piece arrive in one of two
// shared buffers filled by the producer.
template <typename T, int D, int MT, typename TO>
__global__ void __launch_bounds__(kThreads, 1)
    pa_mma_kernel(const __grid_constant__ SplitParams p, const __grid_constant__ CUtensorMap kmap,
                  const __grid_constant__ CUtensorMap vmap)
{
    constexpr bool kBf = std::is_same<T, __nv_bfloat16>::value;
    constexpr int KS = D / 16;  // k-steps of Q K^T
    constexpr int NT = D / 8;   // 8-column tiles of O
    constexpr int ROWS = 16 * MT;
    constexpr int TG = mma_token_groups(D, MT);  // 16-token groups per warp and stage
    constexpr int TPW = kMmaTokens * TG;     // tokens per warp and stage

    extern __shared__ __align__(1024) unsigned char smem_raw[];
    const Smem sm = carve(p, smem_raw);
    float2* ml_buf = reinterpret_cast<float2*>(sm.scratch);         // [warps][16] (max, sum)
    float2* tot = reinterpret_cast<float2*>(sm.scratch + 1024);     // [ROWS] merged (max, sum)
    float* obuf = reinterpret_cast<float*>(sm.scratch + 2048);      // kObufFloats: split-merge factors

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int S = p.stages;

    // inputs may be produced by the previous kernel on the stream
    kernel_entry(p, kmap, vmap, sm);
    const Sched sc = setup_cta(p, sm);

    if (warp >= kConsumerWarps) {
        produce<T, D, true>(p, sc, sm, &kmap, &vmap, warp - kConsumerWarps, lane);
        return;
    }
    // consumers: with p.early (the inputs read before the previous kernel
    // completed), the grid-dependency wait comes at the first piece end,
    // before any write of the output or the workspace
    bool dep_ok = !p.early;

    const int g = lane >> 2, qd = lane & 3;
    const int rg = warp % MT;
    // A stage of TT tokens is consumed by a set of WS = (TT/TPW)*MT warps (one
    // per TPW tokens and row group); the nsets sets take stages in turn.
    const int TT = p.TT;
    const int WS = (TT / TPW) * MT;
    const int nsets = kConsumerWarps / WS;
    const int my_set = warp / WS;
    const int tb = ((warp % WS) / MT) * TPW;  // this warp's first token in a stage
    const uint32_t zero = smem_u32(sm.zero16);
    const uint32_t qbuf = smem_u32(sm.scratch + p.qbuf_off);
    uint32_t gt = 0;
    int piece = 0;
    int nsplit = 0;  // split pieces listed since the last flush (uniform)
    bool alive = true;

    PieceIter pi;
    for (pi.first(p, sc); pi.ok; pi.next(p, sc), ++piece) {
        const Item& it = pi.it;
        const int ntiles = (it.end - it.start + TT - 1) / TT;
        const int R_cta = min(ROWS, p.R - it.rsg * ROWS);
        const int row0 = rg * 16;  // first row of this warp's group within the CTA pass

        // causal / length limits of this thread's two rows (0 for padding rows)
        int lim[2];
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            const int rl = row0 + g + 8 * h;
            const int rho = it.rsg * ROWS + rl;
            lim[h] = rl < R_cta ? it.past + (p.causal ? (rho % p.NQ) + 1 : p.NQ) : 0;
        }
        const int lim_min = __reduce_min_sync(kFull, min(lim[0] > 0 ? lim[0] : INT_MAX,
                                                         lim[1] > 0 ? lim[1] : INT_MAX));

        // Q fragments (row-major A of m16n8k16) from this piece's query buffer
        uint32_t qa[KS][4];
        {
            const int par = piece & 1;
            if (alive) {
                alive = !*sm.abort_flag &&
                        mbar_wait_bounded(&sm.q_full[par], (piece >> 1) & 1, p.wait_ns);
                alive = __all_sync(kFull, alive);
                if (!alive && lane == 0)
                    flag_timeout(p, sm.abort_flag);
            }
            const int qrow = row0 + (lane & 7) + (((lane >> 3) & 1) << 3);
            const uint32_t qaddr = qbuf + (par * ROWS + qrow) * q_row_bytes(D) + ((lane >> 4) << 4);
            const bool r0ok = row0 + g < R_cta, r1ok = row0 + g + 8 < R_cta;
#pragma unroll
            for (int ks = 0; ks < KS; ++ks) {
                ldsm_x4(qaddr + ks * 32, qa[ks][0], qa[ks][1], qa[ks][2], qa[ks][3]);
                if (!r0ok) {  // rows past the pass hold stale shared memory
                    qa[ks][0] = 0u;
                    qa[ks][2] = 0u;
                }
                if (!r1ok) {
                    qa[ks][1] = 0u;
                    qa[ks][3] = 0u;
                }
            }
        }

        float m[2] = {-FLT_MAX, -FLT_MAX}, lp[2] = {0.f, 0.f};
        float o[NT][4];
#pragma unroll
        for (int i = 0; i < NT; ++i)
#pragma unroll
            for (int e = 0; e < 4; ++e)
                o[i][e] = 0.f;

        // The warps of the piece's last stage keep its slot until the piece-end
        // merge is done: its 64 KB serve as the merge buffer (one round).
        int s_hold = -1;
        for (int j = 0; j < ntiles; ++j, ++gt) {
            if (static_cast<int>(gt % nsets) != my_set)
                continue;  // another warp set's stage
            const int s = gt % S;
            if (alive) {
                alive = !*sm.abort_flag &&
                        mbar_wait_bounded(&sm.full[s], (gt / S) & 1, p.wait_ns);
                alive = __all_sync(kFull, alive);
                if (!alive && lane == 0)
                    flag_timeout(p, sm.abort_flag);
            }
            if (!alive)
                continue;
            const uint32_t st = smem_u32(sm.ring) + s * p.stage_bytes;
            const uint32_t k_tile = st, v_tile = st + p.v_off;
            const uint32_t k_new = st + p.knew_off, v_new = st + p.vnew_off;
            const int t0 = it.start + j * TT;
            const int n_tile = min(TT, it.end - t0);
            if (tb >= n_tile) {  // the stage ends before this warp's tokens
                __syncwarp();
                if (j + 1 < ntiles) {
                    if (lane == 0)
                        mbar_arrive(&sm.empty[s]);
                } else {
                    s_hold = s;
                }
                continue;
            }
            // a group whose every token is visible to every row of the warp
            bool full_tile[TG];
#pragma unroll
            for (int u = 0; u < TG; ++u) {
                const int tu = tb + u * kMmaTokens;
                full_tile[u] = tu + kMmaTokens <= n_tile && t0 + tu + kMmaTokens <= lim_min;
            }

            // ---- S = Q K^T (per group, two accumulator sets per 8-token tile:
            // shorter chains; the groups' MMAs interleave)
            float sa[TG][2][2][4];
#pragma unroll
            for (int u = 0; u < TG; ++u)
#pragma unroll
                for (int a = 0; a < 2; ++a)
#pragma unroll
                    for (int nt = 0; nt < 2; ++nt)
#pragma unroll
                        for (int e = 0; e < 4; ++e)
                            sa[u][a][nt][e] = 0.f;
            RowAddr kr[TG];
#pragma unroll
            for (int u = 0; u < TG; ++u)
                kr[u] = row_addr<D>(k_tile, k_new, zero,
                                    tb + u * kMmaTokens + (lane & 7) + ((lane >> 4) << 3), n_tile,
                                    t0, it.past);
#pragma unroll
            for (int ks = 0; ks < KS; ++ks)
#pragma unroll
                for (int u = 0; u < TG; ++u) {
                    uint32_t b00, b01, b10, b11;
                    ldsm_x4(kr[u].at(2 * ks + ((lane >> 3) & 1)), b00, b01, b10, b11);
                    mma_16816<kBf>(sa[u][ks & 1][0], qa[ks], b00, b01);
                    mma_16816<kBf>(sa[u][ks & 1][1], qa[ks], b10, b11);
                }
            // scale, mask, row maxima of the stage
            float sv[TG][2][4];
            float mx[2] = {-INFINITY, -INFINITY};
#pragma unroll
            for (int u = 0; u < TG; ++u)
#pragma unroll
                for (int nt = 0; nt < 2; ++nt)
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        const int h = e >> 1;
                        const int tk = tb + u * kMmaTokens + nt * 8 + 2 * qd + (e & 1);
                        const float v = (sa[u][0][nt][e] + sa[u][1][nt][e]) * p.qscale;
                        const bool valid = full_tile[u] || (tk < n_tile && t0 + tk < lim[h]);
                        sv[u][nt][e] = valid ? v : -INFINITY;
                        mx[h] = fmaxf(mx[h], sv[u][nt][e]);
                    }
            bool grow = false;
#pragma unroll
            for (int h = 0; h < 2; ++h) {
                mx[h] = fmaxf(mx[h], __shfl_xor_sync(kFull, mx[h], 1));
                mx[h] = fmaxf(mx[h], __shfl_xor_sync(kFull, mx[h], 2));
                grow |= mx[h] > m[h];
            }
            if (__any_sync(kFull, grow)) {  // rescale only when a row maximum grew
                float f[2];
#pragma unroll
                for (int h = 0; h < 2; ++h) {
                    const float mn = fmaxf(m[h], mx[h]);
                    f[h] = fast_exp2(m[h] - mn);
                    m[h] = mn;
                    lp[h] *= f[h];
                }
#pragma unroll
                for (int i = 0; i < NT; ++i)
#pragma unroll
                    for (int e = 0; e < 4; ++e)
                        o[i][e] *= f[e >> 1];
            }
            // P as A fragments (high part and remainder)
            uint32_t ahi[TG][4], alo[TG][4];
#pragma unroll
            for (int u = 0; u < TG; ++u)
#pragma unroll
                for (int nt = 0; nt < 2; ++nt)
#pragma unroll
                    for (int h = 0; h < 2; ++h) {
                        const float p0 = fast_exp2(sv[u][nt][2 * h] - m[h]);
                        const float p1 = fast_exp2(sv[u][nt][2 * h + 1] - m[h]);
                        lp[h] += p0 + p1;
                        Pack<T>::split(p0, p1, ahi[u][2 * nt + h], alo[u][2 * nt + h]);
                    }
            // ---- O += P V
            RowAddr vr[TG];
#pragma unroll
            for (int u = 0; u < TG; ++u)
                vr[u] = row_addr<D>(v_tile, v_new, zero,
                                    tb + u * kMmaTokens + (lane & 7) + (((lane >> 3) & 1) << 3),
                                    n_tile, t0, it.past);
#pragma unroll
            for (int pp = 0; pp < NT / 2; ++pp)
#pragma unroll
                for (int u = 0; u < TG; ++u) {
                    uint32_t v00, v01, v10, v11;
                    ldsm_x4_t(vr[u].at(2 * pp + (lane >> 4)), v00, v01, v10, v11);
                    mma_16816<kBf>(o[2 * pp], ahi[u], v00, v01);
                    mma_16816<kBf>(o[2 * pp + 1], ahi[u], v10, v11);
                    mma_16816<kBf>(o[2 * pp], alo[u], v00, v01);
                    mma_16816<kBf>(o[2 * pp + 1], alo[u], v10, v11);
                }
            __syncwarp();
            if (j + 1 < ntiles) {
                if (lane == 0)
                    mbar_arrive(&sm.empty[s]);
            } else {
                s_hold = s;
            }
        }
        // Release the query buffer only now.  ldmatrix completes asynchronously
        // and the fragments are first consumed by the MMAs of the tile loop: a
        // release right after the load let the producer's copy of the piece two
        // ahead land before the read had been performed.  Every MMA reading qa
        // has issued here (a warp that computed no tile never uses qa).
        __syncwarp();
        if (lane == 0)
            mbar_arrive(&sm.q_free[piece & 1]);

        if (!dep_ok) {
            grid_dependency_wait();
            dep_ok = true;
        }
        // ---- piece end: merge the TS warps of each row group.  Each warp
        // leaves its running (max, sum) and its unscaled accumulators in
        // shared memory; the summing threads apply the factors 2^(m_t - M).
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            lp[h] += __shfl_xor_sync(kFull, lp[h], 1);
            lp[h] += __shfl_xor_sync(kFull, lp[h], 2);
        }
        // the previous piece's readers are done with the buffers; uniform abort
        if (consumer_bar_or(*sm.abort_flag != 0))
            break;
        if (qd == 0) {
            ml_buf[warp * 16 + g] = make_float2(m[0], lp[0]);
            ml_buf[warp * 16 + g + 8] = make_float2(m[1], lp[1]);
        }
        const int rows_used = min(16, max(0, R_cta - row0));
        // Rounds of DRr columns: each warp writes its rows (at most RU) of the
        // round's columns to the merge buffer, then all threads sum the TS
        // warps of each row.  The buffer is the piece's last stage (every warp
        // is past its tile loop here, and the stage's slot is not yet
        // released), so one round covers all D columns.
        float* mbuf = reinterpret_cast<float*>(sm.ring + static_cast<size_t>((gt - 1) % S) * p.stage_bytes);
        const int mcap = p.stage_bytes / 4;
        const int RU = min(16, R_cta);
        const int lg = obuf_lg(D, RU, mcap);
        const int DRr = 1 << lg, TPR = DRr / 8, rounds = D >> lg;
        for (int r = 0; r < rounds; ++r) {
            if (r > 0)
                consumer_bar_sync();  // readers of the previous round are done
#pragma unroll
            for (int i = 0; i < NT; ++i) {
                if (i < r * TPR || i >= (r + 1) * TPR)
                    continue;
                const int dd = (i - r * TPR) * 8 + 2 * qd;
                if (g < rows_used)
                    *reinterpret_cast<float2*>(
                        &mbuf[((warp * RU + g) << lg) + ((dd ^ obuf_swz(g)) & (DRr - 1))]) =
                        make_float2(o[i][0], o[i][1]);
                if (g + 8 < rows_used)
                    *reinterpret_cast<float2*>(
                        &mbuf[((warp * RU + g + 8) << lg) + ((dd ^ obuf_swz(g + 8)) & (DRr - 1))]) =
                        make_float2(o[i][2], o[i][3]);
            }
            consumer_bar_sync();
            sum_warps<D, MT, TO>(p, it, R_cta, RU, lg, r, ml_buf, mbuf);
        }
        // the stage goes back to the producer (its TMA writes follow these
        // generic-proxy accesses)
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0 && s_hold >= 0)
            mbar_arrive(&sm.empty[s_hold]);
        // automatic schedule: the CTA's first and last pieces at most
        if (!it.whole && p.counters && nsplit < kSplitList) {
            if (threadIdx.x == 0)
                sm.split_list[nsplit] = make_int4(it.b, it.rsg, it.kh, 0);
            ++nsplit;
        }
    }
    // uniform over the consumer warps (a late abort flag must not split them)
    if (nsplit > 0 && !consumer_bar_or(*sm.abort_flag != 0))
        flush_split_pieces<D, TO>(p, sc, sm.split_list, nsplit, tot, 2 * ROWS, obuf, kObufFloats);
}

// T: __half or __nv_bfloat16; D: head size; TO: output element type.  The
// tensor-core kernel for at most 8 query rows per KV head and pass (GQA
// decode): with rows this few, the 16-row side of the m16n8k16 MMA is put on
// the tokens and the 8-column side on the rows.  Each warp takes TPW tokens of
// a stage and computes S^T = K Q^T (tokens x 8 rows), its running row maxima
// and sums (reduced over the lanes of a row), and O^T += V^T P^T (D x 8 rows),
// the P fragments moved from the accumulator layout into the operand layout by
// movmatrix transposes.  Half the MMAs and half the accumulator registers of
// the 16-row kernel; pipeline, schedule, piece-end and split merges are the
// same.
template <typename T, int D, typename TO>
__global__ void __launch_bounds__(kThreads, 1)
    pa_mmat_kernel(const __grid_constant__ SplitParams p, const __grid_constant__ CUtensorMap kmap,
                   const __grid_constant__ CUtensorMap vmap)
{
    constexpr bool kBf = std::is_same<T, __nv_bfloat16>::value;
    constexpr int KS = D / 16;  // k-steps of K Q^T; also 16-column tiles of O^T
    constexpr int ROWS = 8;     // query rows per CTA pass
    constexpr int TG = mma_token_groups(D, 0);  // 16-token groups per warp and stage
    constexpr int TPW = kMmaTokens * TG;        // tokens per warp and stage

    extern __shared__ __align__(1024) unsigned char smem_raw[];
    const Smem sm = carve(p, smem_raw);
    float2* ml_buf = reinterpret_cast<float2*>(sm.scratch);      // [warps][16] (max, sum)
    float2* tot = reinterpret_cast<float2*>(sm.scratch + 1024);  // split merges: (max, sum)
    float* obuf = reinterpret_cast<float*>(sm.scratch + 2048);   // kObufFloats merge rounds

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int S = p.stages;

    // inputs may be produced by the previous kernel on the stream
    kernel_entry(p, kmap, vmap, sm);
    const Sched sc = setup_cta(p, sm);

    if (warp >= kConsumerWarps) {
        produce<T, D, true>(p, sc, sm, &kmap, &vmap, warp - kConsumerWarps, lane);
        return;
    }
    // consumers: with p.early (the inputs read before the previous kernel
    // completed), the grid-dependency wait comes at the first piece end,
    // before any write of the output or the workspace
    bool dep_ok = !p.early;

    // MMA fragment coordinates: g = lane / 4 (accumulator row: token; operand
    // column: query row), qd = lane % 4 (accumulator columns 2 qd, 2 qd + 1:
    // this thread's two query rows)
    const int g = lane >> 2, qd = lane & 3;
    const int TT = p.TT;
    const int WS = TT / TPW;  // warps per stage
    const int nsets = kConsumerWarps / WS;
    const int my_set = warp / WS;
    const int tb = (warp % WS) * TPW;  // this warp's first token in a stage
    const uint32_t zero = smem_u32(sm.zero16);
    const uint32_t qbuf = smem_u32(sm.scratch + p.qbuf_off);
    uint32_t gt = 0;
    int piece = 0;
    int nsplit = 0;  // split pieces listed since the last flush (uniform)
    bool alive = true;

    PieceIter pi;
    for (pi.first(p, sc); pi.ok; pi.next(p, sc), ++piece) {
        const Item& it = pi.it;
        const int ntiles = (it.end - it.start + TT - 1) / TT;
        const int R_cta = min(ROWS, p.R - it.rsg * ROWS);

        // causal / length limits of this thread's rows 2 qd + e (0 for padding rows)
        int lim[2];
#pragma unroll
        for (int e = 0; e < 2; ++e) {
            const int rl = 2 * qd + e;
            const int rho = it.rsg * ROWS + rl;
            lim[e] = rl < R_cta ? it.past + (p.causal ? (rho % p.NQ) + 1 : p.NQ) : 0;
        }
        const int lim_min = __reduce_min_sync(kFull, min(lim[0] > 0 ? lim[0] : INT_MAX,
                                                         lim[1] > 0 ? lim[1] : INT_MAX));

        // Q^T fragments (operand B: k = head columns, n = query row g) from this
        // piece's query buffer, [8 rows][D] row-major
        uint32_t qb[KS][2];
        {
            const int par = piece & 1;
            if (alive) {
                alive = !*sm.abort_flag &&
                        mbar_wait_bounded(&sm.q_full[par], (piece >> 1) & 1, p.wait_ns);
                alive = __all_sync(kFull, alive);
                if (!alive && lane == 0)
                    flag_timeout(p, sm.abort_flag);
            }
            const uint32_t qaddr = qbuf + (par * ROWS + (lane & 7)) * q_row_bytes(D) + ((lane >> 3) << 4);
            const bool rok = g < R_cta;  // rows past the pass hold stale shared memory
#pragma unroll
            for (int kk = 0; kk < KS / 2; ++kk) {
                ldsm_x4(qaddr + kk * 64, qb[2 * kk][0], qb[2 * kk][1], qb[2 * kk + 1][0],
                        qb[2 * kk + 1][1]);
                if (!rok) {
                    qb[2 * kk][0] = 0u;
                    qb[2 * kk][1] = 0u;
                    qb[2 * kk + 1][0] = 0u;
                    qb[2 * kk + 1][1] = 0u;
                }
            }
        }

        float m[2] = {-FLT_MAX, -FLT_MAX}, lp[2] = {0.f, 0.f};
        float o[KS][4];  // O^T tile mt: (column 16 mt + g (+8), rows 2 qd, 2 qd + 1)
#pragma unroll
        for (int i = 0; i < KS; ++i)
#pragma unroll
            for (int e = 0; e < 4; ++e)
                o[i][e] = 0.f;

        for (int j = 0; j < ntiles; ++j, ++gt) {
            if (static_cast<int>(gt % nsets) != my_set)
                continue;  // another warp set's stage
            const int s = gt % S;
            if (alive) {
                alive = !*sm.abort_flag &&
                        mbar_wait_bounded(&sm.full[s], (gt / S) & 1, p.wait_ns);
                alive = __all_sync(kFull, alive);
                if (!alive && lane == 0)
                    flag_timeout(p, sm.abort_flag);
            }
            if (!alive)
                continue;
            const uint32_t st = smem_u32(sm.ring) + s * p.stage_bytes;
            const uint32_t k_tile = st, v_tile = st + p.v_off;
            const uint32_t k_new = st + p.knew_off, v_new = st + p.vnew_off;
            const int t0 = it.start + j * TT;
            const int n_tile = min(TT, it.end - t0);
            if (tb >= n_tile) {  // the stage ends before this warp's tokens
                __syncwarp();
                if (lane == 0)
                    mbar_arrive(&sm.empty[s]);
                continue;
            }
            // a group whose every token is visible to every row of the pass
            bool full_tile[TG];
#pragma unroll
            for (int u = 0; u < TG; ++u) {
                const int tu = tb + u * kMmaTokens;
                full_tile[u] = tu + kMmaTokens <= n_tile && t0 + tu + kMmaTokens <= lim_min;
            }

            // ---- S^T = K Q^T: operand A = 16 token rows of K (ldmatrix gives
            // (tokens 0-7 | 8-15) x (columns 0-7 | 8-15) as a0 a2 a1 a3); two
            // accumulator sets per group (even / odd k-steps) for shorter chains
            float sa[TG][2][4];
#pragma unroll
            for (int u = 0; u < TG; ++u)
#pragma unroll
                for (int a = 0; a < 2; ++a)
#pragma unroll
                    for (int e = 0; e < 4; ++e)
                        sa[u][a][e] = 0.f;
            RowAddr kr[TG];
#pragma unroll
            for (int u = 0; u < TG; ++u)
                kr[u] = row_addr<D>(k_tile, k_new, zero,
                                    tb + u * kMmaTokens + (lane & 7) + ((lane >> 4) << 3), n_tile,
                                    t0, it.past);
#pragma unroll
            for (int ks = 0; ks < KS; ++ks)
#pragma unroll
                for (int u = 0; u < TG; ++u) {
                    uint32_t a[4];
                    ldsm_x4(kr[u].at(2 * ks + ((lane >> 3) & 1)), a[0], a[2], a[1], a[3]);
                    mma_16816<kBf>(sa[u][ks & 1], a, qb[ks][0], qb[ks][1]);
                }
            // scale, mask, row maxima of the stage: element e of group u is
            // token tb + 16 u + g + 8 (e / 2), row 2 qd + e % 2
            float sv[TG][4];
            float mx[2] = {-INFINITY, -INFINITY};
#pragma unroll
            for (int u = 0; u < TG; ++u)
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    const int h = e & 1;
                    const int tk = tb + u * kMmaTokens + g + ((e >> 1) << 3);
                    const float v = (sa[u][0][e] + sa[u][1][e]) * p.qscale;
                    const bool valid = full_tile[u] || (tk < n_tile && t0 + tk < lim[h]);
                    sv[u][e] = valid ? v : -INFINITY;
                    mx[h] = fmaxf(mx[h], sv[u][e]);
                }
            bool grow = false;
#pragma unroll
            for (int h = 0; h < 2; ++h) {
                mx[h] = fmaxf(mx[h], __shfl_xor_sync(kFull, mx[h], 4));
                mx[h] = fmaxf(mx[h], __shfl_xor_sync(kFull, mx[h], 8));
                mx[h] = fmaxf(mx[h], __shfl_xor_sync(kFull, mx[h], 16));
                grow |= mx[h] > m[h];
            }
            if (__any_sync(kFull, grow)) {  // rescale only when a row maximum grew
                float f[2];
#pragma unroll
                for (int h = 0; h < 2; ++h) {
                    const float mn = fmaxf(m[h], mx[h]);
                    f[h] = fast_exp2(m[h] - mn);
                    m[h] = mn;
                    lp[h] *= f[h];
                }
#pragma unroll
                for (int i = 0; i < KS; ++i)
#pragma unroll
                    for (int e = 0; e < 4; ++e)
                        o[i][e] *= f[e & 1];
            }
            // P^T as operand B (k = tokens, n = row g): the accumulator layout
            // holds (token g, rows 2 qd, 2 qd + 1) per 8x8 block; a movmatrix
            // transpose gives (tokens 2 qd, 2 qd + 1, row g).  High part and
            // remainder.
            uint32_t bh[TG][2], bl[TG][2];
#pragma unroll
            for (int u = 0; u < TG; ++u) {
                const float p0 = fast_exp2(sv[u][0] - m[0]);
                const float p1 = fast_exp2(sv[u][1] - m[1]);
                const float p2 = fast_exp2(sv[u][2] - m[0]);
                const float p3 = fast_exp2(sv[u][3] - m[1]);
                lp[0] += p0 + p2;
                lp[1] += p1 + p3;
                uint32_t h01, l01, h23, l23;
                Pack<T>::split(p0, p1, h01, l01);
                Pack<T>::split(p2, p3, h23, l23);
                bh[u][0] = movm_trans(h01);
                bh[u][1] = movm_trans(h23);
                bl[u][0] = movm_trans(l01);
                bl[u][1] = movm_trans(l23);
            }
            // ---- O^T += V^T P^T: operand A = 16 columns x 16 tokens of V
            // (ldmatrix.trans gives (columns 0-7 | 8-15) x (tokens 0-7 | 8-15)
            // as a0 a2 a1 a3)
            RowAddr vr[TG];
#pragma unroll
            for (int u = 0; u < TG; ++u)
                vr[u] = row_addr<D>(v_tile, v_new, zero,
                                    tb + u * kMmaTokens + (lane & 7) + (((lane >> 3) & 1) << 3),
                                    n_tile, t0, it.past);
#pragma unroll
            for (int mt = 0; mt < KS; ++mt)
#pragma unroll
                for (int u = 0; u < TG; ++u) {
                    uint32_t a[4];
                    ldsm_x4_t(vr[u].at(2 * mt + (lane >> 4)), a[0], a[2], a[1], a[3]);
                    mma_16816<kBf>(o[mt], a, bh[u][0], bh[u][1]);
                    mma_16816<kBf>(o[mt], a, bl[u][0], bl[u][1]);
                }
            __syncwarp();
            if (lane == 0)
                mbar_arrive(&sm.empty[s]);
        }
        // release the query buffer once every MMA reading qb has issued
        __syncwarp();
        if (lane == 0)
            mbar_arrive(&sm.q_free[piece & 1]);

        if (!dep_ok) {
            grid_dependency_wait();
            dep_ok = true;
        }
        // ---- piece end: row sums over the lanes of a row, then the merge of
        // the eight warps through shared memory
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            lp[h] += __shfl_xor_sync(kFull, lp[h], 4);
            lp[h] += __shfl_xor_sync(kFull, lp[h], 8);
            lp[h] += __shfl_xor_sync(kFull, lp[h], 16);
        }
        // the previous piece's readers are done with the buffers; uniform abort
        if (consumer_bar_or(*sm.abort_flag != 0))
            break;
        if (g == 0) {
            ml_buf[warp * 16 + 2 * qd] = make_float2(m[0], lp[0]);
            ml_buf[warp * 16 + 2 * qd + 1] = make_float2(m[1], lp[1]);
        }
        const int RU = R_cta;
        const int lg = obuf_lg(D, RU);
        const int DRr = 1 << lg, rounds = D >> lg;
        for (int r = 0; r < rounds; ++r) {
            if (r > 0)
                consumer_bar_sync();  // readers of the previous round are done
#pragma unroll
            for (int mt = 0; mt < KS; ++mt)
#pragma unroll
                for (int hh = 0; hh < 2; ++hh) {
                    const int d = 16 * mt + g + 8 * hh;
                    if ((d >> lg) != r)
                        continue;
                    const int dd = d & (DRr - 1);
#pragma unroll
                    for (int e = 0; e < 2; ++e) {
                        const int row = 2 * qd + e;
                        if (row < RU)
                            obuf[((warp * RU + row) << lg) + ((dd ^ obuf_swz(row)) & (DRr - 1))] =
                                o[mt][2 * hh + e];
                    }
                }
            consumer_bar_sync();
            sum_warps<D, 1, TO>(p, it, R_cta, RU, lg, r, ml_buf, obuf);
        }
        // automatic schedule: the CTA's first and last pieces at most
        if (!it.whole && p.counters && nsplit < kSplitList) {
            if (threadIdx.x == 0)
                sm.split_list[nsplit] = make_int4(it.b, it.rsg, it.kh, 0);
            ++nsplit;
        }
    }
    // uniform over the consumer warps (a late abort flag must not split them)
    if (nsplit > 0 && !consumer_bar_or(*sm.abort_flag != 0))
        flush_split_pieces<D, TO>(p, sc, sm.split_list, nsplit, tot, 2 * ROWS, obuf, kObufFloats);
}

// -------------------------------------------------------------- merge kernel
// One CTA of 128 threads per (segment = sequence, row group, KV head; row).
// It finds the partial records of the segment (automatic mode: the CTAs whose
// unit ranges overlap the segment, from the schedule the partition kernel
// left; fixed partitions: records (b P + c) for its ranges c, the range count
// following from the sequence length) and merges them: M = max m,
// L = sum l 2^(m - M), O = sum o 2^(m - M), out = L == 0 ? O : O / L.  The
// accumulator loads of up to eight records per thread are issued with the
// (max, sum) loads (with fixed partitions, also with the length load, for all
// P records), so a merge of up to 32 (D = 128) or 64 (D = 64) records costs
// about one L2 round trip.  Whole segments were finished by the partition
// kernel and are skipped.
constexpr int kCombineFac = 1024;  // records whose factors are kept in shared memory

template <int D, typename TO>
__global__ void __launch_bounds__(128) pa_combine_kernel(const __grid_constant__ CombineParams p)
{
    grid_dependency_wait();
    grid_dependents_launch();
    const int idx = blockIdx.x, rl = blockIdx.y;
    const int kh = idx % p.KV;
    const int rsg = (idx / p.KV) % p.NRS;
    const int b = idx / (p.KV * p.NRS);
    const int U = p.NRS * p.KV;
    const int R_cta = min(p.rows_per_cta, p.R - rsg * p.rows_per_cta);
    if (rl >= R_cta)
        return;
    int n, k0 = 0, rec_first = 0;
    int2 sc = make_int2(0, 0);
    int len = 0;
    if (p.stream) {
        sc = p.sched[b];
        const int2 last = p.sched[p.B - 1];
        const long long W = static_cast<long long>(last.x) + static_cast<long long>(last.y) * U;
        const int C = static_cast<int>(W + static_cast<long long>(p.vunits) * p.B * U);
        const int G = active_ctas(p.grid, C, static_cast<long long>(p.B) * U);
        const int gl = rsg * p.KV + kh;
        const SegSpan ss = seg_span(sc.x + gl * sc.y, sc.y, b * U + gl, p.vunits, C, G);
        k0 = ss.k0;
        n = ss.n;
        rec_first = ss.rec_first;
    } else {
        // fixed partitions: the count follows from the length, which is
        // loaded together with the records (all P are loaded; those past the
        // count are never used)
        len = p.seq_lens[b];
        n = p.partitions;
    }
    auto row_of = [&](int c) -> size_t {  // workspace row of record c
        const size_t rec = p.stream ? (c == 0 ? static_cast<size_t>(rec_first)
                                              : static_cast<size_t>(2 * (k0 + c)))
                                    : (static_cast<size_t>(b) * p.partitions + c) * U +
                                          static_cast<size_t>(rsg) * p.KV + kh;
        return rec * p.row_stride + rl;
    };
    __shared__ float fac[kCombineFac];
    __shared__ float red[4];
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    constexpr int D4 = D / 4;
    constexpr int TPI = 128 / D4;  // threads per 4-column item
    const int d4 = tid / TPI, sub = tid % TPI;
    float4 v[8];
#pragma unroll
    for (int u = 0; u < 8; ++u) {
        const int c = sub + u * TPI;
        if (c < n)
            v[u] = __ldcg(reinterpret_cast<const float4*>(p.ws_o + row_of(c) * D) + d4);
    }
    // this thread's first (max, sum) pair, loaded with the accumulators
    float2 first = tid < n ? __ldcg(&p.ws_ml[row_of(tid)]) : make_float2(-FLT_MAX, 0.f);
    if (!p.stream) {
        const int s = len < 0 ? 0 : len > p.cap ? p.cap : len;  // the partition kernel's clamp
        const int total = s + p.NQ;
        const int per = (total + p.partitions - 1) / p.partitions;
        const int chunk = ((per + p.BLOCK - 1) / p.BLOCK) * p.BLOCK;
        n = (total + chunk - 1) / chunk;
        if (tid >= n)
            first = make_float2(-FLT_MAX, 0.f);
    }
    if (n <= 1)
        return;  // a whole segment: written by the partition kernel
    // M and L over the records (threads split them; block reductions)
    float M = -FLT_MAX;
    for (int c = tid; c < n; c += 128) {
        const float2 ml = c == tid ? first : __ldcg(&p.ws_ml[row_of(c)]);
        M = fmaxf(M, ml.x);
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1)
        M = fmaxf(M, __shfl_xor_sync(kFull, M, o));
    if (lane == 0)
        red[warp] = M;
    __syncthreads();
    M = fmaxf(fmaxf(red[0], red[1]), fmaxf(red[2], red[3]));
    __syncthreads();
    float L = 0.f;
    for (int c = tid; c < n; c += 128) {
        const float2 ml = c == tid ? first : __ldcg(&p.ws_ml[row_of(c)]);
        const float f = fast_exp2(ml.x - M);
        L = fmaf(ml.y, f, L);
        if (c < kCombineFac)
            fac[c] = f;
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1)
        L += __shfl_xor_sync(kFull, L, o);
    if (lane == 0)
        red[warp] = L;
    __syncthreads();
    L = (red[0] + red[1]) + (red[2] + red[3]);
    auto factor = [&](int c) {
        return c < kCombineFac ? fac[c] : fast_exp2(__ldcg(&p.ws_ml[row_of(c)]).x - M);
    };
    float4 O = make_float4(0.f, 0.f, 0.f, 0.f);
    auto fma4 = [&](float f, const float4& x) {
        O.x = fmaf(f, x.x, O.x);
        O.y = fmaf(f, x.y, O.y);
        O.z = fmaf(f, x.z, O.z);
        O.w = fmaf(f, x.w, O.w);
    };
#pragma unroll
    for (int u = 0; u < 8; ++u) {
        const int c = sub + u * TPI;
        if (c < n)
            fma4(factor(c), v[u]);
    }
    for (int c0 = sub + 8 * TPI; c0 < n; c0 += 8 * TPI) {  // more than 8 records per thread
#pragma unroll
        for (int u = 0; u < 8; ++u) {
            const int c = c0 + u * TPI;
            if (c < n)
                v[u] = __ldcg(reinterpret_cast<const float4*>(p.ws_o + row_of(c) * D) + d4);
        }
#pragma unroll
        for (int u = 0; u < 8; ++u) {
            const int c = c0 + u * TPI;
            if (c < n)
                fma4(factor(c), v[u]);
        }
    }
#pragma unroll
    for (int o = 1; o < TPI; o <<= 1) {
        O.x += __shfl_xor_sync(kFull, O.x, o);
        O.y += __shfl_xor_sync(kFull, O.y, o);
        O.z += __shfl_xor_sync(kFull, O.z, o);
        O.w += __shfl_xor_sync(kFull, O.w, o);
    }
    if (sub == 0) {
        const float inv = L == 0.f ? 1.f : 1.f / L;
        const size_t orow = (static_cast<size_t>(b) * p.KV + kh) * p.R + rsg * p.rows_per_cta + rl;
        TO* dst = static_cast<TO*>(p.out) + orow * D + 4 * d4;
        dst[0] = from_float<TO>(O.x * inv);
        dst[1] = from_float<TO>(O.y * inv);
        dst[2] = from_float<TO>(O.z * inv);
        dst[3] = from_float<TO>(O.w * inv);
    }
}

template <typename T, typename TO>
SplitFn pick_split_simt(int D, int RG)
{
    if (D == 64)
        return RG == 4 ? pa_split_kernel<T, 64, 4, TO> : pa_split_kernel<T, 64, 8, TO>;
    return RG == 4 ? pa_split_kernel<T, 128, 4, TO> : pa_split_kernel<T, 128, 8, TO>;
}

// MT = 0: the transposed kernel (at most 8 rows per pass); 1 or 2: 16 * MT rows
template <typename T, typename TO>
SplitFn pick_split_mma(int D, int MT)
{
    if (D == 64)
        return MT == 0   ? pa_mmat_kernel<T, 64, TO>
               : MT == 1 ? pa_mma_kernel<T, 64, 1, TO>
                         : pa_mma_kernel<T, 64, 2, TO>;
    return MT == 0   ? pa_mmat_kernel<T, 128, TO>
           : MT == 1 ? pa_mma_kernel<T, 128, 1, TO>
                     : pa_mma_kernel<T, 128, 2, TO>;
}

template <typename TO>
CombineFn pick_combine_typed(int D)
{
    return D == 64 ? pa_combine_kernel<64, TO> : pa_combine_kernel<128, TO>;
}

}  // namespace pa
