// pa_decode_tc.cu -- the partition kernel for 32 query rows per KV head and
// pass (a GQA group times several new tokens, D = 128) on tcgen05 tensor cores.
//
// What it computes is the decode of onnxruntime-ep-mlx 0.31.1,
// src/ops/paged_attention.rs (VECTOR_BODY: scores against the cached and the
// new keys, online softmax, the weighted sum of the values, the causal bound
// total = past + row + 1), for the persistent split schedule of pa_kernels.cuh
// (same pieces, records and in-kernel merge as the mma.sync kernels).
//
// Per 128-token stage (M = 128 tokens, N = 32 query rows):
//   S^T  = K Q^T                 8 MMAs, K-major K tile and Q, into tensor memory
//   P    = 2^(S^T scale - m)     eight softmax warps: per tensor-memory lane
//                                quarter (32 tokens) two warps of 16 rows
//   O^T += V^T [P_hi | P_lo]^T   8 MMAs of N = 64: the 16-bit high part of P in
//                                columns 0-31, the remainder in 32-63 (P keeps
//                                about 22 bits; O = the two halves summed)
// The running row maximum m is shared by the 128 tokens of a stage: it moves
// only when a score exceeds it by more than 2^8 (the rows' values then stay
// below 256 in P), so the cross-lane maximum and the rescale of O in tensor
// memory are rare; the row sums stay per thread until the piece ends.
//
// Warps: 0-7 softmax (two per lane quarter, 16 rows each; also the split
// merge's consumer warps), 8-9 the TMA producers of pa_kernels.cuh (K and V
// released separately by the MMAs' commits), 10 the MMA issuer (it also
// swizzles each piece's query rows and writes the new rows into the stage).
#include "pa_kernels.cuh"
#include "pa_tc.cuh"

namespace pa {
namespace {
using namespace tc;

constexpr int kTcRows = 32;   // query rows per pass (the MMA's N)
constexpr int kTcTT = 128;    // tokens per stage (the MMA's M)
constexpr int kTcD = 128;     // head size
constexpr int kSoftWarps = 8;        // two per tensor-memory lane quarter
constexpr int kWarpRows = 16;        // query rows per softmax warp
constexpr int kMmaWarp = kConsumerWarps + kProducerWarps;  // after the producers
constexpr float kGrowth = 8.f;        // log2 units a score may exceed m before m moves
constexpr uint32_t kColO = 128;       // S buffers at columns 0 and 64, O buffers at 128 and 192
constexpr uint32_t kTmemCols = 256;
constexpr uint32_t kPBytes = kTcTT * 128;           // one P^T buffer: 128 tokens x (32 hi + 32 lo)
constexpr uint32_t kQBytes = 2 * kTcRows * 128;     // one swizzled query tile: 2 halves x 32 rows
constexpr uint32_t kHalfBytes = kTcTT * 128;        // one 64-column half of a K or V tile

// Layout of the kernel's own region (kTcRegionBytes from base + tc_off).
struct TcSmem {
    unsigned char* pbuf;  // [2][128 tokens][128 B]: P^T, columns 0-31 high, 32-63 remainder
    unsigned char* qsw;   // [2][2 halves][32 rows][128 B]: query rows, 128-byte swizzle
    uint64_t* s_full;     // [2] S^T of a stage is in tensor memory (MMA commit)
    uint64_t* s_free;     // [2] the softmax warps have read it (4 arrivals)
    uint64_t* p_full;     // [2] P^T of a stage is in shared memory (4 arrivals)
    uint64_t* pv_done;    // [2] O^T += V^T P^T of a stage has completed (MMA commit)
    uint64_t* o_free;     // [2] O of a piece has been read (4 arrivals)
    uint64_t* fin;        // every MMA of the CTA has completed
    uint32_t* tmem_slot;
    float* red_max;       // [32 rows][4 lane quarters]
    float* red_sum;       // [32 rows][4 lane quarters]
    float* red_fac;       // [8 warps][16 rows]
};

__device__ __forceinline__ TcSmem carve_tc(const SplitParams& p, unsigned char* raw)
{
    unsigned char* base = raw + ((1024u - (smem_u32(raw) & 1023u)) & 1023u) + p.tc_off;
    TcSmem t;
    t.pbuf = base;
    t.qsw = base + 2 * kPBytes;
    uint64_t* bars = reinterpret_cast<uint64_t*>(base + 2 * kPBytes + 2 * kQBytes);
    t.s_full = bars;
    t.s_free = bars + 2;
    t.p_full = bars + 4;
    t.pv_done = bars + 6;
    t.o_free = bars + 8;
    t.fin = bars + 10;
    t.tmem_slot = reinterpret_cast<uint32_t*>(bars + 12);
    t.red_max = reinterpret_cast<float*>(bars + 16);
    t.red_sum = t.red_max + kTcRows * 4;
    t.red_fac = t.red_sum + kTcRows * 4;
    return t;
}

// Named barrier `id` of the four softmax warps of a row half.
__device__ __forceinline__ void soft_bar_sync(int id)
{
    asm volatile("bar.sync %0, %1;" ::"r"(id), "n"(4 * 32) : "memory");
}

// The same, returning the OR of v over the four warps.
__device__ __forceinline__ bool soft_bar_or(int id, bool v)
{
    uint32_t r;
    asm volatile(
        "{\n\t.reg .pred pi, po;\n\t"
        "setp.ne.u32 pi, %1, 0;\n\t"
        "bar.red.or.pred po, %2, %3, pi;\n\t"
        "selp.u32 %0, 1, 0, po;\n\t}"
        : "=r"(r)
        : "r"(static_cast<uint32_t>(v)), "r"(id), "n"(4 * 32)
        : "memory");
    return r != 0;
}

__device__ __forceinline__ void mbar_arrive_n(uint64_t* bar, uint32_t n)
{
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)), "r"(n) : "memory");
}

__device__ __forceinline__ void st_shared4(uint32_t addr, uint32_t a, uint32_t b, uint32_t c, uint32_t d)
{
    asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(a), "r"(b), "r"(c), "r"(d)
                 : "memory");
}

__device__ __forceinline__ uint4 ld_shared4(uint32_t addr)
{
    uint4 v;
    asm volatile("ld.shared.v4.b32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "r"(addr)
                 : "memory");
    return v;
}

// Byte offset of 16-byte chunk c (0-7) of token row `tok` in one 64-column
// half of a tile of 128-byte rows with the 128-byte swizzle.
__device__ __forceinline__ uint32_t swz_row(int tok, int c)
{
    return static_cast<uint32_t>(tok) * 128 + ((static_cast<uint32_t>(c) ^ (tok & 7)) << 4);
}

// ------------------------------------------------------------------ MMA warp
// The piece's query rows, from the producer's row buffer (rows padded to
// q_row_bytes) into the swizzled K-major operand tile; rows past the pass
// are zero.  All 32 lanes.
__device__ __forceinline__ void swizzle_query(const SplitParams& p, const Smem& sm, const TcSmem& ts, int par,
                                              int R_cta, int lane)
{
    const uint32_t src = smem_u32(sm.scratch + p.qbuf_off) + par * kTcRows * q_row_bytes(kTcD);
    const uint32_t dst = smem_u32(ts.qsw) + par * kQBytes;
#pragma unroll 4
    for (int idx = lane; idx < kTcRows * 16; idx += 32) {
        const int r = idx >> 4, ch = idx & 15, h = ch >> 3, c = ch & 7;
        const uint4 v = r < R_cta ? ld_shared4(src + r * q_row_bytes(kTcD) + ch * 16) : make_uint4(0, 0, 0, 0);
        st_shared4(dst + h * (kTcRows * 128) + swz_row(r, c), v.x, v.y, v.z, v.w);
    }
}

// The stage's new rows (tokens past the cache, from the stage's new-row
// area) written into the K and V tiles, and the V rows from the stage's end
// up to the next multiple of 16 zeroed (the cache box may hold anything
// there, and the last MMA of the stage reads them with P = 0).  All lanes.
__device__ __forceinline__ void fix_stage(const SplitParams& p, uint32_t st, int t0, int n_tile, int past, int lane)
{
    const int a0 = max(past - t0, 0);
    const int nnew = n_tile - a0;
    for (int idx = lane; idx < nnew * 32; idx += 32) {
        const int row = idx >> 5, which = (idx >> 4) & 1, ch = idx & 15;
        const int tok = a0 + row;
        const uint32_t src = st + (which ? p.vnew_off : p.knew_off) + (t0 + tok - past) * (kTcD * 2) + ch * 16;
        const uint32_t dst = st + (which ? p.v_off : 0) + (ch >> 3) * kHalfBytes + swz_row(tok, ch & 7);
        const uint4 v = ld_shared4(src);
        st_shared4(dst, v.x, v.y, v.z, v.w);
    }
    const int z1 = (n_tile + 15) & ~15;
    for (int idx = lane; idx < (z1 - n_tile) * 16; idx += 32) {
        const int tok = n_tile + (idx >> 4), ch = idx & 15;
        st_shared4(st + p.v_off + (ch >> 3) * kHalfBytes + swz_row(tok, ch & 7), 0, 0, 0, 0);
    }
}

// Issues, as the barriers allow, S^T of each stage (once its tiles have
// landed and its S buffer is free) and O^T += V^T P^T (once the softmax has
// written P), polling both, so that S of the next stage runs while the
// softmax works on this one.  Lane 0 issues; the warp swizzles the query rows
// and fixes the stages.  Gives up (abort flag, status) after wait_ns without
// progress.
template <bool kBf>
__device__ void mma_warp(const SplitParams& p, const Sched& sc, const Smem& sm, const TcSmem& ts, uint32_t tmem,
                         int lane)
{
    const int S = p.stages;
    const uint32_t id_s = idesc<kBf>(kTcRows, false);      // S^T: N 32 rows, K and Q K-major
    const uint32_t id_o = idesc<kBf>(64, true, true);      // O^T: N 64 (hi | lo), V^T and P^T MN-major
    const uint32_t ring = smem_u32(sm.ring);
    const uint32_t pbuf = smem_u32(ts.pbuf), qsw = smem_u32(ts.qsw);
    struct Pend {
        int s, pc, first, nks;
    } pend[4];
    TileIter ti;
    ti.start(p, sc);
    uint32_t ns = 0, npv = 0;  // stages whose S, whose PV is issued
    int piece = -1;
    uint64_t last = global_timer_ns();
    while (true) {
        bool prog = false;
        if (ti.valid() && ns - npv < 3) {
            const Item& it = ti.pc.it;
            const int s = static_cast<int>(ns % S), b = ns & 1;
            const bool first = ti.j == 0;
            const int pc = piece + (first ? 1 : 0);
            bool ready = true;
            if (lane == 0) {
                ready = mbar_test_wait(&sm.full[s], (ns / S) & 1);
                // S(ns - 2), and with it every earlier MMA (the query tile of
                // piece pc - 2 included), has completed once its readers are done
                if (ready && ns >= 2)
                    ready = mbar_test_wait(&ts.s_free[b], ((ns >> 1) - 1) & 1);
                if (ready && first)
                    ready = mbar_test_wait(&sm.q_full[pc & 1], (pc >> 1) & 1);
            }
            if (__shfl_sync(kFull, ready ? 1 : 0, 0)) {
                const int t0 = it.start + (ti.j << 7);
                const int n_tile = min(kTcTT, it.end - t0);
                const uint32_t st = ring + s * p.stage_bytes;
                if (first) {
                    piece = pc;
                    swizzle_query(p, sm, ts, pc & 1, min(kTcRows, p.R - it.rsg * kTcRows), lane);
                }
                if (t0 + n_tile > it.past || (n_tile & 15))
                    fix_stage(p, st, t0, n_tile, it.past, lane);
                fence_proxy_async_smem();
                __syncwarp();
                if (lane == 0) {
                    if (first)
                        mbar_arrive_n(&sm.q_free[pc & 1], kConsumerWarps);
                    tc_fence_after();
                    const uint64_t dk = smem_desc(st, 16, 1024);
                    const uint64_t dq = smem_desc(qsw + (pc & 1) * kQBytes, 16, 1024);
#pragma unroll
                    for (int ks = 0; ks < kTcD / 16; ++ks) {
                        const uint32_t ka = (ks >> 2) * kHalfBytes + (ks & 3) * 32;
                        const uint32_t qa = (ks >> 2) * (kTcRows * 128) + (ks & 3) * 32;
                        umma(tmem + b * 64, dk + (ka >> 4), dq + (qa >> 4), id_s, ks > 0);
                    }
                    umma_commit(&ts.s_full[b]);
                    umma_commit(&sm.empty[s]);  // K part of the stage
                }
                __syncwarp();
                pend[ns & 3] = Pend{s, pc, first ? 1 : 0, (n_tile + 15) >> 4};
                ++ns;
                ti.next(p, sc);
                prog = true;
            }
        }
        if (npv < ns) {
            const Pend pd = pend[npv & 3];
            const int b = npv & 1;
            bool ready = true;
            if (lane == 0) {
                ready = mbar_test_wait(&ts.p_full[b], (npv >> 1) & 1);
                if (ready && pd.first && pd.pc >= 2)
                    ready = mbar_test_wait(&ts.o_free[pd.pc & 1], ((pd.pc >> 1) - 1) & 1);
            }
            if (__shfl_sync(kFull, ready ? 1 : 0, 0)) {
                if (lane == 0) {
                    tc_fence_after();
                    const uint64_t dv = smem_desc(ring + pd.s * p.stage_bytes + p.v_off, kHalfBytes, 1024);
                    const uint64_t dp = smem_desc(pbuf + b * kPBytes, kPBytes, 1024);
                    const uint32_t to = tmem + kColO + (pd.pc & 1) * 64;
                    for (int ks = 0; ks < pd.nks; ++ks)
                        umma(to, dv + ((ks * 2048) >> 4), dp + ((ks * 2048) >> 4), id_o, !(pd.first && ks == 0));
                    umma_commit(&ts.pv_done[b]);
                    umma_commit(&sm.empty[kMaxStages / 2 + pd.s]);  // V part
                }
                __syncwarp();
                ++npv;
                prog = true;
            }
        }
        if (!ti.valid() && npv == ns)
            break;
        const uint64_t now = global_timer_ns();
        if (prog) {
            last = now;
        } else if (*sm.abort_flag || now - last > p.wait_ns) {
            if (lane == 0)
                flag_timeout(p, sm.abort_flag);
            break;
        }
    }
    // every MMA complete before the tensor memory is released
    if (lane == 0 && ns > 0) {
        umma_commit(ts.fin);
        mbar_wait_bounded(ts.fin, 0, p.wait_ns);
    }
    __syncwarp();
}

// 16 values (one per row) in every lane, reduced over the warp's lanes by
// halving exchanges and a last full exchange (19 shuffles): lanes L and L + 16
// return row L's result.
template <typename Op>
__device__ __forceinline__ float reduce_rows(const float (&v)[kWarpRows], int lane, Op op)
{
    float b[8], c[4], d[2];
    const bool h8 = lane & 8, h4 = lane & 4, h2 = lane & 2, h1 = lane & 1;
#pragma unroll
    for (int k = 0; k < 8; ++k)
        b[k] = op(h8 ? v[k + 8] : v[k], __shfl_xor_sync(kFull, h8 ? v[k] : v[k + 8], 8));
#pragma unroll
    for (int k = 0; k < 4; ++k)
        c[k] = op(h4 ? b[k + 4] : b[k], __shfl_xor_sync(kFull, h4 ? b[k] : b[k + 4], 4));
#pragma unroll
    for (int k = 0; k < 2; ++k)
        d[k] = op(h2 ? c[k + 2] : c[k], __shfl_xor_sync(kFull, h2 ? c[k] : c[k + 2], 2));
    const float e = op(h1 ? d[1] : d[0], __shfl_xor_sync(kFull, h1 ? d[0] : d[1], 1));
    return op(e, __shfl_xor_sync(kFull, e, 16));
}

// ------------------------------------------------------------ softmax warps
// Warp w (0-7): lane quarter qt = w % 4 of S^T and O^T (tokens 32 qt ..
// 32 qt + 31 of every stage, O^T rows d = 32 qt + lane) and row half
// h = w / 4 (query rows 16 h .. 16 h + 15, one per register).  The four warps
// of a row half share m and synchronise on named barrier 4 + h; the halves
// are independent.
template <typename T, typename TO>
__device__ void softmax_warps(const SplitParams& p, const Sched& sc, const Smem& sm, const TcSmem& ts,
                              uint32_t tmem, int w, int lane, int& nsplit, bool& dep_ok)
{
    const int qt = w & 3, h = w >> 2;
    const uint32_t tl = tmem + (static_cast<uint32_t>(32 * qt) << 16);
    const int tok = 32 * qt + lane;
    const uint32_t prow = smem_u32(ts.pbuf) + tok * 128;
    const int swz = tok & 7;
    const int bar = 4 + h;
    float* fac = ts.red_fac + w * kWarpRows;
    uint32_t gt = 0;
    int piece = 0;
    bool dead = false;
    auto give_up = [&](bool ok) {
        if (!ok && lane == 0)
            flag_timeout(p, sm.abort_flag);
        dead = true;
    };
    PieceIter pi;
    for (pi.first(p, sc); pi.ok; pi.next(p, sc), ++piece) {
        const Item& it = pi.it;
        const int ntiles = (it.end - it.start + kTcTT - 1) >> 7;
        const int R_cta = min(kTcRows, p.R - it.rsg * kTcRows);
        const int q0 = (it.rsg * kTcRows + h * kWarpRows) % p.NQ;  // new-token index of this warp's row 0
        const int vis = it.past + (p.causal ? 1 : p.NQ);  // keys below this: visible to every row
        float m[kWarpRows], l[kWarpRows];
#pragma unroll
        for (int r = 0; r < kWarpRows; ++r) {
            m[r] = -FLT_MAX;
            l[r] = 0.f;
        }
        for (int j = 0; j < ntiles; ++j, ++gt) {
            const int b = gt & 1;
            bool ok = !*sm.abort_flag && mbar_wait_bounded(&ts.s_full[b], (gt >> 1) & 1, p.wait_ns);
            ok = __all_sync(kFull, ok);
            float x[kWarpRows];
            if (ok) {
                tc_fence_after();
                Cols16 c;
                tmem_ld16(c, tl + b * 64 + h * kWarpRows);
                tc_fence_before();
                __syncwarp();
                if (lane == 0)
                    mbar_arrive(&ts.s_free[b]);
#pragma unroll
                for (int r = 0; r < kWarpRows; ++r)
                    x[r] = __uint_as_float(c.r[r]) * p.qscale;
            } else {
#pragma unroll
                for (int r = 0; r < kWarpRows; ++r)
                    x[r] = -INFINITY;
            }
            const int t0 = it.start + (j << 7);
            const int n_tile = min(kTcTT, it.end - t0);
            if (n_tile < kTcTT || t0 + kTcTT > vis) {
                // keys past the stage, and (causal) new keys after a row's own
                const bool in = tok < n_tile;
                const int dt = t0 + tok - it.past;  // index among the new keys when >= 0
                int q = q0;
#pragma unroll
                for (int r = 0; r < kWarpRows; ++r) {
                    const bool v = in && (!p.causal || dt <= q);
                    x[r] = v ? x[r] : -INFINITY;
                    q = q + 1 == p.NQ ? 0 : q + 1;
                }
            }
            bool need = false;
#pragma unroll
            for (int r = 0; r < kWarpRows; ++r)
                need |= x[r] > m[r] + kGrowth;
            if (ok && gt >= 2)  // PV of stage gt - 2 has read P buffer b
                ok = !*sm.abort_flag && mbar_wait_bounded(&ts.pv_done[b], ((gt >> 1) - 1) & 1, p.wait_ns);
            ok = __all_sync(kFull, ok);
            if (soft_bar_or(bar, need || !ok)) {
                if (soft_bar_or(bar, !ok)) {
                    give_up(ok);
                    break;
                }
                // the stage's row maxima over its 128 tokens
                const float mx = reduce_rows(x, lane, [](float a, float b) { return fmaxf(a, b); });
                if (lane < kWarpRows)
                    ts.red_max[(h * kWarpRows + lane) * 4 + qt] = mx;
                soft_bar_sync(bar);
                // the factors 2^(m_old - m_new), kept in this warp's row of
                // red_fac for the rescale of O
                bool shrink = false;
#pragma unroll
                for (int r = 0; r < kWarpRows; ++r) {
                    const float4 v = reinterpret_cast<const float4*>(ts.red_max)[h * kWarpRows + r];
                    const float mn = fmaxf(m[r], fmaxf(fmaxf(v.x, v.y), fmaxf(v.z, v.w)));
                    const float f = fast_exp2(m[r] - mn);
                    shrink |= f != 1.f;
                    m[r] = mn;
                    l[r] *= f;
                    if (lane == 0)
                        fac[r] = f;
                }
                __syncwarp();
                if (j > 0 && shrink) {  // uniform over the row half: m is
                    // O of the piece's stages so far, once the last one's PV is done
                    const uint32_t gp = gt - 1;
                    bool ok2 = !*sm.abort_flag && mbar_wait_bounded(&ts.pv_done[gp & 1], (gp >> 1) & 1, p.wait_ns);
                    ok2 = __all_sync(kFull, ok2);
                    if (soft_bar_or(bar, !ok2)) {
                        give_up(ok2);
                        break;
                    }
                    tc_fence_after();
                    const uint32_t to = tl + kColO + (piece & 1) * 64 + h * kWarpRows;
#pragma unroll
                    for (int part = 0; part < 2; ++part) {  // high part, remainder
                        Cols16 o;
                        tmem_ld16(o, to + part * kTcRows);
#pragma unroll
                        for (int r = 0; r < kWarpRows; ++r)
                            o.r[r] = __float_as_uint(__uint_as_float(o.r[r]) * fac[r]);
                        tmem_st16(o.r, to + part * kTcRows);
                    }
                    asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
                }
            }
            // P = 2^(x - m): the row sums, and P^T (high | remainder) of this
            // warp's rows into buffer b (chunks 2h, 2h + 1 and 4 + 2h, 5 + 2h)
            const uint32_t pr = prow + b * kPBytes;
#pragma unroll
            for (int cc = 0; cc < 2; ++cc) {
                uint32_t hi[4], lo[4];
#pragma unroll
                for (int k = 0; k < 4; ++k) {
                    const int r0 = 8 * cc + 2 * k;
                    const float p0 = fast_exp2(x[r0] - m[r0]);
                    const float p1 = fast_exp2(x[r0 + 1] - m[r0 + 1]);
                    l[r0] += p0;
                    l[r0 + 1] += p1;
                    split_pair<T>(p0, p1, hi[k], lo[k]);
                }
                st_shared4(pr + (((2 * h + cc) ^ swz) << 4), hi[0], hi[1], hi[2], hi[3]);
                st_shared4(pr + (((4 + 2 * h + cc) ^ swz) << 4), lo[0], lo[1], lo[2], lo[3]);
            }
            fence_proxy_async_smem();
            tc_fence_before();
            __syncwarp();
            if (lane == 0)
                mbar_arrive(&ts.p_full[b]);
        }
        if (dead)
            break;

        // ---- piece end: row sums over the 128 tokens, O, then the output
        // (whole segment) or the partial record
        const float ls = reduce_rows(l, lane, [](float a, float b) { return a + b; });
        if (lane < kWarpRows)
            ts.red_sum[(h * kWarpRows + lane) * 4 + qt] = ls;
        const uint32_t gl = gt - 1;
        bool ok = !*sm.abort_flag && mbar_wait_bounded(&ts.pv_done[gl & 1], (gl >> 1) & 1, p.wait_ns);
        ok = __all_sync(kFull, ok);
        if (soft_bar_or(bar, !ok)) {  // also publishes red_sum
            give_up(ok);
            break;
        }
        tc_fence_after();
        Cols16 oh;
        float o[kWarpRows];
        const uint32_t to = tl + kColO + (piece & 1) * 64 + h * kWarpRows;
        tmem_ld16(oh, to);
#pragma unroll
        for (int r = 0; r < kWarpRows; ++r)
            o[r] = __uint_as_float(oh.r[r]);
        tmem_ld16(oh, to + kTcRows);
#pragma unroll
        for (int r = 0; r < kWarpRows; ++r)
            o[r] += __uint_as_float(oh.r[r]);
        tc_fence_before();
        __syncwarp();
        if (lane == 0)
            mbar_arrive(&ts.o_free[piece & 1]);
        if (!dep_ok) {
            grid_dependency_wait();
            dep_ok = true;
        }
        const int rows = R_cta - h * kWarpRows;  // this warp's rows of the pass
        const float4* tot = reinterpret_cast<const float4*>(ts.red_sum) + h * kWarpRows;
        const size_t row0 = (static_cast<size_t>(it.b) * p.KV + it.kh) * p.R +
                            static_cast<size_t>(it.rsg) * kTcRows + h * kWarpRows;
        if (it.whole) {
            TO* dst = static_cast<TO*>(p.out) + row0 * kTcD + tok;
#pragma unroll
            for (int r = 0; r < kWarpRows; ++r)
                if (r < rows) {
                    const float4 v = tot[r];
                    const float L = (v.x + v.y) + (v.z + v.w);
                    dst[static_cast<size_t>(r) * kTcD] = from_float<TO>(L == 0.f ? o[r] : o[r] / L);
                }
        } else {
            const size_t wrow0 = static_cast<size_t>(it.rec) * p.row_stride + h * kWarpRows;
            float* dst = p.ws_o + wrow0 * kTcD + tok;
#pragma unroll
            for (int r = 0; r < kWarpRows; ++r)
                if (r < rows)
                    dst[static_cast<size_t>(r) * kTcD] = o[r];
            if (qt == 0)
#pragma unroll
                for (int r = 0; r < kWarpRows; ++r)
                    if (r == lane && r < rows) {
                        const float4 v = tot[r];
                        p.ws_ml[wrow0 + r] = make_float2(m[r], (v.x + v.y) + (v.z + v.w));
                    }
            if (p.counters && nsplit < kSplitList) {
                if (threadIdx.x == 0)
                    sm.split_list[nsplit] = make_int4(it.b, it.rsg, it.kh, 0);
                ++nsplit;
            }
        }
    }
}

// T: __half or __nv_bfloat16; TO: output element type.  One CTA of
// kUmmaThreads per SM.
template <typename T, typename TO>
__global__ void __launch_bounds__(kUmmaThreads, 1)
    pa_umma32_kernel(const __grid_constant__ SplitParams p, const __grid_constant__ CUtensorMap kmap,
                     const __grid_constant__ CUtensorMap vmap)
{
    constexpr bool kBf = std::is_same<T, __nv_bfloat16>::value;
    extern __shared__ __align__(1024) unsigned char smem_raw[];
    const Smem sm = carve(p, smem_raw);
    const TcSmem ts = carve_tc(p, smem_raw);
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;

    kernel_entry(p, kmap, vmap, sm);
    if (threadIdx.x == 0) {
        for (int s = 0; s < p.stages; ++s)
            mbar_init(&sm.empty[kMaxStages / 2 + s], 1);  // V parts (K parts: init_cta)
        for (int i = 0; i < 2; ++i) {
            mbar_init(&ts.s_full[i], 1);
            mbar_init(&ts.s_free[i], kSoftWarps);
            mbar_init(&ts.p_full[i], kSoftWarps);
            mbar_init(&ts.pv_done[i], 1);
            mbar_init(&ts.o_free[i], kSoftWarps);
        }
        mbar_init(ts.fin, 1);
        fence_mbar_init();
    }
    if (warp == kMmaWarp) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                         smem_u32(ts.tmem_slot)),
                     "r"(kTmemCols)
                     : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    }
    tc_fence_before();
    const Sched sc = setup_cta(p, sm);  // one CTA barrier
    tc_fence_after();
    const uint32_t tmem = *ts.tmem_slot;

    if (warp == kMmaWarp) {
        mma_warp<kBf>(p, sc, sm, ts, tmem, lane);
        // tensor memory is freed once the softmax warps are done with it
        asm volatile("bar.sync 6, %0;" ::"n"((kSoftWarps + 1) * 32) : "memory");
        tc_fence_after();
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(kTmemCols)
                     : "memory");
        return;
    }
    if (warp >= kConsumerWarps) {
        produce<T, kTcD, kHalvesSwizzled>(p, sc, sm, &kmap, &vmap, warp - kConsumerWarps, lane);
        return;
    }
    // the softmax warps are the consumer warps of the split merge
    bool dep_ok = !p.early;  // see pa_mma_kernel
    int nsplit = 0;
    softmax_warps<T, TO>(p, sc, sm, ts, tmem, warp, lane, nsplit, dep_ok);
    // Without an abort every warp has seen every piece (nsplit is uniform);
    // the last PV has completed, so the P buffers serve the merge.
    tc_fence_before();
    const bool aborted = consumer_bar_or(*sm.abort_flag != 0);
    asm volatile("bar.arrive 6, %0;" ::"n"((kSoftWarps + 1) * 32) : "memory");
    if (nsplit > 0 && !aborted) {
        if (!dep_ok)
            grid_dependency_wait();
        flush_split_pieces<kTcD, TO>(p, sc, sm.split_list, nsplit, reinterpret_cast<float2*>(sm.scratch + 1024),
                                     2 * kTcRows, reinterpret_cast<float*>(ts.pbuf), kObufFloats);
    }
}

}  // namespace

SplitFn pick_split_tc(int dtype, bool f32_out)
{
    if (dtype == PA_BF16)
        return f32_out ? pa_umma32_kernel<__nv_bfloat16, float> : pa_umma32_kernel<__nv_bfloat16, __nv_bfloat16>;
    return f32_out ? pa_umma32_kernel<__half, float> : pa_umma32_kernel<__half, __half>;
}

}  // namespace pa
