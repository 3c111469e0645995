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
// The stream is latency-bound: a tile lands some 3 us after its copy is
// issued, so throughput is the bytes in flight per SM.  K and V therefore
// have rings of their own (three 32 KB tiles each where shared memory allows),
// land and are released apart (K once its S MMAs complete, V once its PV MMAs
// do), and everything else is kept small: one P^T tile, one query tile
// (loaded by TMA straight into the swizzled operand layout once the previous
// piece's S MMAs are done), the new rows written into the tiles from L2.
//
// Warps: 0-7 softmax (two per lane quarter, 16 rows each; also the split
// merge's consumer warps), 8-9 the TMA producers (K, V), 10 the MMA issuer
// (it also writes the new rows into the tiles).
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
constexpr uint32_t kPBytes = kTcTT * 128;           // P^T: 128 tokens x (32 hi + 32 lo) 16-bit
constexpr uint32_t kQBytes = 2 * kTcRows * 128;     // the query tile: 2 halves x 32 rows
constexpr uint32_t kHalfBytes = kTcTT * 128;        // one 64-column half of a K or V tile
constexpr int kVRing = kMaxStages / 2;              // V ring barriers: full/empty[kVRing + s]

// Layout of the kernel's own region (kTcRegionBytes from base + tc_off).
struct TcSmem {
    unsigned char* pbuf;  // [128 tokens][128 B]: P^T, columns 0-31 high, 32-63 remainder
    unsigned char* qsw;   // [2 halves][32 rows][128 B]: query rows, 128-byte swizzle
    uint64_t* s_full;     // [2] S^T of a stage is in tensor memory (MMA commit)
    uint64_t* s_free;     // [2] the softmax warps have read it (8 arrivals)
    uint64_t* p_full;     // P^T of a stage is in shared memory (8 arrivals)
    uint64_t* pv_done;    // O^T += V^T P^T of a stage has completed (MMA commit)
    uint64_t* o_free;     // [2] O of a piece has been read (8 arrivals)
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
    t.qsw = base + kPBytes;
    uint64_t* bars = reinterpret_cast<uint64_t*>(base + kPBytes + kQBytes);
    t.s_full = bars;
    t.s_free = bars + 2;
    t.p_full = bars + 4;
    t.pv_done = bars + 5;
    t.o_free = bars + 6;
    t.fin = bars + 8;
    t.tmem_slot = reinterpret_cast<uint32_t*>(bars + 10);
    t.red_max = reinterpret_cast<float*>(bars + 16);
    t.red_sum = t.red_max + kTcRows * 4;
    t.red_fac = t.red_sum + kTcRows * 4;
    return t;
}
static_assert(kPBytes + kQBytes + 128 + 3 * 512 <= static_cast<uint32_t>(kTcRegionBytes), "tcgen05 region");

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

__device__ __forceinline__ void st_shared4(uint32_t addr, uint32_t a, uint32_t b, uint32_t c, uint32_t d)
{
    asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(a), "r"(b), "r"(c), "r"(d)
                 : "memory");
}

// Byte offset of 16-byte chunk c (0-7) of token row `tok` in one 64-column
// half of a tile of 128-byte rows with the 128-byte swizzle.
__device__ __forceinline__ uint32_t swz_row(int tok, int c)
{
    return static_cast<uint32_t>(tok) * 128 + ((static_cast<uint32_t>(c) ^ (tok & 7)) << 4);
}

// ------------------------------------------------------------------ producers
// A producer warp (role 0: K, role 1: V): for every tile of this CTA's
// pieces, wait for a free slot of its ring and issue, per cache block, one TMA
// box per 64-column half (half h of the tile at h * kHalfBytes: the canonical
// K-major / MN-major operand layout).  Role 0 also loads each piece's query
// rows (two boxes into the swizzled query tile, once the MMA warp has
// committed the previous piece's S) and, for a segment's last stage, both
// roles prefetch its new rows into L2 for the MMA warp.  Table entries come
// kTableAhead tiles ahead by cp.async (fetch_entries).
template <typename T>
__device__ void produce_tc(const SplitParams& p, const Sched& sc, const Smem& sm, const TcSmem& ts,
                           const CUtensorMap* kmap, const CUtensorMap* vmap, const CUtensorMap* qmap, int role,
                           int lane)
{
    const CUtensorMap* map = role == 0 ? kmap : vmap;
    const int S = role == 0 ? p.stages : p.stages_v;
    uint64_t* full = sm.full + (role ? kVRing : 0);
    uint64_t* empty = sm.empty + (role ? kVRing : 0);
    unsigned char* ring = sm.ring + static_cast<size_t>(role ? p.stages : 0) * p.stage_bytes;
    const T* news = static_cast<const T*>(role == 0 ? p.k_new : p.v_new);
    const uint32_t half_bytes = static_cast<uint32_t>(p.box_rows) * 128;  // one half of a box
    int* entries = sm.entries + role * (kTableSlots * kSlotInts);
    const int HB = p.box_rows;

    TileIter cur, ahead;
    cur.start(p, sc);
    ahead = cur;
    fetch_entries(p, ahead, entries, lane);
    if (ahead.valid())
        ahead.next(p, sc);
    uint32_t gt = 0;  // tiles issued by this role
    int s = 0;        // ring slot of tile gt
    uint32_t ph = 0;  // completed passes over the ring
    int piece = -1, q_issued = 0;
    for (; cur.valid(); cur.next(p, sc), ++gt) {
        if (gt == 0) {
            asm volatile("cp.async.wait_group 0;" ::: "memory");
        } else {
            fetch_entries(p, ahead, entries + ((gt + kTableAhead) % kTableSlots) * kSlotInts, lane);
            if (ahead.valid())
                ahead.next(p, sc);
            asm volatile("cp.async.wait_group %0;" ::"n"(kTableAhead) : "memory");
        }
        if (ph > 0) {
            bool ok = !*sm.abort_flag && mbar_wait_bounded(&empty[s], (ph - 1) & 1, p.wait_ns);
            ok = __all_sync(kFull, ok);
            if (!ok) {
                if (lane == 0)
                    flag_timeout(p, sm.abort_flag);
                break;
            }
        }
        const Item& it = cur.pc.it;
        if (cur.j == 0) {
            ++piece;
            if (role == 0) {
                // the one query tile is free once the previous piece's S MMAs are done
                if (piece >= 1) {
                    bool ok = !*sm.abort_flag && mbar_wait_bounded(&sm.q_free[0], (piece - 1) & 1, p.wait_ns);
                    ok = __all_sync(kFull, ok);
                    if (!ok) {
                        if (lane == 0)
                            flag_timeout(p, sm.abort_flag);
                        break;
                    }
                }
                if (lane == 0) {
                    const int row0 = (it.b * p.KV + it.kh) * p.R + it.rsg * kTcRows;
                    mbar_arrive_expect_tx(&sm.q_full[0], kQBytes);
                    tma_load_3d(ts.qsw, qmap, 0, 0, row0, &sm.q_full[0]);
                    tma_load_3d(ts.qsw + kTcRows * 128, qmap, 0, 1, row0, &sm.q_full[0]);
                }
                ++q_issued;
                // the next piece's query rows into L2 (its load waits for this
                // piece's S MMAs): 64 lines of 128 bytes, two a lane
                PieceIter nx = cur.pc;
                nx.next(p, sc);
                if (nx.ok) {
                    const int rows = min(kTcRows, p.R - nx.it.rsg * kTcRows);
                    const char* src = static_cast<const char*>(p.q) +
                                      ((static_cast<size_t>(nx.it.b) * p.KV + nx.it.kh) * p.R +
                                       static_cast<size_t>(nx.it.rsg) * kTcRows) * (kTcD * 2);
#pragma unroll
                    for (int u = 0; u < 2; ++u)
                        if (lane + 32 * u < 2 * rows)
                            asm volatile("prefetch.global.L2 [%0];" ::"l"(src + (lane + 32 * u) * 128));
                }
            }
        }
        const int t0 = it.start + (cur.j << p.lg_tt);
        const int t1 = min(t0 + p.TT, it.end);
        const int cache_end = min(t1, it.past);
        const int nb = cache_end > t0 ? (cache_end - t0 + HB - 1) >> p.lg_box : 0;
        const int* ent = entries + (gt % kTableSlots) * kSlotInts;
        if (role == 0 && lane < nb && p.checked) {
            const int phys = ent[lane];  // own cp.async
            if ((phys < 0 || phys >= p.num_blocks) && p.status)
                atomicOr(p.status, PA_STATUS_BAD_BLOCK);
        }
        unsigned char* st = ring + static_cast<size_t>(s) * p.stage_bytes;
        // test switch (pa_opts.debug_withhold_stage): every CTA's V producer
        // leaves one stage out, so that the waits for it run out
        const bool withheld = p.withhold > 0 && role == 1 && gt + 1 == static_cast<uint32_t>(p.withhold);
        if (lane == 0 && !withheld)
            mbar_arrive_expect_tx(&full[s], static_cast<uint32_t>(nb) * 2 * half_bytes);
        __syncwarp();  // entries written by other lanes' cp.async are visible
        if (lane < nb && !withheld) {
            const int phys = ent[lane];
            // out-of-pool coordinates read as zeros: the copy never faults
            const int z = (phys << p.lg_block) + ((t0 + (lane << p.lg_box)) & (p.BLOCK - 1));
#pragma unroll
            for (int h = 0; h < kTcD / 64; ++h)
                tma_load_4d(st + h * kHalfBytes + lane * half_bytes, map, 0, h, it.kh, z, &full[s]);
        }
        if (t1 > it.past && lane < 2 * p.NQ) {  // the new rows, 128 bytes a lane
            const char* src = reinterpret_cast<const char*>(news + (static_cast<size_t>(it.b) * p.KV + it.kh) * p.NQ * kTcD);
            asm volatile("prefetch.global.L2 [%0];" ::"l"(src + lane * 128));
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
    // no copy left in flight when the pipeline was abandoned
    __syncwarp();
    if (*sm.abort_flag && lane == 0) {
        const uint32_t first = gt > static_cast<uint32_t>(S) ? gt - S : 0u;
        for (uint32_t g = first; g < gt; ++g)
            mbar_wait_bounded(&full[g % S], (g / S) & 1, p.wait_ns);
        if (q_issued > 0)
            mbar_wait_bounded(&sm.q_full[0], (q_issued - 1) & 1, p.wait_ns);
    }
}

// ------------------------------------------------------------------ MMA warp
// A stage's new rows (tokens past the cache; `rows` = the segment's new rows
// [NQ][D] in global memory, prefetched into L2 by the producer) written into
// its K or V tile; with zero_tail also the rows from the stage's end up to the
// next multiple of 16 zeroed (the cache box may hold anything there, and the
// stage's last PV MMA reads them with P = 0).  All lanes; up to 16 new rows.
template <typename T>
__device__ __forceinline__ void fix_tile(uint32_t tile, const T* rows, int t0, int n_tile, int past, bool zero_tail,
                                         int lane)
{
    const int a0 = max(past - t0, 0);
    const int n = (n_tile - a0) * 16;  // 16-byte chunks of the stage's new rows
    uint4 v[8];
#pragma unroll
    for (int u = 0; u < 8; ++u) {
        const int idx = lane + 32 * u;
        if (idx < n)
            v[u] = __ldg(reinterpret_cast<const uint4*>(rows + static_cast<size_t>(t0 + a0 - past) * kTcD) + idx);
    }
#pragma unroll
    for (int u = 0; u < 8; ++u) {
        const int idx = lane + 32 * u;
        if (idx < n) {
            const int tok = a0 + (idx >> 4), ch = idx & 15;
            st_shared4(tile + (ch >> 3) * kHalfBytes + swz_row(tok, ch & 7), v[u].x, v[u].y, v[u].z, v[u].w);
        }
    }
    if (zero_tail) {
        const int z1 = (n_tile + 15) & ~15;
        for (int idx = lane; idx < (z1 - n_tile) * 16; idx += 32) {
            const int tok = n_tile + (idx >> 4), ch = idx & 15;
            st_shared4(tile + (ch >> 3) * kHalfBytes + swz_row(tok, ch & 7), 0, 0, 0, 0);
        }
    }
}

// Issues, as the barriers allow, O^T += V^T P^T of each stage (once its V
// tile has landed and the softmax has written P; first, as the softmax of the
// next stage waits for it) and S^T (once its K tile has landed and its S
// buffer is free), polling both, so that S of the next stage runs while the
// softmax works on this one.  After the last S of a
// piece it commits the query tile free.  Lane 0 issues; the warp writes the
// new rows.  Gives up (abort flag, status) after wait_ns without progress.
template <typename T>
__device__ void mma_warp(const SplitParams& p, const Sched& sc, const Smem& sm, const TcSmem& ts, uint32_t tmem,
                         int lane)
{
    constexpr bool kBf = std::is_same<T, __nv_bfloat16>::value;
    const int SK = p.stages, SV = p.stages_v;
    const uint32_t id_s = idesc<kBf>(kTcRows, false);      // S^T: N 32 rows, K and Q K-major
    const uint32_t id_o = idesc<kBf>(64, true, true);      // O^T: N 64 (hi | lo), V^T and P^T MN-major
    const uint32_t ring_k = smem_u32(sm.ring);
    const uint32_t ring_v = ring_k + SK * p.stage_bytes;
    const uint64_t dq = smem_desc(smem_u32(ts.qsw), 16, 1024);
    const uint64_t dp = smem_desc(smem_u32(ts.pbuf), kPBytes, 1024);
    struct Pend {
        int pc, first, nks, t0, n_tile, past;
        size_t nrow;  // the segment's first new row in v_new
    } pend[4];
    TileIter ti;
    ti.start(p, sc);
    uint32_t ns = 0, npv = 0;  // stages whose S, whose PV is issued
    int piece = -1;
    uint64_t last = global_timer_ns();
    while (true) {
        bool prog = false;
        if (npv < ns) {
            const Pend pd = pend[npv & 3];
            const int sv = static_cast<int>(npv % SV);
            bool ready = true;
            if (lane == 0) {
                ready = mbar_test_wait(ts.p_full, npv & 1) &&
                        mbar_test_wait(&sm.full[kVRing + sv], (npv / SV) & 1);
                if (ready && pd.first && pd.pc >= 2)
                    ready = mbar_test_wait(&ts.o_free[pd.pc & 1], ((pd.pc >> 1) - 1) & 1);
            }
            if (__shfl_sync(kFull, ready ? 1 : 0, 0)) {
                const uint32_t st = ring_v + sv * p.stage_bytes;
                if (pd.t0 + pd.n_tile > pd.past || (pd.n_tile & 15)) {
                    fix_tile(st, static_cast<const T*>(p.v_new) + pd.nrow * kTcD, pd.t0, pd.n_tile, pd.past, true,
                             lane);
                    fence_proxy_async_smem();
                }
                __syncwarp();
                if (lane == 0) {
                    tc_fence_after();
                    const uint64_t dv = smem_desc(st, kHalfBytes, 1024);
                    const uint32_t to = tmem + kColO + (pd.pc & 1) * 64;
                    for (int ks = 0; ks < pd.nks; ++ks)
                        umma(to, dv + ((ks * 2048) >> 4), dp + ((ks * 2048) >> 4), id_o, !(pd.first && ks == 0));
                    umma_commit(ts.pv_done);
                    umma_commit(&sm.empty[kVRing + sv]);  // the V slot
                }
                __syncwarp();
                ++npv;
                prog = true;
            }
        }
        if (ti.valid() && ns - npv < 3) {
            const Item& it = ti.pc.it;
            const int sk = static_cast<int>(ns % SK), b = ns & 1;
            const bool first = ti.j == 0;
            const int pc = piece + (first ? 1 : 0);
            bool ready = true;
            if (lane == 0) {
                ready = mbar_test_wait(&sm.full[sk], (ns / SK) & 1);
                if (ready && ns >= 2)  // the softmax has read S(ns - 2)
                    ready = mbar_test_wait(&ts.s_free[b], ((ns >> 1) - 1) & 1);
                if (ready && first)
                    ready = mbar_test_wait(&sm.q_full[0], pc & 1);
            }
            if (__shfl_sync(kFull, ready ? 1 : 0, 0)) {
                const int t0 = it.start + (ti.j << 7);
                const int n_tile = min(kTcTT, it.end - t0);
                const uint32_t st = ring_k + sk * p.stage_bytes;
                const size_t nrow = (static_cast<size_t>(it.b) * p.KV + it.kh) * p.NQ;
                if (t0 + n_tile > it.past) {
                    fix_tile(st, static_cast<const T*>(p.k_new) + nrow * kTcD, t0, n_tile, it.past, false, lane);
                    fence_proxy_async_smem();
                }
                __syncwarp();
                piece = pc;
                pend[ns & 3] = Pend{pc, first ? 1 : 0, (n_tile + 15) >> 4, t0, n_tile, it.past, nrow};
                ti.next(p, sc);
                const bool piece_end = !ti.valid() || ti.j == 0;
                if (lane == 0) {
                    tc_fence_after();
                    const uint64_t dk = smem_desc(st, 16, 1024);
#pragma unroll
                    for (int ks = 0; ks < kTcD / 16; ++ks) {
                        const uint32_t ka = (ks >> 2) * kHalfBytes + (ks & 3) * 32;
                        const uint32_t qa = (ks >> 2) * (kTcRows * 128) + (ks & 3) * 32;
                        umma(tmem + b * 64, dk + (ka >> 4), dq + (qa >> 4), id_s, ks > 0);
                    }
                    umma_commit(&ts.s_full[b]);
                    umma_commit(&sm.empty[sk]);  // the K slot
                    if (piece_end)
                        umma_commit(&sm.q_free[0]);  // the query tile
                }
                __syncwarp();
                ++ns;
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
                    bool ok2 = !*sm.abort_flag && mbar_wait_bounded(ts.pv_done, (gt - 1) & 1, p.wait_ns);
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
            // P = 2^(x - m) into registers and the row sums; then, once PV of
            // stage gt - 1 has read the P^T tile, P^T (high | remainder) of this
            // warp's rows (chunks 2h, 2h + 1 and 4 + 2h, 5 + 2h of its token row).
            // A wait that runs out skips the stage; the next barrier of the row
            // half then gives up uniformly (the abort flag is set).
            uint32_t hi[8], lo[8];
#pragma unroll
            for (int k = 0; k < 8; ++k) {
                const float p0 = fast_exp2(x[2 * k] - m[2 * k]);
                const float p1 = fast_exp2(x[2 * k + 1] - m[2 * k + 1]);
                l[2 * k] += p0;
                l[2 * k + 1] += p1;
                split_pair<T>(p0, p1, hi[k], lo[k]);
            }
            bool pv_ok = true;
            if (gt >= 1)
                pv_ok = !*sm.abort_flag && mbar_wait_bounded(ts.pv_done, (gt - 1) & 1, p.wait_ns);
            if (!__all_sync(kFull, pv_ok)) {
                if (lane == 0)
                    flag_timeout(p, sm.abort_flag);
                continue;
            }
#pragma unroll
            for (int cc = 0; cc < 2; ++cc) {
                st_shared4(prow + (((2 * h + cc) ^ swz) << 4), hi[4 * cc], hi[4 * cc + 1], hi[4 * cc + 2],
                           hi[4 * cc + 3]);
                st_shared4(prow + (((4 + 2 * h + cc) ^ swz) << 4), lo[4 * cc], lo[4 * cc + 1], lo[4 * cc + 2],
                           lo[4 * cc + 3]);
            }
            fence_proxy_async_smem();
            tc_fence_before();
            __syncwarp();
            if (lane == 0)
                mbar_arrive(ts.p_full);
        }
        if (dead)
            break;

        // ---- piece end: row sums over the 128 tokens, O, then the output
        // (whole segment) or the partial record
        const float ls = reduce_rows(l, lane, [](float a, float b) { return a + b; });
        if (lane < kWarpRows)
            ts.red_sum[(h * kWarpRows + lane) * 4 + qt] = ls;
        const uint32_t gl = gt - 1;
        bool ok = !*sm.abort_flag && mbar_wait_bounded(ts.pv_done, gl & 1, p.wait_ns);
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
                     const __grid_constant__ CUtensorMap vmap, const __grid_constant__ CUtensorMap qmap)
{
    extern __shared__ __align__(1024) unsigned char smem_raw[];
    const Smem sm = carve(p, smem_raw);
    const TcSmem ts = carve_tc(p, smem_raw);
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;

    if (warp == kMmaWarp && lane == 0)
        tma_prefetch_desc(&qmap);
    kernel_entry(p, kmap, vmap, sm);
    if (threadIdx.x == 0) {
        // K and V rings apart, each slot landing and released by one arrival;
        // one query tile, released by the MMA warp's commit
        for (int s = 0; s < p.stages; ++s)
            mbar_init(&sm.full[s], 1);
        for (int s = 0; s < p.stages_v; ++s) {
            mbar_init(&sm.full[kVRing + s], 1);
            mbar_init(&sm.empty[kVRing + s], 1);
        }
        mbar_init(&sm.q_free[0], 1);
        for (int i = 0; i < 2; ++i) {
            mbar_init(&ts.s_full[i], 1);
            mbar_init(&ts.s_free[i], kSoftWarps);
            mbar_init(&ts.o_free[i], kSoftWarps);
        }
        mbar_init(ts.p_full, kSoftWarps);
        mbar_init(ts.pv_done, 1);
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
        mma_warp<T>(p, sc, sm, ts, tmem, lane);
        // tensor memory is freed once the softmax warps are done with it
        asm volatile("bar.sync 6, %0;" ::"n"((kSoftWarps + 1) * 32) : "memory");
        tc_fence_after();
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(kTmemCols)
                     : "memory");
        return;
    }
    if (warp >= kConsumerWarps) {
        produce_tc<T>(p, sc, sm, ts, &kmap, &vmap, &qmap, warp - kConsumerWarps, lane);
        return;
    }
    // the softmax warps are the consumer warps of the split merge
    bool dep_ok = !p.early;  // see pa_mma_kernel
    int nsplit = 0;
    softmax_warps<T, TO>(p, sc, sm, ts, tmem, warp, lane, nsplit, dep_ok);
    // Without an abort every warp has seen every piece (nsplit is uniform);
    // the last PV has completed, so the P^T tile and the reduction arrays
    // serve the merge.
    tc_fence_before();
    const bool aborted = consumer_bar_or(*sm.abort_flag != 0);
    asm volatile("bar.arrive 6, %0;" ::"n"((kSoftWarps + 1) * 32) : "memory");
    if (nsplit > 0 && !aborted) {
        if (!dep_ok)
            grid_dependency_wait();
        flush_split_pieces<kTcD, TO>(p, sc, sm.split_list, nsplit, reinterpret_cast<float2*>(ts.red_max),
                                     2 * kTcRows, reinterpret_cast<float*>(ts.pbuf), kObufFloats);
    }
}

}  // namespace

SplitTcFn pick_split_tc(int dtype, bool f32_out)
{
    if (dtype == PA_BF16)
        return f32_out ? pa_umma32_kernel<__nv_bfloat16, float> : pa_umma32_kernel<__nv_bfloat16, __nv_bfloat16>;
    return f32_out ? pa_umma32_kernel<__half, float> : pa_umma32_kernel<__half, __half>;
}

}  // namespace pa
