// pa_prefill_tc.cu -- causal prefill on the sm_103a fifth-generation tensor
// cores (tcgen05: MMAs from shared-memory descriptors, accumulators in tensor
// memory), the path pa_prefill takes for 16-bit caches with D = 128.
//
// What is computed is the decode definition of onnxruntime-ep-mlx 0.31.1,
// src/ops/paged_attention.rs (VECTOR_BODY) with many new rows: new row r of
// sequence b (token past + r, past = seq_lens[b]) attends to keys
// 0 .. past + r, the cached ones through the block table and the new ones,
// which pa_prefill stores into the cache first; the engine page
// (src/engine.rs) keeps a prefill configuration next to the decode one.
//
// How: persistent CTAs, one per SM, each walking row tiles (sequence, KV
// head, 128 query rows) in turn; a tile's rows are the g = H / KV query heads
// of the KV head times T = 128 / g consecutive new rows (head-major), so that
// one K/V tile serves all of them.  Per key
// tile of 128 tokens, fetched by TMA one cache block at a time through the
// block table:
//   S  = Q K^T            M 128 (rows), N 128 (keys), K = D; A and B K-major
//   softmax               one thread per row reads its S row from tensor memory,
//                         masks keys past its causal bound, keeps the running
//                         maximum and sum, rescales its O row in tensor memory
//                         when the maximum grew, and writes P as a 16-bit high
//                         part plus a 16-bit remainder (about 22 bits of P) to
//                         shared memory;
//   O += P_hi V + P_lo V  M 128, N = D, K 128 (keys); V as an MN-major operand.
// Warps 0-7: softmax and epilogue, two threads a row (warps w and w + 4 take
// the low and the high 64 columns of tensor-memory lanes 32 (w % 4) ..; they
// exchange the row maximum of each key tile through shared memory); warps 8
// and 9: TMA producers of K and of V (three stages each; a K stage is free again
// once its S is computed, a V stage once its P.V is); warp 10: MMA issuer (one
// thread).  S
// is double-buffered in tensor memory, so that the MMA of key tile t + 1 runs
// while the softmax works on tile t.  The handshakes are mbarriers; every
// wait is bounded, and a wait that gives up reports PA_STATUS_TIMEOUT.  Tensor
// memory (512 columns: S twice, O) is allocated by warp 0 and freed on every
// path.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include <cstdint>
#include <type_traits>

#include "pa_common.cuh"
#include "pa_decode.h"
#include "pa_ptx.cuh"
#include "pa_tc.cuh"
#include "pa_tmem.cuh"

namespace pa {
namespace {

using namespace tc;

constexpr unsigned kFull = 0xffffffffu;
constexpr int kTcD = 128;           // head size of this path
constexpr int kTcTile = 128;        // query rows of a CTA tile, keys of a key tile
constexpr int kTcHalf = 16384;      // one 64-column half of a 128-row tile, bytes
constexpr int kTcSoftmax = 256;     // softmax threads (warps 0-7)
constexpr int kTcThreads = 352;     // warps 0-7 softmax, 8-9 TMA (K, V), 10 MMA
constexpr uint32_t kTcCols = 512;   // tensor-memory columns: S0 | S1 | O | (unused)
constexpr int kTcStages = 3;        // K and V rings
// Q 2 halves, K and V rings (kTcStages x 2 halves each), then the barriers
// and the row-maximum exchange; the dynamic shared-memory base must be
// 1024-aligned (checked at entry)
constexpr int kTcSmem = (2 + 4 * kTcStages) * kTcHalf + 3072;
static_assert(kTcSmem <= 232448, "prefill shared memory");

struct PrefillTcParams {
    const void* q;            // [B][H][NQ][D] (for L2 prefetches; the tiles come by TMA)
    const int32_t* table;     // [B][maxb]
    const int32_t* seq_lens;  // [B] cached tokens before the new rows
    void* out;                // [B][H][NQ][D]
    int* status;
    float qscale;             // scale * log2(e)
    int B, H, KV, NQ, BLOCK, maxb, num_blocks, g, T, tiles;  // tiles: row tiles per (b, kh)
    int total;                // row tiles in all: B * KV * tiles
};

struct TcBars {
    // s_full, p_full and o_done alternate by key-tile parity (the S buffer);
    // the K and V rings have kTcStages stages; q_empty: the row tile's S MMAs
    // are done with the query tile; o_free: its epilogue has read O
    uint64_t q_full, q_empty, o_free, fin, k_full[kTcStages], k_empty[kTcStages], v_full[kTcStages],
        v_empty[kTcStages], s_full[2], p_full[2], o_done[2];
    uint32_t tmem;
    int abort;
    float xchg[2][2][kTcTile];  // [tile parity][column half][row]: partial row maxima, then sums
};
static_assert(sizeof(TcBars) <= 3072, "barrier area");

// Row tile i of the grid's work: the last row tiles see the most keys and come
// first (the row tile is the slowest index).  Persistent CTA c of G takes the
// tiles c, 2G - 1 - c, 2G + c, 4G - 1 - c, ... in turn (a snake over that
// order, so that every CTA gets long and short tiles).
__device__ __forceinline__ int tile_of(int k, int c, int G) { return (k & 1) ? (k + 1) * G - 1 - c : k * G + c; }

struct RowTile {
    int b, kh, r_base, r_last, past, end, ntiles;
};

__device__ __forceinline__ RowTile row_tile(const PrefillTcParams& p, int i, int tid)
{
    RowTile rt;
    const int t = p.tiles - 1 - i / (p.B * p.KV);
    rt.kh = (i % (p.B * p.KV)) % p.KV;
    rt.b = (i % (p.B * p.KV)) / p.KV;
    rt.r_base = t * p.T;
    rt.r_last = min(rt.r_base + p.T, p.NQ) - 1;  // last new row of the tile
    const int cap = p.maxb * p.BLOCK - p.NQ;      // largest past the table can hold
    int past = p.seq_lens[rt.b];
    if (past < 0 || past > cap) {
        if (tid == 0 && t == 0 && rt.kh == 0 && p.status)
            atomicOr(p.status, PA_STATUS_BAD_LENGTH);
        past = past < 0 ? 0 : (cap < 0 ? 0 : cap);
    }
    rt.past = past;
    rt.end = past + p.NQ;                                          // keys of the sequence
    rt.ntiles = (past + rt.r_last + 1 + kTcTile - 1) / kTcTile;  // keys 0 .. past + r_last
    return rt;
}

template <typename T, typename TO>
__global__ void __launch_bounds__(kTcThreads, 1)
    pa_prefill_tc_kernel(const __grid_constant__ PrefillTcParams p, const __grid_constant__ CUtensorMap qmap,
                         const __grid_constant__ CUtensorMap kmap, const __grid_constant__ CUtensorMap vmap)
{
    constexpr bool kBf = std::is_same<T, __nv_bfloat16>::value;
    extern __shared__ __align__(1024) unsigned char smem_raw[];
    if ((smem_u32(smem_raw) & 1023u) != 0) {  // the layout leaves no room to realign
        if (threadIdx.x == 0 && p.status)
            atomicOr(p.status, PA_STATUS_TIMEOUT);
        return;
    }
    unsigned char* base = smem_raw;
    unsigned char* sQ = base;                                // 2 halves
    unsigned char* sK = base + 2 * kTcHalf;                  // kTcStages x 2 halves
    unsigned char* sV = base + (2 + 2 * kTcStages) * kTcHalf;  // kTcStages x 2 halves
    TcBars& bars = *reinterpret_cast<TcBars*>(base + (2 + 4 * kTcStages) * kTcHalf);

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int C = blockIdx.x, G = gridDim.x;

    if (tid == 0) {
        mbar_init(&bars.q_full, 1);
        mbar_init(&bars.q_empty, 1);
        mbar_init(&bars.o_free, kTcSoftmax / 32);  // one arrival per softmax warp
        mbar_init(&bars.fin, 1);
        for (int s = 0; s < kTcStages; ++s) {
            mbar_init(&bars.k_full[s], 1);
            mbar_init(&bars.k_empty[s], 1);
            mbar_init(&bars.v_full[s], 1);
            mbar_init(&bars.v_empty[s], 1);
        }
        for (int s = 0; s < 2; ++s) {
            mbar_init(&bars.s_full[s], 1);
            mbar_init(&bars.p_full[s], kTcSoftmax / 32);  // one arrival per softmax warp
            mbar_init(&bars.o_done[s], 1);
        }
        bars.abort = 0;
        fence_mbar_init();
    }
    if (warp == 0) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                         smem_u32(&bars.tmem)),
                     "r"(kTcCols)
                     : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    // S(t) at tS0 + 128 (t & 1); P(t) overwrites it as 16-bit pairs (see the softmax)
    const uint32_t tS0 = bars.tmem, tO = bars.tmem + 2 * kTcTile;
    volatile int* abort_flag = &bars.abort;
    auto fail = [&]() {
        *abort_flag = 1;
        if (p.status)
            atomicOr(p.status, PA_STATUS_TIMEOUT);
    };
    // Key tiles are counted over all of this CTA's row tiles (g below): the
    // rings, S buffers and their barriers run on across row tiles.

    if (warp == 8 || warp == 9) {
        // ----------------------------------------------------------- TMA producers
        // Warp 8 issues the K boxes (and each row tile's q, once the previous
        // row tile's S MMAs are done with the query tile), warp 9 the V boxes:
        // lane k the boxes (both 64-column halves) of cache block k of each
        // key tile; the table entries of the next tile are loaded while the
        // current one is in flight.
        const bool is_v = warp == 9;
        const CUtensorMap* map = is_v ? &vmap : &kmap;
        unsigned char* ring = is_v ? sV : sK;
        uint64_t* full = is_v ? bars.v_full : bars.k_full;
        uint64_t* empty = is_v ? bars.v_empty : bars.k_empty;
        const int boxes = kTcTile / p.BLOCK;
        if (lane == 0) {
            tma_prefetch_desc(map);
            if (!is_v)
                tma_prefetch_desc(&qmap);
        }
        int issued = 0, q_issued = 0;  // key tiles, query tiles
        bool ok = true;
        for (int k = 0; ok; ++k) {
            const int i = tile_of(k, C, G);
            if (i >= p.total)
                break;
            const RowTile rt = row_tile(p, i, tid);
            if (!is_v) {
                if (q_issued > 0) {
                    ok = !*abort_flag && mbar_wait_bounded(&bars.q_empty, (q_issued - 1) & 1, kWaitLimitNs);
                    ok = __all_sync(kFull, ok);
                    if (!ok) {
                        if (lane == 0)
                            fail();
                        break;
                    }
                }
                if (lane == 0) {
                    mbar_arrive_expect_tx(&bars.q_full, 2 * kTcHalf);
                    for (int h = 0; h < 2; ++h)
                        tma_load_5d(sQ + h * kTcHalf, &qmap, 0, h, rt.r_base, rt.kh * p.g, rt.b, &bars.q_full);
                }
                ++q_issued;
                // the next row tile's query rows into L2 (its load waits for
                // this tile's S MMAs): g heads x T rows of 256 bytes, 128-byte lines
                const int i_next = tile_of(k + 1, C, G);
                if (i_next < p.total) {
                    const int t_n = p.tiles - 1 - i_next / (p.B * p.KV);
                    const int kh_n = (i_next % (p.B * p.KV)) % p.KV, b_n = (i_next % (p.B * p.KV)) / p.KV;
                    const int rows = min(p.T, p.NQ - t_n * p.T);
                    const char* q0 = static_cast<const char*>(p.q) +
                                     ((static_cast<size_t>(b_n) * p.H + kh_n * p.g) * p.NQ + t_n * p.T) * (kTcD * 2);
                    for (int idx = lane; idx < p.g * rows * 2; idx += 32) {
                        const int hh = idx / (rows * 2), w = idx - hh * rows * 2;
                        asm volatile("prefetch.global.L2 [%0];" ::"l"(q0 + static_cast<size_t>(hh) * p.NQ * (kTcD * 2) +
                                                                      w * 128));
                    }
                }
            }
            auto entry = [&](int t) {  // cache row of this lane's block in tile t, or out of range
                const int tok = t * kTcTile + lane * p.BLOCK;
                const int blk = tok / p.BLOCK;
                int row0 = p.num_blocks * p.BLOCK;  // past the pool: the box reads zeros
                if (lane < boxes && t < rt.ntiles && tok < rt.end && blk < p.maxb) {
                    const int phys = p.table[static_cast<size_t>(rt.b) * p.maxb + blk];
                    if (phys >= 0 && phys < p.num_blocks)
                        row0 = phys * p.BLOCK;
                }
                return row0;
            };
            int row_next = entry(0);
            // launched as a programmatic dependent of the store of the new rows:
            // the cache is read only once that grid has completed
            if (k == 0)
                grid_dependency_wait();
            for (int t = 0; t < rt.ntiles; ++t) {
                const int g = issued, s = g % kTcStages;
                const int row0 = row_next;
                if (g >= kTcStages) {
                    ok = !*abort_flag && mbar_wait_bounded(&empty[s], ((g / kTcStages) - 1) & 1, kWaitLimitNs);
                    ok = __all_sync(kFull, ok);
                    if (!ok) {
                        if (lane == 0)
                            fail();
                        break;
                    }
                }
                if (lane == 0)
                    mbar_arrive_expect_tx(&full[s], 2 * kTcHalf);
                __syncwarp();
                if (lane < boxes)
                    for (int h = 0; h < 2; ++h)
                        tma_load_4d(ring + s * 2 * kTcHalf + h * kTcHalf + lane * p.BLOCK * 128, map, 0, h, rt.kh,
                                    row0, &full[s]);
                issued = g + 1;
                row_next = entry(t + 1);
            }
        }
        // no copy may land after the CTA's memory is released: wait (bounded)
        // for the last tile issued on each stage (and for q)
        if (lane == 0) {
            for (int t = issued > kTcStages ? issued - kTcStages : 0; t < issued; ++t)
                mbar_wait_bounded(&full[t % kTcStages], (t / kTcStages) & 1, kWaitLimitNs);
            if (!is_v && q_issued > 0)
                mbar_wait_bounded(&bars.q_full, (q_issued - 1) & 1, kWaitLimitNs);
        }
        __syncwarp();
    } else if (warp == 10) {
        // -------------------------------------------------------------- MMA issuer
        // Over the key tiles of all row tiles in order: S of key tile g + 1
        // (possibly of the next row tile, once its query tile has landed), then
        // P(g).V.  S(g + 1) goes into the S buffer that held P(g - 1): P(g - 1).V
        // was issued before it by this thread, and the MMAs of one thread run in
        // order, so a commit of S(g + 1) also covers P(g - 1).V.  After a row
        // tile's last S the query tile is committed free; before its first P.V,
        // the previous row tile's epilogue must have read O.
        if (lane == 0) {
            const uint32_t qa = smem_u32(sQ), ka = smem_u32(sK), va = smem_u32(sV);
            const uint32_t id_s = idesc<kBf>(kTcTile, false), id_o = idesc<kBf>(kTcD, true);
            // the S cursor (row tile k_s of this CTA, its key tile u_s, global g_s)
            // runs one key tile ahead of the P.V cursor
            int k_s = 0, u_s = 0, g_s = 0;
            RowTile rt_s{};
            bool s_valid = tile_of(0, C, G) < p.total;
            if (s_valid)
                rt_s = row_tile(p, tile_of(0, C, G), tid);
            bool ok = true;
            auto issue_s = [&]() {  // S(g_s) = Q K(g_s)^T, then the cursor moves on
                const int ku = g_s % kTcStages;
                if (u_s == 0 && (*abort_flag || !mbar_wait_bounded(&bars.q_full, k_s & 1, kWaitLimitNs)))
                    return false;
                if (*abort_flag || !mbar_wait_bounded(&bars.k_full[ku], (g_s / kTcStages) & 1, kWaitLimitNs))
                    return false;
                tc_fence_after();
                for (int ks = 0; ks < kTcD / 16; ++ks) {
                    const uint32_t o = (ks >> 2) * kTcHalf + (ks & 3) * 32;
                    umma(tS0 + (g_s & 1) * kTcTile, smem_desc(qa + o, 16, 1024),
                         smem_desc(ka + ku * 2 * kTcHalf + o, 16, 1024), id_s, ks > 0);
                }
                umma_commit(&bars.s_full[g_s & 1]);
                umma_commit(&bars.k_empty[ku]);
                ++g_s;
                if (++u_s == rt_s.ntiles) {
                    umma_commit(&bars.q_empty);  // the query tile, once these S are done
                    u_s = 0;
                    ++k_s;
                    const int i = tile_of(k_s, C, G);
                    s_valid = i < p.total;
                    if (s_valid)
                        rt_s = row_tile(p, i, tid);
                }
                return true;
            };
            if (s_valid)
                ok = issue_s();
            int g = 0;
            for (int k = 0; ok; ++k) {
                const int i = tile_of(k, C, G);
                if (i >= p.total)
                    break;
                const RowTile rt = row_tile(p, i, tid);
                for (int t = 0; t < rt.ntiles && ok; ++t, ++g) {
                    const int sb = g & 1, vs = g % kTcStages;
                    if (s_valid && !issue_s()) {
                        ok = false;
                        break;
                    }
                    ok = mbar_wait_bounded(&bars.p_full[sb], (g >> 1) & 1, kWaitLimitNs);
                    if (ok)
                        ok = mbar_wait_bounded(&bars.v_full[vs], (g / kTcStages) & 1, kWaitLimitNs);
                    if (ok && t == 0 && k > 0)
                        ok = mbar_wait_bounded(&bars.o_free, (k - 1) & 1, kWaitLimitNs);
                    if (!ok)
                        break;
                    tc_fence_after();
                    // O += P_hi V + P_lo V over the tile's keys.  P from tensor memory:
                    // keys 64 h + 16 j + (0 .. 15) of the high part at column
                    // 64 h + 8 j of the S buffer, the remainder 32 columns further;
                    // V is MN-major (its rows are keys, 64 columns of D per half, the
                    // halves 16 KB apart)
                    const uint32_t tP = tS0 + sb * kTcTile;
                    for (int part = 0; part < 2; ++part)
                        for (int ks = 0; ks < kTcTile / 16; ++ks) {
                            const uint32_t pcol = (ks >> 2) * 64 + part * 32 + (ks & 3) * 8;
                            umma_ts(tO, tP + pcol, smem_desc(va + vs * 2 * kTcHalf + ks * 2048, kTcHalf, 1024),
                                    id_o, t > 0 || part > 0 || ks > 0);
                        }
                    umma_commit(&bars.o_done[sb]);
                    umma_commit(&bars.v_empty[vs]);
                }
            }
            if (!ok)
                fail();
            // every MMA complete before the tensor memory is freed
            umma_commit(&bars.fin);
            mbar_wait_bounded(&bars.fin, 0, kWaitLimitNs);
        }
        __syncwarp();
    } else {
        // ---------------------------------------------- softmax and epilogue (rows)
        const int row = (warp & 3) * 32 + lane;  // tile row = tensor-memory lane
        const int part = warp >> 2;              // key columns [64 part, 64 part + 64)
        const uint32_t lane_off = static_cast<uint32_t>((warp & 3) * 32) << 16;
        const uint32_t col0 = part * 64;
        const int pair_bar = 1 + (warp & 3);  // named barrier of warps w, w + 4
        const int hg = row / p.T, tt = row - hg * p.T;
        int g0 = 0;  // key tiles of this CTA's earlier row tiles
        bool ok = true;
        for (int k = 0; ok; ++k) {
            const int i = tile_of(k, C, G);
            if (i >= p.total)
                break;
            const RowTile rt = row_tile(p, i, tid);
            const int r = rt.r_base + tt;
            const bool real = r < p.NQ;
            const int limit = rt.past + r;  // last visible key
            // m: the maximum the exponentials are taken against (the running
            // maximum, moved only when the maximum grows by more than 2^8: P stays
            // at most 256, and O / l is the same for any reference); l: this
            // thread's share of the sum
            float m = -INFINITY, l = 0.f;
            const int vis = rt.past + rt.r_base;  // every row of the tile sees keys 0 .. vis
            // The two warps of a row meet at one barrier per tile (the maximum
            // exchange), and leave the loop only there, together: a wait that gave
            // up (`fault`, warp-uniform) is OR-ed into that barrier.
            bool fault = false;
            for (int t = 0; t < rt.ntiles; ++t) {
                const int g = g0 + t, s = g & 1;
                const bool got = __all_sync(kFull, !fault && !*abort_flag &&
                                                       mbar_wait_bounded(&bars.s_full[s], (g >> 1) & 1, kWaitLimitNs));
                float sc[64];
                float pm = -INFINITY;
                if (got) {
                    tc_fence_after();
                    // both halves of this thread's score columns in flight together;
                    // eight independent partial maxima keep the chains short
                    Cols32 xs[2];
                    tmem_ld32_issue(xs[0], tS0 + s * kTcTile + lane_off + col0);
                    tmem_ld32_issue(xs[1], tS0 + s * kTcTile + lane_off + col0 + 32);
                    tmem_ld_wait(xs[1]);
                    tmem_ld_wait(xs[0]);
                    float pm8[8];
#pragma unroll
                    for (int e = 0; e < 8; ++e)
                        pm8[e] = -INFINITY;
                    if (t * kTcTile + kTcTile - 1 > vis) {  // masked tile, uniform over the CTA
                        const int lim = limit - (t * kTcTile + col0);  // columns 0 .. lim visible
#pragma unroll
                        for (int c = 0; c < 2; ++c)
#pragma unroll
                            for (int j = 0; j < 32; ++j) {
                                const float v = c * 32 + j <= lim ? __uint_as_float(xs[c].r[j]) * p.qscale : -INFINITY;
                                sc[c * 32 + j] = v;
                                pm8[j & 7] = fmaxf(pm8[j & 7], v);
                            }
                    } else {
#pragma unroll
                        for (int c = 0; c < 2; ++c)
#pragma unroll
                            for (int j = 0; j < 32; ++j) {
                                const float v = __uint_as_float(xs[c].r[j]) * p.qscale;
                                sc[c * 32 + j] = v;
                                pm8[j & 7] = fmaxf(pm8[j & 7], v);
                            }
                    }
                    pm = fmaxf(fmaxf(fmaxf(pm8[0], pm8[1]), fmaxf(pm8[2], pm8[3])),
                               fmaxf(fmaxf(pm8[4], pm8[5]), fmaxf(pm8[6], pm8[7])));
                }
                // the other half of the row's maximum
                bars.xchg[s][part][row] = pm;
                if (pair_bar_or(pair_bar, !got)) {
                    ok = false;
                    break;
                }
                const float tile_max = fmaxf(pm, bars.xchg[s][part ^ 1][row]);
                // both threads of the row take the same decision from the same values
                const float mt = tile_max > m + 8.f ? tile_max : m;
                const float alpha = fast_exp2(m - mt);  // 0 at the first tile (m = -inf), else 1 or tiny
                float s8[8];
#pragma unroll
                for (int e = 0; e < 8; ++e)
                    s8[e] = 0.f;
#pragma unroll
                for (int j = 0; j < 64; ++j) {
                    sc[j] = fast_exp2(sc[j] - mt);
                    s8[j & 7] += sc[j];
                }
                const float sum = ((s8[0] + s8[1]) + (s8[2] + s8[3])) + ((s8[4] + s8[5]) + (s8[6] + s8[7]));
                l = l * alpha + sum;
                m = mt;
                // keys past the sequence end inside its last cache block hold other
                // data (not finite for certain): their V rows are zeroed, since
                // P = 0 does not cancel a non-finite value in the MMA
                const int tok = t * kTcTile + row;
                if (t * kTcTile + kTcTile > rt.end) {  // uniform over the CTA
                    // the V stage has landed; the wait orders these stores after the
                    // copy's writes (and they come before p_full, which P.V waits for)
                    const int vs = g % kTcStages;
                    const bool landed = __all_sync(
                        kFull, mbar_wait_bounded(&bars.v_full[vs], (g / kTcStages) & 1, kWaitLimitNs));
                    fault |= !landed;
                    if (landed && tok >= rt.end) {
                        uint4* vrow = reinterpret_cast<uint4*>(sV + vs * 2 * kTcHalf + part * kTcHalf + row * 128);
#pragma unroll
                        for (int c = 0; c < 8; ++c)
                            vrow[c] = make_uint4(0u, 0u, 0u, 0u);
                    }
                }
                // O is rescaled only when a row maximum moved (warp-uniform: tcgen05
                // ld/st are warp-wide), after P(g - 1).V has completed
                if (t > 0 && __any_sync(kFull, alpha != 1.f)) {
                    const bool done = __all_sync(
                        kFull, !fault && mbar_wait_bounded(&bars.o_done[(g - 1) & 1], ((g - 1) >> 1) & 1,
                                                           kWaitLimitNs));
                    fault |= !done;
                    if (done) {
                        tc_fence_after();
#pragma unroll
                        for (int c = 0; c < 2; ++c) {
                            Cols32 x;
                            tmem_ld32(x, tO + lane_off + col0 + c * 32);
#pragma unroll
                            for (int j = 0; j < 32; ++j)
                                x.r[j] = __float_as_uint(__uint_as_float(x.r[j]) * alpha);
                            tmem_st32(x, tO + lane_off + col0 + c * 32);
                        }
                    }
                }
                // P as high part + remainder, packed 16-bit pairs, over this thread's
                // own S columns (it has read them): keys 64 part + 2 e, 2 e + 1 of the
                // high part at column 64 part + e, of the remainder at 64 part + 32 + e.
                // S(g) was committed after P(g - 2).V, so that product is complete.
                {
                    Cols32 hi, lo;
#pragma unroll
                    for (int e = 0; e < 32; ++e)
                        split_pair<T>(sc[2 * e], sc[2 * e + 1], hi.r[e], lo.r[e]);
                    tmem_st32(hi, tS0 + s * kTcTile + lane_off + col0);
                    tmem_st32(lo, tS0 + s * kTcTile + lane_off + col0 + 32);
                    asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
                }
                fence_proxy_async_smem();  // the zeroed V rows
                tc_fence_before();
                __syncwarp();
                if (lane == 0)
                    mbar_arrive(&bars.p_full[s]);
            }
            const int gl = g0 + rt.ntiles - 1;  // the row tile's last key tile
            if (ok)
                ok = __all_sync(kFull, !fault && mbar_wait_bounded(&bars.o_done[gl & 1], (gl >> 1) & 1,
                                                                   kWaitLimitNs));
            // the row sum over both halves, through the exchange slots of parity
            // gl + 1: the partner's last read of them came before the last tile's
            // barrier; a second barrier after the reads keeps the next row tile's
            // first maximum exchange (the same slots) behind them.  Both warps of
            // the row take the decision to go on together (the OR of a failure).
            const int sl = (gl + 1) & 1;
            if (ok)
                bars.xchg[sl][part][row] = l;
            if (pair_bar_or(pair_bar, !ok)) {
                if (!ok && lane == 0)
                    fail();
                ok = false;
                break;
            }
            tc_fence_after();
            const float L = l + bars.xchg[sl][part ^ 1][row];
            const int h = rt.kh * p.g + hg;
            TO* o = static_cast<TO*>(p.out) + ((static_cast<size_t>(rt.b) * p.H + h) * p.NQ + r) * kTcD + col0;
            const float inv = L > 0.f ? 1.f / L : 0.f;
#pragma unroll
            for (int c = 0; c < 2; ++c) {
                Cols32 x;
                tmem_ld32(x, tO + lane_off + col0 + c * 32);
                float v[32];
#pragma unroll
                for (int j = 0; j < 32; ++j)
                    v[j] = __uint_as_float(x.r[j]) * inv;
                if (real)
                    store_row<TO>(o + c * 32, v);
            }
            // O is free for the next row tile's first P.V
            tc_fence_before();
            __syncwarp();
            if (lane == 0)
                mbar_arrive(&bars.o_free);
            asm volatile("bar.sync %0, 64;" ::"r"(pair_bar) : "memory");
            g0 += rt.ntiles;
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 0)
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(bars.tmem), "r"(kTcCols)
                     : "memory");
}

using PrefillTcFn = void (*)(PrefillTcParams, CUtensorMap, CUtensorMap, CUtensorMap);

PrefillTcFn pick_prefill_tc(int dtype, bool f32_out)
{
    if (dtype == PA_BF16)
        return f32_out ? pa_prefill_tc_kernel<__nv_bfloat16, float>
                       : pa_prefill_tc_kernel<__nv_bfloat16, __nv_bfloat16>;
    return f32_out ? pa_prefill_tc_kernel<__half, float> : pa_prefill_tc_kernel<__half, __half>;
}

}  // namespace

bool prefill_tc_supported(int dtype, int D, int H, int KV, int NQ)
{
    const int g = H / KV;
    return (dtype == PA_F16 || dtype == PA_BF16) && D == kTcD && g >= 1 && g <= kTcTile &&
           kTcTile % g == 0 && NQ > PA_MAX_NQ;
}

// Enqueues the tensor-core prefill on `st` (the new rows must already be in
// the cache).  Returns PA_OK or a PA_ERR_* code before any launch.
int launch_prefill_tc(const void* q, const void* k_cache, const void* v_cache, const int32_t* table,
                      const int32_t* seq_lens, void* out, float scale, int B, int H, int KV, int BLOCK,
                      int NQ, int maxb, int num_blocks, int dtype, int out_dtype, int* status,
                      cudaStream_t st, uint64_t* launches)
{
    auto enc = tc_encoder();
    if (!enc)
        return PA_ERR_DRIVER;
    const int g = H / KV, T = kTcTile / g;
    const CUtensorMapDataType dt =
        dtype == PA_BF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16;
    CUtensorMap qmap, kmap, vmap;
    {
        // q [B][H][NQ][D] as {64, 2, NQ, H, B}; box {64, 1, T, g, 1}: one
        // 64-column half of the tile's 128 rows (g heads x T new rows)
        cuuint64_t dims[5] = {64u, 2u, static_cast<cuuint64_t>(NQ), static_cast<cuuint64_t>(H),
                              static_cast<cuuint64_t>(B)};
        cuuint64_t str[4] = {128u, kTcD * 2u, static_cast<cuuint64_t>(NQ) * kTcD * 2,
                             static_cast<cuuint64_t>(H) * NQ * kTcD * 2};
        cuuint32_t box[5] = {64u, 1u, static_cast<cuuint32_t>(T), static_cast<cuuint32_t>(g), 1u};
        cuuint32_t es[5] = {1u, 1u, 1u, 1u, 1u};
        if (enc(&qmap, dt, 5, const_cast<void*>(q), dims, str, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE,
                CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_128B,
                CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
            return PA_ERR_CUDA;
    }
    for (int w = 0; w < 2; ++w) {
        // caches [rows][KV][D] as {64, 2, KV, rows}; box {64, 1, 1, BLOCK}: one
        // half of one cache block of one KV head
        cuuint64_t dims[4] = {64u, 2u, static_cast<cuuint64_t>(KV),
                              static_cast<cuuint64_t>(num_blocks) * BLOCK};
        cuuint64_t str[3] = {128u, kTcD * 2u, static_cast<cuuint64_t>(KV) * kTcD * 2};
        cuuint32_t box[4] = {64u, 1u, 1u, static_cast<cuuint32_t>(BLOCK)};
        cuuint32_t es[4] = {1u, 1u, 1u, 1u};
        if (enc(w ? &vmap : &kmap, dt, 4, const_cast<void*>(w ? v_cache : k_cache), dims, str, box, es,
                CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
            return PA_ERR_CUDA;
    }
    PrefillTcParams prm{};
    prm.q = q;
    prm.table = table;
    prm.seq_lens = seq_lens;
    prm.out = out;
    prm.status = status;
    prm.qscale = scale * kLog2e;
    prm.B = B;
    prm.H = H;
    prm.KV = KV;
    prm.NQ = NQ;
    prm.BLOCK = BLOCK;
    prm.maxb = maxb;
    prm.num_blocks = num_blocks;
    prm.g = g;
    prm.T = T;
    prm.tiles = (NQ + T - 1) / T;
    const PrefillTcFn fn = pick_prefill_tc(dtype, out_dtype == PA_F32);
    if (cudaFuncSetAttribute(reinterpret_cast<const void*>(fn), cudaFuncAttributeMaxDynamicSharedMemorySize,
                             kTcSmem) != cudaSuccess)
        return PA_ERR_CUDA;
    const long long total = static_cast<long long>(B) * KV * prm.tiles;
    if (total >= (1ll << 31) / 4)
        return PA_ERR_BAD_DIMS;
    prm.total = static_cast<int>(total);
    // persistent: one CTA per SM (shared and tensor memory allow no more)
    static int sms = 0;
    if (sms == 0) {
        int dev = 0;
        if (cudaGetDevice(&dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || sms < 1)
            return PA_ERR_CUDA;
    }
    const long long grid = total < sms ? total : sms;
    // programmatic dependent launch: the CTAs set up (barriers, tensor memory,
    // the query tile) while the store of the new rows finishes; the TMA
    // producers wait for it before reading the cache
    cudaLaunchConfig_t cfg{};
    cfg.gridDim = dim3(static_cast<unsigned>(grid));
    cfg.blockDim = dim3(kTcThreads);
    cfg.dynamicSmemBytes = kTcSmem;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    if (cudaLaunchKernelEx(&cfg, fn, prm, qmap, kmap, vmap) != cudaSuccess)
        return PA_ERR_CUDA;
    if (launches)
        ++*launches;
    return PA_OK;
}

}  // namespace pa
