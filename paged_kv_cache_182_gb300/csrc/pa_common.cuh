// pa_common.cuh -- constants and launch-parameter blocks shared by the host
// launcher (pa_host.cu) and the kernel instantiations (pa_inst_*.cu).
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>

#include <cstdint>

namespace pa {

constexpr int kConsumerWarps = 8;                     // compute warps per CTA
constexpr int kProducerWarps = 2;                     // TMA issue: K (+ query, new rows), V
constexpr int kThreads = (kConsumerWarps + kProducerWarps) * 32;
constexpr int kMaxStages = 32;                        // shared-memory ring depth limit
constexpr int kMinRing = 3;                           // stages kept before widening scratch
constexpr int kSubBatch = 4;        // token steps per online-softmax update
constexpr int kStageBytes = 32768;     // CUDA-core path: K + V tile bytes per stage (target)
constexpr int kMmaStageBytes = 65536;  // tensor-core path: K + V tile bytes per stage (target)
constexpr int kHeaderBytes = 3584;  // barriers, scalars, zero row, table entries, split list
constexpr int kMaxBatch = 4096;     // sequences per call (the schedule lives in smem)
constexpr int kMaxGrid = 1024;      // partition-kernel CTAs at most (sizes the workspace)
constexpr int kPieceStages = 1;   // automatic schedule: stages charged per segment
constexpr int kPieceStages2 = 6;  // the same with two 16-row groups per CTA pass
constexpr long long kMinCtaCost = 4;  // automatic schedule: stages of cost a CTA takes at least
constexpr long long kMergeStages = 4;  // automatic schedule: what the in-kernel merge of a split
                                       // segment costs its last CTA, in stages (measured)

// Automatic schedule with the in-kernel merge: whole segments, one per CTA
// (none split, nothing merged), when the S segments are no more than the G
// CTAs the split would use and the longest, max_units stages, is at most a
// CTA's share of the W real stages plus the merge that a split costs.
__host__ __device__ inline bool whole_segments(long long S, long long G, long long W, long long max_units)
{
    return S <= G && max_units * G <= W + kMergeStages * G;
}

// CTAs of `grid` that the automatic schedule gives units to, for total cost C
// over `segments` segments: every CTA at least kMinCtaCost stages of cost (a
// short batch is not cut into pieces whose merges cost more than their work),
// unless there are more segments than that, and never more than C (so that
// every CTA inside a segment holds a unit of it).
__host__ __device__ inline int active_ctas(long long grid, long long C, long long segments)
{
    long long want = (C + kMinCtaCost - 1) / kMinCtaCost;
    if (want < segments)
        want = segments;
    if (want > C)
        want = C;
    return static_cast<int>(grid < want ? grid : want);
}
constexpr uint64_t kWaitLimitNs = 2000000000ull;
constexpr float kLog2e = 1.4426950408889634f;

struct SplitParams {
    const void* q;
    const void* k_new;
    const void* v_new;
    void* out;
    const int32_t* table;
    const int32_t* seq_lens;
    int2* sched;    // [B] (prefix, count) for the merge kernel, or NULL for one pass
    int* counters;  // [B * NRS * KV] finished pieces per split segment (in-kernel merge), or NULL
    float2* ws_ml;  // [items][row_stride] (max, sum) in base-2 units
    float* ws_o;    // [items][row_stride][D]
    int* status;
    float qscale;   // scale * log2(e)
    int B, H, KV, NQ, BLOCK, maxb, num_blocks;
    int causal, partitions, checked;
    int qbuf_off;      // tensor-core kernel: scratch offset of the two query-row buffers
    int box_rows;      // rows of one TMA box (cache tokens); divides BLOCK and TT
    int empty_count;   // consumer warps that release each stage
    int R;             // query rows per KV head = (H / KV) * NQ
    int rows_per_cta;  // kConsumerWarps * RG
    int NRS;           // row groups per KV head = ceil(R / rows_per_cta)
    int TT;            // tokens per pipeline stage, a multiple of BLOCK
    int lg_block, lg_box, lg_tt;  // log2 of BLOCK, box_rows and TT (all powers of two)
    int vunits;        // automatic schedule: virtual units charged per segment
    int row_stride;    // workspace rows per item = min(R, rows_per_cta)
    int stages;        // ring depth (<= kMaxStages)
    int stage_bytes;   // bytes of one stage: K tile | K new rows | V tile | V new rows
    int knew_off;      // byte offsets of the parts within a stage (1024-aligned)
    int v_off;
    int vnew_off;
    int lens_off;      // shared-memory byte offsets from the 1024-aligned base
    int prefix_off;
    int merge_off;
    int stage_off;
    unsigned long long wait_ns;  // limit of every mbarrier wait
    int withhold;      // test switch: each CTA's V producer leaves its stage withhold - 1 out (0: off)
    int early;         // 1: the inputs are read before the grid-dependency wait (see pa_opts)
    int tc_off;        // tcgen05 kernel: byte offset of its region (P, Q, barriers) from the base
    int stages_v;      // tcgen05 kernel: V ring depth (stages: the K ring's; stage_bytes: one tile)
};

struct CombineParams {
    const int2* sched;
    const float2* ws_ml;
    const float* ws_o;
    void* out;
    int B, KV, R, NRS, rows_per_cta, row_stride;
    int stream;  // automatic (balanced) schedule: records are per partition-kernel CTA
    int grid;    // partition-kernel CTAs (automatic schedule)
    int vunits;  // automatic schedule: virtual units charged per segment
    // fixed partitions: the partition count of a segment follows from its length
    const int32_t* seq_lens;
    int partitions, NQ, BLOCK, cap;  // cap = max_blocks * BLOCK (length clamp)
};

using SplitFn = void (*)(SplitParams, CUtensorMap, CUtensorMap);
using SplitTcFn = void (*)(SplitParams, CUtensorMap, CUtensorMap, CUtensorMap);  // + the query map
using CombineFn = void (*)(CombineParams);

// Kernel tables, one per input element type (pa_inst_*.cu).  float32 inputs
// use the CUDA-core kernel (RG query rows per warp); 16-bit inputs use the
// tensor-core kernel (16 * MT query rows per CTA pass).
constexpr int kMmaTokens = 16;  // tokens of one MMA group of the tensor-core kernel
// 16-token groups a consumer warp takes per stage (two at D = 64 or with two
// 16-row groups per pass: 64 KB stages and two independent MMA chains per warp)
__host__ __device__ constexpr int mma_token_groups(int D, int MT) { return D == 64 || MT == 2 ? 2 : 1; }
constexpr int kObufFloats = 4096;  // tensor-core kernel: floats of the piece-end merge buffer
// Bytes per query row in the tensor-core kernels' query buffers: the row plus
// 16 bytes, so that the 8 rows an ldmatrix reads at once fall in 8 different
// bank groups (a 128- or 256-byte stride puts them all in one).
__host__ __device__ constexpr int q_row_bytes(int D) { return D * 2 + 16; }
SplitFn pick_split_f32(int D, int RG);
SplitFn pick_split_f16(bool f32_out, int D, int MT);
SplitFn pick_split_bf16(bool f32_out, int D, int MT);
// Tensor-core prefill (pa_prefill_tc.cu): whether a prefill of these sizes
// takes it, and its launch (the new rows already stored in the cache).
bool prefill_tc_supported(int dtype, int D, int H, int KV, int NQ);
int launch_prefill_tc(const void* q, const void* k_cache, const void* v_cache, const int32_t* table,
                      const int32_t* seq_lens, void* out, float scale, int B, int H, int KV, int BLOCK,
                      int NQ, int maxb, int num_blocks, int dtype, int out_dtype, int* status,
                      cudaStream_t st, uint64_t* launches);
// tcgen05 partition kernel for 32 query rows per pass at D = 128
// (pa_decode_tc.cu): its shared region's bytes (P^T and query tiles,
// barriers, reductions), one K or V tile's bytes, its threads, and the kernel
// of a type pair.
constexpr int kTcRegionBytes = 26624;
constexpr int kTcTileBytes = 32768;
constexpr int kUmmaThreads = kThreads + 32;  // one more warp: the MMA issuer
SplitTcFn pick_split_tc(int dtype, bool f32_out);
CombineFn pick_combine_f32(int D);
CombineFn pick_combine_f16(int D);
CombineFn pick_combine_bf16(int D);

}  // namespace pa
