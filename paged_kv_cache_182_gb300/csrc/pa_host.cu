// pa_host.cu -- host side of libpadecode.so: argument validation, workspace
// layout, tensor-map encoding, kernel choice and launch, and the C ABI of
// include/pa_decode.h.
//
// The launch arguments mirror fn vector of onnxruntime-ep-mlx 0.31.1,
// src/ops/paged_attention.rs (heads, kv_heads, head, block, max_blocks,
// batch, queries, causal, scale, and a partition count); the batch, the
// table stride and the pool size cross the boundary as values instead of
// template constants, and the workspace is caller-owned.
//
// Also here: the cache append kernel, the slot-patched decode (append, then
// decode), the host-buffer entry (gather kernel or copies, decode, copy back)
// and the chunked prefill (store of the new rows, then 16-row chunk decodes
// through staging).

#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>

#include <atomic>
#include <climits>
#include <cmath>
#include <cstdint>
#include <mutex>

#include "pa_common.cuh"
#include "pa_decode.h"
#include "pa_vjp.cuh"

namespace pa {
namespace {

std::atomic<uint64_t> g_launches{0};

size_t elem_size(int dtype) { return dtype == PA_F32 ? 4 : 2; }

// CUDA-core path (float32): query rows per consumer warp, 4 up to 32 rows
// per KV head, else 8; a CTA pass covers kConsumerWarps * RG rows.
int rows_group(int R) { return R <= 32 ? 4 : 8; }

// Tensor-core path (16-bit): 0 = the transposed kernel (at most 8 rows per
// pass, the MMA's 16-row side on the tokens), else 16-row MMA tiles per pass.
int mma_tiles(int R) { return R <= 8 ? 0 : R <= 16 ? 1 : 2; }

// 16-row groups of the warps of a stage (the transposed kernel has one)
int row_groups(int MT) { return MT > 1 ? MT : 1; }

int rows_per_pass(int dtype, int R)
{
    if (dtype == PA_F32)
        return kConsumerWarps * rows_group(R);
    const int MT = mma_tiles(R);
    return MT == 0 ? 8 : 16 * MT;
}

int tokens_per_stage(int D, int es, int BLOCK)
{
    int tt = kStageBytes / (2 * D * es);
    if (tt < BLOCK)
        tt = BLOCK;
    return tt;
}

size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

// Tokens per pipeline stage (the automatic schedule's unit).  Tensor-core
// path: up to 64 KB stages, at most 8 warps (TPW tokens x row groups) per
// stage: 128 tokens at D = 128, 256 at D = 64 (128 with 32 rows per pass); at
// most 16 cache blocks per stage.
int stage_tokens(int dtype, int D, int BLOCK, int MT)
{
    const int es = static_cast<int>(elem_size(dtype));
    if (dtype == PA_F32)
        return tokens_per_stage(D, es, BLOCK);
    int TT = kMmaStageBytes / (2 * D * es);
    const int TPW = kMmaTokens * mma_token_groups(D, MT);  // tokens per consumer warp and stage
    if ((TT / TPW) * row_groups(MT) > kConsumerWarps)
        TT = kConsumerWarps / row_groups(MT) * TPW;
    if (TT > 16 * BLOCK)  // at most 16 boxes (one per block) per stage and role
        TT = 16 * BLOCK;
    return TT;
}

int ilog2(int x)  // x is a power of two
{
    int l = 0;
    while ((1 << l) < x)
        ++l;
    return l;
}

// Workspace records of one call: automatic schedule, two per partition-kernel
// CTA (its first and last piece); fixed partitions, one per item.
long long record_bound(int B, int KV, int NRS, int partitions)
{
    const long long per_seq = static_cast<long long>(KV) * NRS;
    if (partitions == 0)
        return 2ll * kMaxGrid;
    return B * per_seq * partitions;
}

// Workspace: split counters (in-kernel merge) | per-sequence schedule |
// (max, sum) of every partial record | accumulators of every partial record.
struct WsLayout {
    size_t counters, sched, ml, o, total;
};

WsLayout ws_layout(int B, int D, int segments, int row_stride, long long records)
{
    WsLayout w;
    w.counters = 0;
    w.sched = align_up(static_cast<size_t>(segments) * sizeof(int), 256);
    w.ml = w.sched + align_up(static_cast<size_t>(B) * sizeof(int2), 256);
    w.o = w.ml + align_up(static_cast<size_t>(records) * row_stride * sizeof(float2), 256);
    w.total = w.o + static_cast<size_t>(records) * row_stride * D * sizeof(float);
    return w;
}

// --- tensor maps --------------------------------------------------------------
PFN_cuTensorMapEncodeTiled_v12000 encoder()
{
    static PFN_cuTensorMapEncodeTiled_v12000 fn = [] {
        void* ptr = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000,
                                             cudaEnableDefault, &q) != cudaSuccess ||
            q != cudaDriverEntryPointSuccess)
            ptr = nullptr;
        return reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(ptr);
    }();
    return fn;
}

struct MapKey {
    const void* ptr;
    long long rows;
    int KV, D, BLOCK, dtype, halves;
    bool operator==(const MapKey& o) const
    {
        return ptr == o.ptr && rows == o.rows && KV == o.KV && D == o.D && BLOCK == o.BLOCK &&
               dtype == o.dtype && halves == o.halves;
    }
};

std::mutex g_map_mutex;
constexpr int kMapCache = 32;
MapKey g_map_keys[kMapCache];
CUtensorMap g_maps[kMapCache];
int g_map_count = 0, g_map_next = 0;

// Cache pool [num_blocks * BLOCK rows][KV][D] as a 3-D tensor; one box is one
// block of one KV head: {D, 1, BLOCK}.
int cache_map(const void* base, int num_blocks, int BLOCK, int KV, int D, int dtype, int box_rows,
              bool halves, CUtensorMap* out)
{
    // 16-bit caches feed the tensor-core kernels: 64-column boxes, 128-byte swizzle.
    const bool swz = dtype != PA_F32;
    const MapKey key{base, static_cast<long long>(num_blocks) * BLOCK, KV, D, box_rows, dtype, halves ? 1 : 0};
    std::lock_guard<std::mutex> lock(g_map_mutex);
    for (int i = 0; i < g_map_count; ++i)
        if (g_map_keys[i] == key) {
            *out = g_maps[i];
            return PA_OK;
        }
    auto enc = encoder();
    if (!enc)
        return PA_ERR_DRIVER;
    const size_t es = elem_size(dtype);
    const CUtensorMapDataType dt = dtype == PA_F32   ? CU_TENSOR_MAP_DATA_TYPE_FLOAT32
                                   : dtype == PA_F16 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT16
                                                     : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
    // float32 (CUDA-core path): 3-D {D, KV, rows}, box {D, 1, box_rows}, no swizzle.
    // 16-bit (tensor-core path): 4-D {64, D/64, KV, rows}, box {64, D/64, 1,
    // box_rows} -- one box brings both 64-column halves of box_rows token rows
    // -- or, with `halves` (the tcgen05 kernel), box {64, 1, 1, box_rows}: one
    // half, so that each half of a tile is a run of 128-byte rows.
    // L2 fills no wider than one token row of one KV head: with 128-byte rows
    // (D = 64, 16-bit) a 256-byte promotion would also fetch the neighbouring
    // head's row, which another CTA reads at another time
    const CUtensorMapL2promotion promo = static_cast<size_t>(D) * es >= 256
                                             ? CU_TENSOR_MAP_L2_PROMOTION_L2_256B
                                             : CU_TENSOR_MAP_L2_PROMOTION_L2_128B;
    CUtensorMap map;
    CUresult rc;
    if (swz) {
        cuuint64_t dims[4] = {64u, static_cast<cuuint64_t>(D / 64), static_cast<cuuint64_t>(KV),
                              static_cast<cuuint64_t>(key.rows)};
        cuuint64_t strides[3] = {128u, static_cast<cuuint64_t>(D) * es,
                                 static_cast<cuuint64_t>(KV) * D * es};
        cuuint32_t box[4] = {64u, halves ? 1u : static_cast<cuuint32_t>(D / 64), 1u,
                             static_cast<cuuint32_t>(box_rows)};
        cuuint32_t estr[4] = {1u, 1u, 1u, 1u};
        rc = enc(&map, dt, 4, const_cast<void*>(base), dims, strides, box, estr,
                 CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                 promo, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    } else {
        cuuint64_t dims[3] = {static_cast<cuuint64_t>(D), static_cast<cuuint64_t>(KV),
                              static_cast<cuuint64_t>(key.rows)};
        cuuint64_t strides[2] = {static_cast<cuuint64_t>(D) * es,
                                 static_cast<cuuint64_t>(KV) * D * es};
        cuuint32_t box[3] = {static_cast<cuuint32_t>(D), 1u, static_cast<cuuint32_t>(box_rows)};
        cuuint32_t estr[3] = {1u, 1u, 1u};
        rc = enc(&map, dt, 3, const_cast<void*>(base), dims, strides, box, estr,
                 CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
                 promo, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    }
    if (rc != CUDA_SUCCESS)
        return PA_ERR_CUDA;
    const int slot = g_map_count < kMapCache ? g_map_count++ : (g_map_next++ % kMapCache);
    g_map_keys[slot] = key;
    g_maps[slot] = map;
    *out = map;
    return PA_OK;
}

// The query rows [rows][D] (16-bit) for the tcgen05 kernel: 3-D {64, D/64,
// rows}, box {64, 1, 32} with the 128-byte swizzle -- one 64-column half of a
// 32-row pass, in the canonical K-major operand layout; rows past the end
// read as zeros.
int query_map(const void* q, long long rows, int D, int dtype, CUtensorMap* out)
{
    const MapKey key{q, rows, 0, D, -1, dtype, 1};
    std::lock_guard<std::mutex> lock(g_map_mutex);
    for (int i = 0; i < g_map_count; ++i)
        if (g_map_keys[i] == key) {
            *out = g_maps[i];
            return PA_OK;
        }
    auto enc = encoder();
    if (!enc)
        return PA_ERR_DRIVER;
    const CUtensorMapDataType dt = dtype == PA_F16 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT16
                                                   : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
    cuuint64_t dims[3] = {64u, static_cast<cuuint64_t>(D / 64), static_cast<cuuint64_t>(rows)};
    cuuint64_t strides[2] = {128u, static_cast<cuuint64_t>(D) * 2};
    cuuint32_t box[3] = {64u, 1u, 32u};
    cuuint32_t estr[3] = {1u, 1u, 1u};
    CUtensorMap map;
    if (enc(&map, dt, 3, const_cast<void*>(q), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
            CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_128B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
        return PA_ERR_CUDA;
    const int slot = g_map_count < kMapCache ? g_map_count++ : (g_map_next++ % kMapCache);
    g_map_keys[slot] = key;
    g_maps[slot] = map;
    *out = map;
    return PA_OK;
}

// --- kernel table -----------------------------------------------------------------
SplitFn pick_split(int dtype, bool f32_out, int D, int RG)
{
    switch (dtype) {
    case PA_F32:
        return pick_split_f32(D, RG);
    case PA_F16:
        return pick_split_f16(f32_out, D, RG);
    default:
        return pick_split_bf16(f32_out, D, RG);
    }
}

CombineFn pick_combine(int out_dtype, int D)
{
    switch (out_dtype) {
    case PA_F32:
        return pick_combine_f32(D);
    case PA_F16:
        return pick_combine_f16(D);
    default:
        return pick_combine_bf16(D);
    }
}

struct FuncState {
    const void* fn;
    int device;
    int smem_set;
    int occupancy;
    int sms;
};
std::mutex g_func_mutex;
constexpr int kFuncCache = 64;
FuncState g_funcs[kFuncCache];
int g_func_count = 0;

// Raises the dynamic shared-memory limit of `fn` on the current device when
// needed; returns its occupancy (CTAs per SM) and the SM count.
int prepare_func(const void* fn, int threads, int smem, int* occ, int* sms)
{
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess)
        return PA_ERR_CUDA;
    std::lock_guard<std::mutex> lock(g_func_mutex);
    FuncState* st = nullptr;
    for (int i = 0; i < g_func_count; ++i)
        if (g_funcs[i].fn == fn && g_funcs[i].device == dev)
            st = &g_funcs[i];
    if (!st) {
        if (g_func_count == kFuncCache)
            g_func_count = 0;
        st = &g_funcs[g_func_count++];
        *st = FuncState{fn, dev, 0, 0, 0};
        if (cudaDeviceGetAttribute(&st->sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
            return PA_ERR_CUDA;
    }
    if (smem > st->smem_set) {
        if (cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, smem) !=
            cudaSuccess)
            return PA_ERR_CUDA;
        st->smem_set = smem;
        st->occupancy = 0;
    }
    if (st->occupancy == 0) {
        int n = 0;
        if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, fn, threads, smem) != cudaSuccess)
            return PA_ERR_CUDA;
        st->occupancy = n < 1 ? 1 : n;
    }
    *occ = st->occupancy;
    *sms = st->sms;
    return PA_OK;
}

// The opt-in shared-memory limit per block of the current device, asked of the
// runtime once per device.
int device_smem_optin(int* out)
{
    constexpr int kDevices = 64;
    static std::atomic<int> cached[kDevices] = {};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess)
        return PA_ERR_CUDA;
    if (dev >= 0 && dev < kDevices) {
        const int v = cached[dev].load(std::memory_order_relaxed);
        if (v > 0) {
            *out = v;
            return PA_OK;
        }
    }
    int v = 0;
    if (cudaDeviceGetAttribute(&v, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev) != cudaSuccess)
        return PA_ERR_CUDA;
    if (dev >= 0 && dev < kDevices)
        cached[dev].store(v, std::memory_order_relaxed);
    *out = v;
    return PA_OK;
}

bool aligned(const void* p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

}  // namespace

void count_launches(uint64_t n) { g_launches.fetch_add(n); }

}  // namespace pa

using namespace pa;

extern "C" {

int pa_version(void) { return 100; }

uint64_t pa_kernel_launches(void) { return g_launches.load(); }

const char* pa_strerror(int code)
{
    switch (code) {
    case PA_OK:
        return "success";
    case PA_ERR_NULL_POINTER:
        return "PagedAttention: a required pointer is NULL; verify q, caches, block table, "
               "seq_lens, k_new, v_new, out and opts";
    case PA_ERR_BAD_DIMS:
        return "PagedAttention: invalid sizes; verify H % KV == 0, batch >= 0, max_blocks >= 1, "
               "num_blocks * BLOCK < 2^31 and a finite scale";
    case PA_ERR_UNSUPPORTED:
        return "PagedAttention: unsupported configuration; verify D in {64,128}, BLOCK in "
               "{8,16,32,64}, 1 <= NQ <= 16, batch <= 4096, dtype and out_dtype";
    case PA_ERR_ALIGNMENT:
        return "PagedAttention: misaligned pointer; verify 16-byte aligned tensors and a "
               "256-byte aligned workspace";
    case PA_ERR_WORKSPACE:
        return "PagedAttention: workspace missing or too small; verify pa_workspace_bytes()";
    case PA_ERR_CUDA:
        return "PagedAttention: CUDA call failed; verify the device, the stream and GPU limits";
    case PA_ERR_DRIVER:
        return "PagedAttention: cannot reach the driver's tensor-map encoder; verify the CUDA "
               "driver version";
    case PA_ERR_NOT_PINNED:
        return "PagedAttention: the host range is not page-locked memory mapped for the device; "
               "verify cudaHostAlloc / cudaHostRegister (or a pinned tensor) covers all of it";
    case PA_ERR_STATIC_LIMIT:
        return "PagedAttention: the call needs more scratch than the library's built-in "
               "PA_STATIC_WORKSPACE_BYTES; verify pa_workspace_bytes(), use fewer partitions, "
               "or call pa_decode with a workspace of your own";
    default:
        return "PagedAttention: unknown error code";
    }
}

// Largest layout over the two paths (the row grouping differs by dtype), so
// that the sizes do not depend on the dtype.
static WsLayout ws_bound(int batch, int H, int KV, int D, int NQ, int partitions)
{
    const int R = (H / KV) * NQ;
    WsLayout best{};
    for (int dtype : {PA_F32, PA_F16}) {
        const int rpc = rows_per_pass(dtype, R);
        const int NRS = (R + rpc - 1) / rpc;
        const int row_stride = R < rpc ? R : rpc;
        const WsLayout w = ws_layout(batch, D, batch * NRS * KV, row_stride,
                                     record_bound(batch, KV, NRS, partitions));
        if (w.total > best.total)
            best.total = w.total;
        if (w.sched > best.sched)
            best.sched = w.sched;  // = bytes of the counters region
    }
    return best;
}

// Sizes pa_decode accepts (batch up to kMaxBatch: the partition kernels keep
// the schedule in shared memory); the size queries return 0 for the rest.
static bool ws_args_ok(int batch, int H, int KV, int D, int NQ, int partitions)
{
    return batch >= 0 && batch <= kMaxBatch && H >= 1 && KV >= 1 && H % KV == 0 &&
           (D == 64 || D == 128) && NQ >= 1 && NQ <= PA_MAX_NQ && partitions >= 0;
}

int pa_choose_partitions(const int32_t* host_seq_lens, int max_len, int batch, int H, int KV, int D,
                         int BLOCK, int NQ, int dtype, int sms, pa_split_plan* plan)
{
    if (!plan)
        return PA_ERR_NULL_POINTER;
    *plan = pa_split_plan{};
    if (batch < 0 || H < 1 || KV < 1 || H % KV != 0 || max_len < 0 || sms < 0)
        return PA_ERR_BAD_DIMS;
    if ((D != 64 && D != 128) || (BLOCK != 8 && BLOCK != 16 && BLOCK != 32 && BLOCK != 64) || NQ < 1 ||
        NQ > PA_MAX_NQ || (dtype != PA_F32 && dtype != PA_F16 && dtype != PA_BF16) || batch > kMaxBatch)
        return PA_ERR_UNSUPPORTED;
    if (sms == 0) {
        int dev = 0;
        if (cudaGetDevice(&dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
            return PA_ERR_CUDA;
    }
    // the partition kernel's choices (decode_impl): rows per pass, stage size,
    // charge per segment, one persistent CTA per SM
    const int R = (H / KV) * NQ;
    const int MT = mma_tiles(R);
    const int rows_per_cta = rows_per_pass(dtype, R);
    const int NRS = (R + rows_per_cta - 1) / rows_per_cta;
    const int U = NRS * KV;
    const int TT = stage_tokens(dtype, D, BLOCK, MT);
    const long long V = dtype != PA_F32 && MT > 1 ? kPieceStages2 : kPieceStages;
    long long grid = sms < kMaxGrid ? sms : kMaxGrid;
    const long long cost_bound = static_cast<long long>(batch) * U * ((static_cast<long long>(max_len) + NQ + TT - 1) / TT + V);
    if (grid > cost_bound && batch > 0)
        grid = cost_bound;  // as pa_decode launches it (with max_len = max_blocks * BLOCK)
    plan->grid = static_cast<int>(grid);
    plan->segments = batch * U;
    if (batch == 0)
        return 1;
    auto length = [&](int b) {
        const long long s = host_seq_lens ? host_seq_lens[b] : max_len;
        return s < 0 ? 0 : s > max_len ? max_len : s;  // the kernel's clamp
    };
    // cost: real unit x of segment g sits at x + V (g + 1); CTA k of G owns the
    // cost positions [ceil(k C / G), ceil((k + 1) C / G))
    long long W = 0;
    for (int b = 0; b < batch; ++b)
        W += (length(b) + NQ + TT - 1) / TT * U;
    const long long C = W + V * batch * U;
    if (C >= (1ll << 31))
        return PA_ERR_BAD_DIMS;
    const long long G = active_ctas(grid, C, static_cast<long long>(batch) * U);
    plan->active = static_cast<int>(G);
    long long max_units = 0;
    for (int b = 0; b < batch; ++b) {
        const long long nu = (length(b) + NQ + TT - 1) / TT;
        max_units = nu > max_units ? nu : max_units;
    }
    if (whole_segments(static_cast<long long>(batch) * U, G, W, max_units)) {
        plan->active = batch * U;  // one whole segment per CTA
        plan->pieces = batch * U;
        plan->max_pieces = 1;
        return 1;
    }
    auto owner = [&](long long c) { return c * G / C < G - 1 ? c * G / C : G - 1; };
    long long x0 = 0, g = 0;
    int most = 1;
    for (int b = 0; b < batch; ++b) {
        const long long nu = (length(b) + NQ + TT - 1) / TT;
        for (int s = 0; s < U; ++s, ++g, x0 += nu) {
            const long long c0 = x0 + V * (g + 1);
            const int n = static_cast<int>(owner(c0 + nu - 1) - owner(c0) + 1);
            plan->pieces += n;
            if (n > 1) {
                ++plan->split_segments;
                plan->records += n;
            }
            most = n > most ? n : most;
        }
    }
    plan->max_pieces = most;
    return most;
}

size_t pa_workspace_bytes(int batch, int H, int KV, int D, int NQ, int partitions)
{
    if (!ws_args_ok(batch, H, KV, D, NQ, partitions) || partitions == 1 || batch == 0)
        return 0;
    return ws_bound(batch, H, KV, D, NQ, partitions).total;
}

size_t pa_workspace_zero_bytes(int batch, int H, int KV, int D, int NQ, int partitions)
{
    if (!ws_args_ok(batch, H, KV, D, NQ, partitions) || partitions != 0 || batch == 0)
        return 0;
    return ws_bound(batch, H, KV, D, NQ, partitions).sched;
}

static int launch_append(void* k_cache, void* v_cache, const void* k_new, const void* v_new,
                         const int32_t* slots, long long rows, int vpr, int KV, int NQ,
                         long long num_slots, int* status, cudaStream_t stream);

// pa_decode, and pa_decode_positions when `positions` is not NULL: then the
// new rows are first stored at their slots in the (writable) caches, after
// every argument has been checked.  With launch == false: the checks alone.
static int decode_impl(const void* q, const void* k_cache, const void* v_cache,
                       const int32_t* block_table, const int32_t* seq_lens, const void* k_new,
                       const void* v_new, const int32_t* positions, void* out, float scale,
                       int H, int KV, int D, int BLOCK, int NQ, int causal, const pa_opts* opts,
                       void* stream, bool launch = true)
{
    if (!opts)
        return PA_ERR_NULL_POINTER;
    const int B = opts->batch;
    if (B < 0 || H < 1 || KV < 1 || H % KV != 0 || opts->max_blocks < 1 ||
        opts->num_blocks < 1 || opts->partitions < 0)
        return PA_ERR_BAD_DIMS;
    if ((D != 64 && D != 128) || (BLOCK != 8 && BLOCK != 16 && BLOCK != 32 && BLOCK != 64) ||
        NQ < 1 || NQ > PA_MAX_NQ)
        return PA_ERR_UNSUPPORTED;
    if (static_cast<long long>(opts->num_blocks) * BLOCK >= (1ll << 31) ||
        static_cast<long long>(opts->max_blocks) * BLOCK >= (1ll << 30))
        return PA_ERR_BAD_DIMS;
    const int dtype = opts->dtype;
    if (dtype != PA_F32 && dtype != PA_F16 && dtype != PA_BF16)
        return PA_ERR_UNSUPPORTED;
    const int out_dtype = opts->out_dtype < 0 ? dtype : opts->out_dtype;
    if (out_dtype != dtype && out_dtype != PA_F32)
        return PA_ERR_UNSUPPORTED;
    if (!std::isfinite(scale))
        return PA_ERR_BAD_DIMS;
    if (opts->kernel != 0 && opts->kernel != 1)
        return PA_ERR_UNSUPPORTED;
    if (B == 0)
        return PA_OK;
    if (B > kMaxBatch)
        return PA_ERR_UNSUPPORTED;
    if (!q || !k_cache || !v_cache || !block_table || !seq_lens || !k_new || !v_new || !out)
        return PA_ERR_NULL_POINTER;
    if (!aligned(q, 16) || !aligned(k_cache, 16) || !aligned(v_cache, 16) ||
        !aligned(k_new, 16) || !aligned(v_new, 16) || !aligned(out, 16) ||
        !aligned(block_table, 4) || !aligned(seq_lens, 4) || !aligned(positions, 4))
        return PA_ERR_ALIGNMENT;
    if (positions && static_cast<long long>(B) * KV * NQ * D * 8 >= (1ll << 38))
        return PA_ERR_BAD_DIMS;  // threads of the append kernel

    const int R = (H / KV) * NQ;
    const bool mma = dtype != PA_F32;
    const int RG = rows_group(R);
    const int MT = mma_tiles(R);
    const int rows_per_cta = rows_per_pass(dtype, R);
    const int NRS = (R + rows_per_cta - 1) / rows_per_cta;
    const int partitions = opts->partitions;
    const int row_stride = R < rows_per_cta ? R : rows_per_cta;
    const long long records = record_bound(B, KV, NRS, partitions);
    if (records >= (1ll << 31))
        return PA_ERR_BAD_DIMS;
    const int es = static_cast<int>(elem_size(dtype));
    const int TT = stage_tokens(dtype, D, BLOCK, MT);
    const int TPW = kMmaTokens * mma_token_groups(D, MT);  // tokens per consumer warp and stage
    // automatic schedule: units of one stage.  Each segment is charged the
    // measured cost of a piece in stages (the consumer warps' merge and the
    // start of the next piece): about one, six with two row groups per pass
    // (four merge rounds)
    const int vunits = MT > 1 ? kPieceStages2 : kPieceStages;
    // (the units of all segments are counted in int32)
    const long long units = static_cast<long long>(B) *
                            (opts->max_blocks + 1 + NQ / BLOCK + 1 + vunits) * NRS * KV;
    if (partitions == 0 && units >= (1ll << 31))
        return PA_ERR_BAD_DIMS;
    WsLayout ws{};
    if (partitions != 1) {
        ws = ws_layout(B, D, B * NRS * KV, row_stride, records);
        if (!opts->workspace || opts->workspace_bytes < ws.total)
            return PA_ERR_WORKSPACE;
        if (!aligned(opts->workspace, 256))
            return PA_ERR_ALIGNMENT;
    }

    // one TMA box per cache block (per tile when a block spans several tiles):
    // the issue cost of a box is fixed, so fewer, larger boxes stream faster
    const int box_rows = mma ? (BLOCK < TT ? BLOCK : TT) : BLOCK;
    const int ROWS = rows_per_cta;  // tensor-core path: query-row buffer rows
    // shared memory: header | lens[B] | prefix[B+1] | consumer scratch | ring
    const int lens_off = kHeaderBytes;
    const int prefix_off = static_cast<int>(align_up(lens_off + 4 * B, 16));
    const int merge_off = static_cast<int>(align_up(prefix_off + 4 * (B + 1), 128));
    // stage: tensor-core path K tile | V tile | K new rows | V new rows (tiles
    // 1024-aligned for the swizzle); CUDA-core path K tile | K new | V tile | V new
    int v_off, knew_off, vnew_off, stage_end;
    if (mma) {
        v_off = TT * D * es;
        knew_off = 2 * TT * D * es;
        vnew_off = knew_off + NQ * D * es;
        stage_end = vnew_off + NQ * D * es;
    } else {
        knew_off = TT * D * es;
        v_off = static_cast<int>(align_up(knew_off + NQ * D * es, 1024));
        vnew_off = v_off + TT * D * es;
        stage_end = vnew_off + NQ * D * es;
    }
    int stage_bytes = static_cast<int>(align_up(stage_end, 1024));
    int smem_optin = 0;
    if (device_smem_optin(&smem_optin) != PA_OK)
        return PA_ERR_CUDA;
    const int slack = 1024;  // alignment of the dynamic shared-memory base
    // consumer scratch: tensor-core path, (max, sum) tables, one merge round of
    // kObufFloats floats of merge rounds and two query-row buffers; CUDA-core
    // path, per-warp states
    const int qbuf_off = 2048 + kObufFloats * 4;
    const int merge_bytes = mma ? qbuf_off + 2 * ROWS * q_row_bytes(D)
                                : (kConsumerWarps * RG * D + 2 * kConsumerWarps * RG) * 4 +
                                      kConsumerWarps * RG * 8;
    int stage_off = static_cast<int>(align_up(merge_off + merge_bytes, 1024));
    // The tcgen05 kernel (32-row passes at D = 128): its region (P^T and
    // query tiles, barriers, reductions) after the lengths, then a K ring and
    // a V ring of 32 KB tiles, half of the remaining tiles each (the new rows
    // stay in global memory), when each ring gets two tiles at least.
    int tc_off = 0, stages_v = 0;
    bool tc32 = false;
    if (mma && MT == 2 && D == 128 && opts->kernel == 0) {
        const int t_off = static_cast<int>(align_up(merge_off, 1024));
        const int t_stage = static_cast<int>(align_up(t_off + kTcRegionBytes, 1024));
        const int tiles = (smem_optin - slack - t_stage) / kTcTileBytes;
        if (tiles >= 4) {
            tc32 = true;
            tc_off = t_off;
            stage_off = t_stage;
            stage_bytes = kTcTileBytes;
            stages_v = (tiles + 1) / 2 < kMaxStages / 2 ? (tiles + 1) / 2 : kMaxStages / 2;
        }
    }
    int stages = (smem_optin - slack - stage_off) / stage_bytes;
    if (tc32)
        stages -= stages_v;  // the K ring: the tiles the V ring leaves
    if (stages > (tc32 ? kMaxStages / 2 : kMaxStages))
        stages = tc32 ? kMaxStages / 2 : kMaxStages;
    if (stages < 2)
        return PA_ERR_UNSUPPORTED;
    const int smem = slack + stage_off + (stages + stages_v) * stage_bytes;

    CUtensorMap kmap, vmap, qmap;
    int rc = cache_map(k_cache, opts->num_blocks, BLOCK, KV, D, dtype, box_rows, tc32, &kmap);
    if (rc == PA_OK)
        rc = cache_map(v_cache, opts->num_blocks, BLOCK, KV, D, dtype, box_rows, tc32, &vmap);
    if (rc == PA_OK && tc32)
        rc = query_map(q, static_cast<long long>(B) * H * NQ, D, dtype, &qmap);
    if (rc != PA_OK)
        return rc;

    const bool f32_out = out_dtype == PA_F32 && dtype != PA_F32;
    const void* split = tc32 ? reinterpret_cast<const void*>(pick_split_tc(dtype, f32_out))
                             : reinterpret_cast<const void*>(pick_split(dtype, f32_out, D, mma ? MT : RG));
    int occ = 1, sms = 1;
    const int threads = tc32 ? kUmmaThreads : kThreads;
    rc = prepare_func(split, threads, smem, &occ, &sms);
    if (rc != PA_OK)
        return rc;

    SplitParams p{};
    p.q = q;
    p.k_new = k_new;
    p.v_new = v_new;
    p.out = out;
    p.table = block_table;
    p.seq_lens = seq_lens;
    unsigned char* wsb = static_cast<unsigned char*>(opts->workspace);
    p.sched = partitions != 1 ? reinterpret_cast<int2*>(wsb + ws.sched) : nullptr;
    // the in-kernel merge serves the automatic schedule; fixed partitions
    // always use the merge kernel
    const bool merge_in_kernel = partitions == 0 && !opts->merge_kernel;
    p.counters = merge_in_kernel ? reinterpret_cast<int*>(wsb + ws.counters) : nullptr;
    p.ws_ml = partitions != 1 ? reinterpret_cast<float2*>(wsb + ws.ml) : nullptr;
    p.ws_o = partitions != 1 ? reinterpret_cast<float*>(wsb + ws.o) : nullptr;
    p.status = opts->status;
    p.qscale = scale * kLog2e;
    p.B = B;
    p.H = H;
    p.KV = KV;
    p.NQ = NQ;
    p.BLOCK = BLOCK;
    p.maxb = opts->max_blocks;
    p.num_blocks = opts->num_blocks;
    p.causal = causal ? 1 : 0;
    p.partitions = partitions;
    long long grid = static_cast<long long>(sms) * occ;  // persistent CTAs
    if (grid > kMaxGrid)
        grid = kMaxGrid;
    if (partitions == 0) {
        // no more CTAs than the schedule's cost (at most this, as every length
        // is clamped to the table): the device uses min(CTAs, cost) of them, so
        // a small batch no longer starts a CTA on every SM for nothing
        const long long seg_units = (static_cast<long long>(opts->max_blocks) * BLOCK + NQ + TT - 1) / TT;
        const long long cost_bound = static_cast<long long>(B) * NRS * KV * (seg_units + vunits);
        if (grid > cost_bound)
            grid = cost_bound;
    }
    if (partitions != 0 && grid > records)  // fixed partitions: no more CTAs than items
        grid = records;
    p.qbuf_off = qbuf_off;
    p.box_rows = box_rows;
    // warps that release a stage; the tcgen05 kernel's MMA commits release
    // its K and V parts (one arrival each)
    p.empty_count = tc32 ? 1 : mma ? (TT / TPW) * row_groups(MT) : kConsumerWarps;
    p.tc_off = tc_off;
    p.stages_v = stages_v;
    p.checked = opts->checked ? 1 : 0;
    p.R = R;
    p.rows_per_cta = rows_per_cta;
    p.NRS = NRS;
    p.TT = TT;
    p.lg_block = ilog2(BLOCK);
    p.lg_box = ilog2(box_rows);
    p.lg_tt = ilog2(TT);
    p.vunits = vunits;
    p.row_stride = row_stride;
    p.stages = stages;
    p.stage_bytes = stage_bytes;
    p.knew_off = knew_off;
    p.v_off = v_off;
    p.vnew_off = vnew_off;
    p.lens_off = lens_off;
    p.prefix_off = prefix_off;
    p.merge_off = merge_off;
    p.stage_off = stage_off;
    p.wait_ns = opts->wait_limit_ns ? opts->wait_limit_ns : kWaitLimitNs;
    p.withhold = opts->debug_withhold_stage > 0 ? opts->debug_withhold_stage : 0;
    // the slot-patched decode runs right after its own append kernel
    p.early = opts->inputs_unchanged && !positions ? 1 : 0;

    if (!launch)
        return PA_OK;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    if (positions) {
        const int es_row = D * es;
        rc = launch_append(const_cast<void*>(k_cache), const_cast<void*>(v_cache), k_new, v_new,
                           positions, static_cast<long long>(B) * KV * NQ, es_row / 16, KV, NQ,
                           static_cast<long long>(opts->num_blocks) * BLOCK, opts->status, st);
        if (rc != PA_OK)
            return rc;
    }
    if (opts->trace_begin &&
        cudaEventRecord(static_cast<cudaEvent_t>(opts->trace_begin), st) != cudaSuccess)
        return PA_ERR_CUDA;

    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;

    cudaLaunchConfig_t cfg{};
    cfg.gridDim = dim3(static_cast<unsigned>(grid));
    cfg.blockDim = dim3(threads);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    void* args[4] = {&p, &kmap, &vmap, &qmap};
    if (cudaLaunchKernelExC(&cfg, split, args) != cudaSuccess)
        return PA_ERR_CUDA;
    g_launches.fetch_add(1);

    if (opts->trace_split &&
        cudaEventRecord(static_cast<cudaEvent_t>(opts->trace_split), st) != cudaSuccess)
        return PA_ERR_CUDA;

    if (partitions != 1 && !merge_in_kernel) {
        CombineParams cp{};
        cp.sched = p.sched;
        cp.ws_ml = p.ws_ml;
        cp.ws_o = p.ws_o;
        cp.out = out;
        cp.B = B;
        cp.KV = KV;
        cp.R = R;
        cp.NRS = NRS;
        cp.rows_per_cta = rows_per_cta;
        cp.row_stride = row_stride;
        cp.stream = partitions == 0 ? 1 : 0;
        cp.grid = static_cast<int>(grid);
        cp.vunits = vunits;
        cp.seq_lens = seq_lens;
        cp.partitions = partitions;
        cp.NQ = NQ;
        cp.BLOCK = BLOCK;
        cp.cap = opts->max_blocks * BLOCK;
        const CombineFn comb = pick_combine(out_dtype, D);
        cudaLaunchConfig_t cc{};
        cc.gridDim = dim3(static_cast<unsigned>(B) * KV * NRS, static_cast<unsigned>(row_stride));
        cc.blockDim = dim3(128);
        cc.dynamicSmemBytes = 0;
        cc.stream = st;
        cc.attrs = attr;
        cc.numAttrs = 1;
        void* cargs[1] = {&cp};
        if (cudaLaunchKernelExC(&cc, reinterpret_cast<const void*>(comb), cargs) != cudaSuccess)
            return PA_ERR_CUDA;
        g_launches.fetch_add(1);
    }
    return PA_OK;
}

int pa_decode(const void* q, const void* k_cache, const void* v_cache, const int32_t* block_table,
              const int32_t* seq_lens, const void* k_new, const void* v_new, void* out,
              float scale, int H, int KV, int D, int BLOCK, int NQ, int causal,
              const pa_opts* opts, void* stream)
{
    return decode_impl(q, k_cache, v_cache, block_table, seq_lens, k_new, v_new, nullptr, out,
                       scale, H, KV, D, BLOCK, NQ, causal, opts, stream);
}

int pa_decode_positions(const void* q, void* k_cache, void* v_cache, const int32_t* block_table,
                        const int32_t* seq_lens, const void* k_new, const void* v_new,
                        const int32_t* positions, void* out, float scale, int H, int KV, int D,
                        int BLOCK, int NQ, int causal, const pa_opts* opts, void* stream)
{
    return decode_impl(q, k_cache, v_cache, block_table, seq_lens, k_new, v_new, positions, out,
                       scale, H, KV, D, BLOCK, NQ, causal, opts, stream);
}

// ------------------------------------------------------------ cache append
// One thread per 16 bytes of one new row of K or V (rows in k_new order
// [B][KV][NQ]): the slot of the row's (sequence, new row) names the cache row.
// When several new rows of one sequence name one slot, only the last of them
// (largest j) is stored, so the result does not depend on thread order.
struct AppendParams {
    uint4* k_cache;
    uint4* v_cache;
    const uint4* k_new;
    const uint4* v_new;
    const int32_t* slots;  // [B][NQ]
    int* status;
    long long rows;        // B * KV * NQ
    int vpr;               // 16-byte vectors per row (D * element bytes / 16)
    int KV, NQ;
    long long num_slots;   // num_blocks * BLOCK
};

__global__ void __launch_bounds__(256) pa_append_kernel(const __grid_constant__ AppendParams a)
{
    // a decode launched after it may start (it waits for this grid before
    // reading anything this kernel writes)
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    const long long i = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x;
    const long long per = a.rows * a.vpr;  // vectors of K (or V)
    if (i >= 2 * per)
        return;
    const bool is_v = i >= per;
    const long long k = is_v ? i - per : i;
    const long long row = k / a.vpr;
    const int v = static_cast<int>(k - row * a.vpr);
    const int j = static_cast<int>(row % a.NQ);
    const long long bk = row / a.NQ;  // b * KV + kh
    const int kh = static_cast<int>(bk % a.KV);
    const long long b = bk / a.KV;
    const int s = a.slots[b * a.NQ + j];
    if (s == -1)
        return;
    if (s < -1 || s >= a.num_slots) {
        if (a.status && !is_v && v == 0 && kh == 0)
            atomicOr(a.status, PA_STATUS_BAD_SLOT);
        return;
    }
    for (int jj = j + 1; jj < a.NQ; ++jj)
        if (a.slots[b * a.NQ + jj] == s)
            return;  // a later new row of this sequence lands here
    const uint4* src = (is_v ? a.v_new : a.k_new) + row * a.vpr + v;
    uint4* dst = (is_v ? a.v_cache : a.k_cache) + (static_cast<long long>(s) * a.KV + kh) * a.vpr + v;
    *dst = *src;
}

// ------------------------------------------------------- host-buffer entry
// Inputs in page-locked host memory are readable by the device (unified
// addressing): one gather kernel then moves all of them into the staging area,
// in place of one copy per input.  Segment k of blockIdx.y: 16-byte words when
// both ends are 16-byte aligned, else 4-byte words.
struct GatherParams {
    const void* src[5];
    void* dst[5];
    int bytes[5];
};

__global__ void __launch_bounds__(256) pa_gather_kernel(const __grid_constant__ GatherParams g)
{
    // the decode launched next sets up while the inputs move (it waits for
    // this grid before reading them)
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    const int k = blockIdx.y;
    const int n = g.bytes[k];
    const int t = blockIdx.x * blockDim.x + threadIdx.x, nt = gridDim.x * blockDim.x;
    if (((reinterpret_cast<uintptr_t>(g.src[k]) | reinterpret_cast<uintptr_t>(g.dst[k])) & 15) == 0) {
        const uint4* s = static_cast<const uint4*>(g.src[k]);
        uint4* d = static_cast<uint4*>(g.dst[k]);
        for (int i = t; i < n / 16; i += nt)
            d[i] = s[i];
        const int* s4 = static_cast<const int*>(g.src[k]);
        int* d4 = static_cast<int*>(g.dst[k]);
        for (int i = (n / 16) * 4 + t; i < n / 4; i += nt)
            d4[i] = s4[i];
    } else {
        const int* s4 = static_cast<const int*>(g.src[k]);
        int* d4 = static_cast<int*>(g.dst[k]);
        for (int i = t; i < n / 4; i += nt)
            d4[i] = s4[i];
    }
}

int pa_cache_append(void* k_cache, void* v_cache, const void* k_new, const void* v_new,
                    const int32_t* slot_mapping, int B, int KV, int D, int NQ, int BLOCK,
                    int num_blocks, int dtype, int* status, void* stream)
{
    if (B < 0 || KV < 1 || D < 1 || NQ < 1 || BLOCK < 1 || num_blocks < 1)
        return PA_ERR_BAD_DIMS;
    if (dtype != PA_F32 && dtype != PA_F16 && dtype != PA_BF16)
        return PA_ERR_UNSUPPORTED;
    const long long row_bytes = static_cast<long long>(D) * elem_size(dtype);
    if (row_bytes % 16 != 0)
        return PA_ERR_UNSUPPORTED;
    const long long num_slots = static_cast<long long>(num_blocks) * BLOCK;
    const long long rows = static_cast<long long>(B) * KV * NQ;
    if (num_slots >= (1ll << 31) || rows * (row_bytes / 16) * 2 >= (1ll << 38))
        return PA_ERR_BAD_DIMS;
    if (B == 0)
        return PA_OK;
    if (!k_cache || !v_cache || !k_new || !v_new || !slot_mapping)
        return PA_ERR_NULL_POINTER;
    if (!aligned(k_cache, 16) || !aligned(v_cache, 16) || !aligned(k_new, 16) ||
        !aligned(v_new, 16) || !aligned(slot_mapping, 4))
        return PA_ERR_ALIGNMENT;
    return launch_append(k_cache, v_cache, k_new, v_new, slot_mapping, rows,
                         static_cast<int>(row_bytes / 16), KV, NQ, num_slots, status,
                         static_cast<cudaStream_t>(stream));
}

static int launch_append(void* k_cache, void* v_cache, const void* k_new, const void* v_new,
                         const int32_t* slots, long long rows, int vpr, int KV, int NQ,
                         long long num_slots, int* status, cudaStream_t stream)
{
    AppendParams a{};
    a.k_cache = static_cast<uint4*>(k_cache);
    a.v_cache = static_cast<uint4*>(v_cache);
    a.k_new = static_cast<const uint4*>(k_new);
    a.v_new = static_cast<const uint4*>(v_new);
    a.slots = slots;
    a.status = status;
    a.rows = rows;
    a.vpr = vpr;
    a.KV = KV;
    a.NQ = NQ;
    a.num_slots = num_slots;
    const long long threads = 2 * rows * a.vpr;
    pa_append_kernel<<<static_cast<unsigned>((threads + 255) / 256), 256, 0, stream>>>(a);
    if (cudaGetLastError() != cudaSuccess)
        return PA_ERR_CUDA;
    g_launches.fetch_add(1);
    return PA_OK;
}

// Page-locked host regions declared by pa_host_register: their device
// addresses are taken from here, without a runtime query per call.
namespace {
struct HostRegion {
    const char* lo;
    size_t bytes;
    const char* dev;
};
std::mutex g_host_mutex;
constexpr int kHostRegions = 64;
HostRegion g_host[kHostRegions];
int g_host_count = 0;

// Device address of [host, host + bytes) when it lies inside one registered
// region, else nullptr.
const void* registered_view(const void* host, size_t bytes)
{
    const char* p = static_cast<const char*>(host);
    std::lock_guard<std::mutex> lock(g_host_mutex);
    for (int i = 0; i < g_host_count; ++i) {
        const HostRegion& r = g_host[i];
        if (p >= r.lo && bytes <= r.bytes && static_cast<size_t>(p - r.lo) <= r.bytes - bytes)
            return r.dev + (p - r.lo);
    }
    return nullptr;
}

// The runtime's device address of a host pointer in page-locked memory, else
// nullptr (a pageable pointer is not an error for the caller).
const void* query_view(const void* host)
{
    cudaPointerAttributes a{};
    if (cudaPointerGetAttributes(&a, host) == cudaSuccess && a.type == cudaMemoryTypeHost)
        return a.devicePointer;
    cudaGetLastError();
    return nullptr;
}
}  // namespace

// Device address of [host, host + bytes) when it lies in page-locked memory:
// from a registered region, else asked of the runtime (on every call: an
// answer cached without registration could outlive the buffer it was taken for).
static const void* device_view(const void* host, size_t bytes)
{
    const void* r = registered_view(host, bytes);
    return r ? r : query_view(host);
}

int pa_host_register(const void* ptr, size_t bytes)
{
    if (!ptr || bytes == 0)
        return PA_ERR_NULL_POINTER;
    const char* lo = static_cast<const char*>(ptr);
    const char* d0 = static_cast<const char*>(query_view(lo));
    const char* d1 = static_cast<const char*>(query_view(lo + bytes - 1));
    if (!d0 || d1 != d0 + (bytes - 1))  // the whole range page-locked, mapped contiguously
        return PA_ERR_NOT_PINNED;
    std::lock_guard<std::mutex> lock(g_host_mutex);
    for (int i = 0; i < g_host_count; ++i)
        if (g_host[i].lo == lo) {  // registered again: the new extent replaces the old
            g_host[i].bytes = bytes;
            g_host[i].dev = d0;
            return PA_OK;
        }
    if (g_host_count == kHostRegions)
        return PA_ERR_BAD_DIMS;
    g_host[g_host_count++] = HostRegion{lo, bytes, d0};
    return PA_OK;
}

int pa_host_unregister(const void* ptr)
{
    std::lock_guard<std::mutex> lock(g_host_mutex);
    for (int i = 0; i < g_host_count; ++i)
        if (g_host[i].lo == ptr) {
            g_host[i] = g_host[--g_host_count];
            return PA_OK;
        }
    return PA_ERR_NULL_POINTER;
}

// Device workspace of pa_decode_host: the split workspace first (so that its
// leading zero bytes stay at offset 0), then 256-aligned staging for q, the
// table, the lengths, k_new, v_new and the output.
struct HostLayout {
    size_t q, table, lens, knew, vnew, out, total;
};

static HostLayout host_layout(size_t split_bytes, int batch, int max_blocks, int H, int KV, int D,
                              int NQ, int dtype, int out_dtype)
{
    const size_t es = elem_size(dtype), eo = elem_size(out_dtype < 0 ? dtype : out_dtype);
    HostLayout l{};
    size_t off = align_up(split_bytes, 256);
    l.q = off;
    off = align_up(off + static_cast<size_t>(batch) * H * NQ * D * es, 256);
    l.table = off;
    off = align_up(off + static_cast<size_t>(batch) * max_blocks * 4, 256);
    l.lens = off;
    off = align_up(off + static_cast<size_t>(batch) * 4, 256);
    l.knew = off;
    off = align_up(off + static_cast<size_t>(batch) * KV * NQ * D * es, 256);
    l.vnew = off;
    off = align_up(off + static_cast<size_t>(batch) * KV * NQ * D * es, 256);
    l.out = off;
    off = align_up(off + static_cast<size_t>(batch) * H * NQ * D * eo, 256);
    l.total = off;
    return l;
}

size_t pa_host_workspace_bytes(int batch, int max_blocks, int H, int KV, int D, int NQ,
                               int partitions, int dtype, int out_dtype)
{
    if (!ws_args_ok(batch, H, KV, D, NQ, partitions) || max_blocks < 1 || batch == 0 ||
        (dtype != PA_F32 && dtype != PA_F16 && dtype != PA_BF16))
        return 0;
    return host_layout(pa_workspace_bytes(batch, H, KV, D, NQ, partitions), batch, max_blocks, H,
                       KV, D, NQ, dtype, out_dtype)
        .total;
}

int pa_decode_host(const void* q, const void* k_cache, const void* v_cache,
                   const int32_t* block_table, const int32_t* seq_lens, const void* k_new,
                   const void* v_new, void* out, float scale, int H, int KV, int D, int BLOCK,
                   int NQ, int causal, const pa_opts* opts, void* stream)
{
    if (!opts)
        return PA_ERR_NULL_POINTER;
    const int B = opts->batch;
    if (B < 0 || H < 1 || KV < 1 || H % KV != 0 || opts->max_blocks < 1 || NQ < 1 ||
        NQ > PA_MAX_NQ || opts->partitions < 0)
        return PA_ERR_BAD_DIMS;
    if (B == 0)
        return PA_OK;
    if (!q || !block_table || !seq_lens || !k_new || !v_new || !out || !opts->workspace)
        return PA_ERR_NULL_POINTER;
    if (opts->dtype != PA_F32 && opts->dtype != PA_F16 && opts->dtype != PA_BF16)
        return PA_ERR_UNSUPPORTED;
    if (D != 64 && D != 128)
        return PA_ERR_UNSUPPORTED;
    const size_t split = pa_workspace_bytes(B, H, KV, D, NQ, opts->partitions);
    const HostLayout l = host_layout(split, B, opts->max_blocks, H, KV, D, NQ, opts->dtype,
                                     opts->out_dtype);
    if (opts->workspace_bytes < l.total)
        return PA_ERR_WORKSPACE;
    if (!aligned(opts->workspace, 256))
        return PA_ERR_ALIGNMENT;
    const size_t es = elem_size(opts->dtype);
    const size_t eo = elem_size(opts->out_dtype < 0 ? opts->dtype : opts->out_dtype);
    unsigned char* ws = static_cast<unsigned char*>(opts->workspace);
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    const size_t qb = static_cast<size_t>(B) * H * NQ * D * es;
    const size_t nb = static_cast<size_t>(B) * KV * NQ * D * es;
    struct {
        void* dst;
        const void* src;
        size_t bytes;
    } in[5] = {{ws + l.q, q, qb},
               {ws + l.table, block_table, static_cast<size_t>(B) * opts->max_blocks * 4},
               {ws + l.lens, seq_lens, static_cast<size_t>(B) * 4},
               {ws + l.knew, k_new, nb},
               {ws + l.vnew, v_new, nb}};
    // page-locked inputs (4-byte aligned): one gather kernel; else one copy each
    GatherParams g{};
    bool mapped = true;
    for (int i = 0; i < 5 && mapped; ++i) {
        const void* dv = device_view(in[i].src, in[i].bytes);
        mapped = dv && (reinterpret_cast<uintptr_t>(dv) & 3) == 0 && in[i].bytes < (1u << 30);
        g.src[i] = dv;
        g.dst[i] = in[i].dst;
        g.bytes[i] = static_cast<int>(in[i].bytes);
    }
    if (mapped) {
        size_t big = 0;
        for (const auto& c : in)
            big = c.bytes > big ? c.bytes : big;
        unsigned gx = static_cast<unsigned>((big / 16 + 255) / 256);
        gx = gx < 1 ? 1 : gx > 64 ? 64 : gx;
        pa_gather_kernel<<<dim3(gx, 5), 256, 0, st>>>(g);
        if (cudaGetLastError() != cudaSuccess)
            return PA_ERR_CUDA;
        g_launches.fetch_add(1);
    } else {
        for (const auto& c : in)
            if (cudaMemcpyAsync(c.dst, c.src, c.bytes, cudaMemcpyHostToDevice, st) != cudaSuccess)
                return PA_ERR_CUDA;
    }
    pa_opts dev = *opts;
    dev.inputs_unchanged = 0;  // the gather kernel just before writes the inputs
    dev.workspace = split ? ws : nullptr;
    dev.workspace_bytes = split;
    // a registered output is written by the kernels in place (no copy back)
    const size_t out_bytes = static_cast<size_t>(B) * H * NQ * D * eo;
    void* out_dev = const_cast<void*>(registered_view(out, out_bytes));
    const int rc = pa_decode(ws + l.q, k_cache, v_cache, reinterpret_cast<const int32_t*>(ws + l.table),
                             reinterpret_cast<const int32_t*>(ws + l.lens), ws + l.knew, ws + l.vnew,
                             out_dev ? out_dev : ws + l.out, scale, H, KV, D, BLOCK, NQ, causal, &dev, stream);
    if (rc != PA_OK || out_dev)
        return rc;
    if (cudaMemcpyAsync(out, ws + l.out, out_bytes, cudaMemcpyDeviceToHost, st) != cudaSuccess)
        return PA_ERR_CUDA;
    return PA_OK;
}

// ------------------------------------------------------------------ prefill
// A prefill of NQ new tokens per sequence runs as the cache append of all new
// rows (slots from the block table), then
//   - for 16-bit caches with D = 128 and more than PA_MAX_NQ new rows, one
//     tensor-core launch (pa_prefill_tc.cu) over 128-row query tiles;
//   - otherwise causal decodes of chunks of at most PA_MAX_NQ rows: chunk
//     [r0, r0 + n) sees seq_lens[b] + r0 cached tokens (the earlier chunks'
//     rows are in the cache by then) and its own rows as new rows.
// Either way row r attends to keys 0 .. seq_lens[b] + r.

// New row j of sequence b is token seq_lens[b] + j: its slot comes from the
// block table.  One thread per 16 bytes of one new row of K or V.
struct PrefillAppendParams {
    uint4* k_cache;
    uint4* v_cache;
    const uint4* k_new;
    const uint4* v_new;
    const int32_t* table;     // [B][maxb]
    const int32_t* seq_lens;  // [B]
    int* status;
    long long rows;           // B * KV * NQ
    int vpr, KV, NQ, BLOCK, maxb, num_blocks;
};

__global__ void __launch_bounds__(256)
    pa_prefill_append_kernel(const __grid_constant__ PrefillAppendParams a)
{
    // the tensor-core prefill that follows may start its set-up now; it waits
    // for this grid's completion before it reads the cache
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    const long long i = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x;
    const long long per = a.rows * a.vpr;
    if (i >= 2 * per)
        return;
    const bool is_v = i >= per;
    const long long k = is_v ? i - per : i;
    const long long row = k / a.vpr;
    const int v = static_cast<int>(k - row * a.vpr);
    const int j = static_cast<int>(row % a.NQ);
    const long long bk = row / a.NQ;  // b * KV + kh
    const int kh = static_cast<int>(bk % a.KV);
    const long long b = bk / a.KV;
    const bool reporter = a.status && !is_v && v == 0 && kh == 0;
    const int past = a.seq_lens[b];
    if (past < 0) {
        if (reporter)
            atomicOr(a.status, PA_STATUS_BAD_LENGTH);
        return;
    }
    const long long t = static_cast<long long>(past) + j;
    const long long blk = t / a.BLOCK;
    const int phys = blk < a.maxb ? a.table[b * a.maxb + blk] : -1;
    if (phys < 0 || phys >= a.num_blocks) {
        if (reporter)
            atomicOr(a.status, PA_STATUS_BAD_SLOT);
        return;
    }
    const long long slot = static_cast<long long>(phys) * a.BLOCK + (t - blk * a.BLOCK);
    const uint4* src = (is_v ? a.v_new : a.k_new) + row * a.vpr + v;
    uint4* dst = (is_v ? a.v_cache : a.k_cache) + (slot * a.KV + kh) * a.vpr + v;
    *dst = *src;
}

// Rows [src_r0, src_r0 + n) of each of `outer` groups of src_rows rows to rows
// [dst_r0, dst_r0 + n) of groups of dst_rows rows (vpr 16-byte vectors a row):
// a chunk's q, k_new, v_new into staging, or its output back.
struct RowCopy {
    const uint4* src;
    uint4* dst;
    long long outer;
    int src_rows, src_r0, dst_rows, dst_r0, n, vpr;
};

struct ChunkCopyParams {
    RowCopy seg[3];           // blockIdx.y selects one
    const int32_t* lens_in;   // with lens_out: lens_out[b] = lens_in[b] + add
    int32_t* lens_out;        // (a negative length is kept, for the decode to report)
    int B, add;
};

__global__ void __launch_bounds__(256) pa_chunk_copy_kernel(const __grid_constant__ ChunkCopyParams c)
{
    const RowCopy s = c.seg[blockIdx.y];
    const long long total = s.outer * s.n * s.vpr;
    const long long step = static_cast<long long>(gridDim.x) * blockDim.x;
    for (long long i = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x; i < total;
         i += step) {
        const long long rest = i / s.vpr;
        const int v = static_cast<int>(i - rest * s.vpr);
        const long long o = rest / s.n;
        const int r = static_cast<int>(rest - o * s.n);
        s.dst[(o * s.dst_rows + s.dst_r0 + r) * s.vpr + v] =
            s.src[(o * s.src_rows + s.src_r0 + r) * s.vpr + v];
    }
    if (c.lens_out && blockIdx.x == 0 && blockIdx.y == 0)
        for (int b = threadIdx.x; b < c.B; b += blockDim.x) {
            const long long len = c.lens_in[b];
            const long long moved = len < 0 ? len : len + c.add;
            c.lens_out[b] = static_cast<int32_t>(moved > INT32_MAX ? INT32_MAX : moved);
        }
}

static int launch_chunk_copy(const ChunkCopyParams& c, int nseg, cudaStream_t st)
{
    long long most = 0;
    for (int k = 0; k < nseg; ++k) {
        const long long t = c.seg[k].outer * c.seg[k].n * c.seg[k].vpr;
        most = t > most ? t : most;
    }
    long long gx = (most + 255) / 256;
    gx = gx < 1 ? 1 : gx > 1216 ? 1216 : gx;  // grid-stride beyond 8 CTAs per SM
    pa_chunk_copy_kernel<<<dim3(static_cast<unsigned>(gx), static_cast<unsigned>(nseg)), 256, 0,
                           st>>>(c);
    if (cudaGetLastError() != cudaSuccess)
        return PA_ERR_CUDA;
    g_launches.fetch_add(1);
    return PA_OK;
}

// Workspace of pa_prefill: the decode workspace of the largest chunk layout
// first (its leading zero bytes at offset 0), then 256-aligned staging for a
// chunk's q, k_new, v_new, output and lengths.
struct PrefillLayout {
    size_t split, zero, q, knew, vnew, out, lens, total;
};

static bool prefill_dtypes_ok(int dtype, int out_dtype)
{
    const bool in = dtype == PA_F32 || dtype == PA_F16 || dtype == PA_BF16;
    return in && (out_dtype < 0 || out_dtype == dtype || out_dtype == PA_F32);
}

static PrefillLayout prefill_layout(int B, int H, int KV, int D, int NQ, int partitions, int dtype,
                                    int out_dtype)
{
    PrefillLayout l{};
    const int C = NQ < PA_MAX_NQ ? NQ : PA_MAX_NQ;
    for (int n = 1; n <= C; ++n) {
        const size_t w = pa_workspace_bytes(B, H, KV, D, n, partitions);
        const size_t z = pa_workspace_zero_bytes(B, H, KV, D, n, partitions);
        l.split = w > l.split ? w : l.split;
        l.zero = z > l.zero ? z : l.zero;
    }
    const size_t es = elem_size(dtype), eo = elem_size(out_dtype < 0 ? dtype : out_dtype);
    size_t off = align_up(l.split, 256);
    l.q = off;
    off = align_up(off + static_cast<size_t>(B) * H * C * D * es, 256);
    l.knew = off;
    off = align_up(off + static_cast<size_t>(B) * KV * C * D * es, 256);
    l.vnew = off;
    off = align_up(off + static_cast<size_t>(B) * KV * C * D * es, 256);
    l.out = off;
    off = align_up(off + static_cast<size_t>(B) * H * C * D * eo, 256);
    l.lens = off;
    off = align_up(off + static_cast<size_t>(B) * 4, 256);
    l.total = off;
    return l;
}

static bool prefill_args_ok(int batch, int H, int KV, int D, int NQ, int partitions, int dtype,
                            int out_dtype)
{
    return ws_args_ok(batch, H, KV, D, 1, partitions) && NQ >= 1 && NQ <= PA_MAX_PREFILL &&
           batch <= kMaxBatch && prefill_dtypes_ok(dtype, out_dtype);
}

size_t pa_prefill_workspace_bytes(int batch, int H, int KV, int D, int NQ, int partitions,
                                  int dtype, int out_dtype)
{
    if (!prefill_args_ok(batch, H, KV, D, NQ, partitions, dtype, out_dtype) || batch == 0)
        return 0;
    return prefill_layout(batch, H, KV, D, NQ, partitions, dtype, out_dtype).total;
}

size_t pa_prefill_workspace_zero_bytes(int batch, int H, int KV, int D, int NQ, int partitions,
                                       int dtype, int out_dtype)
{
    if (!prefill_args_ok(batch, H, KV, D, NQ, partitions, dtype, out_dtype) || batch == 0)
        return 0;
    return prefill_layout(batch, H, KV, D, NQ, partitions, dtype, out_dtype).zero;
}

int pa_prefill(const void* q, void* k_cache, void* v_cache, const int32_t* block_table,
               const int32_t* seq_lens, const void* k_new, const void* v_new, void* out,
               float scale, int H, int KV, int D, int BLOCK, int NQ, const pa_opts* opts,
               void* stream)
{
    if (!opts)
        return PA_ERR_NULL_POINTER;
    const int B = opts->batch;
    if (B < 0 || H < 1 || KV < 1 || H % KV != 0 || NQ < 1 || opts->partitions < 0 ||
        opts->max_blocks < 1 || opts->num_blocks < 1)
        return PA_ERR_BAD_DIMS;
    if (NQ > PA_MAX_PREFILL || (D != 64 && D != 128) || !prefill_dtypes_ok(opts->dtype, opts->out_dtype))
        return PA_ERR_UNSUPPORTED;
    if (B == 0)
        return PA_OK;
    if (B > kMaxBatch)
        return PA_ERR_UNSUPPORTED;
    if (!q || !k_cache || !v_cache || !block_table || !seq_lens || !k_new || !v_new || !out)
        return PA_ERR_NULL_POINTER;
    if (!aligned(q, 16) || !aligned(k_cache, 16) || !aligned(v_cache, 16) ||
        !aligned(k_new, 16) || !aligned(v_new, 16) || !aligned(out, 16) ||
        !aligned(block_table, 4) || !aligned(seq_lens, 4))
        return PA_ERR_ALIGNMENT;
    const int dtype = opts->dtype;
    const int out_dtype = opts->out_dtype < 0 ? dtype : opts->out_dtype;
    const int vpr = D * static_cast<int>(elem_size(dtype)) / 16;
    const int vpr_o = D * static_cast<int>(elem_size(out_dtype)) / 16;
    const long long rows = static_cast<long long>(B) * KV * NQ;
    if (rows * vpr * 2 >= (1ll << 38))
        return PA_ERR_BAD_DIMS;
    const int C = NQ < PA_MAX_NQ ? NQ : PA_MAX_NQ;
    const int last = NQ - (NQ - 1) / C * C;  // rows of the last chunk, 1 .. C
    pa_opts dopts = *opts;
    dopts.trace_begin = nullptr;
    dopts.trace_split = nullptr;
    dopts.inputs_unchanged = 0;  // the store of the new rows (and chunk copies) come just before
    unsigned char* ws = static_cast<unsigned char*>(opts->workspace);
    const bool direct = NQ <= PA_MAX_NQ;  // one chunk: the caller's buffers serve the decode
    PrefillLayout l{};
    if (!direct) {
        l = prefill_layout(B, H, KV, D, NQ, opts->partitions, dtype, opts->out_dtype);
        if (!ws || opts->workspace_bytes < l.total)
            return PA_ERR_WORKSPACE;
        if (!aligned(ws, 256))
            return PA_ERR_ALIGNMENT;
        dopts.workspace = l.split ? ws : nullptr;
        dopts.workspace_bytes = l.split;
    }
    const void* cq = direct ? q : ws + l.q;
    const void* ckn = direct ? k_new : ws + l.knew;
    const void* cvn = direct ? v_new : ws + l.vnew;
    void* cout = direct ? out : ws + l.out;
    const int32_t* clens = direct ? seq_lens : reinterpret_cast<const int32_t*>(ws + l.lens);
    // every decode of the call is checked before the first launch
    for (int n : {C, last}) {
        const int rc = decode_impl(cq, k_cache, v_cache, block_table, clens, ckn, cvn, nullptr,
                                   cout, scale, H, KV, D, BLOCK, n, 1, &dopts, stream, false);
        if (rc != PA_OK)
            return rc;
    }

    cudaStream_t st = static_cast<cudaStream_t>(stream);
    PrefillAppendParams a{};
    a.k_cache = static_cast<uint4*>(k_cache);
    a.v_cache = static_cast<uint4*>(v_cache);
    a.k_new = static_cast<const uint4*>(k_new);
    a.v_new = static_cast<const uint4*>(v_new);
    a.table = block_table;
    a.seq_lens = seq_lens;
    a.status = opts->status;
    a.rows = rows;
    a.vpr = vpr;
    a.KV = KV;
    a.NQ = NQ;
    a.BLOCK = BLOCK;
    a.maxb = opts->max_blocks;
    a.num_blocks = opts->num_blocks;
    const long long threads = 2 * rows * vpr;
    pa_prefill_append_kernel<<<static_cast<unsigned>((threads + 255) / 256), 256, 0, st>>>(a);
    if (cudaGetLastError() != cudaSuccess)
        return PA_ERR_CUDA;
    g_launches.fetch_add(1);
    if (direct)
        return decode_impl(q, k_cache, v_cache, block_table, seq_lens, k_new, v_new, nullptr, out,
                           scale, H, KV, D, BLOCK, NQ, 1, &dopts, stream);
    if (prefill_tc_supported(dtype, D, H, KV, NQ)) {
        // 16-bit caches, D = 128: one tensor-core launch over all rows
        uint64_t n = 0;
        const int rc = launch_prefill_tc(q, k_cache, v_cache, block_table, seq_lens, out, scale, B, H,
                                         KV, BLOCK, NQ, opts->max_blocks, opts->num_blocks, dtype,
                                         out_dtype, opts->status, st, &n);
        g_launches.fetch_add(n);
        return rc;
    }

    for (int r0 = 0; r0 < NQ; r0 += C) {
        const int n = NQ - r0 < C ? NQ - r0 : C;
        ChunkCopyParams in{};
        in.seg[0] = {static_cast<const uint4*>(q), reinterpret_cast<uint4*>(ws + l.q),
                     static_cast<long long>(B) * H, NQ, r0, n, 0, n, vpr};
        in.seg[1] = {static_cast<const uint4*>(k_new), reinterpret_cast<uint4*>(ws + l.knew),
                     static_cast<long long>(B) * KV, NQ, r0, n, 0, n, vpr};
        in.seg[2] = {static_cast<const uint4*>(v_new), reinterpret_cast<uint4*>(ws + l.vnew),
                     static_cast<long long>(B) * KV, NQ, r0, n, 0, n, vpr};
        in.lens_in = seq_lens;
        in.lens_out = reinterpret_cast<int32_t*>(ws + l.lens);
        in.B = B;
        in.add = r0;
        int rc = launch_chunk_copy(in, 3, st);
        if (rc == PA_OK)
            rc = decode_impl(cq, k_cache, v_cache, block_table, clens, ckn, cvn, nullptr, cout,
                             scale, H, KV, D, BLOCK, n, 1, &dopts, stream);
        if (rc != PA_OK)
            return rc;
        ChunkCopyParams back{};
        back.seg[0] = {reinterpret_cast<const uint4*>(ws + l.out), static_cast<uint4*>(out),
                       static_cast<long long>(B) * H, n, 0, NQ, r0, n, vpr_o};
        rc = launch_chunk_copy(back, 1, st);
        if (rc != PA_OK)
            return rc;
    }
    return PA_OK;
}

}  // extern "C"
