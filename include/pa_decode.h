/*
 * pa_decode.h -- C ABI of libpadecode.so: decode-step attention over a paged
 * KV cache on NVIDIA GB300 (sm_103a).
 *
 * The operation is the one defined by onnxruntime-ep-mlx 0.31.1,
 * src/ops/paged_attention.rs (VECTOR_BODY: paged gather, grouped-query map,
 * causal bound, online softmax; VECTOR_PARTIALS / PARTIALS_REDUCE: the split
 * into partitions and their log-sum-exp merge; fn vector: the arguments).
 * For every sequence b, query head h and new row r:
 *
 *   kh    = h / (H / KV)
 *   past  = seq_lens[b]
 *   total = past + (causal ? r + 1 : NQ)
 *   key i = k_cache row (block_table[b][i / BLOCK] * BLOCK + i % BLOCK, kh)
 *           for i < past, else k_new[b][kh][i - past]   (values likewise)
 *   out[b][h][r] = sum_i softmax_i(scale * q[b][h][r] . key_i) * value_i
 *
 * Layouts (row-major, element offsets, no padding):
 *   q, out           [B][H][NQ][D]
 *   k_cache, v_cache [num_blocks][BLOCK][KV][D]
 *   block_table      [B][max_blocks]   int32 physical block ids
 *   seq_lens         [B]               int32 cached tokens per sequence
 *   k_new, v_new     [B][KV][NQ][D]    the NQ rows appended this step
 *
 * Ownership: every pointer argument is a caller-owned DEVICE pointer (the
 * library allocates no memory and never synchronises); every call is
 * asynchronous on `stream` (a cudaStream_t, NULL = legacy default stream).
 * Table entries are read only for blocks that hold visible keys; entries past
 * a sequence's last block and cache slots past its length are never read.
 *
 * Entry points: pa_decode, pa_decode_static_workspace and pa_decode_host
 * read the caches; pa_cache_append (the step's new rows into their slots),
 * pa_decode_positions (a decode step with slot patching) and pa_prefill (a
 * causal prefill of up to PA_MAX_PREFILL new rows, in chunks) also write the
 * new rows into them.
 *
 * Errors: functions return PA_OK (0) or a negative PA_ERR_* code before
 * anything is launched; pa_strerror() names what to verify.  Conditions that
 * only the device can see (a table entry outside the pool in checked mode, a
 * length larger than max_blocks * BLOCK) are OR-ed into *opts->status as
 * PA_STATUS_* bits and become visible after the caller synchronises; the
 * kernels never trap.
 */
#ifndef PA_DECODE_H
#define PA_DECODE_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* element types of q, caches, k_new, v_new (and out) */
#define PA_F32 0
#define PA_F16 1
#define PA_BF16 2

/* return codes */
#define PA_OK 0
#define PA_ERR_NULL_POINTER (-1) /* a required pointer (or opts) is NULL */
#define PA_ERR_BAD_DIMS (-2)     /* H % KV != 0, a size < 1, or a size too large */
#define PA_ERR_UNSUPPORTED (-3)  /* D, BLOCK, NQ, dtype or out_dtype outside the built set */
#define PA_ERR_ALIGNMENT (-4)    /* a data pointer is not 16-byte aligned (workspace: 256) */
#define PA_ERR_WORKSPACE (-5)    /* workspace NULL or smaller than pa_workspace_bytes() */
#define PA_ERR_CUDA (-6)         /* a CUDA runtime call or kernel launch failed */
#define PA_ERR_DRIVER (-7)       /* the tensor-map encoder of the driver is unavailable */
#define PA_ERR_STATIC_LIMIT (-8) /* pa_decode_static_workspace: the call needs more
                                    scratch than PA_STATIC_WORKSPACE_BYTES */
#define PA_ERR_NOT_PINNED (-9)   /* pa_host_register: the range is not page-locked host
                                    memory mapped for the device */

/* device status bits, OR-ed into *opts->status when it is not NULL */
#define PA_STATUS_BAD_BLOCK 1  /* checked mode: a table entry outside [0, num_blocks) */
#define PA_STATUS_BAD_LENGTH 2 /* seq_lens[b] < 0 or > max_blocks * BLOCK (clamped) */
#define PA_STATUS_TIMEOUT 4    /* an internal wait gave up (the output is undefined) */
#define PA_STATUS_BAD_SLOT 8   /* a new row's slot < -1 or >= num_blocks * BLOCK, or (pa_prefill)
                                  its token beyond the table: the row is not stored */

/* supported sizes */
#define PA_MAX_NQ 16           /* new rows per sequence of one decode call */
#define PA_MAX_PREFILL 65536   /* new rows per sequence of one pa_prefill call */

/* scratch built into the library for pa_decode_static_workspace (16 MiB) */
#define PA_STATIC_WORKSPACE_BYTES ((size_t)16 << 20)

typedef struct pa_opts {
    int batch;       /* B, sequences in this call (0 = nothing to do) */
    int max_blocks;  /* row stride of block_table (entries per sequence) */
    int num_blocks;  /* physical blocks in each of k_cache and v_cache */
    int dtype;       /* PA_F32, PA_F16 or PA_BF16: q, k_cache, v_cache, k_new, v_new */
    int out_dtype;   /* -1 = same as dtype; or PA_F32 for a float32 output */
    int partitions;  /* 0 = automatic split, 1 = one pass per sequence,
                        P >= 2 = each sequence split into P key ranges */
    int checked;     /* nonzero: report table entries outside the pool */
    void *workspace; /* device scratch of >= pa_workspace_bytes() bytes, 256-aligned;
                        may be NULL when partitions == 1.  With partitions == 0
                        and merge_kernel == 0 its first pa_workspace_zero_bytes()
                        bytes (split counters) must be zero before its first
                        use; every call that completes leaves them zero again
                        (after a call that reports PA_STATUS_TIMEOUT, zero them
                        once more) */
    size_t workspace_bytes;
    int *status;        /* device int32 for PA_STATUS_* bits, or NULL */
    void *trace_begin;  /* optional cudaEvent_t recorded before the partition kernel */
    void *trace_split;  /* optional cudaEvent_t recorded after it (before the merge) */
    int merge_kernel;   /* automatic split (partitions == 0): 0 (default), the
                           partition kernel's last CTA to finish a split segment
                           merges its partial states; 1, a separate log-sum-exp
                           merge kernel does (no counters needed).  Fixed
                           partitions (P >= 2) always use the merge kernel */
    /* Failure testing (0 = off, the default of a zero-filled pa_opts):
     * wait_limit_ns        limit of every wait inside the partition kernel
     *                      (0: 2 seconds); a wait that runs out sets
     *                      PA_STATUS_TIMEOUT, every warp of the CTA leaves, and
     *                      no copy is left in flight when it exits
     * debug_withhold_stage k > 0: the V-issuing warp of each partition-kernel
     *                      CTA leaves its k-th pipeline stage out, so that the
     *                      waits for that stage run out (the output is then
     *                      undefined; zero the split counters again after it) */
    unsigned long long wait_limit_ns;
    int debug_withhold_stage;
    /* inputs_unchanged = 1: the caller guarantees that the kernel enqueued on
     * `stream` just before this call writes none of q, k_cache, v_cache,
     * block_table, seq_lens, k_new, v_new (for example: the previous decode
     * step of the same batch).  The partition kernel then reads them (the
     * lengths, the schedule, the table, the first stages of K and V) before
     * that kernel has completed; it still waits for it before writing out or
     * the workspace.  0 (default): every input is read after it.  Ignored by
     * pa_decode_positions, pa_decode_host and pa_prefill, which run their
     * own kernels just before the decode. */
    int inputs_unchanged;
    /* kernel = 0 (default): 16-bit inputs with D = 128 and more than 16 query
     * rows per KV head (H/KV * NQ > 16) run the tcgen05 partition kernel
     * (S^T = K Q^T and O^T += V^T P^T on the tensor cores, accumulators in
     * tensor memory), when its shared memory fits beside two pipeline stages;
     * every other case runs the mma.sync kernels.  1: the mma.sync kernels
     * for every 16-bit case (same results within the tolerance; for
     * comparison).  Other values: PA_ERR_UNSUPPORTED. */
    int kernel;
} pa_opts;

/*
 * Decode attention for `opts->batch` sequences (see the definition above).
 * Launches the partition kernel (persistent CTAs, one per SM, each taking
 * (sequence, KV head) segments or key ranges of them; a CTA serves all
 * H/KV * NQ query rows of its KV head, so each K/V row is read from memory
 * once) and, with fixed partitions (partitions >= 2) or merge_kernel = 1, the
 * log-sum-exp merge kernel for sequences that were split.
 *   scale     multiplies q . k, applied in float32 exactly as given
 *   H, KV     query heads and KV heads, H % KV == 0
 *   D         head size, 64 or 128
 *   BLOCK     tokens per cache block, 8, 16, 32 or 64
 *   NQ        new rows this step, 1 .. PA_MAX_NQ
 *   causal    nonzero: new row r sees the past and new rows 0..r only
 *   stream    cudaStream_t to launch on
 * Returns PA_OK or a PA_ERR_* code.
 */
int pa_decode(const void *q, const void *k_cache, const void *v_cache,
              const int32_t *block_table, const int32_t *seq_lens,
              const void *k_new, const void *v_new, void *out, float scale,
              int H, int KV, int D, int BLOCK, int NQ, int causal,
              const pa_opts *opts, void *stream);

/*
 * pa_decode for callers that cannot allocate device memory.  The paged
 * attention page has no counterpart to this entry point; it exists for
 * callers such as an engine plugin that is handed only its input and output
 * buffers (the host framework owns every device allocation), a serving loop
 * that reserved all device memory up front, or latency-critical code that
 * must not pay the device-wide synchronisation a cudaMalloc/cudaFree brings.
 *
 * Same arguments and results as pa_decode, except that opts->workspace and
 * opts->workspace_bytes are ignored: the split scratch is a fixed array
 * inside the library, PA_STATIC_WORKSPACE_BYTES per GPU, which every GPU that
 * loads the library holds until the process exits.  The call allocates and
 * frees nothing.
 *   - A call whose pa_workspace_bytes() exceeds PA_STATIC_WORKSPACE_BYTES
 *     returns PA_ERR_STATIC_LIMIT and launches nothing (use fewer partitions,
 *     partitions == 1, or pa_decode with your own workspace).
 *   - The first call on a device looks up the array's device address with
 *     that device current, and so does the first call after the device's
 *     context was reset or replaced (the address is cached per context); make
 *     those calls before any stream capture starts.
 *   - All calls on a device share the array, which keeps whatever the last
 *     call left in it.  Nothing in it has to start at zero (this entry point
 *     always merges split sequences with the separate merge kernel, and each
 *     call writes every value it later reads), but two calls whose kernels
 *     overlap on the GPU (different streams, or host threads racing on one
 *     device) corrupt each other's results: issue them on one stream.
 */
int pa_decode_static_workspace(const void *q, const void *k_cache, const void *v_cache,
                               const int32_t *block_table, const int32_t *seq_lens,
                               const void *k_new, const void *v_new, void *out, float scale,
                               int H, int KV, int D, int BLOCK, int NQ, int causal,
                               const pa_opts *opts, void *stream);

/*
 * pa_decode for a step whose inputs and output live in host memory, as in a
 * serving loop that assembles each step's queries, block table and lengths on
 * the CPU.  The paged attention page passes its arrays through the host
 * framework; this entry point keeps that shape without allocating.
 *
 * q, block_table, seq_lens, k_new, v_new (read) and out (written) are HOST
 * pointers with the layouts of pa_decode; pinned (page-locked) memory makes
 * the copies asynchronous.  k_cache and v_cache are device pointers (the cache
 * stays resident).  opts->workspace is a device buffer of at least
 * pa_host_workspace_bytes() bytes, 256-byte aligned: it holds the split
 * workspace of pa_decode first (its leading pa_workspace_zero_bytes() bytes
 * follow the same zero rule), then the device copies of the inputs and of the
 * output.
 *
 * Enqueues on `stream`: the inputs' move to the device, the decode, and the
 * device-to-host copy of the output.  When every input lies in page-locked
 * memory (cudaHostAlloc / cudaHostRegister, 4-byte aligned), one gather kernel
 * reads them through their device addresses; otherwise each input gets its
 * own host-to-device copy.  Returns without waiting: `out` holds the result
 * once the stream has passed that copy (synchronise the stream before reading
 * it, and do not modify the inputs before then).  Errors as pa_decode;
 * PA_ERR_WORKSPACE when the workspace is too small.
 */
int pa_decode_host(const void *q, const void *k_cache, const void *v_cache,
                   const int32_t *block_table, const int32_t *seq_lens, const void *k_new,
                   const void *v_new, void *out, float scale, int H, int KV, int D, int BLOCK,
                   int NQ, int causal, const pa_opts *opts, void *stream);

/*
 * Declares the page-locked host memory [ptr, ptr + bytes) (cudaHostAlloc,
 * cudaHostRegister, a pinned framework tensor) to pa_decode_host, which then
 * takes its device address from this record instead of asking the runtime on
 * every call, and writes an `out` that lies in such a region directly from
 * the kernels (no separate copy back).  The whole range must be page-locked
 * and mapped for the device (else PA_ERR_NOT_PINNED); registering the same
 * ptr again replaces its extent; at most 64 regions (else PA_ERR_BAD_DIMS).
 * Call pa_host_unregister(ptr) before the memory is freed or unpinned: a
 * record that outlives its buffer makes the kernels read or write memory that
 * no longer belongs to it.  Host-side bookkeeping only (thread-safe); nothing
 * is enqueued.
 */
int pa_host_register(const void *ptr, size_t bytes);
int pa_host_unregister(const void *ptr);  /* PA_OK, or PA_ERR_NULL_POINTER if unknown */

/*
 * Device workspace bytes of pa_decode_host for these sizes (opts->max_blocks,
 * opts->dtype and opts->out_dtype as in the call; -1 = same as dtype).
 * Returns 0 for invalid arguments.
 */
size_t pa_host_workspace_bytes(int batch, int max_blocks, int H, int KV, int D, int NQ,
                               int partitions, int dtype, int out_dtype);

/*
 * How the automatic split (partitions == 0) of pa_decode divides a batch: the
 * counterpart of the paged attention page's partition chooser
 * (onnxruntime-ep-mlx 0.31.1, src/ops/paged_attention.rs: fn partitions, and
 * fn vector, which launches one threadgroup per partition).  Where the page
 * picks one partition count from a table of Apple GPU sizes, the partition
 * kernel here lays every (sequence, row group, KV head) segment end to end,
 * cut into stage-sized units, and gives each of its persistent CTAs an equal
 * share of the cost (units plus a fixed charge per segment); a segment is
 * split where a CTA's share ends inside it.  Splits are merged by the last
 * CTA to finish a piece of the segment, which costs it about four stages, so
 * when the segments are no more than those CTAs and the longest is at most a
 * CTA's share of the stages plus four, every CTA takes one whole segment
 * instead (none split; this assumes the default in-kernel merge).  This call
 * repeats that arithmetic on the host for given lengths.
 *   host_seq_lens  HOST int32 [batch] cached tokens per sequence, or NULL: all
 *                  sequences hold max_len tokens
 *   max_len        the table's capacity in tokens (max_blocks * BLOCK): lengths
 *                  are clamped to [0, max_len] as the kernel does
 *   sms            CTAs of the partition kernel (one per SM), or 0: the SM count
 *                  of the current device
 * Fills *plan and returns plan->max_pieces (>= 1: the effective partition
 * count, the most pieces one segment is split into), or a PA_ERR_* code
 * (PA_ERR_CUDA when sms == 0 and no device answers).
 */
typedef struct pa_split_plan {
    int grid;            /* partition-kernel CTAs launched */
    int active;          /* CTAs that receive units: each at least 4 stages of cost,
                            unless the segments are more; at most grid and the cost */
    int segments;        /* (sequence, row group, KV head) segments */
    int pieces;          /* pieces over all segments (a segment's piece per CTA) */
    int split_segments;  /* segments cut between two or more CTAs */
    int records;         /* partial records those pieces write (merged after) */
    int max_pieces;      /* the most pieces of one segment */
} pa_split_plan;

int pa_choose_partitions(const int32_t *host_seq_lens, int max_len, int batch, int H, int KV, int D,
                         int BLOCK, int NQ, int dtype, int sms, pa_split_plan *plan);

/*
 * Bytes of workspace pa_decode needs for these sizes (0 when partitions == 1).
 * Depends only on the arguments, not on the device or the lengths: it holds
 * a per-sequence schedule and one float32 partial state (max, sum, D
 * accumulators) per query row for every key range the split can produce.
 * Returns 0 for arguments pa_decode rejects (including batch > 4096, which
 * pa_decode reports as PA_ERR_UNSUPPORTED).
 */
size_t pa_workspace_bytes(int batch, int H, int KV, int D, int NQ, int partitions);

/*
 * Leading bytes of the workspace that must be zero before its first use with
 * the in-kernel merge (per-segment split counters; see pa_opts.workspace).
 * 0 unless partitions == 0.  Returns 0 for invalid arguments.
 */
size_t pa_workspace_zero_bytes(int batch, int H, int KV, int D, int NQ, int partitions);

/*
 * Writes the step's new rows into the paged cache: for every sequence b, new
 * row j and KV head kh with s = slot_mapping[b * NQ + j] >= 0,
 *     k_cache[s / BLOCK][s % BLOCK][kh][:] = k_new[b][kh][j][:]
 *     v_cache[s / BLOCK][s % BLOCK][kh][:] = v_new[b][kh][j][:]
 * (a slot is physical_block * BLOCK + offset, the cache position that the
 * block table gives a logical token: table[b][t / BLOCK] * BLOCK + t % BLOCK).
 * This is the cache update that follows a decode step on the paged-attention
 * page, where the host framework writes the rows back after evaluation; here
 * it is one kernel.  Rows are copied as stored (no conversion).
 *
 * k_cache, v_cache: device, [num_blocks][BLOCK][KV][D], written.  k_new,
 * v_new: device, [B][KV][NQ][D], read.  slot_mapping: device int32 [B][NQ];
 * -1 skips a row; a slot < -1 or >= num_blocks * BLOCK skips it and ORs
 * PA_STATUS_BAD_SLOT into *status (device int32, may be NULL).  When several
 * new rows of one sequence name one slot, the last of them (largest j) is
 * stored; when rows of different sequences name one slot, one of them lands,
 * unspecified which.  dtype: PA_F32, PA_F16 or PA_BF16 (D * element bytes a
 * multiple of 16).  Pointers of the caches and new rows 16-byte aligned,
 * slot_mapping 4-byte aligned.
 *
 * Enqueues one kernel on `stream` (B == 0: nothing) and returns PA_OK, or a
 * PA_ERR_* code before any launch (NULL pointer, sizes, alignment, dtype).
 */
int pa_cache_append(void *k_cache, void *v_cache, const void *k_new, const void *v_new,
                    const int32_t *slot_mapping, int B, int KV, int D, int NQ, int BLOCK,
                    int num_blocks, int dtype, int *status, void *stream);

/*
 * A decode step with slot patching (onnxruntime-ep-mlx 0.31.1,
 * src/ops/paged_attention.rs, VECTOR_BODY: entry 1 + j of the position
 * vector).  positions[b * NQ + j] is the cache slot (physical_block * BLOCK +
 * offset) that new row j of sequence b is bound for, or -1.  On that page the
 * kernel reads a cached key i < past whose slot a new row of its sequence is
 * bound for from that new row instead (the last such row wins), and the host
 * writes the new rows into the cache after the step.  Here the write comes
 * first: this call enqueues pa_cache_append(k_cache, v_cache, k_new, v_new,
 * positions, ...) and then pa_decode over the updated cache, so once the
 * stream has run, the caches hold the new rows and `out` is the page's
 * read-time substitution, provided no sequence's past covers a slot that a
 * new row of another sequence is bound for and no two sequences name one
 * slot (both hold when every sequence owns the blocks it writes).
 *
 * Arguments as pa_decode, except: k_cache and v_cache are written (the rows
 * named by positions); positions is device int32 [batch][NQ], 4-byte aligned,
 * NULL for a plain pa_decode.  Slots < -1 or >= num_blocks * BLOCK are skipped
 * and OR PA_STATUS_BAD_SLOT into *opts->status.  Every argument is checked
 * before the first launch; returns PA_OK or a PA_ERR_* code.
 */
int pa_decode_positions(const void *q, void *k_cache, void *v_cache,
                        const int32_t *block_table, const int32_t *seq_lens,
                        const void *k_new, const void *v_new, const int32_t *positions,
                        void *out, float scale, int H, int KV, int D, int BLOCK, int NQ,
                        int causal, const pa_opts *opts, void *stream);

/*
 * Causal prefill of NQ new tokens per sequence over the paged cache (the
 * chunked form of the decode step: onnxruntime-ep-mlx 0.31.1,
 * src/ops/paged_attention.rs, VECTOR_BODY with its causal bound, for any
 * number of new rows).  New row j of sequence b is token past + j, past =
 * seq_lens[b]; its output row r attends to keys 0 .. past + r: the cached
 * keys through the block table and new rows 0 .. r.  The call also stores the
 * new rows in the cache at the slots the block table gives those tokens,
 * table[b][t / BLOCK] * BLOCK + t % BLOCK for t = past + j, so the table must
 * hold blocks for past + NQ tokens (a token beyond it, or an entry outside
 * [0, num_blocks), skips that row's store and ORs PA_STATUS_BAD_SLOT into
 * *opts->status; the decode then reports PA_STATUS_BAD_LENGTH).
 *
 * It enqueues the store of all new rows, then causal decodes of chunks of at
 * most PA_MAX_NQ rows: chunk [r0, r0 + n) attends to past + r0 cached tokens
 * (the earlier rows are in the cache by then) and its n rows as new rows.
 * With NQ > PA_MAX_NQ the chunk's q, k_new, v_new and output pass through
 * staging in the workspace.
 *
 * Arguments as pa_decode with causal = 1, except: NQ is 1 .. PA_MAX_PREFILL;
 * k_cache and v_cache are written; opts->workspace holds at least
 * pa_prefill_workspace_bytes() bytes (256-aligned; its first
 * pa_prefill_workspace_zero_bytes() bytes zero before the first use, and left
 * zero by every call that completes), or, for NQ <= PA_MAX_NQ, what pa_decode
 * needs; opts->trace_begin / trace_split are ignored.  Every argument of every
 * chunk is checked before the first launch; returns PA_OK or a PA_ERR_* code.
 */
int pa_prefill(const void *q, void *k_cache, void *v_cache, const int32_t *block_table,
               const int32_t *seq_lens, const void *k_new, const void *v_new, void *out,
               float scale, int H, int KV, int D, int BLOCK, int NQ, const pa_opts *opts,
               void *stream);

/* Workspace of pa_prefill and its leading bytes that must be zero (0 for
 * invalid arguments or batch == 0).  out_dtype as in pa_opts (-1 = dtype). */
size_t pa_prefill_workspace_bytes(int batch, int H, int KV, int D, int NQ, int partitions,
                                  int dtype, int out_dtype);
size_t pa_prefill_workspace_zero_bytes(int batch, int H, int KV, int D, int NQ, int partitions,
                                       int dtype, int out_dtype);

/* A sentence naming what to verify for a PA_ERR_* code (static storage). */
const char *pa_strerror(int code);

/* Library version: major * 10000 + minor * 100 + patch. */
int pa_version(void);

/* Kernels this library has launched since it was loaded (all devices). */
uint64_t pa_kernel_launches(void);

#ifdef __cplusplus
}
#endif

#endif /* PA_DECODE_H */
