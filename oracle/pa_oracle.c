/*
 * pa_oracle.c -- float64 CPU oracle for decode-step attention over a paged
 * KV cache.
 *
 * TEST INFRASTRUCTURE ONLY.  Only the tests, the smoke check and the CPU
 * baseline leg of the bench may load this library.  It shares no code,
 * header, table or helper with the CUDA path, and the CUDA path never calls
 * it.
 *
 * What it computes (the plain definition, no blocking, fusion or splitting):
 *
 *   onnxruntime-ep-mlx 0.31.1, src/ops/paged_attention.rs, VECTOR_BODY,
 *   VECTOR_REDUCE and PARTIALS_REDUCE together compute, for every query head
 *   h and new query row r of a sequence,
 *
 *     kh     = h / (H / KV)                      (grouped-query map)
 *     total  = past + (causal ? r + 1 : NQ)       (keys visible to row r)
 *     key i  = cache row table[i / BLOCK] * BLOCK + i % BLOCK   if i <  past
 *              (new row j instead when that cache row is the slot
 *              positions[j] names, for the last such j)
 *            = new row i - past                                  if i >= past
 *     s_i    = sum_d (scale * q[h][r][d]) * k_i[d]
 *     out    = sum_i softmax(s)_i * v_i ,   out = 0 when no key is visible.
 *
 *   The page's online softmax (running maximum, rescaled sum) and its split
 *   into partitions merged by a log-sum-exp reduction change only rounding,
 *   so the oracle evaluates the definition directly: one pass for the
 *   maximum, then exponentials, their sum, and the weighted sum of values,
 *   all in double precision and in logical key order.
 *
 * Readings of points the page leaves open:
 *   - The page handles one sequence per dispatch with position[0] as its
 *     cached length; here seq_lens[b] is the cached length of sequence b and
 *     each sequence has its own row of the block table.
 *   - The NQ new rows always come from k_new / v_new (the page's i >= past
 *     branch).  Slot patching (the page's position[1 + j]: new row j is
 *     bound for cache slot position[1 + j], and a cached key i < past whose
 *     slot offset / (KV * D) equals it reads new row j instead; the last
 *     such j wins) is modelled by pa_oracle_decode_positions, with
 *     positions[b][j] for sequence b; pa_oracle_decode is the same with no
 *     positions.
 *   - The empty-row convention (sum == 0 -> output the zero accumulator)
 *     follows the `sum == 0` guards of VECTOR_REDUCE and PARTIALS_REDUCE.
 *
 * Layouts (row-major, element offsets):
 *   q, out        [B][H][NQ][D]
 *   k_cache, v_c. [num_blocks][BLOCK][KV][D]
 *   block_table   [B][max_blocks]   (int32)
 *   seq_lens      [B]               (int32, cached tokens per sequence)
 *   k_new, v_new  [B][KV][NQ][D]
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#ifdef _OPENMP
#include <omp.h>
#endif

/* Error codes of the oracle (independent of the CUDA library's codes). */
#define ORACLE_OK 0
#define ORACLE_BAD_DIMS -1
#define ORACLE_BAD_LEN -2
#define ORACLE_BAD_BLOCK -3
#define ORACLE_NO_MEMORY -4

int pa_oracle_version(void) { return 1; }

int pa_oracle_max_threads(void)
{
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

/* Returns a pointer to the D values of key (or value) i of sequence b and KV
 * head kh, or NULL when the block table points outside the pool.  With
 * `positions` (NULL: none), a cached key whose slot a new row is bound for
 * reads that new row. */
static const double *key_row(const double *cache, const double *fresh,
                             const int32_t *block_table, const int32_t *positions,
                             int b, int kh, int i, int past, int KV, int D,
                             int BLOCK, int NQ, int max_blocks, int64_t num_blocks)
{
    if (i < past) {
        int32_t physical = block_table[(int64_t)b * max_blocks + i / BLOCK];
        if (physical < 0 || (int64_t)physical >= num_blocks)
            return NULL;
        int64_t slot = (int64_t)physical * BLOCK + i % BLOCK;
        int bound = -1; /* the last new row bound for this slot */
        if (positions)
            for (int p = 0; p < NQ; ++p) {
                int32_t target = positions[(int64_t)b * NQ + p];
                if (target >= 0 && (int64_t)target == slot)
                    bound = p;
            }
        if (bound >= 0)
            return fresh + (((int64_t)b * KV + kh) * NQ + bound) * D;
        return cache + (slot * KV + kh) * D;
    }
    int j = i - past; /* new row j of this step */
    return fresh + (((int64_t)b * KV + kh) * NQ + j) * D;
}

/*
 * Full decode step.  `positions`, when not NULL, is int32 [B][NQ]: the cache
 * slot new row j of sequence b is bound for, or a negative value for none.
 * `row_mask`, when not NULL, has B*H*NQ bytes; rows whose byte is 0 are
 * skipped and left untouched in `out` (used to sample rows of very large
 * cases).  `threads` <= 0 means the OpenMP default.
 */
int pa_oracle_decode_positions(const double *q, const double *k_cache,
                               const double *v_cache, const int32_t *block_table,
                               const int32_t *seq_lens, const double *k_new,
                               const double *v_new, const int32_t *positions,
                               double *out, double scale, int B, int H, int KV,
                               int D, int BLOCK, int NQ, int causal,
                               int max_blocks, int64_t num_blocks,
                               const uint8_t *row_mask, int threads)
{
    if (B < 0 || H < 1 || KV < 1 || H % KV != 0 || D < 1 || BLOCK < 1 ||
        NQ < 1 || max_blocks < 0 || num_blocks < 0)
        return ORACLE_BAD_DIMS;
    for (int b = 0; b < B; ++b)
        if (seq_lens[b] < 0 || (int64_t)seq_lens[b] > (int64_t)max_blocks * BLOCK)
            return ORACLE_BAD_LEN;

    const int group = H / KV;
    const int64_t rows = (int64_t)B * H * NQ;
    int status = ORACLE_OK;

#ifdef _OPENMP
    if (threads > 0)
        omp_set_num_threads(threads);
#pragma omp parallel for schedule(dynamic, 1)
#endif
    for (int64_t flat = 0; flat < rows; ++flat) {
        if (row_mask && !row_mask[flat])
            continue;
        const int r = (int)(flat % NQ);
        const int h = (int)((flat / NQ) % H);
        const int b = (int)(flat / ((int64_t)NQ * H));
        const int kh = h / group;
        const int past = seq_lens[b];
        const int total = past + (causal ? r + 1 : NQ);
        const double *qrow = q + flat * D;
        double *orow = out + flat * D;

        double *s = (double *)malloc(sizeof(double) * (size_t)(total > 0 ? total : 1));
        if (!s) {
#ifdef _OPENMP
#pragma omp atomic write
#endif
            status = ORACLE_NO_MEMORY;
            continue;
        }

        /* scores s_i = sum_d (scale * q_d) * k_i[d] */
        int bad = 0;
        for (int i = 0; i < total && !bad; ++i) {
            const double *k = key_row(k_cache, k_new, block_table, positions, b,
                                      kh, i, past, KV, D, BLOCK, NQ, max_blocks,
                                      num_blocks);
            if (!k) {
                bad = 1;
                break;
            }
            double dot = 0.0;
            for (int d = 0; d < D; ++d)
                dot += (scale * qrow[d]) * k[d];
            s[i] = dot;
        }
        if (bad) {
            free(s);
#ifdef _OPENMP
#pragma omp atomic write
#endif
            status = ORACLE_BAD_BLOCK;
            continue;
        }

        /* softmax(s) . V, stabilised by the maximum score */
        double m = -INFINITY;
        for (int i = 0; i < total; ++i)
            if (s[i] > m)
                m = s[i];
        double denom = 0.0;
        for (int i = 0; i < total; ++i) {
            s[i] = exp(s[i] - m);
            denom += s[i];
        }
        for (int d = 0; d < D; ++d)
            orow[d] = 0.0;
        for (int i = 0; i < total; ++i) {
            const double *v = key_row(v_cache, v_new, block_table, positions, b,
                                      kh, i, past, KV, D, BLOCK, NQ, max_blocks,
                                      num_blocks);
            for (int d = 0; d < D; ++d)
                orow[d] += s[i] * v[d];
        }
        if (denom != 0.0)
            for (int d = 0; d < D; ++d)
                orow[d] /= denom;
        free(s);
    }
    return status;
}

int pa_oracle_decode(const double *q, const double *k_cache,
                     const double *v_cache, const int32_t *block_table,
                     const int32_t *seq_lens, const double *k_new,
                     const double *v_new, double *out, double scale, int B,
                     int H, int KV, int D, int BLOCK, int NQ, int causal,
                     int max_blocks, int64_t num_blocks,
                     const uint8_t *row_mask, int threads)
{
    return pa_oracle_decode_positions(q, k_cache, v_cache, block_table, seq_lens,
                                      k_new, v_new, NULL, out, scale, B, H, KV,
                                      D, BLOCK, NQ, causal, max_blocks,
                                      num_blocks, row_mask, threads);
}
