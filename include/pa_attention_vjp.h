/*
 * pa_attention_vjp.h -- C ABI of the dense attention backward (VJP).
 *
 * The operation is onnxruntime-ep-mlx 0.31.1, src/ops/attention_vjp/dense.rs,
 * fn execute: given the forward inputs q, k, v, the forward output y and the
 * gradient g arriving at y, it returns dq, dk and dv of
 *
 *   y = softmax(scale * q k^T + bias) v     (per query head h, with key/value
 *                                           head h / (HQ / HK))
 *
 * evaluated as that page does it:
 *
 *   p     = the softmax above, 0 on a row with no visible key
 *   dv    = sum over the query heads of a group of p^T g
 *   dp    = g v^T
 *   delta = rowsum(y * g)                  (the y passed in, not a recomputed one)
 *   ds    = p * (dp - delta)
 *   dq    = scale * ds k
 *   dk    = scale * sum over the group of ds^T q
 *
 * (the page scales q and k by sqrt(scale) each; that is the same product).
 *
 * Masks (pa_vjp_opts.mask_kind):
 *   PA_VJP_MASK_NONE  no bias.
 *   PA_VJP_MASK_BOOL  uint8 mask, nonzero = the key is visible (bias 0),
 *                     zero = hidden (bias -inf).
 *   PA_VJP_MASK_ADD   float32 additive bias (natural-log units, -inf hides).
 *   The mask is dense, row-major, of dims {MB, MH, MQ, W} = mask_dims with
 *   MB in {1, B}, MH in {1, HQ}, MQ in {1, SQ}, 1 <= W <= SK; a dim of 1
 *   broadcasts.  W == 1 broadcasts over keys; 1 < W < SK hides keys W..SK-1
 *   (the page pads the mask with -inf).  causal = 1 also hides key j from
 *   query row i when j > i (top-left aligned: row i sees keys 0..i).
 *
 * Layouts (row-major, contiguous, device memory, 16-byte aligned):
 *   q, y, g, dq : [B][HQ][SQ][D]      k, v, dk, dv : [B][HK][SK][D]
 *   q, k, v, y, g in opts->dtype; dq, dk, dv in opts->out_dtype.
 * Ownership: every pointer is the caller's; nothing is kept after the call.
 * The call only enqueues work on `stream` (a cudaStream_t, NULL = legacy
 * default stream) and returns; results are ready when the stream reaches
 * that point.  dq, dk and dv are fully overwritten (rows with no visible key
 * get dq = 0; keys no row sees get dk = dv = 0).
 *
 * Returns PA_OK or a PA_ERR_* code of pa_decode.h, checked before any launch:
 *   PA_ERR_NULL_POINTER  a tensor, opts, the mask (mask_kind != 0) or a needed
 *                        workspace is NULL;
 *   PA_ERR_BAD_DIMS      a size < 0 (HQ, HK, D < 1), HQ % HK != 0, scale not
 *                        positive and finite, bad mask dims, or a tensor of
 *                        2^31 elements or more;
 *   PA_ERR_UNSUPPORTED   D > 256, a dtype / out_dtype outside the set below,
 *                        B > 65535 or HQ > 65535;
 *   PA_ERR_ALIGNMENT     a tensor not 16-byte aligned, a workspace not 256;
 *   PA_ERR_WORKSPACE     workspace smaller than pa_attention_vjp_workspace_bytes;
 *   PA_ERR_DRIVER / PA_ERR_CUDA as for pa_decode.
 * dtype: PA_F32, PA_F16 or PA_BF16.  out_dtype: -1 (= dtype) or PA_F32.
 * Arithmetic: float32 accumulation.  float32 inputs use CUDA-core kernels;
 * 16-bit inputs with D = 128 (or 64) use tcgen05 tensor-core kernels whose
 * products take p and ds rounded to the input's 16-bit type.
 */
#ifndef PA_ATTENTION_VJP_H
#define PA_ATTENTION_VJP_H

#include <stddef.h>
#include <stdint.h>

#include "pa_decode.h"

#ifdef __cplusplus
extern "C" {
#endif

#define PA_VJP_MASK_NONE 0
#define PA_VJP_MASK_BOOL 1
#define PA_VJP_MASK_ADD 2

typedef struct pa_vjp_opts {
    int dtype;         /* PA_F32, PA_F16, PA_BF16: q, k, v, y, g */
    int out_dtype;     /* -1 (= dtype) or PA_F32: dq, dk, dv */
    int causal;        /* 1: row i sees keys 0..i only */
    int mask_kind;     /* PA_VJP_MASK_* */
    int mask_dims[4];  /* MB, MH, MQ, W (ignored without a mask) */
    void *workspace;   /* device, 256-aligned, >= pa_attention_vjp_workspace_bytes() */
    size_t workspace_bytes;
    int *status;       /* device int or NULL: PA_STATUS_TIMEOUT is ORed in when an
                          internal wait of a tensor-core kernel gave up (the results
                          are then undefined); never cleared by the library */
    int kernel;        /* 0 = automatic; 1 = CUDA-core kernels for any dtype (a
                          cross-check of the tensor-core path) */
    unsigned long long wait_limit_ns; /* 0 = default (1 s): bound of every internal wait */
} pa_vjp_opts;

/* Scratch of pa_attention_vjp: per-row softmax statistics and, when dq is
 * 16-bit, a float32 accumulator of dq.  0 for invalid sizes. */
size_t pa_attention_vjp_workspace_bytes(int B, int HQ, int SQ, int D, int dtype, int out_dtype);

int pa_attention_vjp(const void *q, const void *k, const void *v, const void *y, const void *g,
                     const void *mask, void *dq, void *dk, void *dv, float scale, int B, int HQ,
                     int HK, int SQ, int SK, int D, const pa_vjp_opts *opts, void *stream);

#ifdef __cplusplus
}
#endif

#endif /* PA_ATTENTION_VJP_H */
