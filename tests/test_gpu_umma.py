"""The tcgen05 partition kernel (16-bit inputs, D = 128, more than 16 query
rows per KV head) against the float64 oracle, element by element, and the
mma.sync kernels on the same inputs (pa_opts.kernel = 1).  Needs a GPU.

The cases cover the stage boundaries (128 tokens), padding rows in a pass
(24 rows; a second pass of 18 rows), 8-, 16-, 32- and 64-token blocks (one
TMA box per block and 64-column half), empty sequences, the new rows
straddling two stages, and value laws with 1% of the K/V entries times 20
and q times 2, whose running row maxima move in the middle of a piece (the
rescale of O in tensor memory).  Unused pool blocks and slots past each
length are NaN, so a stray read shows up as a non-finite output.
"""
import pytest
import torch

import parity_util as pu
from paged_kv_cache_182_gb300 import workloads as W

pytestmark = pytest.mark.gpu

# dtype, H, KV, BLOCK, NQ, causal, lens, outliers
CASES = [
    ("f16", 64, 8, 32, 4, True, [333, 2048, 0, 5000], False),   # the causal-append shape
    ("bf16", 64, 8, 32, 4, True, [1, 126, 127, 128, 129, 255], False),  # new rows across stages
    ("f16", 24, 8, 16, 8, True, [700, 70], False),        # 24 rows: padding rows in the pass
    ("f16", 40, 4, 64, 5, True, [1000, 64, 3], False),    # 50 rows: passes of 32 and 18
    ("bf16", 32, 1, 8, 1, False, [4096], False),           # MQA: 32 rows, 8-token blocks
    ("f16", 64, 8, 32, 4, True, [3000, 2500], True),       # the maximum moves mid-piece
    ("bf16", 16, 2, 16, 3, False, [1500, 9, 300], True),   # 24 rows, non-causal
    ("f16", 16, 8, 64, 16, True, [40, 700], False),        # 2 heads x 16 new rows, 64-token blocks
    ("bf16", 32, 1, 32, 1, False, [2049, 1, 128], True),   # 32 heads on one KV head
]


def _case_id(c):
    return f"{c[0]}-H{c[1]}-KV{c[2]}-B{c[3]}-NQ{c[4]}-{'c' if c[5] else 'n'}{'-out' if c[7] else ''}"


def _make(case, seed):
    dt, H, KV, BLOCK, NQ, causal, lens, outliers = case
    law = dict(q_mult=2.0, outlier_frac=0.01, outlier_mult=20.0) if outliers else {}
    spec = W.Spec("umma", dt, B=len(lens), H=H, KV=KV, D=128, BLOCK=BLOCK, NQ=NQ, causal=causal,
                  extra_table_cols=2, **law)
    return W.make(spec, seed=seed, lens=lens)


@pytest.mark.parametrize("case", CASES, ids=_case_id)
@pytest.mark.parametrize("P", [0, 1, 3])
def test_umma_kernel_matches_oracle(case, P):
    w = _make(case, seed=11)
    got = pu.run_gpu(w, partitions=P, out_dtype=torch.float32)
    pu.check(got, pu.run_oracle(w), w.spec.dtype, "f32", f"tcgen05 {case} P={P}")


@pytest.mark.parametrize("case", CASES, ids=_case_id)
def test_umma_kernel_native_output_and_mma_sync_kernel(case):
    """Native 16-bit output; and the same inputs through the mma.sync kernel."""
    w = _make(case, seed=12)
    want = pu.run_oracle(w)
    got = pu.run_gpu(w)
    pu.check(got, want, w.spec.dtype, w.spec.dtype, f"tcgen05 native {case}")
    legacy = pu.run_gpu(w, out_dtype=torch.float32, kernel=1)
    pu.check(legacy, want, w.spec.dtype, "f32", f"mma.sync {case}")


def test_umma_kernel_separate_merge_kernel():
    w = _make(CASES[0], seed=13)
    got = pu.run_gpu(w, partitions=0, out_dtype=torch.float32, merge_kernel=True)
    pu.check(got, pu.run_oracle(w), "f16", "f32", "tcgen05 with the merge kernel")


def test_umma_kernel_repeat_calls_are_bitwise_equal():
    """The schedule and every sum's order depend on the lengths only."""
    w = _make(CASES[5], seed=14)
    a = pu.run_gpu(w, out_dtype=torch.float32)
    b = pu.run_gpu(w, out_dtype=torch.float32)
    assert torch.equal(a, b)
