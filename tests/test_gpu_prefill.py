"""Causal prefill (pa_prefill) against the oracle (needs a GPU).

New row j of sequence b is token seq_lens[b] + j; output row r attends to keys
0 .. seq_lens[b] + r.  The oracle evaluates that definition over the caches as
given (the new tokens' slots hold NaN there, so a read of a slot before the
prefill stored it shows up); the library stores the new rows, then decodes in
chunks.  The output must agree within the parity tolerance and the caches must
equal the oracle's append of the new rows at the slots the block table gives
their tokens, bit for bit.
"""
import numpy as np
import pytest
import torch

import oracle
import parity_util as pu
from paged_kv_cache_182_gb300 import workloads as W

pytestmark = pytest.mark.gpu

BITS = {torch.float32: torch.int32, torch.float16: torch.int16, torch.bfloat16: torch.int16}


def bits(t):
    return t.contiguous().cpu().view(BITS[t.dtype]).numpy()


def prefill_slots(w):
    s = w.spec
    slots = np.empty((s.B, s.NQ), dtype=np.int32)
    for b, past in enumerate(w.seq_lens.tolist()):
        for j in range(s.NQ):
            t = past + j
            slots[b, j] = int(w.block_table[b, t // s.BLOCK]) * s.BLOCK + t % s.BLOCK
    return slots


def run_case(w, partitions, out_dtype=torch.float32):
    from paged_kv_cache_182_gb300 import binding

    dev = w.to("cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    got = binding.prefill(*dev.tensors(), scale=w.spec.scale, partitions=partitions,
                          out_dtype=out_dtype, status=status)
    torch.cuda.synchronize()
    want = oracle.decode(*w.tensors(), scale=w.spec.scale, causal=True)
    out_fmt = "f32" if out_dtype == torch.float32 else w.spec.dtype
    pu.check(got, want, w.spec.dtype, out_fmt, f"{w.spec.name} NQ={w.spec.NQ} P={partitions}")
    want_k, want_v, bad = oracle.cache_append(bits(w.k_cache), bits(w.v_cache), bits(w.k_new),
                                              bits(w.v_new), prefill_slots(w))
    assert not bad and int(status.item()) == 0
    assert np.array_equal(bits(dev.k_cache), want_k)
    assert np.array_equal(bits(dev.v_cache), want_v)


CASES = [
    # dtype, H, KV, D, BLOCK, NQ, past per sequence
    ("f16", 32, 8, 128, 16, 100, [0, 37, 300]),  # 7 chunks, the last of 4 rows
    ("bf16", 8, 1, 64, 32, 40, [129, 5]),        # MQA: 128 query rows per chunk
    ("f32", 4, 2, 64, 16, 33, [1, 70]),
    ("f16", 16, 8, 128, 8, 16, [20, 0, 64]),     # one chunk: no staging
    ("f16", 8, 2, 64, 16, 1, [300]),             # one new row
    # the tensor-core path (16-bit, D = 128, more than 16 new rows)
    ("bf16", 16, 16, 128, 32, 45, [0, 130]),     # one head per tile: 128 rows, partial
    ("bf16", 64, 4, 128, 64, 70, [9, 1000]),     # 16 heads x 8 rows a tile, BLOCK 64
    ("f16", 16, 2, 128, 8, 130, [250, 3]),       # 8 heads x 16 rows, 16 blocks a key tile
    ("f16", 32, 8, 128, 16, 630, [0, 300]),      # 320 row tiles: several per persistent CTA, ragged last
]


@pytest.mark.parametrize("case", CASES, ids=lambda c: f"{c[0]}-H{c[1]}-KV{c[2]}-D{c[3]}-NQ{c[5]}")
@pytest.mark.parametrize("P", [0, 1, 3])
def test_prefill_small(case, P):
    dt, H, KV, D, BLOCK, NQ, lens = case
    spec = W.Spec("prefill", dt, B=len(lens), H=H, KV=KV, D=D, BLOCK=BLOCK, NQ=NQ, causal=True)
    run_case(W.make_prefill(spec, seed=21, lens=lens), P)


def test_prefill_tensor_core_native_output():
    spec = W.Spec("prefill", "bf16", B=2, H=32, KV=8, D=128, BLOCK=16, NQ=77, causal=True)
    run_case(W.make_prefill(spec, seed=24, lens=[513, 64]), 0, out_dtype=None)


def test_prefill_full_workload():
    w = W.make_prefill("prefill_fp16", seed=22)
    run_case(w, 0, out_dtype=None)


def test_prefill_repeat_is_bitwise_stable():
    from paged_kv_cache_182_gb300 import binding

    w = W.make_prefill(W.Spec("prefill", "f16", B=2, H=16, KV=4, D=128, BLOCK=16, NQ=50,
                              causal=True), seed=23, lens=[70, 200])
    dev = w.to("cuda")
    plan = binding.PrefillPlan(*dev.tensors(), scale=w.spec.scale)
    a = plan.run().clone()
    b = plan.run().clone()  # the caches already hold the new rows: same values again
    torch.cuda.synchronize()
    assert torch.equal(a, b)
