"""Decode with slot patching (pa_decode_positions) against the oracle (needs a GPU).

New row j of sequence b is bound for cache slot positions[b, j].  The oracle
applies the page's read-time rule (a cached key of sequence b whose slot a new
row of b is bound for reads that row, the last such row winning) over the
unchanged cache; the library stores the new rows first and attends over the
updated cache.  The outputs must agree within the parity tolerance and the
updated caches must equal the oracle's cache append bit for bit.  Every
sequence names only slots of its own blocks: cached tokens (an in-place
rewrite, with two rows of one sequence naming one slot), the tail of its last
block, or none.
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


def own_positions(w, seed):
    s = w.spec
    rng = np.random.default_rng(seed)
    table = w.block_table.numpy()
    pos = np.full((s.B, s.NQ), -1, dtype=np.int32)
    for b in range(s.B):
        past = int(w.seq_lens[b])
        owned = -(-past // s.BLOCK) * s.BLOCK  # tokens of the blocks the sequence holds
        for j in range(s.NQ):
            kind = rng.integers(3)
            if kind == 0 and past > 0:
                t = int(rng.integers(past))  # a cached token: rewritten in place
            elif kind == 1 and past + j < owned:
                t = past + j  # the tail of its last block: a plain append
            else:
                continue
            pos[b, j] = int(table[b, t // s.BLOCK]) * s.BLOCK + t % s.BLOCK
        if s.NQ >= 2 and past > 0:
            t = int(rng.integers(past))
            pos[b, 0] = pos[b, s.NQ - 1] = int(table[b, t // s.BLOCK]) * s.BLOCK + t % s.BLOCK
    return pos


def run_case(w, partitions, seed, out_dtype=torch.float32):
    from paged_kv_cache_182_gb300 import binding

    pos = own_positions(w, seed)
    assert (pos >= 0).any()
    dev = w.to("cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    got = binding.decode_positions(*dev.tensors(), torch.from_numpy(pos).cuda(),
                                   scale=w.spec.scale, causal=w.spec.causal,
                                   partitions=partitions, out_dtype=out_dtype, status=status)
    torch.cuda.synchronize()
    want = oracle.decode(*w.tensors(), scale=w.spec.scale, causal=w.spec.causal, positions=pos)
    out_fmt = "f32" if out_dtype == torch.float32 else w.spec.dtype
    pu.check(got, want, w.spec.dtype, out_fmt, f"{w.spec.name} P={partitions}")
    want_k, want_v, bad = oracle.cache_append(bits(w.k_cache), bits(w.v_cache), bits(w.k_new),
                                              bits(w.v_new), pos)
    assert not bad and int(status.item()) == 0
    assert np.array_equal(bits(dev.k_cache), want_k)
    assert np.array_equal(bits(dev.v_cache), want_v)


CASES = [
    # dtype, H, KV, D, BLOCK, NQ, causal, lens
    ("f16", 8, 2, 128, 16, 2, True, [0, 37, 300]),      # 8 rows per KV head
    ("bf16", 16, 2, 64, 32, 3, False, [64, 129, 1000]),  # 24 rows: two row groups
    ("f16", 12, 3, 128, 8, 3, True, [5, 513]),          # 12 rows
    ("f32", 8, 2, 64, 16, 4, True, [1, 77, 300]),
]


@pytest.mark.parametrize("case", CASES, ids=lambda c: f"{c[0]}-H{c[1]}-KV{c[2]}-D{c[3]}-NQ{c[5]}")
@pytest.mark.parametrize("P", [0, 1, 3])
def test_slot_patch_small(case, P):
    dt, H, KV, D, BLOCK, NQ, causal, lens = case
    spec = W.Spec("positions", dt, B=len(lens), H=H, KV=KV, D=D, BLOCK=BLOCK, NQ=NQ,
                  causal=causal, pool_blocks=0, extra_table_cols=2)
    run_case(W.make(spec, seed=11, lens=lens), P, seed=12)


def test_slot_patch_full_causal_workload():
    w = W.make("causal_append_fp16", seed=13)
    run_case(w, 0, seed=14, out_dtype=None)


def test_no_positions_named_equals_plain_decode():
    from paged_kv_cache_182_gb300 import binding

    w = W.make(W.shrink(W.SPECS["gqa_fp16"], B=3, past=150, past_hi=900), seed=15)
    dev = w.to("cuda")
    pos = torch.full((w.spec.B, w.spec.NQ), -1, dtype=torch.int32, device="cuda")
    a = binding.decode_positions(*dev.tensors(), pos, scale=w.spec.scale, causal=w.spec.causal)
    b = binding.decode(*dev.tensors(), scale=w.spec.scale, causal=w.spec.causal)
    torch.cuda.synchronize()
    assert torch.equal(a, b)
