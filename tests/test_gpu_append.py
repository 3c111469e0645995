"""pa_cache_append on the GPU against the oracle's cache append, bit for bit."""
import numpy as np
import pytest
import torch

import oracle
from paged_kv_cache_182_gb300 import workloads as W

pytestmark = pytest.mark.gpu

DT = {"f32": torch.float32, "f16": torch.float16, "bf16": torch.bfloat16}
BITS = {torch.float32: torch.int32, torch.float16: torch.int16, torch.bfloat16: torch.int16}


def bits(t):
    """The stored bit patterns (exact comparison, NaN-safe, bfloat16 included)."""
    return t.contiguous().cpu().view(BITS[t.dtype]).numpy()


def run_case(dt, B, KV, D, NQ, BLOCK, NB, slots, seed):
    from paged_kv_cache_182_gb300 import binding

    g = torch.Generator().manual_seed(seed)
    kc = torch.randn(NB, BLOCK, KV, D, generator=g).to(DT[dt])
    vc = torch.randn(NB, BLOCK, KV, D, generator=g).to(DT[dt])
    kn = torch.randn(B, KV, NQ, D, generator=g).to(DT[dt])
    vn = torch.randn(B, KV, NQ, D, generator=g).to(DT[dt])
    sl = torch.tensor(slots, dtype=torch.int32).reshape(B, NQ)
    kc_d, vc_d = kc.cuda(), vc.cuda()
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    binding.cache_append(kc_d, vc_d, kn.cuda(), vn.cuda(), sl.cuda(), status=status)
    torch.cuda.synchronize()
    want_k, want_v, bad = oracle.cache_append(bits(kc), bits(vc), bits(kn), bits(vn), sl.numpy())
    assert np.array_equal(bits(kc_d), want_k)
    assert np.array_equal(bits(vc_d), want_v)
    assert bool(int(status.item()) & binding.PA_STATUS_BAD_SLOT) == bad


CASES = [
    # dtype, B, KV, D, NQ, BLOCK, pool blocks
    ("f16", 16, 8, 128, 4, 32, 40),
    ("bf16", 5, 4, 64, 1, 16, 9),
    ("f32", 3, 2, 64, 16, 16, 8),
    ("f16", 1, 1, 128, 3, 32, 2),
]


@pytest.mark.parametrize("case", CASES, ids=lambda c: f"{c[0]}-B{c[1]}-KV{c[2]}-D{c[3]}-NQ{c[4]}")
def test_random_distinct_slots(case):
    dt, B, KV, D, NQ, BLOCK, NB = case
    rng = np.random.default_rng(B * 100 + NQ)
    n = B * NQ
    slots = rng.choice(NB * BLOCK, size=n, replace=False).astype(np.int64)
    slots[rng.random(n) < 0.2] = -1  # skipped rows
    run_case(dt, B, KV, D, NQ, BLOCK, NB, slots.tolist(), seed=1)


def test_bad_slots_are_skipped_and_reported():
    B, NQ, BLOCK, NB = 2, 3, 16, 4
    slots = [5, NB * BLOCK, -1, -7, 63, 0]  # one past the end, one below -1
    run_case("f16", B, 2, 64, NQ, BLOCK, NB, slots, seed=2)


def test_append_at_logical_positions_of_a_workload():
    """The full-size causal-append workload's new rows written over the slots
    of each sequence's last NQ cached tokens (slots through its block table:
    table[b][t // BLOCK] * BLOCK + t % BLOCK)."""
    from paged_kv_cache_182_gb300 import binding

    w = W.make("causal_append_fp16", seed=3)
    s = w.spec
    slots = torch.full((s.B, s.NQ), -1, dtype=torch.int32)
    for b in range(s.B):
        past = int(w.seq_lens[b])
        for j in range(s.NQ):
            t = past - s.NQ + j
            if t >= 0:
                slots[b, j] = int(w.block_table[b, t // s.BLOCK]) * s.BLOCK + t % s.BLOCK
    kc_d, vc_d = w.k_cache.cuda(), w.v_cache.cuda()
    binding.cache_append(kc_d, vc_d, w.k_new.cuda(), w.v_new.cuda(), slots.cuda())
    torch.cuda.synchronize()
    want_k, want_v, bad = oracle.cache_append(bits(w.k_cache), bits(w.v_cache), bits(w.k_new),
                                              bits(w.v_new), slots.numpy())
    assert not bad and (slots >= 0).any()
    assert np.array_equal(bits(kc_d), want_k)
    assert np.array_equal(bits(vc_d), want_v)


def test_empty_batch_launches_nothing():
    from paged_kv_cache_182_gb300 import binding

    kc = torch.zeros(2, 16, 1, 64, dtype=torch.float16, device="cuda")
    before = binding.kernel_launches()
    binding.cache_append(kc, kc.clone(), torch.zeros(0, 1, 1, 64, dtype=torch.float16, device="cuda"),
                         torch.zeros(0, 1, 1, 64, dtype=torch.float16, device="cuda"),
                         torch.zeros(0, 1, dtype=torch.int32, device="cuda"))
    assert binding.kernel_launches() == before


def test_rows_of_one_sequence_naming_one_slot():
    """Two new rows of one sequence bound for one slot: the later row lands."""
    B, NQ, BLOCK, NB = 3, 4, 16, 4
    slots = [7, 20, 7, 7,  33, -1, 33, 2,  50, 51, 52, 50]
    run_case("bf16", B, 2, 128, NQ, BLOCK, NB, slots, seed=4)


def test_golden_writeback_rows():
    """The engine page's printed write-back example (cache [3][4][2][8] of
    2-byte elements, rows 9, 2, 1, 2 at axis 1) as a slot mapping; the oracle
    side is pinned to the printed byte ranges by the CPU tests."""
    run_case("f16", 1, 2, 8, 4, 4, 3, [9, 2, 1, 2], seed=5)
