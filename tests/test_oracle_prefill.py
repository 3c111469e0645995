"""The chunked prefill schedule against the definition, on the oracle (CPU only).

A causal prefill of NQ new rows per sequence is the decode definition with NQ
new rows and the causal bound (row r sees past + r + 1 keys).  The library
runs it as the store of all new rows into the cache followed by causal
decodes of chunks of at most 16 rows, chunk [r0, r0 + n) seeing past + r0
cached tokens.  Written with the oracle's own append and decode, that
schedule must reproduce the definition bit for bit: the same key values in
the same logical order."""
import numpy as np
import pytest

import oracle
from paged_kv_cache_182_gb300 import workloads as W

CHUNK = 16


def prefill_slots(w):
    s = w.spec
    slots = np.empty((s.B, s.NQ), dtype=np.int32)
    for b, past in enumerate(w.seq_lens.tolist()):
        for j in range(s.NQ):
            t = past + j
            slots[b, j] = int(w.block_table[b, t // s.BLOCK]) * s.BLOCK + t % s.BLOCK
    return slots


@pytest.mark.parametrize("NQ", [1, 16, 17, 37])
def test_chunked_schedule_equals_definition(NQ):
    spec = W.Spec("pf", "f32", B=3, H=8, KV=2, D=16, BLOCK=8, NQ=NQ, causal=True)
    w = W.make_prefill(spec, seed=NQ, lens=[0, 13, 40])
    q, kc, vc, table, lens, kn, vn = (x.numpy() for x in w.tensors())
    full = oracle.decode(q, kc, vc, table, lens, kn, vn, scale=spec.scale, causal=True)
    assert np.all(np.isfinite(full))
    kc2, vc2, bad = oracle.cache_append(kc, vc, kn, vn, prefill_slots(w))
    assert not bad
    for r0 in range(0, NQ, CHUNK):
        n = min(CHUNK, NQ - r0)
        part = oracle.decode(np.ascontiguousarray(q[:, :, r0:r0 + n]), kc2, vc2, table,
                             lens + r0, np.ascontiguousarray(kn[:, :, r0:r0 + n]),
                             np.ascontiguousarray(vn[:, :, r0:r0 + n]), scale=spec.scale,
                             causal=True)
        assert np.array_equal(part, full[:, :, r0:r0 + n]), f"chunk at row {r0}"


def test_prefill_workload_table_covers_new_tokens():
    w = W.make_prefill(W.Spec("pf", "f16", B=2, H=4, KV=2, D=64, BLOCK=16, NQ=40,
                              causal=True), seed=1, lens=[5, 32])
    slots = prefill_slots(w)
    assert len(set(slots.ravel().tolist())) == slots.size  # distinct, inside the pool
    assert slots.min() >= 0 and slots.max() < w.num_blocks * w.spec.BLOCK
    nanrows = np.isnan(w.k_cache.float().numpy()).all(axis=(2, 3))
    for s in slots.ravel().tolist():  # poisoned until the prefill writes them
        assert nanrows[s // 16, s % 16]
