"""Pins of the float64 oracle to facts that do not come from the oracle itself.

Each ``pin_*`` takes an ``oracle.Oracle`` and raises AssertionError when the
oracle disagrees with:

  * torch's float64 ``scaled_dot_product_attention`` (a library routine) on
    dense, contiguous K/V that the test scatters into a paged pool -- this
    checks the block-table gather, the grouped-query map, the new-row branch
    and the causal bound at once;
  * bitwise invariance under any permutation of the physical blocks;
  * closed forms: a single visible key returns its value row; a zero query
    returns the mean of the visible values; two keys with scores 0 and ln 3
    weigh their values 1/4 and 3/4; a huge scale returns the value row of the
    arg-max key (and no overflow);
  * the grouped-query map (query head h reads KV head h // (H / KV)) with
    constant value rows;
  * causal truncation: causal row r equals row r of a non-causal call that
    sees only new rows 0..r;
  * slot patching (the position vector's entries 1 + j on the same page,
    VECTOR_BODY): torch SDPA on dense keys/values in which every cached token
    whose slot a new row of its own sequence is bound for holds that row (the
    last such row), and bitwise equality with a plain call when no position
    names a cached slot of its sequence.

The semantics pinned are those of onnxruntime-ep-mlx 0.31.1,
src/ops/paged_attention.rs (VECTOR_BODY, VECTOR_REDUCE, PARTIALS_REDUCE), with
the grouping and the causal rule also stated by the dense attention VJP page
(src/ops/attention_vjp/dense.rs, fn execute: the [b, hk, groups, sq, d]
reshape and the ki <= qi mask).
"""
from __future__ import annotations

import math

import numpy as np
import torch
import torch.nn.functional as F


# --------------------------------------------------------------------------
# test-side construction of a paged case from dense per-sequence K/V
# --------------------------------------------------------------------------

def dense_case(B, H, KV, D, BLOCK, NQ, lens, seed, spare_blocks=3, q_zero=False):
    """Dense keys/values per sequence, scattered into a shuffled paged pool."""
    rng = np.random.default_rng(seed)
    lens = [int(x) for x in lens]
    q = np.zeros((B, H, NQ, D)) if q_zero else rng.standard_normal((B, H, NQ, D))
    dense_k = [rng.standard_normal((KV, n, D)) for n in lens]
    dense_v = [rng.standard_normal((KV, n, D)) for n in lens]
    k_new = rng.standard_normal((B, KV, NQ, D))
    v_new = rng.standard_normal((B, KV, NQ, D))
    nblk = [(n + BLOCK - 1) // BLOCK for n in lens]
    pool = sum(nblk) + spare_blocks
    perm = rng.permutation(pool)
    maxb = max(nblk + [1]) + 1
    table = -np.ones((B, maxb), dtype=np.int32)
    k_cache = np.full((pool, BLOCK, KV, D), np.nan)
    v_cache = np.full((pool, BLOCK, KV, D), np.nan)
    at = 0
    for b, n in enumerate(lens):
        for j in range(nblk[b]):
            phys = int(perm[at + j])
            table[b, j] = phys
            for slot in range(BLOCK):
                t = j * BLOCK + slot
                if t < n:
                    k_cache[phys, slot] = dense_k[b][:, t, :]
                    v_cache[phys, slot] = dense_v[b][:, t, :]
        at += nblk[b]
    return dict(q=q, k_cache=k_cache, v_cache=v_cache, block_table=table,
                seq_lens=np.array(lens, dtype=np.int32), k_new=k_new, v_new=v_new,
                dense_k=dense_k, dense_v=dense_v, H=H, KV=KV, NQ=NQ)


def run(orc, c, scale, causal, **kw):
    return orc.decode(c["q"], c["k_cache"], c["v_cache"], c["block_table"], c["seq_lens"],
                      c["k_new"], c["v_new"], scale=scale, causal=causal, **kw)


def sdpa_reference(c, scale, causal):
    """torch float64 SDPA per sequence on [cached ; new] keys, GQA via enable_gqa."""
    B, H, NQ, D = c["q"].shape
    out = np.zeros_like(c["q"])
    for b, n in enumerate(c["seq_lens"].tolist()):
        k = np.concatenate([c["dense_k"][b], c["k_new"][b]], axis=1)  # [KV, n+NQ, D]
        v = np.concatenate([c["dense_v"][b], c["v_new"][b]], axis=1)
        L = n + NQ
        allowed = np.ones((NQ, L), dtype=bool)
        if causal:
            for r in range(NQ):
                allowed[r, n + r + 1:] = False
        o = F.scaled_dot_product_attention(
            torch.from_numpy(c["q"][b][None]), torch.from_numpy(k[None]),
            torch.from_numpy(v[None]), attn_mask=torch.from_numpy(allowed), scale=scale,
            enable_gqa=True)
        out[b] = o[0].numpy()
    return out


SDPA_CASES = [
    # B, H, KV, D, BLOCK, NQ, causal, lens
    (2, 4, 2, 16, 4, 1, False, [5, 9]),
    (2, 8, 2, 8, 8, 3, True, [0, 13]),
    (3, 6, 3, 32, 16, 2, False, [17, 1, 32]),
    (1, 2, 1, 64, 16, 4, True, [100]),
    (2, 8, 1, 8, 2, 2, True, [7, 3]),
    (2, 4, 2, 16, 8, 40, True, [0, 21]),  # a prefill-sized chunk of new rows
]


def pin_sdpa_dense(orc):
    for i, (B, H, KV, D, BLOCK, NQ, causal, lens) in enumerate(SDPA_CASES):
        c = dense_case(B, H, KV, D, BLOCK, NQ, lens, seed=100 + i)
        scale = 1.0 / math.sqrt(D)
        got = run(orc, c, scale, causal)
        want = sdpa_reference(c, scale, causal)
        assert np.all(np.isfinite(got)), f"case {i}: non-finite oracle output"
        err = float(np.max(np.abs(got - want)))
        assert err < 1e-12, f"case {i}: oracle vs torch SDPA max abs err {err}"


def pin_permutation_bitwise(orc):
    c = dense_case(3, 8, 2, 16, 4, 2, [11, 0, 23], seed=7)
    base = run(orc, c, 0.25, True)
    rng = np.random.default_rng(8)
    pool = c["k_cache"].shape[0]
    perm = rng.permutation(pool)  # new position of each old block
    inv = np.argsort(perm)
    c2 = dict(c)
    c2["k_cache"] = c["k_cache"][inv]
    c2["v_cache"] = c["v_cache"][inv]
    t = c["block_table"].copy()
    t[t >= 0] = perm[t[t >= 0]]
    c2["block_table"] = t.astype(np.int32)
    again = run(orc, c2, 0.25, True)
    assert np.array_equal(base, again), "output changed under a block permutation"


def pin_single_key(orc):
    c = dense_case(2, 6, 3, 16, 8, 1, [0, 0], seed=9)
    got = run(orc, c, 0.3, False)
    g = 6 // 3
    for b in range(2):
        for h in range(6):
            assert np.array_equal(got[b, h, 0], c["v_new"][b, h // g, 0]), \
                "one visible key must return its value row exactly"


def pin_equal_scores(orc):
    c = dense_case(2, 4, 2, 8, 4, 3, [6, 10], seed=11, q_zero=True)
    for causal in (False, True):
        got = run(orc, c, 0.5, causal)
        for b, n in enumerate(c["seq_lens"].tolist()):
            for h in range(4):
                kh = h // 2
                for r in range(3):
                    vis = n + (r + 1 if causal else 3)
                    rows = np.concatenate([c["dense_v"][b][kh], c["v_new"][b][kh]])[:vis]
                    want = rows.mean(axis=0)
                    err = np.max(np.abs(got[b, h, r] - want))
                    assert err < 1e-13, f"zero query must average the visible values ({err})"


def pin_two_keys_closed_form(orc):
    # one cached key with score 0 and one new key with score ln 3:
    # weights 1/4 and 3/4
    q = np.array([[[[1.0, 0.0, 0.0, 0.0]]]])
    k_cache = np.zeros((2, 1, 1, 4))
    v_cache = np.zeros((2, 1, 1, 4))
    k_cache[1, 0, 0] = [0.0, 5.0, -3.0, 2.0]  # score 0 (only d=0 counts)
    v_cache[1, 0, 0] = [4.0, 8.0, -4.0, 1.0]
    k_cache[0] = np.nan
    v_cache[0] = np.nan
    k_new = np.array([[[[2.0 * math.log(3.0), 1.0, 1.0, 1.0]]]])
    v_new = np.array([[[[0.0, 4.0, 8.0, -1.0]]]])
    table = np.array([[1]], dtype=np.int32)
    lens = np.array([1], dtype=np.int32)
    got = orc.decode(q, k_cache, v_cache, table, lens, k_new, v_new, scale=0.5, causal=False)
    want = np.array([1.0, 5.0, 5.0, -0.5])
    err = np.max(np.abs(got[0, 0, 0] - want))
    assert err < 1e-14, f"two-key closed form off by {err}"


def pin_hard_max(orc):
    c = dense_case(2, 4, 2, 16, 4, 2, [9, 14], seed=13)
    scale = 1.0e6
    got = run(orc, c, scale, False)
    assert np.all(np.isfinite(got)), "huge scores must not overflow"
    for b, n in enumerate(c["seq_lens"].tolist()):
        for h in range(4):
            kh = h // 2
            keys = np.concatenate([c["dense_k"][b][kh], c["k_new"][b][kh]])
            vals = np.concatenate([c["dense_v"][b][kh], c["v_new"][b][kh]])
            for r in range(2):
                s = keys @ c["q"][b, h, r]
                top = np.sort(s)
                assert top[-1] - top[-2] > 1e-3  # the limit is a single key
                want = vals[int(np.argmax(s))]
                assert np.array_equal(got[b, h, r], want), "hard-max limit must pick the arg-max value"


def pin_gqa_map(orc):
    B, H, KV, D, BLOCK = 2, 12, 3, 8, 4
    c = dense_case(B, H, KV, D, BLOCK, 2, [5, 8], seed=17)
    for kh in range(KV):
        c["v_cache"][:, :, kh, :] = kh + 1.0
        c["v_new"][:, kh] = kh + 1.0
        for b in range(B):
            c["dense_v"][b][kh] = kh + 1.0
    got = run(orc, c, 0.4, True)
    g = H // KV
    for h in range(H):
        err = np.max(np.abs(got[:, h] - (h // g + 1.0)))
        assert err < 1e-13, f"query head {h} must read KV head {h // g}"


def pin_causal_truncation(orc):
    c = dense_case(2, 4, 2, 16, 8, 4, [12, 3], seed=19)
    full = run(orc, c, 0.25, True)
    for r in range(4):
        c2 = dict(c)
        c2["q"] = np.ascontiguousarray(c["q"][:, :, : r + 1])
        c2["k_new"] = np.ascontiguousarray(c["k_new"][:, :, : r + 1])
        c2["v_new"] = np.ascontiguousarray(c["v_new"][:, :, : r + 1])
        part = run(orc, c2, 0.25, False)
        assert np.array_equal(full[:, :, r], part[:, :, r]), \
            f"causal row {r} must see exactly the past plus new rows 0..{r}"
    one = dict(c)
    for key in ("q", "k_new", "v_new"):
        one[key] = np.ascontiguousarray(c[key][:, :, :1])
    assert np.array_equal(run(orc, one, 0.25, True), run(orc, one, 0.25, False))


def slot_of(c, b, t):
    """Cache slot (physical block * BLOCK + offset) of token t of sequence b."""
    BLOCK = c["k_cache"].shape[1]
    return int(c["block_table"][b, t // BLOCK]) * BLOCK + t % BLOCK


def patched_dense(c, positions):
    """Dense per-sequence keys/values with the slot patch applied token by
    token: cached token t of sequence b takes new row j when positions[b, j]
    is its slot, later j overriding earlier ones."""
    dk = [x.copy() for x in c["dense_k"]]
    dv = [x.copy() for x in c["dense_v"]]
    for b, n in enumerate(c["seq_lens"].tolist()):
        for t in range(n):
            for j in range(positions.shape[1]):
                if positions[b, j] >= 0 and positions[b, j] == slot_of(c, b, t):
                    dk[b][:, t] = c["k_new"][b][:, j]
                    dv[b][:, t] = c["v_new"][b][:, j]
    out = dict(c)
    out["dense_k"], out["dense_v"] = dk, dv
    return out


def positions_case():
    c = dense_case(3, 8, 2, 16, 4, 4, [9, 14, 0], seed=23)
    s = lambda b, t: slot_of(c, b, t)
    positions = np.array([
        [s(0, 3), -1, s(0, 3), s(0, 9)],          # rows 0 and 2 name one cached slot; 9 = past
        [s(1, 0), s(0, 5), s(1, 13), 1 << 30],    # another sequence's slot; out of the pool
        [s(0, 1), -5, -1, s(1, 2)],               # no past: nothing to patch
    ], dtype=np.int32)
    return c, positions


def pin_positions_sdpa(orc):
    c, positions = positions_case()
    for causal in (False, True):
        got = run(orc, c, 0.3, causal, positions=positions)
        want = sdpa_reference(patched_dense(c, positions), 0.3, causal)
        assert np.all(np.isfinite(got)), "non-finite oracle output with positions"
        err = float(np.max(np.abs(got - want)))
        assert err < 1e-12, f"slot patching (causal={causal}): max abs err {err}"


def pin_positions_neutral(orc):
    c, positions = positions_case()
    base = run(orc, c, 0.3, True)
    none = -np.ones_like(positions)
    assert np.array_equal(run(orc, c, 0.3, True, positions=none), base)
    # slots at or past each sequence's length, or in another sequence's blocks
    away = np.array([[slot_of(c, 0, 9), slot_of(c, 0, 10), -1, slot_of(c, 1, 4)],
                     [slot_of(c, 1, 14), slot_of(c, 0, 0), -1, -1],
                     [slot_of(c, 1, 1), -1, -1, -1]], dtype=np.int32)
    assert np.array_equal(run(orc, c, 0.3, True, positions=away), base)


ALL_PINS = [
    pin_sdpa_dense,
    pin_permutation_bitwise,
    pin_single_key,
    pin_equal_scores,
    pin_two_keys_closed_form,
    pin_hard_max,
    pin_gqa_map,
    pin_causal_truncation,
    pin_positions_sdpa,
    pin_positions_neutral,
]


def run_all(orc) -> list[str]:
    """Names of the pins that fail (an exception of any kind counts)."""
    failed = []
    for pin in ALL_PINS:
        try:
            pin(orc)
        except Exception as exc:  # noqa: BLE001 - any failure counts as caught
            failed.append(f"{pin.__name__}: {type(exc).__name__}: {exc}")
    return failed
