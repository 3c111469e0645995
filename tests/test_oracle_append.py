"""The oracle's cache append (the cache update of a decode step) against a
hand-worked example, its skip rules, and the decode it feeds (CPU only)."""
from pathlib import Path

import numpy as np

import oracle
import oracle_pins


def test_hand_worked_example():
    # 3 blocks of 2 slots, 1 KV head, D = 2; two sequences, two new rows each
    kc = np.zeros((3, 2, 1, 2))
    vc = np.zeros((3, 2, 1, 2))
    kn = np.array([[[[1.0, 2.0], [3.0, 4.0]]], [[[5.0, 6.0], [7.0, 8.0]]]])  # [B=2][KV=1][NQ=2][D=2]
    vn = -kn
    slots = np.array([[3, -1], [0, 5]], dtype=np.int32)  # slot 3 = block 1, offset 1; 5 = block 2, offset 1
    k2, v2, bad = oracle.cache_append(kc, vc, kn, vn, slots)
    want_k = np.zeros((3, 2, 1, 2))
    want_k[1, 1, 0] = [1.0, 2.0]  # sequence 0, new row 0 -> slot 3
    want_k[0, 0, 0] = [5.0, 6.0]  # sequence 1, new row 0 -> slot 0
    want_k[2, 1, 0] = [7.0, 8.0]  # sequence 1, new row 1 -> slot 5
    assert np.array_equal(k2, want_k)
    assert np.array_equal(v2, -want_k)
    assert not bad
    assert not kc.any()  # the inputs are not modified


def test_skips_and_reports_bad_slots():
    rng = np.random.default_rng(1)
    kc = rng.standard_normal((4, 4, 2, 8))
    vc = rng.standard_normal((4, 4, 2, 8))
    kn = rng.standard_normal((3, 2, 2, 8))
    vn = rng.standard_normal((3, 2, 2, 8))
    slots = np.array([[-1, 16], [-5, 2], [15, -1]], dtype=np.int32)  # 16 slots in all
    k2, v2, bad = oracle.cache_append(kc, vc, kn, vn, slots)
    assert bad
    touched = {2: (1, 1), 15: (2, 0)}  # slot -> (sequence, new row)
    for s in range(16):
        if s in touched:
            b, j = touched[s]
            assert np.array_equal(k2[s // 4, s % 4], kn[b, :, j])
            assert np.array_equal(v2[s // 4, s % 4], vn[b, :, j])
        else:
            assert np.array_equal(k2[s // 4, s % 4], kc[s // 4, s % 4])
            assert np.array_equal(v2[s // 4, s % 4], vc[s // 4, s % 4])


def test_append_then_decode_equals_decode_with_new_rows():
    """Appending new row 0 at the slot of logical token past (table[b][past //
    BLOCK] * BLOCK + past % BLOCK) and decoding rows 1.. with past + 1 gives
    bitwise the rows 1.. of decoding all new rows as new rows: the append puts
    a row exactly where the decode's block-table gather reads token past."""
    orc = oracle.default()
    for causal in (False, True):
        B, H, KV, D, BLOCK, NQ = 3, 4, 2, 8, 4, 3
        lens = [7, 8, 0]  # 8 and 0 end on a block boundary: the next token needs a new block
        c = oracle_pins.dense_case(B, H, KV, D, BLOCK, NQ, lens, seed=11, spare_blocks=6)
        table = c["block_table"].copy()
        used = set(table[table >= 0].tolist())
        spare = [p for p in range(c["k_cache"].shape[0]) if p not in used]
        slots = np.zeros((B, 1), dtype=np.int32)
        for b, n in enumerate(lens):
            if table[b, n // BLOCK] < 0:
                table[b, n // BLOCK] = spare.pop()
            slots[b, 0] = table[b, n // BLOCK] * BLOCK + n % BLOCK
        full = orc.decode(c["q"], c["k_cache"], c["v_cache"], table, c["seq_lens"], c["k_new"],
                          c["v_new"], scale=0.3, causal=causal)
        kc2, vc2, bad = oracle.cache_append(c["k_cache"], c["v_cache"], c["k_new"][:, :, :1],
                                            c["v_new"][:, :, :1], slots)
        assert not bad
        part = orc.decode(np.ascontiguousarray(c["q"][:, :, 1:]), kc2, vc2, table,
                          c["seq_lens"] + 1, np.ascontiguousarray(c["k_new"][:, :, 1:]),
                          np.ascontiguousarray(c["v_new"][:, :, 1:]), scale=0.3, causal=causal)
        assert np.array_equal(full[:, :, 1:], part), f"causal={causal}"


def test_later_row_of_a_sequence_wins():
    kc = np.zeros((2, 2, 1, 2))
    vc = np.zeros((2, 2, 1, 2))
    kn = np.array([[[[1.0, 1.0], [2.0, 2.0], [3.0, 3.0]]]])  # [B=1][KV=1][NQ=3][D=2]
    k2, _, _ = oracle.cache_append(kc, vc, kn, -kn, np.array([[1, 2, 1]], dtype=np.int32))
    assert np.array_equal(k2[0, 1, 0], [3.0, 3.0])  # rows 0 and 2 name slot 1: row 2 lands
    assert np.array_equal(k2[1, 0, 0], [2.0, 2.0])


def test_slot_patch_equals_decode_after_append():
    """Decode with the slot patch over the old cache equals a plain decode over
    the cache with the new rows stored at their slots, when every sequence
    names only slots of its own blocks: the page's read-time substitution and
    its write-back describe one step."""
    c, _ = oracle_pins.positions_case()
    s = lambda b, t: oracle_pins.slot_of(c, b, t)
    positions = np.array([[s(0, 3), -1, s(0, 3), s(0, 9)],
                          [s(1, 0), s(1, 7), s(1, 13), s(1, 14)],
                          [-1, -1, -1, -1]], dtype=np.int32)
    for causal in (False, True):
        got = oracle_pins.run(oracle.default(), c, 0.3, causal, positions=positions)
        kc, vc, bad = oracle.cache_append(c["k_cache"], c["v_cache"], c["k_new"], c["v_new"],
                                          positions)
        assert not bad
        after = dict(c, k_cache=kc, v_cache=vc)
        want = oracle_pins.run(oracle.default(), after, 0.3, causal)
        assert np.array_equal(got, want)


GOLDEN = Path(__file__).resolve().parent / "golden" / "writeback_ranges.txt"


def golden_writebacks():
    cases = []
    for line in GOLDEN.read_text().splitlines():
        if not line.strip() or line.startswith("#"):
            continue
        shape, itemsize, axis, rows, ranges = (f.strip() for f in line.split("|"))
        cases.append(dict(
            shape=[int(x) for x in shape.split(",")], itemsize=int(itemsize), axis=int(axis),
            rows=[] if rows == "-" else [int(x) for x in rows.split(",")],
            ranges=None if ranges == "error" else
            [] if ranges == "-" else [tuple(int(y) for y in r.split("-")) for r in ranges.split(",")]))
    return cases


def as_cache_shape(shape, axis):
    """A paged cache [num_blocks][BLOCK][KV][D] whose rows at its axis 1 (the
    slots, physical block * BLOCK + offset) are the page's rows at `axis`: a
    rank-4 shape cut at axis 1 is one as it stands."""
    if len(shape) == 4 and axis == 1:
        return tuple(shape)
    lead = int(np.prod(shape[:axis + 1]))
    block = shape[axis] if axis >= 1 else 1
    return (lead // block, block, 1, int(np.prod(shape[axis + 1:])))


def test_writeback_ranges_golden():
    """The cache rows the append writes for a slot mapping are exactly the
    byte ranges the engine page prints for its write-back of those rows."""
    dt = {2: np.float16, 4: np.float32}
    cases = golden_writebacks()
    assert len(cases) == 4
    for c in cases:
        shape = as_cache_shape(c["shape"], c["axis"])
        kc = np.zeros(shape, dtype=dt[c["itemsize"]])
        n = max(len(c["rows"]), 1)
        kn = np.zeros((1, shape[2], n, shape[3]), dtype=kc.dtype)
        kn.view(np.uint8)[...] = 0x5A  # every byte of a new row nonzero
        slots = np.array([c["rows"] or [-1]], dtype=np.int32)
        k2, _, bad = oracle.cache_append(kc, kc.copy(), kn, kn, slots)
        written = np.flatnonzero(k2.view(np.uint8).reshape(-1))
        if c["ranges"] is None:
            assert bad and written.size == 0
            continue
        want = np.concatenate([np.arange(a, b) for a, b in c["ranges"]] or [np.zeros(0, int)])
        assert not bad
        assert np.array_equal(written, want), (c, written)
