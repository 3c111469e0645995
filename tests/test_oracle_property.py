"""Randomised pins of the oracle (CPU only): over drawn shapes, lengths, block
sizes, causal flags and slot positions, the oracle must equal torch's float64
scaled_dot_product_attention on the dense keys and values that the test
scatters into a shuffled paged pool (with the slot patch applied token by
token where positions are drawn).  The fixed pins in oracle_pins.py name the
individual facts; these sweep their combinations."""
import math

import numpy as np
import pytest

import oracle
import oracle_pins as op

hypothesis = pytest.importorskip("hypothesis")
st = hypothesis.strategies


@st.composite
def cases(draw):
    KV = draw(st.integers(1, 3))
    group = draw(st.integers(1, 4))
    B = draw(st.integers(1, 3))
    D = draw(st.sampled_from([4, 8, 16]))
    BLOCK = draw(st.sampled_from([1, 2, 4, 8]))
    NQ = draw(st.integers(1, 6))
    lens = draw(st.lists(st.integers(0, 40), min_size=B, max_size=B))
    causal = draw(st.booleans())
    seed = draw(st.integers(0, 2**31 - 1))
    return dict(B=B, H=KV * group, KV=KV, D=D, BLOCK=BLOCK, NQ=NQ, lens=lens, causal=causal,
                seed=seed)


SETTINGS = hypothesis.settings(max_examples=60, deadline=None, derandomize=True)


@SETTINGS
@hypothesis.given(cases())
def test_oracle_equals_sdpa(c):
    case = op.dense_case(c["B"], c["H"], c["KV"], c["D"], c["BLOCK"], c["NQ"], c["lens"],
                         seed=c["seed"])
    scale = 1.0 / math.sqrt(c["D"])
    got = op.run(oracle.default(), case, scale, c["causal"])
    want = op.sdpa_reference(case, scale, c["causal"])
    assert np.max(np.abs(got - want)) < 1e-12


@SETTINGS
@hypothesis.given(cases(), st.data())
def test_slot_patch_equals_sdpa(c, data):
    case = op.dense_case(c["B"], c["H"], c["KV"], c["D"], c["BLOCK"], c["NQ"], c["lens"],
                         seed=c["seed"])
    positions = np.full((c["B"], c["NQ"]), -1, dtype=np.int32)
    for b, n in enumerate(c["lens"]):
        for j in range(c["NQ"]):
            kind = data.draw(st.sampled_from(["none", "own", "other"]))
            if kind == "own" and n > 0:
                positions[b, j] = op.slot_of(case, b, data.draw(st.integers(0, n - 1)))
            elif kind == "other":
                others = [(bb, nn) for bb, nn in enumerate(c["lens"]) if bb != b and nn > 0]
                if others:
                    bb, nn = data.draw(st.sampled_from(others))
                    positions[b, j] = op.slot_of(case, bb, data.draw(st.integers(0, nn - 1)))
    scale = 1.0 / math.sqrt(c["D"])
    got = op.run(oracle.default(), case, scale, c["causal"], positions=positions)
    want = op.sdpa_reference(op.patched_dense(case, positions), scale, c["causal"])
    assert np.max(np.abs(got - want)) < 1e-12
