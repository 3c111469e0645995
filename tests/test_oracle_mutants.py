"""Plausible mistakes planted in a copy of the oracle must each fail a pin.

Each mutant is a one-spot textual edit of ``oracle/pa_oracle.c`` (a wrong
index, a dropped term, a swapped operand), compiled into a temporary library
and run against every pin in a child process, so that a mutant that reads out
of bounds cannot take the test run down with it.  The real oracle source is
never modified.
"""
import os
import subprocess
import sys
from pathlib import Path

import pytest

ROOT = Path(__file__).resolve().parent.parent
SOURCE = ROOT / "oracle" / "pa_oracle.c"

MUTANTS = {
    "gqa_modulo": ("const int kh = h / group;", "const int kh = h % KV;"),
    "causal_off_by_one": ("int total = past + (causal ? r + 1 : NQ);", "int total = past + (causal ? r : NQ);"),
    "causal_ignored": ("int total = past + (causal ? r + 1 : NQ);", "int total = past + NQ;"),
    "new_row_index": ("int j = i - past;", "int j = 0;"),
    "table_index_mod": ("[(int64_t)b * max_blocks + i / BLOCK]", "[(int64_t)b * max_blocks + i % BLOCK]"),
    "table_row_ignored": ("[(int64_t)b * max_blocks + i / BLOCK]", "[i / BLOCK]"),
    "slot_offset_div": ("(int64_t)physical * BLOCK + i % BLOCK", "(int64_t)physical * BLOCK + i / BLOCK"),
    "cache_layout_head_major": ("return cache + (slot * KV + kh) * D;",
                                "return cache + ((int64_t)kh * num_blocks * BLOCK + slot) * D;"),
    "scale_dropped": ("dot += (scale * qrow[d]) * k[d];", "dot += qrow[d] * k[d];"),
    "no_max_shift": ("s[i] = exp(s[i] - m);", "s[i] = exp(s[i]);"),
    "min_instead_of_max": ("if (s[i] > m)", "if (s[i] < m || m == -INFINITY)"),
    "no_normalisation": ("if (denom != 0.0)", "if (0)"),
    "values_from_keys": ("const double *v = key_row(v_cache, v_new,", "const double *v = key_row(k_cache, k_new,"),
    "new_rows_from_head_zero": ("fresh + (((int64_t)b * KV + kh) * NQ + j) * D", "fresh + (((int64_t)b * KV) * NQ + j) * D"),
    "positions_first_wins": ("bound = p;", "if (bound < 0) bound = p;"),
    "positions_sequence_ignored": ("positions[(int64_t)b * NQ + p]", "positions[p]"),
    "positions_ignored": ("if (bound >= 0)", "if (0)"),
    "patched_row_zero": ("NQ + bound) * D", "NQ + 0) * D"),
    "patched_from_head_zero": ("fresh + (((int64_t)b * KV + kh) * NQ + bound) * D",
                               "fresh + (((int64_t)b * KV) * NQ + bound) * D"),
    "head_row_swapped": ("const int r = (int)(flat % NQ);\n        const int h = (int)((flat / NQ) % H);",
                         "const int h = (int)(flat % H);\n        const int r = (int)((flat / H) % NQ);"),
}

CHILD = r"""
import sys
sys.path[:0] = [{root!r}, {tests!r}]
import oracle, oracle_pins
failed = oracle_pins.run_all(oracle.Oracle({lib!r}))
print("\n".join(failed))
sys.exit(3 if failed else 0)
"""


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_mutant_is_caught(name, tmp_path):
    import oracle

    old, new = MUTANTS[name]
    text = SOURCE.read_text()
    assert text.count(old) == 1, f"mutation anchor for {name} not found exactly once"
    src = tmp_path / f"mutant_{name}.c"
    src.write_text(text.replace(old, new))
    lib = oracle.build(src, tmp_path / f"libmutant_{name}.so", force=True)
    code = CHILD.format(root=str(ROOT), tests=str(ROOT / "tests"), lib=str(lib))
    proc = subprocess.run([sys.executable, "-c", code], capture_output=True, text=True,
                          timeout=300, env=dict(os.environ, OMP_NUM_THREADS="2"))
    assert proc.returncode != 0, f"mutant {name} passed every pin:\n{proc.stdout}{proc.stderr}"


def test_unmutated_copy_passes(tmp_path):
    import oracle

    src = tmp_path / "copy.c"
    src.write_text(SOURCE.read_text())
    lib = oracle.build(src, tmp_path / "libcopy.so", force=True)
    code = CHILD.format(root=str(ROOT), tests=str(ROOT / "tests"), lib=str(lib))
    proc = subprocess.run([sys.executable, "-c", code], capture_output=True, text=True, timeout=300)
    assert proc.returncode == 0, proc.stdout + proc.stderr
