"""The bench's oracle arm (`bench.py --impl reference`), run on the CPU: one
JSON line with the device arm's `config`, whole decode steps timed, and the
keys the line contract asks of that arm."""
import json
import subprocess
import sys
from pathlib import Path

ROOT = Path(__file__).resolve().parents[1]


def test_reference_line_matches_device_config():
    out = subprocess.run(
        [sys.executable, "bench.py", "--impl", "reference", "--workload", "tiny_fp32",
         "--steps", "2", "--warmup", "1"],
        cwd=ROOT, capture_output=True, text=True, timeout=300, check=True).stdout
    lines = [ln for ln in out.splitlines() if ln.startswith("{")]
    assert len(lines) == 1, out
    line = json.loads(lines[0])

    sys.path.insert(0, str(ROOT))
    import bench
    from paged_kv_cache_182_gb300 import workloads as W

    w = W.make("tiny_fp32", seed=0, poison=False)
    assert line["impl"] == "reference"
    assert line["config"] == json.loads(json.dumps(bench.workload_config(w, 1)))
    assert line["config"]["seq_lens"] == w.seq_lens.tolist()
    assert line["config"]["partitions"] == (w.spec.partitions or "auto")
    assert line["steps"] == 2 and line["warmup"] == 1 and line["n_gpus"] == 1
    assert line["metric"] == bench.METRIC and line["unit"] == "GB/s"
    assert line["higher_is_better"] is True
    # value is the workload's algorithmic bytes over the measured time of a
    # whole step (no sampled fraction scaled up)
    by = W.algorithmic_bytes(w)
    assert abs(line["value"] - by / (line["ms_per_step"] * 1e-3) / 1e9) <= 1e-3 * line["value"] + 1e-3
    cb = line["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["value"] == line["value"] and cb["cores"] >= 1
    assert "whole decode steps" in cb["sample"]
    assert line["e2e"] == {"value": line["value"], "unit": "GB/s",
                           "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}
