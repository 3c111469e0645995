"""Benchmark of paged decode attention on GB300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

One step = one decode call over one batch of the ragged large-batch workload
(B=64 sequences, H=32, KV=4, D=64, BLOCK=32, fp16, past lengths
log-uniform in [64, 16384], blocks randomly permuted over a pool sized to the
blocks in use, 1% of the K/V entries x20, NQ=1): the partition kernel, whose
last CTA on each split segment also merges its partial states (the automatic
split; fixed partitions add the log-sum-exp merge kernel).  It is the largest
of the five workloads and one of the two the HBM target is stated for; the
others are timed in the per-workload table.  The metric is decode-attention
throughput in GB/s of algorithmic bytes (every visible K and V row once, q,
the output, the table entries and lengths) divided by device time, with the
fraction of the measured HBM copy bandwidth.

Sequences are independent, so N GPUs run N independent batches (weak
scaling, no collective on the data path); ``value`` is the bytes of all ranks
over the slowest rank's time.

Pools smaller than L2 (gqa_fp16's are 75 MB) would be served from the
129 MB L2, so the bench keeps copies of the pools (together larger than 3x
L2) and rotates through them step by step: every step reads its K/V from HBM.

``--impl reference`` times the float64 CPU oracle on the host cores on a
bounded sample of the same workload (rank 0 only).
"""
from __future__ import annotations

import argparse
import ctypes
import json
import math
import os
import statistics
import subprocess
import sys
import time
from pathlib import Path

import torch

ROOT = Path(__file__).resolve().parent
sys.path.insert(0, str(ROOT))

WORKLOAD = "ragged_fp16"
METRIC = "decode attention HBM GB/s"
L2_BYTES = 129 * 1024 * 1024


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--workload", default=WORKLOAD)
    ap.add_argument("--no-extras", action="store_true",
                    help="skip the per-workload table and the CPU baseline")
    ap.add_argument("--vjp", action="store_true",
                    help="time only the attention backward on its benchmarked shape (one JSON "
                         "line, --steps timed calls after --warmup)")
    ap.add_argument("--prefill", action="store_true",
                    help="time only the causal prefill of the prefill workload (one JSON "
                         "line, --steps timed calls after --warmup)")
    return ap.parse_args()


def dist_setup(n):
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist

        backend = "nccl" if torch.cuda.is_available() else "gloo"
        if backend == "nccl":
            torch.cuda.set_device(local)
        dist.init_process_group(backend)
    elif torch.cuda.is_available():
        torch.cuda.set_device(local)
    return rank, world, local


def barrier(world):
    if world > 1:
        import torch.distributed as dist

        dist.barrier()


def _all_reduce(x: float, world: int, op: str) -> float:
    if world == 1:
        return x
    import torch.distributed as dist

    dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([x], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX if op == "max" else dist.ReduceOp.SUM)
    return float(t.item())


def reduce_max(x: float, world: int) -> float:
    """Largest value over ranks (the slowest rank's time)."""
    return _all_reduce(x, world, "max")


def reduce_sum(x: float, world: int) -> float:
    """Sum over ranks (the bytes of all ranks' batches)."""
    return _all_reduce(x, world, "sum")


def aggregate(rank_bytes: int, rank_ms: float, world: int):
    """Weak scaling: every rank runs its own batch.  Returns (GB/s of all
    ranks' bytes over the slowest rank's time, that time in ms, total bytes)."""
    ms_max = reduce_max(rank_ms, world)
    total = reduce_sum(float(rank_bytes), world)
    return total / (ms_max * 1e-3) / 1e9, ms_max, int(total)


# The sources each kernel family is built from: a capture stays valid while
# these are unchanged (comments and whitespace aside).
KERNEL_SOURCES = {
    "decode": ["pa_kernels.cuh", "pa_common.cuh", "pa_ptx.cuh", "pa_inst_f32.cu", "pa_inst_f16.cu",
               "pa_inst_bf16.cu", "pa_decode_tc.cu", "pa_tc.cuh", "pa_host.cu",
               "../../include/pa_decode.h"],
    "prefill_tc": ["pa_prefill_tc.cu", "pa_tc.cuh", "pa_tmem.cuh", "pa_ptx.cuh", "pa_common.cuh",
                   "pa_host.cu"],
    "vjp": ["pa_vjp.cu", "pa_vjp_tc.cu", "pa_vjp.cuh", "pa_tc.cuh", "pa_tmem.cuh", "pa_ptx.cuh",
            "../../include/pa_attention_vjp.h"],
}


def kernel_sources_sha256(family: str = "decode") -> str:
    """Hash of the sources of one kernel family with comments and whitespace
    removed, so that a comment edit does not retire a capture of the same code."""
    import hashlib
    import re

    token = re.compile(r'("(?:\\.|[^"\\\n])*")|(//[^\n]*)|(/\*.*?\*/)', re.S)
    csrc = ROOT / "paged_kv_cache_182_gb300" / "csrc"
    h = hashlib.sha256()
    for name in KERNEL_SOURCES[family]:
        f = (csrc / name).resolve()
        code = token.sub(lambda m: m.group(1) or " ", f.read_text())
        h.update(f.name.encode())
        h.update(" ".join(code.split()).encode())
    return h.hexdigest()


def partition_kernel_name(spec):
    """Which partition kernel runs a workload: float32 caches take the
    CUDA-core kernel; 16-bit caches the transposed mma.sync kernel at 8 or
    fewer query rows per KV head, the tcgen05 kernel above 16 rows at D = 128,
    else the 16-row mma.sync one."""
    if spec.dtype == "f32":
        return "pa_split_kernel"
    rows = spec.group * spec.NQ
    if rows <= 8:
        return "pa_mmat_kernel"
    return "pa_umma32_kernel" if rows > 16 and spec.D == 128 else "pa_mma_kernel"


def captured_traffic(kernel: str, workload: str, family: str = "decode"):
    """DRAM bytes per launch from the committed ncu summary of this kernel and
    workload, or None when there is none or the kernel sources changed since."""
    path = ROOT / "profiles" / f"{kernel}_{workload}.md"
    if not path.exists():
        return None
    fields = {}
    for line in path.read_text().splitlines():
        key, sep, val = line.strip().partition(": ")
        if sep and key in ("csrc_sha256", "traffic_bytes_per_launch"):
            fields[key] = val.strip()
    if fields.get("csrc_sha256") != kernel_sources_sha256(family):
        return None
    v = fields.get("traffic_bytes_per_launch")
    return int(v) if v else None


def measured_peaks():
    path = ROOT / "MEASURED_PEAKS.json"
    if path.exists():
        d = json.loads(path.read_text())
        return float(d["hbm_gbs"]), "measured"
    return 6800.0, "fallback"


# ------------------------------------------------------------------ clocks
class Clocks:
    """nvidia-smi sampling of SM clocks and throttle reasons during a region."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.lines = []

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
        time.sleep(0.3)
        return self

    def __exit__(self, *exc):
        if self.proc is not None:
            time.sleep(0.2)
            self.proc.terminate()
            try:
                out, _ = self.proc.communicate(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
                out, _ = self.proc.communicate()
            self.lines = [ln for ln in out.splitlines() if ln.strip()]

    def summary(self):
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                mx.append(float(parts[2]))
            except ValueError:
                continue
            for name, flag in zip(names, parts[5:9]):
                if flag.lower() == "active":
                    reasons.add(name)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"]}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx),
                "reasons": sorted(reasons), "samples": len(sm)}


# -------------------------------------------------------------- our kernels
def rotation_copies(w, device):
    """Enough copies of the KV pools that consecutive steps never hit in L2."""
    pool = 2 * w.k_cache.numel() * w.k_cache.element_size()
    n = max(1, math.ceil(3 * L2_BYTES / pool))
    kc = [w.k_cache.to(device)]
    vc = [w.v_cache.to(device)]
    for _ in range(n - 1):
        kc.append(kc[0].clone())
        vc.append(vc[0].clone())
    return kc, vc, n * pool


def workload_config(w, world):
    """The line's `config`, the same for the device arm and the oracle arm: the
    workload's sizes and lengths, and how the device arm keeps L2 out of it."""
    from paged_kv_cache_182_gb300 import workloads as W

    s = w.spec
    pool = 2 * w.k_cache.numel() * w.k_cache.element_size()
    n = max(1, math.ceil(3 * L2_BYTES / pool))
    return {"workload": s.name, "B": s.B, "H": s.H, "KV": s.KV, "D": s.D, "BLOCK": s.BLOCK,
            "NQ": s.NQ, "causal": s.causal, "partitions": s.partitions or "auto",
            "seq_lens": w.seq_lens.tolist(), "bytes_per_step": W.algorithmic_bytes(w),
            "l2": f"inputs larger than L2 on the device: {n} copies of the KV pools "
                  f"({n * pool // 2**20} MiB) rotated step by step",
            "inputs_unchanged": "on: each device step reads its inputs while the previous "
                                "step finishes (none of them is written between steps); "
                                "per_workload gives the step times with it off too",
            "parallelism": f"independent batches x{world}"}


def make_plans(w, device, partitions=None, inputs_unchanged=False):
    from paged_kv_cache_182_gb300 import binding

    kc, vc, pool_bytes = rotation_copies(w, device)
    q, table, lens, kn, vn = (t.to(device) for t in (w.q, w.block_table, w.seq_lens,
                                                      w.k_new, w.v_new))
    P = w.spec.partitions if partitions is None else partitions
    out = torch.empty(q.shape, dtype=q.dtype, device=device)
    ws = binding.new_workspace(w.spec.B, w.spec.H, w.spec.KV, w.spec.D, w.spec.NQ, P, device)
    plans = []
    for k, v in zip(kc, vc):
        p = binding.Plan(q, k, v, table, lens, kn, vn, scale=w.spec.scale, causal=w.spec.causal,
                         partitions=P, out=out, workspace=ws, inputs_unchanged=inputs_unchanged)
        p.bind_stream(torch.cuda.current_stream(device))
        plans.append(p)
    return plans, pool_bytes


def time_steps(plans, steps, warmup, world, trace=True):
    """Times `steps` decode calls (rotating over the pool copies) on the current
    stream.  Returns (ms per step over the whole region, mean partition-kernel
    ms, kernels launched).  With ``trace`` an event pair brackets each partition
    kernel (its duration for the roofline); events between launches also
    serialise them, so the step time of a traced run is not the headline."""
    from paged_kv_cache_182_gb300 import binding

    stream = torch.cuda.current_stream()
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
           for _ in range(steps)] if trace else []
    for a, b in evs:  # create the events before the timed region
        a.record(stream)
        b.record(stream)
    for i in range(warmup):
        plans[i % len(plans)].set_trace()
        plans[i % len(plans)].run_bound()
    torch.cuda.synchronize()
    barrier(world)
    torch.cuda.synchronize()
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    launches0 = binding.kernel_launches()
    start.record(stream)
    for i in range(steps):
        p = plans[i % len(plans)]
        if trace:
            p.set_trace(*evs[i])
        p.run_bound()
    end.record(stream)
    torch.cuda.synchronize()
    barrier(world)
    torch.cuda.synchronize()
    launches = binding.kernel_launches() - launches0
    for p in plans:
        p.set_trace()
    ms = start.elapsed_time(end) / steps
    split_ms = statistics.mean(a.elapsed_time(b) for a, b in evs) if trace else None
    return ms, split_ms, launches


def e2e_steps(w, device, steps, warmup):
    """Same metric end to end through the public host-buffer call
    (binding.HostPlan -> pa_decode_host): per step the step's inputs (q, table,
    lengths, new rows) go host->device from pinned memory, the kernels run, the
    output comes back to pinned host memory and the host waits for it; the KV
    cache stays resident in HBM, rotated over copies larger than L2 in all."""
    from paged_kv_cache_182_gb300 import binding

    kc, vc, _ = rotation_copies(w, device)  # more than 3x L2, as for the device-timed value
    host = [t.pin_memory() for t in (w.q, w.block_table, w.seq_lens, w.k_new, w.v_new)]
    out = torch.empty(w.q.shape, dtype=w.q.dtype, pin_memory=True)
    h2d = sum(t.numel() * t.element_size() for t in host)
    d2h = out.numel() * out.element_size()
    s = w.spec
    stream = torch.cuda.current_stream(device)
    plans = [binding.HostPlan(k, v, B=s.B, H=s.H, NQ=s.NQ, max_blocks=int(w.block_table.shape[1]),
                              scale=s.scale, causal=s.causal, partitions=s.partitions)
             for k, v in zip(kc, vc)]
    # the step's pinned buffers are declared once (pa_host_register) and bound:
    # each step is one foreign call; the kernels write the output in place
    plans[0].register(*host, out)
    for pl in plans:
        pl.bind(*host, out, stream)

    def step(i):
        plans[i % len(plans)].run_bound()
        stream.synchronize()

    for i in range(warmup):
        step(i)
    t0 = time.perf_counter()
    for i in range(steps):
        step(i)
    el = (time.perf_counter() - t0) / steps * 1e3
    plans[0].close()
    return el, h2d, d2h


def cpu_baseline(w, budget_s=10.0):
    """The float64 oracle as it stands on the host cores, on whole sequences of
    the workload until about `budget_s` seconds have passed."""
    import numpy as np

    import oracle
    from paged_kv_cache_182_gb300 import workloads as W

    orc = oracle.default()
    threads = orc.max_threads()
    args = [np.ascontiguousarray(t.to(torch.float64).numpy()) if t.is_floating_point() else
            t.numpy() for t in w.tensors()]
    done_bytes, t0, calls = 0, time.perf_counter(), 0
    per = W.algorithmic_bytes(w)
    while True:
        orc.decode(*args, scale=w.spec.scale, causal=w.spec.causal, threads=threads)
        calls += 1
        done_bytes += per
        el = time.perf_counter() - t0
        if el >= budget_s or calls >= 2000:
            break
    return {"value": round(done_bytes / el / 1e9, 4), "unit": "GB/s", "cores": threads,
            "kind": "oracle",
            "sample": f"{calls} full decode steps of {w.spec.name} (B={w.spec.B}) in {el:.1f} s, "
                      f"float64, OpenMP over (sequence, head, row)"}


def per_workload_table(device, steps, warmup, peak, peak_kind):
    from paged_kv_cache_182_gb300 import workloads as W

    rows = []
    for name in W.ORDER:
        w = W.make(name, seed=0, poison=False)
        plans, _ = make_plans(w, device)
        ms_wait, _, _ = time_steps(plans, steps, warmup, 1, trace=False)
        del plans
        plans, _ = make_plans(w, device, inputs_unchanged=True)
        ms, _, _ = time_steps(plans, steps, warmup, 1, trace=False)
        _, split_ms, _ = time_steps(plans, steps, warmup, 1)
        by = W.algorithmic_bytes(w)
        gbs = by / (ms * 1e-3) / 1e9
        kernel = partition_kernel_name(w.spec)
        achieved = by / (split_ms * 1e-3) / 1e9
        rows.append({"workload": name, "us_per_step": round(ms * 1e3, 2),
                     "us_per_step_inputs_read_after_wait": round(ms_wait * 1e3, 2),
                     "partition_kernel_us": round(split_ms * 1e3, 2),
                     "GB_per_s": round(gbs, 1), "frac_of_measured_hbm": round(gbs / peak, 3),
                     "tokens_per_s": round(w.spec.B * w.spec.NQ / (ms * 1e-3), 1),
                     "bytes_per_step": by, "partitions": w.spec.partitions or "auto",
                     "roofline": {"bound": "hbm", "kernel": kernel, "achieved": round(achieved, 1),
                                  "peak": peak, "unit": "GB/s", "frac": round(achieved / peak, 4),
                                  "traffic": captured_traffic(kernel, name),
                                  "peak_kind": peak_kind}})
        del plans
        torch.cuda.empty_cache()
    return rows


def append_timing(device, steps=200, warmup=10):
    """pa_cache_append on the causal-append workload: the step's new rows
    written over the slots of each sequence's last NQ cached tokens, back to
    back on rotated copies of the pools; bytes = new rows read + cache rows
    written, K and V."""
    from paged_kv_cache_182_gb300 import binding
    from paged_kv_cache_182_gb300 import workloads as W

    w = W.make("causal_append_fp16", seed=0, poison=False)
    s = w.spec
    slots = torch.full((s.B, s.NQ), -1, dtype=torch.int32)
    for b in range(s.B):
        past = int(w.seq_lens[b])
        for j in range(s.NQ):
            t = past - s.NQ + j
            if t >= 0:
                slots[b, j] = int(w.block_table[b, t // s.BLOCK]) * s.BLOCK + t % s.BLOCK
    kc, vc, _ = rotation_copies(w, device)
    kn, vn, sl = w.k_new.to(device), w.v_new.to(device), slots.to(device)
    stream = torch.cuda.current_stream(device)
    binding.cache_append(kc[0], vc[0], kn, vn, sl, stream=stream)  # argument checks once
    # then the C entry point with prepared arguments, as a bound decode plan does
    args = [[ctypes.c_void_p(k.data_ptr()), ctypes.c_void_p(v.data_ptr()),
             ctypes.c_void_p(kn.data_ptr()), ctypes.c_void_p(vn.data_ptr()),
             ctypes.c_void_p(sl.data_ptr()), s.B, s.KV, s.D, s.NQ, s.BLOCK,
             int(w.k_cache.shape[0]), binding.PA_F16, None, ctypes.c_void_p(stream.cuda_stream)]
            for k, v in zip(kc, vc)]
    for i in range(warmup):
        binding.LIB.pa_cache_append(*args[i % len(args)])
    torch.cuda.synchronize()
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record(stream)
    for i in range(steps):
        binding.LIB.pa_cache_append(*args[i % len(args)])
    b.record(stream)
    torch.cuda.synchronize()
    us = a.elapsed_time(b) / steps * 1e3
    moved = 2 * 2 * int((slots >= 0).sum()) * s.KV * s.D * w.k_new.element_size()
    return {"kernel": "pa_append_kernel", "workload": "causal_append_fp16 new rows",
            "us_per_call": round(us, 2), "bytes_per_call": moved,
            "GB_per_s": round(moved / (us * 1e-6) / 1e9, 1)}


def prefill_flops(w):
    """Algorithmic flops of a causal prefill: row r of sequence b attends to
    past + r + 1 keys, 2 flops per multiply-add in q.k and in p.v."""
    s = w.spec
    keys = sum(s.NQ * past + s.NQ * (s.NQ + 1) // 2 for past in w.seq_lens.tolist())
    return 4 * s.H * s.D * keys


def prefill_timing(device, steps=20, warmup=3):
    """pa_prefill on the prefill workload (NQ = 512 new rows after 1024 cached
    tokens), back to back on rotated copies of the pools; the stores of the
    new rows rewrite the same values each call."""
    from paged_kv_cache_182_gb300 import binding
    from paged_kv_cache_182_gb300 import workloads as W

    w = W.make_prefill("prefill_fp16", seed=0)
    s = w.spec
    kc, vc, pool_bytes = rotation_copies(w, device)
    q, table, lens, kn, vn = (t.to(device) for t in (w.q, w.block_table, w.seq_lens,
                                                      w.k_new, w.v_new))
    out = torch.empty(q.shape, dtype=q.dtype, device=device)
    plans = [binding.PrefillPlan(q, k, v, table, lens, kn, vn, scale=s.scale, out=out)
             for k, v in zip(kc, vc)]
    stream = torch.cuda.current_stream(device)
    for i in range(warmup):
        plans[i % len(plans)].run(stream)
    torch.cuda.synchronize()
    launches = binding.kernel_launches()
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record(stream)
    for i in range(steps):
        plans[i % len(plans)].run(stream)
    b.record(stream)
    torch.cuda.synchronize()
    us = a.elapsed_time(b) / steps * 1e3
    flops = prefill_flops(w)
    peak = float(json.loads((ROOT / "MEASURED_PEAKS.json").read_text())["bf16_tflops"]) \
        if (ROOT / "MEASURED_PEAKS.json").exists() else 1900.0
    tflops = flops / (us * 1e-6) / 1e12
    return {"workload": f"prefill_fp16 (B={s.B}, H={s.H}, KV={s.KV}, D={s.D}, BLOCK={s.BLOCK}, "
                        f"past={int(w.seq_lens[0])}, NQ={s.NQ}, causal)",
            "us_per_call": round(us, 1), "new_tokens_per_s": round(s.B * s.NQ / (us * 1e-6), 1),
            "flops_per_call": flops, "TFLOP_per_s": round(tflops, 2),
            "frac_of_measured_tensor_peak": round(tflops / peak, 4),
            "roofline": {"bound": "tensor", "achieved": round(tflops, 2), "peak": peak,
                         "unit": "TFLOP/s", "frac": round(tflops / peak, 4),
                         "traffic": captured_traffic("pa_prefill_tc_kernel", "prefill_fp16",
                                                     "prefill_tc"),
                         "kernel": "pa_prefill_tc_kernel (and the store of the new rows)",
                         "peak_kind": "bf16_tflops of MEASURED_PEAKS.json (burst); f16 has the "
                                      "same nominal dense rate"},
            "launches_per_call": (binding.kernel_launches() - launches) // steps,
            "l2": f"{len(plans)} copies of the KV pools ({pool_bytes // 2**20} MiB) rotated"}


def vjp_timing(device, steps=10, warmup=3):
    """pa_attention_vjp on the benchmarked backward shape (4 sequences of 2048
    tokens, 32 query heads on 8 key/value heads, D 128, bf16, causal), back to
    back; q, k, v, y, g and the outputs (about 350 MB) are larger than L2."""
    from paged_kv_cache_182_gb300 import binding
    from paged_kv_cache_182_gb300 import workloads as W

    s = W.VJP_SPECS["vjp_bf16"]
    x = W.make_vjp(s, seed=0).to(device)
    plan = binding.VjpPlan(x.q, x.k, x.v, x.y, x.g, scale=1.0 / math.sqrt(s.D), causal=s.causal)
    stream = torch.cuda.current_stream(device)
    for _ in range(warmup):
        plan.run(stream)
    torch.cuda.synchronize()
    launches = binding.kernel_launches()
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record(stream)
    for _ in range(steps):
        plan.run(stream)
    b.record(stream)
    torch.cuda.synchronize()
    us = a.elapsed_time(b) / steps * 1e3
    flops = W.vjp_flops(s)
    peak = float(json.loads((ROOT / "MEASURED_PEAKS.json").read_text())["bf16_tflops"]) \
        if (ROOT / "MEASURED_PEAKS.json").exists() else 1900.0
    tflops = flops / (us * 1e-6) / 1e12
    return {"workload": f"vjp_bf16 (B={s.B}, HQ={s.HQ}, HK={s.HK}, SQ={s.SQ}, SK={s.SK}, "
                        f"D={s.D}, causal)",
            "us_per_call": round(us, 1), "tokens_per_s": round(s.B * s.SQ / (us * 1e-6), 1),
            "flops_per_call": flops, "TFLOP_per_s": round(tflops, 2),
            "frac_of_measured_tensor_peak": round(tflops / peak, 4),
            "roofline": {"bound": "tensor", "achieved": round(tflops, 2), "peak": peak,
                         "unit": "TFLOP/s", "frac": round(tflops / peak, 4),
                         "traffic": captured_traffic("vjp_main_tc", "vjp_bf16", "vjp"),
                         "traffic_kernel": "vjp_main_tc, per launch (the call's largest)",
                         "kernel": "the whole call: vjp_stats_tc, vjp_main_tc, vjp_dq_round",
                         "peak_kind": "bf16_tflops of MEASURED_PEAKS.json (burst)"},
            "launches_per_call": (binding.kernel_launches() - launches) // steps,
            "l2": "inputs and outputs (about 350 MB) larger than L2"}


def run_ours(args, rank, world, local):
    from paged_kv_cache_182_gb300 import binding  # noqa: F401  (fails loudly if not built)
    from paged_kv_cache_182_gb300 import workloads as W

    device = torch.device("cuda", local)
    peak, peak_kind = measured_peaks()
    w = W.make(args.workload, seed=rank, poison=False)
    per_rank_bytes = W.algorithmic_bytes(w)
    # every step reads another copy of the pools and writes only the output and
    # the workspace, so the kernel before a step writes none of its inputs
    # (pa_opts.inputs_unchanged): each step reads them while the previous one
    # finishes, and waits for it before writing
    plans, _ = make_plans(w, device, inputs_unchanged=True)
    with Clocks(local) as clk:
        # the headline: plain back-to-back steps, no events between them
        ms, _, launches = time_steps(plans, args.steps, args.warmup, world, trace=False)
    # the partition kernel's own duration (roofline), from events around each
    # launch in a second timed pass
    _, split_ms, _ = time_steps(plans, max(20, args.steps // 4), args.warmup, world)
    value, ms_max, total_bytes = aggregate(per_rank_bytes, ms, world)
    achieved = per_rank_bytes / (split_ms * 1e-3) / 1e9
    kernel = partition_kernel_name(w.spec)
    traffic = captured_traffic(kernel, w.spec.name)
    del plans
    torch.cuda.empty_cache()
    e2e_ms, h2d, d2h = e2e_steps(w, device, max(20, args.steps // 4), 3)
    e2e_value, e2e_ms, _ = aggregate(per_rank_bytes, e2e_ms, world)
    line = {
        "metric": METRIC, "value": round(value, 1), "unit": "GB/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms_max, 5),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": w.spec.dtype,
        "data": "synthetic (seeded N(0,1), random block permutation)",
        "config": workload_config(w, world),
        "bytes_per_step_all_ranks": total_bytes,
        "tokens_per_s": round(reduce_sum(w.spec.B * w.spec.NQ, world) / (ms_max * 1e-3), 1),
        "roofline": {"bound": "hbm", "achieved": round(achieved, 1), "peak": peak,
                     "unit": "GB/s", "frac": round(achieved / peak, 4), "traffic": traffic,
                     "kernel": kernel, "peak_kind": peak_kind,
                     "algorithmic_bytes": per_rank_bytes},
        "e2e": {"value": round(e2e_value, 2),
                "unit": "GB/s", "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h},
        "gpu_launches": launches,
        "clocks": clk.summary(),
    }
    if rank == 0 and not args.no_extras:
        line["per_workload"] = per_workload_table(device, 50, 5, peak, peak_kind)
        line["cache_append"] = append_timing(device)
        line["prefill"] = prefill_timing(device)
        line["attention_vjp"] = vjp_timing(device)
        line["cpu_baseline"] = cpu_baseline(w)
    if rank == 0:
        print(json.dumps(line), flush=True)


def run_reference(args, rank, world):
    """The float64 oracle on the host cores: every step a whole decode step of
    the workload (all rows of every sequence), on rank 0 only."""
    if rank != 0:
        return
    import numpy as np

    import oracle
    from paged_kv_cache_182_gb300 import workloads as W

    w = W.make(args.workload, seed=0, poison=False)
    s = w.spec
    orc = oracle.default()
    threads = orc.max_threads()
    args_np = [np.ascontiguousarray(t.to(torch.float64).numpy()) if t.is_floating_point() else
               t.numpy() for t in w.tensors()]
    by = W.algorithmic_bytes(w)

    def step():
        orc.decode(*args_np, scale=s.scale, causal=s.causal, threads=threads)

    for _ in range(args.warmup):
        step()
    t0 = time.perf_counter()
    for _ in range(args.steps):
        step()
    el = (time.perf_counter() - t0) / args.steps
    value = by / el / 1e9
    line = {
        "metric": METRIC, "value": round(value, 4), "unit": "GB/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(el * 1e3, 5),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic (seeded N(0,1), random block permutation)",
        "config": workload_config(w, world),
        "impl": "reference",
        "cpu_baseline": {"value": round(value, 4), "unit": "GB/s", "cores": threads,
                         "kind": "oracle",
                         "sample": f"{args.steps} whole decode steps of {s.name} (B={s.B}, all "
                                   f"{s.B * s.H * s.NQ} query rows), float64, OpenMP over "
                                   f"(sequence, head, row)"},
        "e2e": {"value": round(value, 4), "unit": "GB/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def main():
    args = parse()
    rank, world, local = dist_setup(args.gpus)
    if args.impl == "reference":
        run_reference(args, rank, world)
    else:
        if not torch.cuda.is_available():
            raise SystemExit("bench.py --impl ours needs a CUDA device")
        if args.vjp:
            if rank == 0:
                line = vjp_timing(torch.device("cuda", local), args.steps, args.warmup)
                print(json.dumps({"mode": "attention_vjp", **line}), flush=True)
        elif args.prefill:
            if rank == 0:
                line = prefill_timing(torch.device("cuda", local), args.steps, args.warmup)
                print(json.dumps({"mode": "prefill", **line}), flush=True)
        else:
            run_ours(args, rank, world, local)
    if world > 1:
        import torch.distributed as dist

        dist.destroy_process_group()


if __name__ == "__main__":
    main()
