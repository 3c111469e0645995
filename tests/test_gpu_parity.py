"""CUDA path against the float64 oracle, element by element (needs a GPU).

Inputs come from the seeded generators; unused pool blocks and cache slots
past each length are NaN, so any stray read shows up as a non-finite output.
"""
import numpy as np
import pytest
import torch

import parity_util as pu
from paged_kv_cache_182_gb300 import workloads as W

pytestmark = pytest.mark.gpu

FMT_OUT = {"f32": torch.float32, "f16": torch.float16, "bf16": torch.bfloat16}


def small(name, **kw):
    """A reduced copy of a named workload: several tiles, ragged tails."""
    s = W.SPECS[name]
    base = dict(
        tiny_fp32=dict(),
        gqa_fp16=dict(B=3, past=150, past_hi=900),
        long_bf16=dict(past=3000),
        causal_append_fp16=dict(B=3, past=333),
        ragged_fp16=dict(B=7, past=20, past_hi=2500),
    )[name]
    base.update(kw)
    return W.shrink(s, **base)


# ------------------------------------------------------------- full workloads
@pytest.mark.parametrize("name", W.ORDER)
def test_full_workload_f32_output(name):
    w = W.make(name, seed=0)
    got = pu.run_gpu(w, out_dtype=torch.float32)
    want = pu.run_oracle(w)
    pu.check(got, want, w.spec.dtype, "f32", name)


@pytest.mark.parametrize("name", W.ORDER)
def test_full_workload_native_output(name):
    w = W.make(name, seed=1)
    got = pu.run_gpu(w)
    assert got.dtype == FMT_OUT[w.spec.dtype]
    want = pu.run_oracle(w)
    pu.check(got, want, w.spec.dtype, w.spec.dtype, name)


# ---------------------------------------------------------- split invariance
@pytest.mark.parametrize("name", W.ORDER)
@pytest.mark.parametrize("P", [1, 2, 7, 32, 0])
def test_partition_counts(name, P):
    w = W.make(small(name), seed=2)
    got = pu.run_gpu(w, partitions=P, out_dtype=torch.float32)
    pu.check(got, pu.run_oracle(w), w.spec.dtype, "f32", f"{name} P={P}")


@pytest.mark.parametrize("seed", [3, 4])
def test_more_seeds_small(seed):
    for name in W.ORDER:
        w = W.make(small(name), seed=seed)
        got = pu.run_gpu(w, out_dtype=torch.float32)
        pu.check(got, pu.run_oracle(w), w.spec.dtype, "f32", f"{name} seed={seed}")


# ---------------------------------------------------------------- shape sweep
SWEEP = [
    # dtype, H, KV, D, BLOCK, NQ, causal, lens
    ("f32", 8, 2, 128, 8, 1, False, [1, 77, 300]),
    ("bf16", 16, 2, 64, 64, 3, True, [0, 64, 129, 1000]),
    ("f16", 12, 3, 128, 32, 16, True, [5, 40]),
    ("f16", 12, 3, 128, 32, 16, False, [31, 33]),
    ("f16", 40, 5, 64, 16, 2, True, [400, 17]),       # 16 rows per KV head
    ("bf16", 64, 1, 128, 16, 1, False, [700]),        # MQA: 64 rows, two row groups
    ("f32", 4, 4, 64, 16, 1, False, [5000]),           # no grouping, long
    ("f16", 32, 8, 128, 8, 4, True, [2047, 2048, 2049]),
]


@pytest.mark.parametrize("case", SWEEP, ids=lambda c: f"{c[0]}-H{c[1]}-KV{c[2]}-D{c[3]}-B{c[4]}-NQ{c[5]}-{'c' if c[6] else 'n'}")
@pytest.mark.parametrize("P", [0, 1, 3])
def test_shape_sweep(case, P):
    dt, H, KV, D, BLOCK, NQ, causal, lens = case
    spec = W.Spec("sweep", dt, B=len(lens), H=H, KV=KV, D=D, BLOCK=BLOCK, NQ=NQ,
                  causal=causal, pool_blocks=0, extra_table_cols=2)
    w = W.make(spec, seed=5, lens=lens)
    # a few spare (poisoned) pool blocks beyond the referenced ones
    got = pu.run_gpu(w, partitions=P, out_dtype=torch.float32)
    pu.check(got, pu.run_oracle(w), dt, "f32", f"sweep {case} P={P}")


# ------------------------------------------------------------- closed forms
def test_single_key_returns_new_value_exactly():
    spec = W.Spec("one", "f16", B=3, H=8, KV=2, D=128, BLOCK=16, NQ=1)
    w = W.make(spec, seed=6, lens=[0, 0, 0])
    got = pu.run_gpu(w, partitions=0)
    g = spec.group
    want = w.v_new[:, :, 0, :].repeat_interleave(g, dim=1)
    assert torch.equal(got[:, :, 0, :].cpu(), want)


def test_block_permutation_is_bitwise_invariant():
    w = W.make(small("gqa_fp16"), seed=7)
    a = pu.run_gpu(w, out_dtype=torch.float32).cpu()
    g = torch.Generator().manual_seed(8)
    perm = torch.randperm(w.num_blocks, generator=g)  # new slot of each old block
    inv = torch.argsort(perm)
    w2 = W.Workload(w.spec, w.seq_lens, w.block_table.clone(), w.q, w.k_cache[inv].contiguous(),
                    w.v_cache[inv].contiguous(), w.k_new, w.v_new)
    t = w2.block_table
    t[t >= 0] = perm[t[t >= 0].long()].to(torch.int32)
    b = pu.run_gpu(w2, out_dtype=torch.float32).cpu()
    assert torch.equal(a, b)


def test_repeat_calls_are_deterministic():
    w = W.make(small("ragged_fp16"), seed=9)
    a = pu.run_gpu(w, out_dtype=torch.float32).cpu()
    b = pu.run_gpu(w, out_dtype=torch.float32).cpu()
    assert torch.equal(a, b)


# ------------------------------------------------------- streams and graphs
def test_side_stream_and_graph_replay():
    from paged_kv_cache_182_gb300 import binding

    w = W.make(small("gqa_fp16"), seed=10)
    dev = w.to("cuda")
    want = pu.run_oracle(w)
    s = torch.cuda.Stream()
    plan = binding.Plan(*dev.tensors(), scale=w.spec.scale, partitions=0,
                        out_dtype=torch.float32)
    with torch.cuda.stream(s):
        plan.run(s)
    s.synchronize()
    pu.check(plan.out, want, "f16", "f32", "side stream")
    plan.out.zero_()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        plan.run()
    graph.replay()
    torch.cuda.synchronize()
    pu.check(plan.out, want, "f16", "f32", "graph replay")


# ----------------------------------------------------------- device checks
def test_checked_mode_reports_bad_block():
    w = W.make(small("gqa_fp16"), seed=11)
    w.block_table[1, 2] = w.num_blocks + 3
    w.block_table[2, 0] = -2
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    pu.run_gpu(w, out_dtype=torch.float32, status=status, checked=True)
    assert int(status.item()) & 1


def test_length_beyond_table_is_clamped_and_reported():
    w = W.make(small("gqa_fp16"), seed=12)
    lens = w.seq_lens.clone()
    w_ok = W.Workload(w.spec, lens.clone(), w.block_table, w.q, w.k_cache, w.v_cache,
                      w.k_new, w.v_new)
    cap = w.max_blocks * w.spec.BLOCK
    lens[0] = cap + 100
    w.seq_lens = lens
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    pu.run_gpu(w, out_dtype=torch.float32, status=status)
    assert int(status.item()) & 2
    assert w_ok.seq_lens[0] <= cap


def test_checked_mode_clean_run_has_zero_status():
    w = W.make(small("ragged_fp16"), seed=13)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    got = pu.run_gpu(w, out_dtype=torch.float32, status=status, checked=True)
    assert int(status.item()) == 0
    pu.check(got, pu.run_oracle(w), "f16", "f32", "checked clean")


def test_kernel_launch_counter_moves():
    from paged_kv_cache_182_gb300 import binding

    before = binding.kernel_launches()
    w = W.make(small("gqa_fp16"), seed=14)
    pu.run_gpu(w, partitions=1)
    pu.run_gpu(w, partitions=0)
    pu.run_gpu(w, partitions=0, merge_kernel=True)
    pu.run_gpu(w, partitions=3)
    # 1 + 1 (merge in the kernel) + 2 + 2 (fixed partitions: merge kernel)
    assert binding.kernel_launches() - before == 6


# ------------------------------------------------ workspace hygiene
@pytest.mark.parametrize("name", W.ORDER)
@pytest.mark.parametrize("P", [0, 3])
def test_workspace_garbage_is_never_read(name, P):
    """A workspace full of NaN bytes must not leak into the output: every
    partial record the merge reads was written in the same call."""
    from paged_kv_cache_182_gb300 import binding

    w = W.make(small(name), seed=15)
    s = w.spec
    want = pu.run_oracle(w)
    for merge_kernel in (False, True):
        ws = torch.full((binding.workspace_bytes(s.B, s.H, s.KV, s.D, s.NQ, P),), 0xFF,
                        dtype=torch.uint8, device="cuda")
        zb = binding.workspace_zero_bytes(s.B, s.H, s.KV, s.D, s.NQ, P)
        ws[:zb] = 0  # the split counters of the in-kernel merge start at zero
        for rep in range(2):  # the second call reuses the counters the first left
            got = pu.run_gpu(w, partitions=P, out_dtype=torch.float32, workspace=ws,
                             merge_kernel=merge_kernel)
            pu.check(got, want, s.dtype, "f32",
                     f"{name} P={P} merge_kernel={merge_kernel} call {rep} garbage workspace")
        assert int(ws[:zb].count_nonzero()) == 0, "counters must be left at zero"


@pytest.mark.parametrize("name", W.ORDER)
@pytest.mark.parametrize("P", [0, 2, 7])
def test_separate_merge_kernel(name, P):
    w = W.make(small(name), seed=16)
    got = pu.run_gpu(w, partitions=P, out_dtype=torch.float32, merge_kernel=True)
    pu.check(got, pu.run_oracle(w), w.spec.dtype, "f32", f"{name} P={P} merge kernel")


def test_repeated_calls_full_ragged_are_stable():
    """Many short pieces per CTA keep the producer several pieces ahead of
    the consumers: the query-buffer and stage hand-offs are exercised on every
    call.  Twenty calls in a row must all equal the first, which matches the
    oracle."""
    w = W.make("ragged_fp16", seed=17)
    want = pu.run_oracle(w)
    first = pu.run_gpu(w, out_dtype=torch.float32)
    pu.check(first, want, "f16", "f32", "ragged repeated, call 0")
    first = first.cpu()
    for rep in range(1, 20):
        got = pu.run_gpu(w, out_dtype=torch.float32).cpu()
        assert torch.equal(got, first), f"call {rep} differs from call 0"


@pytest.mark.parametrize("name", ["gqa_fp16", "ragged_fp16", "long_bf16", "tiny_fp32"])
@pytest.mark.parametrize("P", [0, 3])
def test_host_entry_point_matches_device_call(name, P):
    """pa_decode_host (inputs and output in pinned host memory, two steps in a
    row on one plan: same cache and table, new queries and new rows) gives
    exactly pa_decode's output, which matches the oracle."""
    from paged_kv_cache_182_gb300 import binding

    w0 = W.make(small(name), seed=20)
    s = w0.spec
    plan = binding.HostPlan(w0.k_cache.cuda(), w0.v_cache.cuda(), B=s.B, H=s.H, NQ=s.NQ,
                            max_blocks=int(w0.block_table.shape[1]), scale=s.scale,
                            causal=s.causal, partitions=P, out_dtype=torch.float32)
    g = torch.Generator().manual_seed(21)
    for rep in range(2):
        if rep == 0:
            w = w0
        else:
            fresh = [torch.randn(t.shape, generator=g).to(t.dtype) for t in (w0.q, w0.k_new, w0.v_new)]
            w = W.Workload(s, w0.seq_lens, w0.block_table, fresh[0], w0.k_cache, w0.v_cache,
                           fresh[1], fresh[2])
        host = [t.pin_memory() for t in (w.q, w.block_table, w.seq_lens, w.k_new, w.v_new)]
        out = torch.full(w.q.shape, float("nan"), dtype=torch.float32).pin_memory()
        plan.run(*host, out)
        torch.cuda.synchronize()
        want_dev = pu.run_gpu(w, partitions=P, out_dtype=torch.float32).cpu()
        assert torch.equal(out, want_dev), f"{name} P={P} step {rep}"
        pu.check(out, pu.run_oracle(w), s.dtype, "f32", f"{name} P={P} host step {rep}")


def test_host_entry_point_pageable_buffers():
    """Inputs and output in pageable host memory take the one-copy-per-input
    path (no device view of them); the result equals that of pinned buffers,
    which the device reads with one gather kernel."""
    from paged_kv_cache_182_gb300 import binding

    w = W.make(small("gqa_fp16"), seed=22)
    s = w.spec
    plan = binding.HostPlan(w.k_cache.cuda(), w.v_cache.cuda(), B=s.B, H=s.H, NQ=s.NQ,
                            max_blocks=int(w.block_table.shape[1]), scale=s.scale,
                            causal=s.causal, partitions=0, out_dtype=torch.float32)
    outs = []
    for pinned in (False, True):
        host = [t.clone().pin_memory() if pinned else t.clone()
                for t in (w.q, w.block_table, w.seq_lens, w.k_new, w.v_new)]
        out = torch.full(w.q.shape, float("nan"), dtype=torch.float32)
        out = out.pin_memory() if pinned else out
        plan.run(*host, out)
        torch.cuda.synchronize()
        outs.append(out.clone())
    assert torch.equal(outs[0], outs[1])
    pu.check(outs[0], pu.run_oracle(w), s.dtype, "f32", "pageable host buffers")


@pytest.mark.parametrize("name", ["gqa_fp16", "ragged_fp16", "tiny_fp32"])
def test_host_entry_point_registered_buffers(name):
    """Registered pinned buffers (pa_host_register): the step's inputs are read
    through their recorded device addresses and the output is written by the
    kernels in place (no copy back); over two steps on one bound plan the
    result equals pa_decode's bit for bit.  After unregistering, the same
    buffers take the per-call path and give the same result."""
    from paged_kv_cache_182_gb300 import binding

    w = W.make(small(name), seed=25)
    s = w.spec
    plan = binding.HostPlan(w.k_cache.cuda(), w.v_cache.cuda(), B=s.B, H=s.H, NQ=s.NQ,
                            max_blocks=int(w.block_table.shape[1]), scale=s.scale,
                            causal=s.causal, partitions=0, out_dtype=torch.float32)
    host = [t.clone().pin_memory() for t in (w.q, w.block_table, w.seq_lens, w.k_new, w.v_new)]
    out = torch.full(w.q.shape, float("nan"), dtype=torch.float32).pin_memory()
    plan.register(*host, out)
    plan.bind(*host, out)
    want = pu.run_gpu(w, partitions=0, out_dtype=torch.float32).cpu()
    for step in range(2):
        out.fill_(float("nan"))
        plan.run_bound()
        torch.cuda.synchronize()
        assert torch.equal(out, want), f"{name} registered step {step}"
    plan.close()
    out.fill_(float("nan"))
    plan.run(*host, out)
    torch.cuda.synchronize()
    assert torch.equal(out, want)
    pu.check(out, pu.run_oracle(w), s.dtype, "f32", f"{name} registered host buffers")


@pytest.mark.parametrize("name,P", [("ragged_fp16", 0), ("long_bf16", 32), ("gqa_fp16", 0),
                                    ("causal_append_fp16", 0), ("tiny_fp32", 0)])
def test_inputs_unchanged_back_to_back(name, P):
    """pa_opts.inputs_unchanged: two batches with different data share the output
    and the workspace and run back to back with no sync, each reading its
    inputs before the previous decode has completed.  The writes still wait,
    so the last call's batch is what out holds, and it matches the oracle."""
    from paged_kv_cache_182_gb300 import binding

    wa = W.make(small(name), seed=21)
    wb = W.make(small(name), seed=22)
    dev = "cuda"
    da, db = wa.to(dev), wb.to(dev)
    out = torch.empty(da.q.shape, dtype=torch.float32, device=dev)
    s = wa.spec
    ws = binding.new_workspace(s.B, s.H, s.KV, s.D, s.NQ, P, dev)
    plans = [binding.Plan(*d.tensors(), scale=s.scale, causal=s.causal, partitions=P, out=out,
                          workspace=ws, out_dtype=torch.float32, inputs_unchanged=True)
             for d in (da, db)]
    want = [pu.run_oracle(w) for w in (wa, wb)]
    for last in (1, 0):
        n = 11
        for i in range(n):  # alternating, ending on plan `last`
            plans[last ^ ((n - 1 - i) & 1)].run()
        torch.cuda.synchronize()
        pu.check(out, want[last], s.dtype, "f32", f"{name} back to back, last = {'ab'[last]}")
