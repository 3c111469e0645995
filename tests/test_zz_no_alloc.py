"""pa_decode_static_workspace: decode attention for callers that may not
allocate device memory (an engine plugin handed only its input and output
buffers, a serving loop that reserved all memory up front, code that cannot
afford the synchronisation of cudaMalloc).  It takes its split scratch from an
array built into the library instead of a caller workspace.

These tests call it through the C ABI with no caller workspace at all and
compare its output with pa_decode's on the same inputs, for two calls in a row
on different workloads (the shared array keeps the first call's contents when
the second runs).  This file is collected last on purpose.
"""
import ctypes

import pytest
import torch

import parity_util as pu
from paged_kv_cache_182_gb300 import workloads as W

pytestmark = pytest.mark.gpu

PA_ERR_STATIC_LIMIT = -8


def static_call(plan):
    """Call the static-scratch entry point with the plan's arguments but with
    no workspace in the options."""
    from paged_kv_cache_182_gb300 import binding

    opts = binding.PaOpts.from_buffer_copy(plan.opts)
    opts.workspace = None
    opts.workspace_bytes = 0
    args = plan._args[:-1] + [ctypes.byref(opts), binding._stream_handle(None)]
    return binding.LIB.pa_decode_static_workspace(*args)


def test_static_workspace_matches_pa_decode_two_calls_in_a_row():
    from paged_kv_cache_182_gb300 import binding

    cases = [
        (W.make(W.shrink("gqa_fp16", B=3, past=150, past_hi=900), seed=31), 0),
        (W.make(W.shrink("ragged_fp16", B=7, past=20, past_hi=2500), seed=32), 5),
    ]
    for w, P in cases:
        dev = w.to("cuda")
        ref = binding.Plan(*dev.tensors(), scale=w.spec.scale, causal=w.spec.causal,
                           partitions=P, out_dtype=torch.float32)
        ref.run()
        out = torch.full_like(ref.out, float("nan"))
        plan = binding.Plan(*dev.tensors(), scale=w.spec.scale, causal=w.spec.causal,
                            partitions=P, out=out, out_dtype=torch.float32,
                            workspace=torch.empty(0, dtype=torch.uint8, device="cuda"))
        before = binding.kernel_launches()
        assert static_call(plan) == 0
        torch.cuda.synchronize()
        assert binding.kernel_launches() - before == 2  # partition + separate merge kernel
        assert torch.isfinite(out).all()
        diff = (out - ref.out).abs().max().item()
        assert diff <= pu.TOL[w.spec.dtype], f"{w.spec.name}: static vs pa_decode {diff}"


def test_static_workspace_rejects_oversized_requests():
    from paged_kv_cache_182_gb300 import binding

    # 4096 sequences, 64 query rows per KV head, 8 partitions: far beyond 16 MiB
    need = binding.workspace_bytes(4096, 64, 8, 128, 4, 8)
    assert need > (16 << 20)
    fake = [ctypes.c_void_p(0x10000 * (i + 1)) for i in range(8)]
    opts = binding.PaOpts(batch=4096, max_blocks=4, num_blocks=8, dtype=binding.PA_F16,
                          out_dtype=-1, partitions=8, checked=0, workspace=None,
                          workspace_bytes=0, status=None, trace_begin=None, trace_split=None)
    before = binding.kernel_launches()
    rc = binding.LIB.pa_decode_static_workspace(*fake, ctypes.c_float(0.1), 64, 8, 128, 16, 4, 1,
                                                ctypes.byref(opts), None)
    assert rc == PA_ERR_STATIC_LIMIT
    assert "PA_STATIC_WORKSPACE_BYTES" in binding.strerror(rc)
    assert binding.kernel_launches() == before
