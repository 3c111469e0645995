"""The bounded-wait failure path of the partition kernels (needs a GPU).

A test switch makes the V-issuing warp of every CTA leave one pipeline stage
out, and a short wait limit (1 ms) makes the consumers' wait for that
stage run out.  The call must complete (every wait is bounded, nothing
traps), report PA_STATUS_TIMEOUT, and leave the context usable: after the
split counters are zeroed again, the next normal call matches the oracle.
"""
import pytest
import torch

import parity_util as pu
from paged_kv_cache_182_gb300 import workloads as W

pytestmark = pytest.mark.gpu

CASES = [
    ("gqa_fp16", dict(B=3, past=150, past_hi=900)),            # <= 8 rows: transposed kernel
    ("causal_append_fp16", dict(B=3, past=333)),               # 32 rows: 16-row tile kernel
    ("tiny_fp32", dict()),                                      # float32: CUDA-core kernel
]


@pytest.mark.parametrize("name,kw", CASES, ids=[c[0] for c in CASES])
@pytest.mark.parametrize("partitions,stage", [(0, 1), (1, 1), (1, 2)])
def test_withheld_stage_times_out_then_recovers(name, kw, partitions, stage):
    """partitions = 1 gives each CTA whole segments (several stages); the
    automatic split (0) may give a CTA a single stage, the first."""
    from paged_kv_cache_182_gb300 import binding

    w = W.make(W.shrink(name, **kw), seed=41)
    s = w.spec
    dev = w.to("cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    plan = binding.Plan(*dev.tensors(), scale=s.scale, causal=s.causal, partitions=partitions,
                        status=status, out_dtype=torch.float32)
    plan.opts.wait_limit_ns = 1_000_000
    plan.opts.debug_withhold_stage = stage
    plan.run()
    torch.cuda.synchronize()
    assert int(status.item()) & binding.PA_STATUS_TIMEOUT

    # the same plan again, switch off, counters zeroed as the header asks
    zero = binding.workspace_zero_bytes(s.B, s.H, s.KV, s.D, s.NQ, partitions)
    if zero:
        plan.workspace[:zero] = 0
    status.zero_()
    plan.opts.wait_limit_ns = 0
    plan.opts.debug_withhold_stage = 0
    got = plan.run().clone()
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    pu.check(got, pu.run_oracle(w), s.dtype, "f32", f"{name} after a timeout")
