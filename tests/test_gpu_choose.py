"""pa_choose_partitions against a launch (needs a GPU): the partial records
the partition kernel writes for the split pieces of the automatic schedule
are counted in a workspace filled with NaN beforehand, and compared with the
plan the host-side chooser makes for the same lengths on this device."""
import pytest
import torch

from paged_kv_cache_182_gb300 import workloads as W

pytestmark = pytest.mark.gpu


def align256(n):
    return (n + 255) // 256 * 256


@pytest.mark.parametrize("name", ["gqa_fp16", "long_bf16", "ragged_fp16"])
def test_choose_partitions_counts_the_records_a_launch_writes(name):
    from paged_kv_cache_182_gb300 import binding

    w = W.make(name, seed=11)
    s = w.spec
    R = s.group * s.NQ
    assert R <= 8  # one row group: the transposed kernel, row stride R
    max_len = int(w.block_table.shape[1]) * s.BLOCK
    dt = {"f16": torch.float16, "bf16": torch.bfloat16}[s.dtype]
    plan = binding.choose_partitions(w.seq_lens, max_len, s.H, s.KV, s.D, s.BLOCK, s.NQ, dt)
    dev = w.to("cuda")
    ws = binding.new_workspace(s.B, s.H, s.KV, s.D, s.NQ, 0, "cuda")
    ws.fill_(0xFF)  # NaN in every float
    ws[:binding.workspace_zero_bytes(s.B, s.H, s.KV, s.D, s.NQ, 0)] = 0
    out = binding.decode(*dev.tensors(), scale=s.scale, causal=s.causal, partitions=0,
                         workspace=ws, merge_kernel=True)
    torch.cuda.synchronize()
    # workspace: split counters [B * KV] | schedule [B] int2 | (max, sum) per record and row | ...
    ml_off = align256(s.B * s.KV * 4) + align256(s.B * 8)
    ml = ws[ml_off:].view(torch.float32)[: 2 * 2 * 1024 * R].view(2 * 1024, R, 2)
    written = int((~torch.isnan(ml[:, 0, 0])).sum())
    assert written == plan.records, (written, plan.records, plan.split_segments)
    assert plan.grid == torch.cuda.get_device_properties(0).multi_processor_count
    assert torch.isfinite(out).all()
