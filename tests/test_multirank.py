"""Multi-rank host logic of bench.py on CPU (gloo, two ranks): each rank runs
its own batch (weak scaling, no collective on the data path); the reported
throughput is all ranks' bytes over the slowest rank's time."""
import os
import socket
import sys
from pathlib import Path

import pytest
import torch
import torch.multiprocessing as mp

ROOT = Path(__file__).resolve().parents[1]


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank: int, world: int, port: int, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), WORLD_SIZE=str(world),
                      RANK=str(rank), LOCAL_RANK=str(rank))
    sys.path.insert(0, str(ROOT))
    import bench
    from paged_kv_cache_182_gb300 import workloads as W

    r, wsz, _ = bench.dist_setup(world)
    assert (r, wsz) == (rank, world)
    spec = W.shrink("gqa_fp16", B=3, past=150, past_hi=900)
    w = W.make(spec, seed=r)  # each rank draws its own batch
    rank_bytes = W.algorithmic_bytes(w)
    rank_ms = 1.0 + r  # rank 1 is the slower one
    value, ms_max, total = bench.aggregate(rank_bytes, rank_ms, wsz)
    bench.barrier(wsz)
    out.put((r, rank_bytes, w.seq_lens.tolist(), value, ms_max, total))
    import torch.distributed as dist

    dist.destroy_process_group()


@pytest.mark.timeout(120)
@pytest.mark.skipif(torch.cuda.is_available(), reason="the CPU (gloo) form of the multi-rank path")
def test_two_ranks_weak_scaling_aggregate():
    ctx = mp.get_context("spawn")
    out = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, out)) for r in range(2)]
    for p in procs:
        p.start()
    res = [out.get(timeout=100) for _ in range(2)]
    for p in procs:
        p.join(timeout=30)
        assert p.exitcode == 0
    res.sort()
    (_, b0, lens0, v0, m0, t0), (_, b1, lens1, v1, m1, t1) = res
    assert lens0 != lens1, "ranks must run independent batches"
    # every rank reports the same aggregate: both ranks' bytes over the slowest time
    assert m0 == m1 == 2.0
    assert t0 == t1 == b0 + b1
    expect = (b0 + b1) / (2.0e-3) / 1e9
    assert v0 == pytest.approx(expect) and v1 == pytest.approx(expect)


def test_single_rank_aggregate_is_plain_throughput():
    sys.path.insert(0, str(ROOT))
    import bench

    value, ms, total = bench.aggregate(1_000_000, 0.5, 1)
    assert (ms, total) == (0.5, 1_000_000)
    assert value == pytest.approx(1_000_000 / 0.5e-3 / 1e9)
