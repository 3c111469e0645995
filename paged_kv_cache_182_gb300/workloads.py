"""Seeded synthetic inputs for paged decode attention.

This module only draws random tensors and lays them out; it holds none of
the attention arithmetic.  Both the CUDA path (tests, bench) and the float64
oracle (tests) take their inputs from here, so neither side depends on the
other.

The five named workloads follow the decode shapes the paged-attention page
describes (onnxruntime-ep-mlx 0.31.1, src/ops/paged_attention.rs, fn vector:
query [H, NQ, D], a block table per sequence, caches of fixed-size blocks,
NQ new rows with an optional causal mask):

  tiny_fp32          B=1  H=4  KV=2 D=64  BLOCK=16 past=100 (7 of a 16-block pool) fp32
  gqa_fp16           B=8  H=32 KV=8 D=128 BLOCK=16 past ~ U{512..4096}            fp16
  long_bf16          B=1  H=32 KV=8 D=128 BLOCK=16 past=32768, 32 partitions, q*2   bf16
  causal_append_fp16 B=16 H=64 KV=8 D=128 BLOCK=32 past=2048, NQ=4 causal          fp16
  ragged_fp16        B=64 H=32 KV=4 D=64  BLOCK=32 past log-uniform [64,16384],
                     1% of K/V entries scaled by 20                                 fp16

Recipe: a CPU ``torch.Generator`` seeded with ``seed`` draws, in this order,
the past lengths, the block permutation, q, K cache, V cache, k_new, v_new
and the outlier masks; values are N(0,1) in float32, multiplied as the
workload says, then cast to the workload dtype.  Physical blocks are a random
permutation of the pool, so logically adjacent blocks are scattered.  With
``poison=True`` every pool block no table references and every cache slot past
a sequence's length is set to NaN, so a stray read of either shows up as NaN
in the output.  Table entries past a sequence's last block are -1.

Prefill workloads (``PREFILL_SPECS``, ``make_prefill``) draw the same way with
the table covering past + NQ tokens per sequence: the blocks of the NQ new
tokens are allocated and their slots poisoned (NaN) until the prefill stores
the new rows there.

  prefill_fp16       B=4  H=32 KV=8 D=128 BLOCK=16 past=1024, NQ=512 causal       fp16
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field, replace

import torch

DTYPES = {"f32": torch.float32, "f16": torch.float16, "bf16": torch.bfloat16}


@dataclass(frozen=True)
class Spec:
    name: str
    dtype: str  # "f32" | "f16" | "bf16"
    B: int
    H: int
    KV: int
    D: int
    BLOCK: int
    NQ: int = 1
    causal: bool = False
    lens: str = "fixed"  # "fixed" | "uniform" | "loguniform"
    past: int = 0  # fixed length, or lower bound
    past_hi: int = 0  # upper bound for "uniform" / "loguniform"
    pool_blocks: int = 0  # 0: exactly the blocks referenced; else total pool size
    partitions: int = 0  # 0 = automatic split, 1 = single pass, P = fixed P
    q_mult: float = 1.0
    outlier_frac: float = 0.0
    outlier_mult: float = 1.0
    extra_table_cols: int = 0  # unused (-1) table columns past the longest sequence

    @property
    def group(self) -> int:
        return self.H // self.KV

    @property
    def scale(self) -> float:
        # 1/sqrt(D) rounded to float32, as the attention call receives it
        return float(torch.tensor(1.0 / math.sqrt(self.D), dtype=torch.float32))

    @property
    def elem_bytes(self) -> int:
        return torch.tensor([], dtype=DTYPES[self.dtype]).element_size()


SPECS = {
    "tiny_fp32": Spec("tiny_fp32", "f32", B=1, H=4, KV=2, D=64, BLOCK=16, past=100,
                      pool_blocks=16),
    "gqa_fp16": Spec("gqa_fp16", "f16", B=8, H=32, KV=8, D=128, BLOCK=16, lens="uniform",
                     past=512, past_hi=4096),
    "long_bf16": Spec("long_bf16", "bf16", B=1, H=32, KV=8, D=128, BLOCK=16, past=32768,
                      partitions=32, q_mult=2.0),
    "causal_append_fp16": Spec("causal_append_fp16", "f16", B=16, H=64, KV=8, D=128,
                               BLOCK=32, past=2048, NQ=4, causal=True),
    "ragged_fp16": Spec("ragged_fp16", "f16", B=64, H=32, KV=4, D=64, BLOCK=32,
                        lens="loguniform", past=64, past_hi=16384, outlier_frac=0.01,
                        outlier_mult=20.0),
}

ORDER = ["tiny_fp32", "gqa_fp16", "long_bf16", "causal_append_fp16", "ragged_fp16"]

PREFILL_SPECS = {
    "prefill_fp16": Spec("prefill_fp16", "f16", B=4, H=32, KV=8, D=128, BLOCK=16, past=1024,
                         NQ=512, causal=True),
}


@dataclass
class Workload:
    spec: Spec
    seq_lens: torch.Tensor  # [B] int32 cached tokens per sequence
    block_table: torch.Tensor  # [B, MAXB] int32, -1 past the last block
    q: torch.Tensor  # [B, H, NQ, D]
    k_cache: torch.Tensor  # [NB, BLOCK, KV, D]
    v_cache: torch.Tensor
    k_new: torch.Tensor  # [B, KV, NQ, D]
    v_new: torch.Tensor
    seed: int = 0
    meta: dict = field(default_factory=dict)

    @property
    def num_blocks(self) -> int:
        return int(self.k_cache.shape[0])

    @property
    def max_blocks(self) -> int:
        return int(self.block_table.shape[1])

    def tensors(self):
        return (self.q, self.k_cache, self.v_cache, self.block_table, self.seq_lens,
                self.k_new, self.v_new)

    def to(self, device) -> "Workload":
        moved = [t.to(device) for t in self.tensors()]
        return Workload(self.spec, moved[4], moved[3], moved[0], moved[1], moved[2], moved[5],
                        moved[6], self.seed, dict(self.meta))

    def kv_tokens(self) -> int:
        """Keys read per step summed over sequences (cached + new rows)."""
        return int(self.seq_lens.to(torch.int64).sum()) + self.spec.B * self.spec.NQ


def _draw_lens(spec: Spec, g: torch.Generator) -> torch.Tensor:
    if spec.lens == "fixed":
        return torch.full((spec.B,), spec.past, dtype=torch.int32)
    if spec.lens == "uniform":
        return torch.randint(spec.past, spec.past_hi + 1, (spec.B,), generator=g,
                             dtype=torch.int64).to(torch.int32)
    if spec.lens == "loguniform":
        u = torch.rand(spec.B, generator=g, dtype=torch.float64)
        lo, hi = math.log(spec.past), math.log(spec.past_hi)
        return torch.exp(lo + (hi - lo) * u).round().to(torch.int32)
    raise ValueError(f"unknown length law {spec.lens!r}")


def _randn(shape, g, mult, dtype, outlier_frac=0.0, outlier_mult=1.0):
    x = torch.randn(shape, generator=g, dtype=torch.float32)
    if mult != 1.0:
        x = x * mult
    if outlier_frac > 0.0:
        hit = torch.rand(shape, generator=g, dtype=torch.float32) < outlier_frac
        x = torch.where(hit, x * outlier_mult, x)
    return x.to(dtype)


def make(spec: Spec | str, seed: int = 0, poison: bool = True, lens=None) -> Workload:
    """Generate one workload on the CPU.  ``lens`` overrides the drawn lengths."""
    if isinstance(spec, str):
        spec = SPECS[spec]
    if spec.H % spec.KV != 0:
        raise ValueError("H must be a multiple of KV")
    g = torch.Generator().manual_seed(int(seed))
    seq_lens = _draw_lens(spec, g)
    if lens is not None:
        seq_lens = torch.as_tensor(lens, dtype=torch.int32).reshape(spec.B)
    nblk = [(int(n) + spec.BLOCK - 1) // spec.BLOCK for n in seq_lens.tolist()]
    used = sum(nblk)
    pool = max(spec.pool_blocks, used, 1)  # the pool is never empty
    perm = torch.randperm(pool, generator=g).to(torch.int32)
    maxb = max(nblk + [1]) + spec.extra_table_cols
    table = torch.full((spec.B, maxb), -1, dtype=torch.int32)
    at = 0
    for b, n in enumerate(nblk):
        table[b, :n] = perm[at:at + n]
        at += n
    dt = DTYPES[spec.dtype]
    q = _randn((spec.B, spec.H, spec.NQ, spec.D), g, spec.q_mult, dt)
    shape = (pool, spec.BLOCK, spec.KV, spec.D)
    k_cache = _randn(shape, g, 1.0, dt, spec.outlier_frac, spec.outlier_mult)
    v_cache = _randn(shape, g, 1.0, dt, spec.outlier_frac, spec.outlier_mult)
    nshape = (spec.B, spec.KV, spec.NQ, spec.D)
    k_new = _randn(nshape, g, 1.0, dt, spec.outlier_frac, spec.outlier_mult)
    v_new = _randn(nshape, g, 1.0, dt, spec.outlier_frac, spec.outlier_mult)
    if poison:
        referenced = torch.zeros(pool, dtype=torch.bool)
        referenced[perm[:used].long()] = True
        nan = float("nan")
        k_cache[~referenced] = nan
        v_cache[~referenced] = nan
        for b, n in enumerate(seq_lens.tolist()):
            tail = n % spec.BLOCK
            if tail:
                last = int(table[b, nblk[b] - 1])
                k_cache[last, tail:] = nan
                v_cache[last, tail:] = nan
    return Workload(spec, seq_lens, table, q, k_cache, v_cache, k_new, v_new, seed,
                    {"pool_blocks": pool, "used_blocks": used})


def shrink(spec: Spec | str, *, past: int | None = None, past_hi: int | None = None,
           B: int | None = None, **kw) -> Spec:
    """A smaller copy of a named workload (same dtype, heads, D, BLOCK, NQ, laws)."""
    if isinstance(spec, str):
        spec = SPECS[spec]
    upd = dict(kw)
    if past is not None:
        upd["past"] = past
    if past_hi is not None:
        upd["past_hi"] = past_hi
    if B is not None:
        upd["B"] = B
    return replace(spec, name=spec.name + "_small", **upd)


def algorithmic_bytes(w: Workload, out_elem_bytes: int | None = None) -> int:
    """Bytes a decode step must move at minimum: every visible K and V row once,
    q, the output, the table entries in use, and the lengths.  The split-K
    workspace is not counted (it is an implementation choice)."""
    s = w.spec
    e = s.elem_bytes
    oe = e if out_elem_bytes is None else out_elem_bytes
    lens = w.seq_lens.to(torch.int64)
    kv = 2 * (int(lens.sum()) + s.B * s.NQ) * s.KV * s.D * e
    qo = s.B * s.H * s.NQ * s.D * (e + oe)
    table = 4 * int(((lens + s.BLOCK - 1) // s.BLOCK).sum())
    return kv + qo + table + 4 * s.B


def make_prefill(spec: Spec | str, seed: int = 0, lens=None) -> Workload:
    """A prefill workload: ``seq_lens`` are the cached tokens, and the block
    table also holds the blocks of the NQ new tokens of every sequence, whose
    cache slots are NaN (the prefill writes them)."""
    if isinstance(spec, str):
        spec = PREFILL_SPECS[spec]
    past = _draw_lens(spec, torch.Generator().manual_seed(int(seed)))
    if lens is not None:
        past = torch.as_tensor(lens, dtype=torch.int32).reshape(spec.B)
    w = make(spec, seed, poison=True, lens=(past + spec.NQ).tolist())
    nan = float("nan")
    for b, n in enumerate(past.tolist()):
        for t in range(n, n + spec.NQ):
            phys = int(w.block_table[b, t // spec.BLOCK])
            w.k_cache[phys, t % spec.BLOCK] = nan
            w.v_cache[phys, t % spec.BLOCK] = nan
    w.seq_lens = past.clone()
    w.meta["prefill"] = True
    return w


# ---------------------------------------------------------------------------
# Dense attention backward (VJP) inputs.
#
# Shapes follow onnxruntime-ep-mlx 0.31.1, src/ops/attention_vjp/dense.rs,
# fn execute: q, y, g [B, HQ, SQ, D]; k, v [B, HK, SK, D]; an optional mask
# of dims [MB, MH, MQ, W] that broadcasts against the scores [B, HQ, SQ, SK]
# (MB in {1, B}, MH in {1, HQ}, MQ in {1, SQ}, W in {1..SK}).
#
# Recipe: a CPU torch.Generator seeded with ``seed`` draws q, k, v, y, g as
# N(0,1) float32 (y scaled by 1/4, the size of a softmax average of unit
# values), cast to the dtype; then the mask: boolean = Bernoulli(keep) as
# uint8, additive = N(0,1) float32 with -inf where a Bernoulli(1 - keep) hits.
# Tests that want y to be the true forward output compute it themselves.
# ---------------------------------------------------------------------------


@dataclass(frozen=True)
class VjpSpec:
    name: str
    dtype: str  # "f32" | "f16" | "bf16"
    B: int
    HQ: int
    HK: int
    SQ: int
    SK: int
    D: int
    causal: bool = False
    mask_kind: int = 0  # 0 none, 1 boolean (uint8), 2 additive (float32)
    mask_dims: tuple = (1, 1, 1, 1)
    keep: float = 0.9

    @property
    def elem_bytes(self) -> int:
        return 4 if self.dtype == "f32" else 2


VJP_SPECS = {
    # Llama-style grouped-query training shape: 4 sequences of 2048 tokens,
    # 32 query heads on 8 key/value heads, causal.
    "vjp_bf16": VjpSpec("vjp_bf16", "bf16", B=4, HQ=32, HK=8, SQ=2048, SK=2048, D=128,
                        causal=True),
}


@dataclass
class VjpInputs:
    spec: VjpSpec
    q: torch.Tensor
    k: torch.Tensor
    v: torch.Tensor
    y: torch.Tensor
    g: torch.Tensor
    mask: torch.Tensor | None
    seed: int = 0

    def tensors(self):
        return (self.q, self.k, self.v, self.y, self.g, self.mask)

    def to(self, device) -> "VjpInputs":
        moved = [None if t is None else t.to(device) for t in self.tensors()]
        return VjpInputs(self.spec, *moved, seed=self.seed)


def make_vjp(spec: VjpSpec | str, seed: int = 0) -> VjpInputs:
    if isinstance(spec, str):
        spec = VJP_SPECS[spec]
    if spec.HQ % spec.HK != 0:
        raise ValueError("HQ must be a multiple of HK")
    g = torch.Generator().manual_seed(int(seed))
    dt = DTYPES[spec.dtype]
    q = _randn((spec.B, spec.HQ, spec.SQ, spec.D), g, 1.0, dt)
    k = _randn((spec.B, spec.HK, spec.SK, spec.D), g, 1.0, dt)
    v = _randn((spec.B, spec.HK, spec.SK, spec.D), g, 1.0, dt)
    y = _randn((spec.B, spec.HQ, spec.SQ, spec.D), g, 0.25, dt)
    grad = _randn((spec.B, spec.HQ, spec.SQ, spec.D), g, 1.0, dt)
    mask = None
    if spec.mask_kind == 1:
        mask = (torch.rand(spec.mask_dims, generator=g) < spec.keep).to(torch.uint8)
    elif spec.mask_kind == 2:
        mask = torch.randn(spec.mask_dims, generator=g, dtype=torch.float32)
        hit = torch.rand(spec.mask_dims, generator=g) >= spec.keep
        mask = torch.where(hit, torch.full_like(mask, float("-inf")), mask)
    return VjpInputs(spec, q, k, v, y, grad, mask, seed)


def vjp_flops(spec: VjpSpec) -> int:
    """Flops of the five products of the backward (scores, dv, dp, dq, dk),
    2 * D each per visible (query row, key) pair: with the causal mask only
    pairs ki <= qi count.  Other masks are not subtracted."""
    if spec.causal:
        n = min(spec.SQ, spec.SK)
        pairs = n * (n + 1) // 2 + max(0, spec.SQ - spec.SK) * spec.SK
    else:
        pairs = spec.SQ * spec.SK
    return 10 * spec.B * spec.HQ * spec.D * pairs
