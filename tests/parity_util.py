"""Shared helpers of the GPU parity tests: run both sides, compare, bounds.

Tolerances (stated by the benchmark spec for this path): max abs error 1e-5 for
float32 inputs and 2e-3 for float16 / bfloat16 inputs, with float32
accumulation.  With a float32 output the kernel result is compared directly.
With a 16-bit output the result is additionally rounded to that format, so
the bound grows by half a unit in the last place of the exact value.
"""
from __future__ import annotations

import numpy as np
import torch

import oracle

TOL = {"f32": 1e-5, "f16": 2e-3, "bf16": 2e-3}
MANT = {"f16": 10, "bf16": 7}  # explicit mantissa bits


def half_ulp(values: np.ndarray, fmt: str) -> np.ndarray:
    """Half a unit in the last place of `fmt` at |values| (0 for float32 outputs)."""
    if fmt == "f32":
        return np.zeros_like(values)
    mag = np.maximum(np.abs(values), 2.0 ** -14)
    e = np.floor(np.log2(mag))
    return 0.5 * 2.0 ** (e - MANT[fmt])


def run_gpu(w, *, partitions=None, out_dtype=None, stream=None, **kw):
    from paged_kv_cache_182_gb300 import binding

    dev = w.to("cuda")
    P = w.spec.partitions if partitions is None else partitions
    out = binding.decode(*dev.tensors(), scale=w.spec.scale, causal=w.spec.causal,
                         partitions=P, out_dtype=out_dtype, stream=stream, **kw)
    torch.cuda.synchronize()
    return out


def run_oracle(w, row_mask=None):
    return oracle.decode(*w.tensors(), scale=w.spec.scale, causal=w.spec.causal,
                         row_mask=row_mask)


def max_err(got: torch.Tensor, want: np.ndarray) -> float:
    g = got.detach().cpu().double().numpy()
    assert np.all(np.isfinite(g)), "non-finite GPU output (a stray read of a poisoned slot?)"
    return float(np.max(np.abs(g - want)))


def check(got: torch.Tensor, want: np.ndarray, in_fmt: str, out_fmt: str, label: str = ""):
    g = got.detach().cpu().double().numpy()
    assert np.all(np.isfinite(g)), f"{label}: non-finite GPU output"
    bound = TOL[in_fmt] + half_ulp(want, out_fmt)
    err = np.abs(g - want)
    worst = int(np.argmax(err - bound))
    assert np.all(err <= bound), (
        f"{label}: |gpu - oracle| = {err.flat[worst]:.3e} exceeds {bound.flat[worst]:.3e} "
        f"at flat index {worst} (oracle {want.flat[worst]:.6f}, gpu {g.flat[worst]:.6f}); "
        f"max abs err {err.max():.3e}")
    return float(err.max())
