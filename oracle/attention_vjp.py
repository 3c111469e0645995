"""float64 CPU oracle for the dense attention backward (VJP) -- TEST INFRASTRUCTURE ONLY.

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this module.  The CUDA library never calls it and
shares no code with it.

What it computes follows onnxruntime-ep-mlx 0.31.1,
src/ops/attention_vjp/dense.rs, fn execute, step by step in that page's
order and notation, with numpy matmul as the only library primitive:

  inputs  q, y, g : [b, hq, sq, d]     k, v : [b, hk, sk, d]
          (y is the forward output, g the gradient arriving at it)
  groups  = hq / hk;  q and g viewed as [b, hk, groups, sq, d], k and v as
          [b, hk, 1, sk, d], so query head h reads key/value head h // groups
  root    = sqrt(scale);  qs = q * root;  ks = k * root
  scores  = qs @ ks^T                      -> [b, hq, sq, sk]
  mask    kind 1 (boolean): bias = 0 where the mask is set, -inf elsewhere;
          kind 2 (additive): bias = the mask itself.  A bias whose last
          extent (its width) is neither 1 nor sk is padded with -inf on the
          right up to sk; scores += bias (numpy broadcasting)
  causal  score (qi, ki) kept where ki <= qi, -inf elsewhere
  maximum = max over keys;  empty = (maximum == -inf)
  p       = softmax(where(empty, 0, scores)), then 0 on empty rows
  dv      = sum over groups of p^T @ g
  dp      = g @ v^T
  delta   = sum over d of y * g           (the supplied y, not a recomputed one)
  ds      = p * (dp - delta)
  dq      = (ds @ ks) * root               -> [b, hq, sq, d]
  dk      = sum over groups of (ds^T @ qs) * root

Readings of points the page leaves open:
  - All arithmetic is float64 on the input values (the page computes in the
    input's own type); the oracle is the exact result up to rounding order.
  - A boolean mask is "set" where it is nonzero; an additive mask is taken
    as given (float).  A mask whose width exceeds sk is an error here (the
    page's addition would fail to broadcast).
  - scale must be positive: the page takes its square root.
  - The maximum over no keys (sk = 0) is -inf, so such rows are empty.

Pins (tests/test_oracle_vjp.py): torch float64 autograd of
scaled_dot_product_attention, central finite differences of a loop-written
forward on tiny shapes, the single-key closed form (which also fixes the
role of y), the grouped-query identity against repeated heads, the padded
mask against its explicit full-width form, and empty rows.  Mutants of this
source must fail a pin.
"""
from __future__ import annotations

import numpy as np


def _bias(mask: np.ndarray, mask_kind: int, sk: int) -> np.ndarray:
    """The additive bias the mask stands for, padded with -inf up to sk keys."""
    if mask_kind == 1:
        bias = np.where(np.asarray(mask) != 0, 0.0, -np.inf)
    elif mask_kind == 2:
        bias = np.asarray(mask, dtype=np.float64)
    else:
        raise ValueError(f"mask_kind {mask_kind}")
    width = bias.shape[-1]
    if width > sk:
        raise ValueError(f"mask width {width} exceeds sk {sk}")
    if width != 1 and width < sk:
        pad = [(0, 0)] * (bias.ndim - 1) + [(0, sk - width)]
        bias = np.pad(bias, pad, mode="constant", constant_values=-np.inf)
    return bias


def probabilities(q, k, scale: float, causal: bool = False, mask=None, mask_kind: int = 0):
    """p [b, hq, sq, sk] of the page's forward recompute, empty rows zero."""
    q = np.asarray(q, dtype=np.float64)
    k = np.asarray(k, dtype=np.float64)
    b, hq, sq, d = q.shape
    hk, sk = k.shape[1], k.shape[2]
    if hq % hk:
        raise ValueError("hq must be a multiple of hk")
    if not scale > 0:
        raise ValueError("scale must be positive")
    groups = hq // hk
    root = np.sqrt(np.float64(scale))
    qs = q.reshape(b, hk, groups, sq, d) * root
    ks = k.reshape(b, hk, 1, sk, d) * root
    scores = np.matmul(qs, np.swapaxes(ks, -1, -2)).reshape(b, hq, sq, sk)
    if mask_kind:
        scores = scores + _bias(mask, mask_kind, sk)
    if causal:
        qi = np.arange(sq).reshape(sq, 1)
        ki = np.arange(sk)
        scores = np.where(ki <= qi, scores, -np.inf)
    maximum = np.max(scores, axis=-1, keepdims=True, initial=-np.inf)
    empty = maximum == -np.inf
    safe = np.where(empty, 0.0, scores)
    shifted = np.exp(safe - np.max(safe, axis=-1, keepdims=True, initial=-np.inf))
    probability = shifted / np.sum(shifted, axis=-1, keepdims=True)
    return np.where(empty, 0.0, probability)


def forward(q, k, v, scale: float, causal: bool = False, mask=None, mask_kind: int = 0):
    """y = p @ v with the same p the backward recomputes (rows with no key give 0)."""
    p = probabilities(q, k, scale, causal, mask, mask_kind)
    b, hq, sq, sk = p.shape
    v = np.asarray(v, dtype=np.float64)
    hk, d = v.shape[1], v.shape[3]
    groups = hq // hk
    y = np.matmul(p.reshape(b, hk, groups, sq, sk), v.reshape(b, hk, 1, sk, d))
    return y.reshape(b, hq, sq, d)


def attention_vjp(q, k, v, y, g, scale: float, causal: bool = False, mask=None,
                  mask_kind: int = 0):
    """(dq, dk, dv) in float64: dq [b, hq, sq, d], dk and dv [b, hk, sk, d]."""
    q = np.asarray(q, dtype=np.float64)
    k = np.asarray(k, dtype=np.float64)
    v = np.asarray(v, dtype=np.float64)
    y = np.asarray(y, dtype=np.float64)
    g = np.asarray(g, dtype=np.float64)
    b, hq, sq, d = q.shape
    hk, sk = k.shape[1], k.shape[2]
    groups = hq // hk
    root = np.sqrt(np.float64(scale))
    qs = q.reshape(b, hk, groups, sq, d) * root
    ks = k.reshape(b, hk, 1, sk, d) * root
    g5 = g.reshape(b, hk, groups, sq, d)
    v5 = v.reshape(b, hk, 1, sk, d)
    p = probabilities(q, k, scale, causal, mask, mask_kind).reshape(b, hk, groups, sq, sk)
    pt = np.swapaxes(p, -1, -2)
    dv = np.sum(np.matmul(pt, g5), axis=2)
    dp = np.matmul(g5, np.swapaxes(v5, -1, -2))
    delta = np.sum(y.reshape(b, hk, groups, sq, d) * g5, axis=-1, keepdims=True)
    ds = p * (dp - delta)
    dq = (np.matmul(ds, ks) * root).reshape(b, hq, sq, d)
    dk = np.sum(np.matmul(np.swapaxes(ds, -1, -2), qs) * root, axis=2)
    return dq, dk, dv
