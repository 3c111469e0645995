"""Pins of the float64 attention-backward oracle to things other than itself.

Each pin takes the oracle module (the real one, or a mutant of its source)
and raises AssertionError when the module disagrees with:

  - torch float64 autograd of scaled_dot_product_attention (plain, causal
    with sq < sk and sq > sk, boolean mask, broadcast additive mask, GQA);
  - central finite differences of a forward written here as loops over the
    definition of attention (tiny shapes);
  - the single-key closed form, where p = 1 and the backward reduces to
    dq = scale (g.(v - y)) k, dk = scale sum (g.(v - y)) q, dv = sum g
    (this also fixes that delta uses the supplied y);
  - the grouped-query identity: hk < hq equals hk = hq with each key/value
    head repeated, dk and dv summed over the repeats;
  - the mask rules of onnxruntime-ep-mlx 0.31.1, src/ops/attention_vjp/
    dense.rs, fn execute: a narrow mask equals its explicit form padded with
    masked keys, a width-1 mask broadcasts over keys (an additive row
    constant changes nothing), and a row with no visible key has p = 0, so
    its dq is zero and it adds nothing to dk and dv.
"""
from __future__ import annotations

import math

import numpy as np
import torch


def _rand(rng, *shape):
    return rng.standard_normal(shape)


def _case(seed, b, hq, hk, sq, sk, d):
    rng = np.random.default_rng(seed)
    return (rng, _rand(rng, b, hq, sq, d), _rand(rng, b, hk, sk, d), _rand(rng, b, hk, sk, d),
            _rand(rng, b, hq, sq, d))


def _torch_vjp(q, k, v, g, scale, causal=False, attn_mask=None):
    """dq, dk, dv and the forward output from torch's own float64 autograd."""
    tq, tk, tv = (torch.tensor(x, dtype=torch.float64, requires_grad=True) for x in (q, k, v))
    mask = None if attn_mask is None else torch.tensor(attn_mask)
    out = torch.nn.functional.scaled_dot_product_attention(
        tq, tk, tv, attn_mask=mask, is_causal=causal, scale=scale,
        enable_gqa=q.shape[1] != k.shape[1])
    out.backward(torch.tensor(g, dtype=torch.float64))
    return (tq.grad.numpy(), tk.grad.numpy(), tv.grad.numpy(), out.detach().numpy())


def _close(got, want, tol, what):
    for name, a, w in zip(("dq", "dk", "dv"), got, want):
        err = float(np.max(np.abs(np.asarray(a) - np.asarray(w)))) if np.size(w) else 0.0
        assert np.all(np.isfinite(a)), f"{what}: {name} not finite"
        assert err <= tol, f"{what}: {name} max err {err:.3e} > {tol:.1e}"


def _against_torch(m, seed, b, hq, hk, sq, sk, d, scale, causal=False, mask=None,
                   mask_kind=0, torch_mask=None, what=""):
    _, q, k, v, g = _case(seed, b, hq, hk, sq, sk, d)
    dq, dk, dv, y = _torch_vjp(q, k, v, g, scale, causal, torch_mask)
    got = m.attention_vjp(q, k, v, y, g, scale, causal, mask, mask_kind)
    _close(got, (dq, dk, dv), 1e-10, what)


def pin_torch_plain(m):
    _against_torch(m, 1, 2, 4, 2, 5, 7, 6, 0.37, what="plain gqa")


def pin_torch_causal_wide(m):
    _against_torch(m, 2, 1, 3, 1, 5, 9, 4, 0.5, causal=True, what="causal sq<sk")


def pin_torch_causal_tall(m):
    _against_torch(m, 3, 2, 2, 2, 9, 5, 4, 0.25, causal=True, what="causal sq>sk")


def pin_torch_bool_mask(m):
    rng = np.random.default_rng(4)
    b, hq, hk, sq, sk, d = 2, 4, 1, 6, 8, 5
    keep = rng.random((b, 1, sq, sk)) < 0.6
    keep[..., 0] = True  # no empty rows: torch gives NaN for those
    _against_torch(m, 5, b, hq, hk, sq, sk, d, 0.3, mask=keep.astype(np.uint8), mask_kind=1,
                   torch_mask=keep, what="boolean mask")


def pin_torch_additive_mask(m):
    rng = np.random.default_rng(6)
    b, hq, hk, sq, sk, d = 1, 4, 2, 5, 6, 3
    bias = rng.standard_normal((1, hq, 1, sk)) * 2.0
    _against_torch(m, 7, b, hq, hk, sq, sk, d, 0.7, mask=bias, mask_kind=2, torch_mask=bias,
                   what="additive broadcast mask")


def _loop_forward(q, k, v, scale, causal, bias):
    """Attention by its definition, one (b, h, i) at a time: softmax over visible keys."""
    b, hq, sq, d = q.shape
    hk, sk = k.shape[1], k.shape[2]
    y = np.zeros_like(q)
    for bb in range(b):
        for h in range(hq):
            kh = h // (hq // hk)
            for i in range(sq):
                s = []
                for j in range(sk):
                    if causal and j > i:
                        s.append(-math.inf)
                        continue
                    s.append(scale * sum(q[bb, h, i, t] * k[bb, kh, j, t] for t in range(d))
                             + bias[i][j])
                top = max(s)
                if top == -math.inf:
                    continue
                w = [math.exp(x - top) for x in s]
                tot = sum(w)
                for t in range(d):
                    y[bb, h, i, t] = sum(w[j] * v[bb, kh, j, t] for j in range(sk)) / tot
    return y


def pin_finite_differences(m):
    rng, q, k, v, g = _case(8, 1, 2, 1, 3, 4, 3)
    scale = 0.6
    bias = rng.standard_normal((3, 4))
    bias[2, 1] = -math.inf

    def loss(q_, k_, v_):
        return float(np.sum(g * _loop_forward(q_, k_, v_, scale, True, bias)))

    y = _loop_forward(q, k, v, scale, True, bias)
    got = m.attention_vjp(q, k, v, y, g, scale, True, bias.reshape(1, 1, 3, 4), 2)
    want = []
    h = 1e-5
    for x, idx in ((q, 0), (k, 1), (v, 2)):
        grad = np.zeros_like(x)
        for pos in np.ndindex(x.shape):
            args = [q.copy(), k.copy(), v.copy()]
            args[idx][pos] += h
            up = loss(*args)
            args[idx][pos] -= 2 * h
            down = loss(*args)
            grad[pos] = (up - down) / (2 * h)
        want.append(grad)
    _close(got, want, 1e-7, "finite differences")


def pin_single_key(m):
    rng, q, k, v, g = _case(9, 2, 4, 2, 3, 1, 5)
    y = _rand(rng, 2, 4, 3, 5)  # any y: delta must use it as given
    scale = 0.45
    groups = 2
    kr = np.repeat(k, groups, axis=1)
    vr = np.repeat(v, groups, axis=1)
    c = np.sum(g * (vr - y), axis=-1, keepdims=True)  # g.(v - y) per row
    dq = scale * c * kr
    dk = (scale * c * q).reshape(2, 2, groups, 3, 5).sum(axis=(2, 3)).reshape(2, 2, 1, 5)
    dv = g.reshape(2, 2, groups, 3, 5).sum(axis=(2, 3)).reshape(2, 2, 1, 5)
    got = m.attention_vjp(q, k, v, y, g, scale)
    _close(got, (dq, dk, dv), 1e-12, "single key")


def pin_gqa_repeat(m):
    rng, q, k, v, g = _case(10, 2, 6, 2, 4, 5, 3)
    y = _rand(rng, 2, 6, 4, 3)
    got = m.attention_vjp(q, k, v, y, g, 0.5, True)
    dq, dk6, dv6 = m.attention_vjp(q, np.repeat(k, 3, axis=1), np.repeat(v, 3, axis=1), y, g,
                                   0.5, True)
    want = (dq, dk6.reshape(2, 2, 3, 5, 3).sum(axis=2), dv6.reshape(2, 2, 3, 5, 3).sum(axis=2))
    _close(got, want, 1e-12, "gqa repeat")


def pin_padded_mask(m):
    rng, q, k, v, g = _case(11, 1, 2, 2, 4, 7, 3)
    y = _rand(rng, 1, 2, 4, 3)
    keep = rng.random((1, 2, 4, 4)) < 0.7
    keep[..., 0] = True
    full = np.zeros((1, 2, 4, 7), dtype=bool)
    full[..., :4] = keep
    got = m.attention_vjp(q, k, v, y, g, 0.4, False, keep.astype(np.uint8), 1)
    want = m.attention_vjp(q, k, v, y, g, 0.4, False, full.astype(np.uint8), 1)
    _close(got, want, 0.0, "boolean mask padded")
    bias = rng.standard_normal((1, 1, 4, 3))
    wide = np.full((1, 1, 4, 7), -np.inf)
    wide[..., :3] = bias
    got = m.attention_vjp(q, k, v, y, g, 0.4, False, bias, 2)
    want = m.attention_vjp(q, k, v, y, g, 0.4, False, wide, 2)
    _close(got, want, 0.0, "additive mask padded")


def pin_width_one(m):
    rng, q, k, v, g = _case(12, 1, 2, 1, 5, 6, 4)
    y = _rand(rng, 1, 2, 5, 4)
    plain = m.attention_vjp(q, k, v, y, g, 0.8)
    shift = rng.standard_normal((1, 2, 5, 1)) * 3.0
    _close(m.attention_vjp(q, k, v, y, g, 0.8, False, shift, 2), plain, 1e-12,
           "width-1 additive row constant")
    keep = np.ones((1, 1, 5, 1), dtype=np.uint8)
    _close(m.attention_vjp(q, k, v, y, g, 0.8, False, keep, 1), plain, 0.0,
           "width-1 boolean mask set everywhere")


def pin_empty_rows(m):
    rng, q, k, v, g = _case(13, 1, 2, 1, 4, 5, 3)
    y = _rand(rng, 1, 2, 4, 3)
    keep = np.ones((1, 2, 4, 5), dtype=np.uint8)
    keep[0, 1, 2, :] = 0  # head 1, row 2 sees no key
    dq, dk, dv = m.attention_vjp(q, k, v, y, g, 0.5, False, keep, 1)
    assert np.all(dq[0, 1, 2] == 0.0), "empty row: dq not zero"
    g0 = g.copy()
    g0[0, 1, 2] = 0.0
    _, dk0, dv0 = m.attention_vjp(q, k, v, y, g0, 0.5)
    _close((dq[0, 1, 2], dk, dv), (np.zeros(3), dk0, dv0), 1e-12, "empty row contributes nothing")
    # a width-1 boolean mask that is clear on a row empties that row
    row = np.ones((1, 1, 4, 1), dtype=np.uint8)
    row[0, 0, 0, 0] = 0
    dq1, _, _ = m.attention_vjp(q, k, v, y, g, 0.5, False, row, 1)
    assert np.all(dq1[:, :, 0] == 0.0), "width-1 clear row: dq not zero"


PINS = [
    pin_torch_plain, pin_torch_causal_wide, pin_torch_causal_tall, pin_torch_bool_mask,
    pin_torch_additive_mask, pin_finite_differences, pin_single_key, pin_gqa_repeat,
    pin_padded_mask, pin_width_one, pin_empty_rows,
]


def run_all(m) -> list[str]:
    failed = []
    for pin in PINS:
        try:
            pin(m)
        except Exception as exc:  # a mutant may also raise: that counts as failing the pin
            failed.append(f"{pin.__name__}: {exc}")
    return failed
