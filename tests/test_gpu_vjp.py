"""Attention backward (pa_attention_vjp) against the float64 oracle.

Inputs come from the seeded generator; y is the oracle's forward output
(rounded to the input type) unless a test says otherwise.  Bounds, as
max |got - want| over a tensor, relative to max(1, max |want|):

  - float32 inputs, or 16-bit inputs on the CUDA-core kernels with float32
    outputs: 2e-5.  Inputs reach both sides exactly; the kernels accumulate
    in float32 over at most a few thousand terms (relative rounding of a
    sum of n terms grows like sqrt(n) * 2^-24 in practice).
  - 16-bit inputs on the tensor-core kernels: p and ds enter the products
    rounded to the input type (unit roundoff u = 2^-8 bf16, 2^-11 f16); the
    sums of those rounded terms are random-signed, so the error stays near
    u times the typical term, bounded here by 4u.
  - 16-bit outputs add half a unit in the last place of the output type.
"""
from __future__ import annotations

from dataclasses import replace

import numpy as np
import pytest
import torch

from oracle import attention_vjp as orc
from paged_kv_cache_182_gb300 import workloads as wl

pytestmark = pytest.mark.gpu

UNIT = {"f32": 2.0 ** -24, "f16": 2.0 ** -11, "bf16": 2.0 ** -8}


def _spec(dtype="f32", B=2, HQ=4, HK=2, SQ=37, SK=53, D=64, causal=False, mask_kind=0,
          mask_dims=(1, 1, 1, 1), keep=0.85):
    return wl.VjpSpec("t", dtype, B, HQ, HK, SQ, SK, D, causal, mask_kind, tuple(mask_dims), keep)


def _np(t):
    return None if t is None else t.to(torch.float64).numpy() if t.dtype != torch.uint8 else t.numpy()


def _oracle(x: wl.VjpInputs, scale, y=None):
    s = x.spec
    return orc.attention_vjp(_np(x.q), _np(x.k), _np(x.v), _np(x.y) if y is None else y, _np(x.g),
                             scale, s.causal, _np(x.mask), s.mask_kind)


def _with_forward_y(x: wl.VjpInputs, scale):
    s = x.spec
    y = orc.forward(_np(x.q), _np(x.k), _np(x.v), scale, s.causal, _np(x.mask), s.mask_kind)
    x.y = torch.from_numpy(y).to(x.q.dtype)
    return x


def _run(x: wl.VjpInputs, scale, **kw):
    from paged_kv_cache_182_gb300 import binding

    d = x.to("cuda")
    out = binding.attention_vjp(d.q, d.k, d.v, d.y, d.g, d.mask, scale=scale,
                                causal=x.spec.causal, **kw)
    torch.cuda.synchronize()
    return [t.cpu() for t in out]


def _check(got, want, tol, out_fmt=None, label=""):
    for name, a, w in zip(("dq", "dk", "dv"), got, want):
        a = a.to(torch.float64).numpy()
        assert a.shape == w.shape, f"{label} {name}: shape {a.shape} != {w.shape}"
        assert np.all(np.isfinite(a)), f"{label} {name}: not finite"
        if w.size == 0:
            continue
        ref = max(1.0, float(np.max(np.abs(w))))
        bound = tol * ref
        if out_fmt in ("f16", "bf16"):
            bound += UNIT[out_fmt] * ref
        err = float(np.max(np.abs(a - w)))
        assert err <= bound, f"{label} {name}: max err {err:.3e} > {bound:.3e} (scale {ref:.2f})"


F32_TOL = 2e-5

CASES = {
    "plain": dict(),
    "gqa4_d128": dict(HQ=8, HK=2, D=128, SQ=70, SK=45),
    "mha_odd_d": dict(HQ=3, HK=3, D=40, SQ=19, SK=33),
    "causal_wide": dict(causal=True, SQ=30, SK=70),
    "causal_tall": dict(causal=True, SQ=90, SK=40),
    "bool_mask_full": dict(mask_kind=1, mask_dims=(2, 4, 37, 53)),
    "bool_mask_narrow": dict(mask_kind=1, mask_dims=(1, 1, 37, 20)),
    "add_mask_heads": dict(mask_kind=2, mask_dims=(1, 4, 1, 53)),
    "add_mask_width1": dict(mask_kind=2, mask_dims=(2, 1, 37, 1)),
    "add_mask_causal": dict(mask_kind=2, mask_dims=(2, 4, 37, 53), causal=True, keep=0.7),
}


@pytest.mark.parametrize("name", sorted(CASES))
def test_f32_cases(name):
    s = _spec(**CASES[name])
    scale = 1.0 / np.sqrt(s.D)
    x = _with_forward_y(wl.make_vjp(s, seed=3), scale)
    _check(_run(x, scale), _oracle(x, scale), F32_TOL, label=name)


@pytest.mark.parametrize("dtype", ["f16", "bf16"])
@pytest.mark.parametrize("out", ["f32", "native"])
def test_16bit_on_cuda_cores(dtype, out):
    s = _spec(dtype=dtype, HQ=8, HK=2, SQ=61, SK=75, D=128, causal=True)
    scale = 1.0 / np.sqrt(s.D)
    x = _with_forward_y(wl.make_vjp(s, seed=4), scale)
    kw = dict(kernel=1)
    if out == "f32":
        kw["out_dtype"] = torch.float32
    _check(_run(x, scale, **kw), _oracle(x, scale), F32_TOL,
           out_fmt=None if out == "f32" else dtype, label=f"{dtype}/{out}")


def test_y_is_taken_as_given():
    """delta uses the y passed in: a y that is not the forward output changes
    dq and dk exactly as the oracle says."""
    s = _spec(SQ=24, SK=31)
    x = wl.make_vjp(s, seed=5)  # y drawn at random, not the forward output
    _check(_run(x, 0.2), _oracle(x, 0.2), F32_TOL, label="random y")


def test_empty_rows_and_unseen_keys():
    s = _spec(SQ=20, SK=24, mask_kind=1, mask_dims=(2, 4, 20, 24))
    x = _with_forward_y(wl.make_vjp(s, seed=6), 0.3)
    x.mask[0, 1, 5, :] = 0      # one row with no visible key
    x.mask[1, :, :, 7] = 0      # key 7 of batch 1 hidden from every row
    x = _with_forward_y(x, 0.3)
    got = _run(x, 0.3)
    _check(got, _oracle(x, 0.3), F32_TOL, label="empty rows")
    assert torch.all(got[0][0, 1, 5] == 0)
    assert torch.all(got[1][1, :, 7] == 0) and torch.all(got[2][1, :, 7] == 0)


def test_degenerate_sizes():
    from paged_kv_cache_182_gb300 import binding

    for sq, sk in ((0, 9), (9, 0), (1, 1)):
        s = _spec(SQ=sq, SK=sk)
        x = wl.make_vjp(s, seed=7)
        d = x.to("cuda")
        out = tuple(torch.full_like(t, float("nan")) for t in (d.q, d.k, d.k))
        binding.attention_vjp(d.q, d.k, d.v, d.y, d.g, scale=0.5, out=out)
        torch.cuda.synchronize()
        _check([t.cpu() for t in out], _oracle(x, 0.5), F32_TOL, label=f"sq={sq} sk={sk}")


def test_repeat_calls_reuse_the_workspace():
    from paged_kv_cache_182_gb300 import binding

    s = _spec(dtype="bf16", HQ=8, HK=2, SQ=50, SK=64, D=128)
    x = _with_forward_y(wl.make_vjp(s, seed=8), 0.125)
    d = x.to("cuda")
    plan = binding.VjpPlan(d.q, d.k, d.v, d.y, d.g, scale=0.125, kernel=1)
    first = [t.clone() for t in plan.run()]
    second = plan.run()
    torch.cuda.synchronize()
    for a, b in zip(first, second):
        assert torch.equal(a, b) or torch.allclose(a.float(), b.float(), atol=0, rtol=2.0 ** -7)


# --------------------------------------------------------------- tensor cores
TC_TOL = {"bf16": 4 * UNIT["bf16"], "f16": 4 * UNIT["f16"]}

TC_CASES = {
    # name: (B, HQ, HK, SQ, SK, causal)
    "one_tile": (1, 2, 1, 64, 128, False),
    "ragged_gqa4": (2, 8, 2, 200, 300, False),
    "ragged_gqa4_causal": (2, 8, 2, 200, 300, True),
    "tall_causal": (1, 4, 4, 300, 130, True),
    "wide_causal_mha": (2, 3, 3, 70, 333, True),
    "single": (1, 2, 2, 1, 1, False),
    "gqa8_square": (1, 16, 2, 256, 256, True),
    # more row tiles than SMs: every CTA of the persistent statistics kernel
    # takes several items of different lengths (snake order), the K ring and
    # the two Q buffers run on across them
    "persistent_causal": (1, 40, 10, 1000, 1000, True),
    "persistent_wide": (1, 64, 16, 700, 300, False),
}


def _status():
    return torch.zeros(1, dtype=torch.int32, device="cuda")


@pytest.mark.parametrize("dtype", ["bf16", "f16"])
@pytest.mark.parametrize("name", sorted(TC_CASES))
def test_tensor_cores_match_the_oracle(name, dtype):
    B, HQ, HK, SQ, SK, causal = TC_CASES[name]
    s = _spec(dtype=dtype, B=B, HQ=HQ, HK=HK, SQ=SQ, SK=SK, D=128, causal=causal)
    scale = 1.0 / np.sqrt(128)
    x = _with_forward_y(wl.make_vjp(s, seed=11), scale)
    st = _status()
    got = _run(x, scale, out_dtype=torch.float32, status=st)
    assert int(st.item()) == 0, f"status {int(st.item())}"
    _check(got, _oracle(x, scale), TC_TOL[dtype], label=f"{name}/{dtype}")


@pytest.mark.parametrize("dtype", ["bf16", "f16"])
def test_tensor_cores_native_outputs(dtype):
    s = _spec(dtype=dtype, B=1, HQ=8, HK=2, SQ=190, SK=170, D=128, causal=True)
    scale = 1.0 / np.sqrt(128)
    x = _with_forward_y(wl.make_vjp(s, seed=12), scale)
    st = _status()
    got = _run(x, scale, status=st)
    assert int(st.item()) == 0
    assert all(t.dtype == x.q.dtype for t in got)
    _check(got, _oracle(x, scale), TC_TOL[dtype], out_fmt=dtype, label=f"native {dtype}")


def test_tensor_cores_agree_with_cuda_cores():
    """The two kernel families on the same inputs: within the tensor-core bound."""
    s = _spec(dtype="bf16", B=1, HQ=4, HK=1, SQ=150, SK=260, D=128, causal=False)
    x = _with_forward_y(wl.make_vjp(s, seed=13), 0.09)
    a = _run(x, 0.09, out_dtype=torch.float32)
    b = _run(x, 0.09, out_dtype=torch.float32, kernel=1)
    _check(a, [t.double().numpy() for t in b], TC_TOL["bf16"], label="tc vs simt")


def test_tensor_cores_empty_key_set_and_rows():
    """SK = 0 (every row empty: dq = 0) and SQ = 0 (dk = dv = 0) on the 16-bit path."""
    from paged_kv_cache_182_gb300 import binding

    for sq, sk in ((0, 200), (130, 0)):
        s = _spec(dtype="bf16", B=1, HQ=2, HK=1, SQ=sq, SK=sk, D=128)
        x = wl.make_vjp(s, seed=14)
        d = x.to("cuda")
        out = tuple(torch.full_like(t, float("nan")) for t in (d.q, d.k, d.k))
        binding.attention_vjp(d.q, d.k, d.v, d.y, d.g, scale=0.1, out=out)
        torch.cuda.synchronize()
        for t in out:
            assert torch.all(t == 0)


@pytest.mark.parametrize("seed", [0, 1])
def test_full_size_sampled(seed):
    """The benchmarked shape (4 x 2048 tokens, 32 query heads on 8 key/value
    heads, D 128, bf16, causal) in the launch configuration the bench times;
    two (batch, key/value head) groups checked against the oracle, which
    needs only that group's rows."""
    from paged_kv_cache_182_gb300 import binding

    s = wl.VJP_SPECS["vjp_bf16"]
    x = wl.make_vjp(s, seed=seed)
    d = x.to("cuda")
    st = _status()
    dq, dk, dv = binding.attention_vjp(d.q, d.k, d.v, d.y, d.g, scale=1 / np.sqrt(s.D),
                                       causal=True, status=st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    rng = np.random.default_rng(seed)
    g = s.HQ // s.HK
    for _ in range(2):
        b, kh = int(rng.integers(s.B)), int(rng.integers(s.HK))
        hs = slice(kh * g, kh * g + g)
        sub = [_np(t[b:b + 1, hs]) for t in (x.q, x.y, x.g)]
        kv = [_np(t[b:b + 1, kh:kh + 1]) for t in (x.k, x.v)]
        want = orc.attention_vjp(sub[0], kv[0], kv[1], sub[1], sub[2], 1 / np.sqrt(s.D), True)
        got = [dq[b:b + 1, hs].cpu(), dk[b:b + 1, kh:kh + 1].cpu(), dv[b:b + 1, kh:kh + 1].cpu()]
        _check(got, want, TC_TOL["bf16"], out_fmt="bf16", label=f"full b={b} kh={kh}")
