"""The attention-backward oracle against its pins, and planted mistakes against the pins.

Each mutant is a one-spot textual edit of ``oracle/attention_vjp.py`` loaded
as a separate module; every mutant must fail at least one pin.  The real
oracle source is never modified.
"""
import importlib.util
from pathlib import Path

import pytest

import vjp_pins
from oracle import attention_vjp

ROOT = Path(__file__).resolve().parent.parent
SOURCE = ROOT / "oracle" / "attention_vjp.py"

MUTANTS = {
    "causal_strict": ("np.where(ki <= qi,", "np.where(ki < qi,"),
    "causal_bottom_right": ("np.where(ki <= qi,", "np.where(ki <= qi + (sk - sq),"),
    "scale_not_rooted": ("root = np.sqrt(np.float64(scale))\n    qs = q.reshape(b, hk, groups, sq, d) * root\n    ks = k.reshape(b, hk, 1, sk, d) * root\n    scores",
                         "root = np.float64(scale)\n    qs = q.reshape(b, hk, groups, sq, d) * root\n    ks = k.reshape(b, hk, 1, sk, d) * root\n    scores"),
    "grad_scale_not_rooted": ("root = np.sqrt(np.float64(scale))\n    qs = q.reshape(b, hk, groups, sq, d) * root\n    ks = k.reshape(b, hk, 1, sk, d) * root\n    g5",
                              "root = np.float64(scale)\n    qs = q.reshape(b, hk, groups, sq, d) * root\n    ks = k.reshape(b, hk, 1, sk, d) * root\n    g5"),
    "delta_dropped": ("ds = p * (dp - delta)", "ds = p * dp"),
    "delta_zero": ("* g5, axis=-1", "* 0.0, axis=-1"),
    "delta_sign": ("ds = p * (dp - delta)", "ds = p * (dp + delta)"),
    "empty_not_zeroed": ("return np.where(empty, 0.0, probability)", "return probability"),
    "gqa_modulo": ("qs = q.reshape(b, hk, groups, sq, d) * root\n    ks = k.reshape(b, hk, 1, sk, d) * root\n    scores",
                   "qs = np.swapaxes(q.reshape(b, groups, hk, sq, d), 1, 2) * root\n    ks = k.reshape(b, hk, 1, sk, d) * root\n    scores"),
    "dk_first_group_only": ("dk = np.sum(np.matmul(np.swapaxes(ds, -1, -2), qs) * root, axis=2)",
                            "dk = np.matmul(np.swapaxes(ds, -1, -2), qs)[:, :, 0] * root"),
    "dv_extra_root": ("dv = np.sum(np.matmul(pt, g5), axis=2)", "dv = np.sum(np.matmul(pt, g5), axis=2) * root"),
    "dq_no_root": ("dq = (np.matmul(ds, ks) * root)", "dq = (np.matmul(ds, ks))"),
    "dk_with_q_unscaled": ("np.swapaxes(ds, -1, -2), qs) * root", "np.swapaxes(ds, -1, -2), qs / root) * root"),
    "dp_from_keys": ("dp = np.matmul(g5, np.swapaxes(v5, -1, -2))", "dp = np.matmul(g5, np.swapaxes(ks, -1, -2))"),
    "pad_with_zero": ("constant_values=-np.inf", "constant_values=0.0"),
    "boolean_inverted": ("np.where(np.asarray(mask) != 0, 0.0, -np.inf)", "np.where(np.asarray(mask) != 0, -np.inf, 0.0)"),
    "width_one_padded": ("if width != 1 and width < sk:", "if width < sk:"),
    "mask_ignored": ("scores = scores + _bias(mask, mask_kind, sk)", "pass"),
}


@pytest.mark.parametrize("pin", vjp_pins.PINS, ids=lambda f: f.__name__)
def test_pin(pin):
    pin(attention_vjp)


def _load_mutant(name, tmp_path):
    old, new = MUTANTS[name]
    text = SOURCE.read_text()
    assert text.count(old) == 1, f"mutant {name}: anchor found {text.count(old)} times"
    path = tmp_path / f"attention_vjp_{name}.py"
    path.write_text(text.replace(old, new))
    spec = importlib.util.spec_from_file_location(f"attention_vjp_{name}", path)
    mod = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(mod)
    return mod


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_mutant_fails_a_pin(name, tmp_path):
    failed = vjp_pins.run_all(_load_mutant(name, tmp_path))
    assert failed, f"mutant {name} passed every pin"
