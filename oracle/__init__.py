"""float64 CPU oracle for paged decode attention -- TEST INFRASTRUCTURE ONLY.

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package.  The CUDA library never calls it and
shares no code with it; the only thing both sides see is the seeded input
generator, which holds none of the method's arithmetic.

The arithmetic lives in ``pa_oracle.c`` (plain C, float64 loops); this module
compiles it with gcc and marshals numpy arrays to it.  What it computes is
the plain definition of decode attention over a paged cache written out
(onnxruntime-ep-mlx 0.31.1, src/ops/paged_attention.rs, VECTOR_BODY /
VECTOR_REDUCE / PARTIALS_REDUCE); see the header of ``pa_oracle.c``.

Pins (tests/test_oracle_pins.py): torch's float64 scaled_dot_product_attention
on dense K/V scattered into a paged pool, bitwise invariance under block
permutation, the single-key and equal-score closed forms, the hard-max limit,
a two-key closed form, the grouped-query map, and causal truncation.
Mutants of this source (tests/test_oracle_mutants.py) must fail a pin.
"""
from __future__ import annotations

import ctypes
import os
import shutil
import subprocess
from pathlib import Path

import numpy as np

HERE = Path(__file__).resolve().parent
SOURCE = HERE / "pa_oracle.c"
LIBRARY = HERE / "_build" / "libpa_oracle.so"


def build(source: Path = SOURCE, library: Path = LIBRARY, force: bool = False) -> Path:
    """Compile ``source`` into ``library`` with gcc (OpenMP when available)."""
    library = Path(library)
    if library.exists() and not force and library.stat().st_mtime >= Path(source).stat().st_mtime:
        return library
    library.parent.mkdir(parents=True, exist_ok=True)
    cc = os.environ.get("CC", shutil.which("gcc") or "cc")
    tmp = library.with_suffix(f".{os.getpid()}.tmp.so")
    base = [cc, "-O2", "-fPIC", "-shared", "-std=c11", str(source), "-o", str(tmp), "-lm"]
    try:
        subprocess.run(base[:1] + ["-fopenmp"] + base[1:], check=True, capture_output=True)
    except subprocess.CalledProcessError:
        subprocess.run(base, check=True, capture_output=True)
    os.replace(tmp, library)
    return library


class Oracle:
    """ctypes handle on one compiled oracle library (the real one or a test mutant)."""

    def __init__(self, library: Path | str | None = None):
        path = Path(library) if library is not None else build()
        self.path = path
        self.lib = ctypes.CDLL(str(path))
        f = self.lib.pa_oracle_decode
        f.restype = ctypes.c_int
        P = ctypes.c_void_p
        I = ctypes.c_int
        f.argtypes = [P, P, P, P, P, P, P, P, ctypes.c_double, I, I, I, I, I, I, I, I,
                      ctypes.c_int64, P, I]
        g = self.lib.pa_oracle_decode_positions
        g.restype = ctypes.c_int
        g.argtypes = f.argtypes[:7] + [P] + f.argtypes[7:]
        self.lib.pa_oracle_max_threads.restype = ctypes.c_int

    def max_threads(self) -> int:
        return int(self.lib.pa_oracle_max_threads())

    def decode(self, q, k_cache, v_cache, block_table, seq_lens, k_new, v_new, *,
               scale: float, causal: bool, row_mask=None, threads: int = 0,
               positions=None) -> np.ndarray:
        """Attention output [B, H, NQ, D] in float64.

        Array shapes: q [B,H,NQ,D]; k_cache/v_cache [NB,BLOCK,KV,D];
        block_table [B,MAXB] int32; seq_lens [B] int32; k_new/v_new [B,KV,NQ,D];
        positions (optional) [B,NQ] int32, the cache slot each new row is bound
        for or -1: a cached key of sequence b whose slot is positions[b, j]
        reads new row j instead (the last such j).
        Any float dtype is accepted and converted exactly to float64.
        """
        q = _f64(q)
        kc, vc = _f64(k_cache), _f64(v_cache)
        kn, vn = _f64(k_new), _f64(v_new)
        table = np.ascontiguousarray(block_table, dtype=np.int32)
        lens = np.ascontiguousarray(seq_lens, dtype=np.int32)
        B, H, NQ, D = q.shape
        NB, BLOCK, KV, D2 = kc.shape
        if D2 != D or vc.shape != kc.shape or kn.shape != (B, KV, NQ, D) or vn.shape != kn.shape:
            raise ValueError("oracle: inconsistent shapes")
        if table.ndim != 2 or table.shape[0] != B or lens.shape != (B,):
            raise ValueError("oracle: block table / seq_lens shape")
        out = np.zeros((B, H, NQ, D), dtype=np.float64)
        mask_ptr = None
        if row_mask is not None:
            row_mask = np.ascontiguousarray(row_mask, dtype=np.uint8).reshape(-1)
            if row_mask.size != B * H * NQ:
                raise ValueError("oracle: row_mask must have B*H*NQ entries")
            mask_ptr = row_mask.ctypes.data
        tail = (out.ctypes.data, float(scale), B, H, KV, D, BLOCK, NQ, int(bool(causal)),
                table.shape[1], NB, mask_ptr, int(threads))
        head = (q.ctypes.data, kc.ctypes.data, vc.ctypes.data, table.ctypes.data,
                lens.ctypes.data, kn.ctypes.data, vn.ctypes.data)
        if positions is None:
            rc = self.lib.pa_oracle_decode(*head, *tail)
        else:
            pos = np.ascontiguousarray(positions, dtype=np.int32)
            if pos.shape != (B, NQ):
                raise ValueError("oracle: positions must be [B, NQ]")
            rc = self.lib.pa_oracle_decode_positions(*head, pos.ctypes.data, *tail)
        if rc != 0:
            raise ValueError(f"oracle: pa_oracle_decode returned {rc}")
        return out


def _f64(a) -> np.ndarray:
    if hasattr(a, "detach"):  # torch tensor: exact upcast of the stored values
        import torch

        a = a.detach().to("cpu", torch.float64).numpy()
    return np.ascontiguousarray(a, dtype=np.float64)


_DEFAULT: Oracle | None = None


def default() -> Oracle:
    global _DEFAULT
    if _DEFAULT is None:
        _DEFAULT = Oracle()
    return _DEFAULT


def decode(*args, **kwargs) -> np.ndarray:
    """Module-level shortcut on the default (unmutated) oracle."""
    return default().decode(*args, **kwargs)


def cache_append(k_cache, v_cache, k_new, v_new, slot_mapping):
    """The cache update of a decode step, written out: copies of the caches in
    which, for every sequence b, new row j and KV head kh whose slot
    s = slot_mapping[b, j] lies in [0, num_blocks * BLOCK),
        cache[s // BLOCK, s % BLOCK, kh, :] = new[b, kh, j, :].
    A slot is a cache row index, physical block * BLOCK + offset, as the
    decode kernel of the paged-attention page names the slot of new row j
    (onnxruntime-ep-mlx 0.31.1, src/ops/paged_attention.rs, VECTOR_BODY,
    position[j + 1]); on that page the host writes these rows back into the
    cache after evaluation (src/engine.rs, write_back_input_rows).  Slot -1
    skips a row; any other slot outside the cache skips it and is reported.
    Works on the stored values (any dtype; bfloat16 as its 16-bit pattern):
    returns (k_cache', v_cache', bad_slot)."""
    kc = np.array(k_cache, copy=True)
    vc = np.array(v_cache, copy=True)
    kn, vn = np.asarray(k_new), np.asarray(v_new)
    slots = np.asarray(slot_mapping)
    NB, BLOCK, KV, _ = kc.shape
    B, _, NQ, _ = kn.shape
    bad = False
    for b in range(B):
        for j in range(NQ):
            s = int(slots[b, j])
            if s == -1:
                continue
            if s < -1 or s >= NB * BLOCK:
                bad = True
                continue
            for kh in range(KV):
                kc[s // BLOCK, s % BLOCK, kh, :] = kn[b, kh, j, :]
                vc[s // BLOCK, s % BLOCK, kh, :] = vn[b, kh, j, :]
    return kc, vc, bad
