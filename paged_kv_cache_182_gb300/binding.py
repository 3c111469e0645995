"""ctypes binding of ``libpadecode.so`` (C ABI in ``include/pa_decode.h``).

Argument marshalling only: every step of the computation runs in the
library's CUDA kernels.  If the library has not been built, importing this
module raises -- there is no Python or CPU fallback.

Tensor layouts (row-major, contiguous):
  q, out           [B, H, NQ, D]            float32 / float16 / bfloat16
  k_cache, v_cache [num_blocks, BLOCK, KV, D]
  block_table      [B, max_blocks]          int32
  seq_lens         [B]                      int32 (cached tokens per sequence)
  k_new, v_new     [B, KV, NQ, D]

Entry points: ``decode`` / ``Plan`` (device tensors), ``decode_host`` /
``HostPlan`` (host tensors, device-resident caches), ``cache_append`` (new
rows into their cache slots), ``decode_positions`` (a decode step with slot
patching), ``prefill`` / ``PrefillPlan`` (causal prefill of any number of
new rows up to PA_MAX_PREFILL) and ``attention_vjp`` / ``VjpPlan`` (dense
attention backward, ``include/pa_attention_vjp.h``: q, y, g [B, HQ, SQ, D],
k, v [B, HK, SK, D]).
"""
from __future__ import annotations

import ctypes
from pathlib import Path

import torch

from . import _build

PA_F32, PA_F16, PA_BF16 = 0, 1, 2
PA_STATUS_BAD_BLOCK, PA_STATUS_BAD_LENGTH, PA_STATUS_TIMEOUT, PA_STATUS_BAD_SLOT = 1, 2, 4, 8
PA_MAX_NQ = 16
PA_MAX_PREFILL = 65536
_DT = {torch.float32: PA_F32, torch.float16: PA_F16, torch.bfloat16: PA_BF16}

LIBRARY = _build.LIBRARY


class PaOpts(ctypes.Structure):
    _fields_ = [
        ("batch", ctypes.c_int),
        ("max_blocks", ctypes.c_int),
        ("num_blocks", ctypes.c_int),
        ("dtype", ctypes.c_int),
        ("out_dtype", ctypes.c_int),
        ("partitions", ctypes.c_int),
        ("checked", ctypes.c_int),
        ("workspace", ctypes.c_void_p),
        ("workspace_bytes", ctypes.c_size_t),
        ("status", ctypes.c_void_p),
        ("trace_begin", ctypes.c_void_p),
        ("trace_split", ctypes.c_void_p),
        ("merge_kernel", ctypes.c_int),
        ("wait_limit_ns", ctypes.c_ulonglong),
        ("debug_withhold_stage", ctypes.c_int),
        ("inputs_unchanged", ctypes.c_int),
        ("kernel", ctypes.c_int),
    ]


class VjpOpts(ctypes.Structure):
    _fields_ = [
        ("dtype", ctypes.c_int),
        ("out_dtype", ctypes.c_int),
        ("causal", ctypes.c_int),
        ("mask_kind", ctypes.c_int),
        ("mask_dims", ctypes.c_int * 4),
        ("workspace", ctypes.c_void_p),
        ("workspace_bytes", ctypes.c_size_t),
        ("status", ctypes.c_void_p),
        ("kernel", ctypes.c_int),
        ("wait_limit_ns", ctypes.c_ulonglong),
    ]


class SplitPlan(ctypes.Structure):
    _fields_ = [(name, ctypes.c_int) for name in (
        "grid", "active", "segments", "pieces", "split_segments", "records", "max_pieces")]


def load(path: Path = LIBRARY) -> ctypes.CDLL:
    """Load the C-ABI library and declare its signatures."""
    if not Path(path).exists():
        raise RuntimeError(
            f"{path} is missing: build it with paged_kv_cache_182_gb300._build.build() "
            "(there is no fallback path)")
    lib = ctypes.CDLL(str(path))
    P, I = ctypes.c_void_p, ctypes.c_int
    lib.pa_decode.restype = I
    lib.pa_decode.argtypes = [P, P, P, P, P, P, P, P, ctypes.c_float, I, I, I, I, I, I,
                              ctypes.POINTER(PaOpts), P]
    lib.pa_decode_positions.restype = I
    lib.pa_decode_positions.argtypes = [P, P, P, P, P, P, P, P, P, ctypes.c_float, I, I, I, I,
                                        I, I, ctypes.POINTER(PaOpts), P]
    lib.pa_prefill.restype = I
    lib.pa_prefill.argtypes = [P, P, P, P, P, P, P, P, ctypes.c_float, I, I, I, I, I,
                               ctypes.POINTER(PaOpts), P]
    lib.pa_prefill_workspace_bytes.restype = ctypes.c_size_t
    lib.pa_prefill_workspace_bytes.argtypes = [I, I, I, I, I, I, I, I]
    lib.pa_prefill_workspace_zero_bytes.restype = ctypes.c_size_t
    lib.pa_prefill_workspace_zero_bytes.argtypes = [I, I, I, I, I, I, I, I]
    lib.pa_decode_static_workspace.restype = I
    lib.pa_decode_static_workspace.argtypes = lib.pa_decode.argtypes
    lib.pa_workspace_bytes.restype = ctypes.c_size_t
    lib.pa_workspace_bytes.argtypes = [I, I, I, I, I, I]
    lib.pa_workspace_zero_bytes.restype = ctypes.c_size_t
    lib.pa_workspace_zero_bytes.argtypes = [I, I, I, I, I, I]
    lib.pa_decode_host.restype = I
    lib.pa_decode_host.argtypes = lib.pa_decode.argtypes
    lib.pa_host_workspace_bytes.restype = ctypes.c_size_t
    lib.pa_host_workspace_bytes.argtypes = [I, I, I, I, I, I, I, I, I]
    lib.pa_strerror.restype = ctypes.c_char_p
    lib.pa_strerror.argtypes = [I]
    lib.pa_version.restype = I
    lib.pa_kernel_launches.restype = ctypes.c_uint64
    lib.pa_host_register.restype = I
    lib.pa_host_register.argtypes = [P, ctypes.c_size_t]
    lib.pa_host_unregister.restype = I
    lib.pa_host_unregister.argtypes = [P]
    lib.pa_choose_partitions.restype = I
    lib.pa_choose_partitions.argtypes = [P, I, I, I, I, I, I, I, I, I, ctypes.POINTER(SplitPlan)]
    lib.pa_attention_vjp.restype = I
    lib.pa_attention_vjp.argtypes = [P, P, P, P, P, P, P, P, P, ctypes.c_float, I, I, I, I, I, I,
                                     ctypes.POINTER(VjpOpts), P]
    lib.pa_attention_vjp_workspace_bytes.restype = ctypes.c_size_t
    lib.pa_attention_vjp_workspace_bytes.argtypes = [I, I, I, I, I, I]
    lib.pa_cache_append.restype = I
    lib.pa_cache_append.argtypes = [P, P, P, P, P, I, I, I, I, I, I, I, P, P]
    return lib


LIB = load()


class PagedAttentionError(RuntimeError):
    def __init__(self, code: int):
        self.code = code
        super().__init__(f"pa_decode returned {code}: {strerror(code)}")


def strerror(code: int) -> str:
    return LIB.pa_strerror(int(code)).decode()


def kernel_launches() -> int:
    return int(LIB.pa_kernel_launches())


def choose_partitions(seq_lens, max_len: int, H: int, KV: int, D: int, BLOCK: int, NQ: int,
                      dtype=torch.float16, sms: int = 0, batch: int | None = None) -> SplitPlan:
    """The automatic split pa_decode makes of a batch with these host lengths
    (pa_choose_partitions); ``seq_lens=None`` means every sequence holds
    ``max_len`` tokens (then ``batch`` gives their number)."""
    if seq_lens is None:
        arr, B = None, int(batch)
    else:
        lens = torch.as_tensor(seq_lens, dtype=torch.int32).contiguous().cpu()
        arr, B = ctypes.c_void_p(lens.data_ptr()), int(lens.numel())
    plan = SplitPlan()
    rc = LIB.pa_choose_partitions(arr, int(max_len), B, H, KV, D, BLOCK, NQ, _DT[dtype], int(sms),
                                  ctypes.byref(plan))
    if rc < 0:
        raise PagedAttentionError(rc)
    return plan


def workspace_bytes(B: int, H: int, KV: int, D: int, NQ: int, partitions: int = 0) -> int:
    return int(LIB.pa_workspace_bytes(B, H, KV, D, NQ, partitions))


def workspace_zero_bytes(B: int, H: int, KV: int, D: int, NQ: int, partitions: int = 0) -> int:
    """Leading workspace bytes that must be zero before first use (in-kernel merge)."""
    return int(LIB.pa_workspace_zero_bytes(B, H, KV, D, NQ, partitions))


def new_workspace(B, H, KV, D, NQ, partitions=0, device="cuda"):
    """A zero-filled workspace of the size pa_decode needs (None when none is needed)."""
    need = workspace_bytes(B, H, KV, D, NQ, partitions)
    return torch.zeros(need, dtype=torch.uint8, device=device) if need > 0 else None


def _ptr(t):
    return None if t is None or t.data_ptr() == 0 else ctypes.c_void_p(t.data_ptr())


def _stream_handle(stream):
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream)


class Plan:
    """One prepared decode call on fixed device tensors.

    Validates shapes once and packs the ctypes arguments, so that repeated
    calls (a decode loop, CUDA-graph capture, the bench) cost one foreign
    call.  The workspace is allocated once, here, with torch.
    """

    def __init__(self, q, k_cache, v_cache, block_table, seq_lens, k_new, v_new, *,
                 scale: float, causal: bool = False, partitions: int = 0, out=None,
                 out_dtype=None, workspace=None, status=None, checked: bool = False,
                 trace=None, merge_kernel: bool = False, inputs_unchanged: bool = False,
                 kernel: int = 0):
        B, H, NQ, D = q.shape
        NB, BLOCK, KV, D2 = k_cache.shape
        if (D2 != D or tuple(v_cache.shape) != tuple(k_cache.shape)
                or tuple(k_new.shape) != (B, KV, NQ, D) or tuple(v_new.shape) != (B, KV, NQ, D)):
            raise ValueError("inconsistent q / cache / new-row shapes")
        if block_table.dim() != 2 or block_table.shape[0] != B or tuple(seq_lens.shape) != (B,):
            raise ValueError("block_table must be [B, max_blocks] and seq_lens [B]")
        if block_table.dtype != torch.int32 or seq_lens.dtype != torch.int32:
            raise TypeError("block_table and seq_lens must be int32")
        dt = q.dtype
        for t in (k_cache, v_cache, k_new, v_new):
            if t.dtype != dt:
                raise TypeError("q, caches and new rows must share one dtype")
        if dt not in _DT:
            raise TypeError(f"unsupported dtype {dt}")
        tensors = (q, k_cache, v_cache, block_table, seq_lens, k_new, v_new)
        for t in tensors:
            if not t.is_cuda:
                raise ValueError("all tensors must be CUDA tensors")
            if not t.is_contiguous():
                raise ValueError("all tensors must be contiguous")
        odt = dt if out_dtype is None else out_dtype
        if out is None:
            out = torch.empty((B, H, NQ, D), dtype=odt, device=q.device)
        elif tuple(out.shape) != (B, H, NQ, D) or not out.is_contiguous() or out.dtype != odt:
            raise ValueError("out must be a contiguous [B, H, NQ, D] tensor of the output dtype")
        if workspace is None:
            workspace = new_workspace(B, H, KV, D, NQ, partitions, q.device)
        self.tensors = tensors
        self.out = out
        self.workspace = workspace
        self.status = status
        self.trace = trace
        self.device = q.device
        self.shape = dict(B=B, H=H, KV=KV, D=D, BLOCK=BLOCK, NQ=NQ, num_blocks=NB,
                          max_blocks=int(block_table.shape[1]))
        self.opts = PaOpts(
            batch=B, max_blocks=int(block_table.shape[1]), num_blocks=NB, dtype=_DT[dt],
            out_dtype=_DT[odt], partitions=int(partitions), checked=int(bool(checked)),
            workspace=None if workspace is None else workspace.data_ptr(),
            workspace_bytes=0 if workspace is None else workspace.numel(),
            status=None if status is None else status.data_ptr(),
            trace_begin=None if trace is None else trace[0].cuda_event,
            trace_split=None if trace is None else trace[1].cuda_event,
            merge_kernel=int(bool(merge_kernel)), inputs_unchanged=int(bool(inputs_unchanged)),
            kernel=int(kernel))
        self._args = [_ptr(t) for t in tensors] + [_ptr(out), ctypes.c_float(scale), H, KV, D,
                                                   BLOCK, NQ, int(bool(causal)),
                                                   ctypes.byref(self.opts)]

    def set_trace(self, begin=None, split=None):
        """Events recorded around the partition kernel by the next run()."""
        self.opts.trace_begin = None if begin is None else begin.cuda_event
        self.opts.trace_split = None if split is None else split.cuda_event

    def bind_stream(self, stream=None):
        """Fix the stream of later run_bound() calls (default: torch's current)."""
        self._bound = self._args + [_stream_handle(stream)]

    def run_bound(self):
        """Launch on the stream fixed by bind_stream(): one foreign call, no lookups."""
        rc = LIB.pa_decode(*self._bound)
        if rc != 0:
            raise PagedAttentionError(rc)
        return self.out

    def run(self, stream=None):
        """Launch on ``stream`` (default: torch's current stream); returns ``out``."""
        if torch.cuda.current_device() == self.device.index:
            rc = LIB.pa_decode(*self._args, _stream_handle(stream))
        else:
            with torch.cuda.device(self.device):
                rc = LIB.pa_decode(*self._args, _stream_handle(stream))
        if rc != 0:
            raise PagedAttentionError(rc)
        return self.out


def decode(q, k_cache, v_cache, block_table, seq_lens, k_new, v_new, *, scale: float,
           causal: bool = False, partitions: int = 0, out=None, out_dtype=None, workspace=None,
           status=None, checked: bool = False, stream=None, merge_kernel: bool = False,
           kernel: int = 0):
    """Decode attention on device tensors (see the module docstring); returns ``out``.

    A caller-provided ``workspace`` must be zero-filled before its first use
    (see pa_opts.workspace); ``new_workspace`` makes one.  ``kernel`` is
    pa_opts.kernel (0 automatic, 1 the mma.sync kernels only)."""
    plan = Plan(q, k_cache, v_cache, block_table, seq_lens, k_new, v_new, scale=scale,
                causal=causal, partitions=partitions, out=out, out_dtype=out_dtype,
                workspace=workspace, status=status, checked=checked, merge_kernel=merge_kernel,
                kernel=kernel)
    return plan.run(stream)


def decode_positions(q, k_cache, v_cache, block_table, seq_lens, k_new, v_new, positions, *,
                     scale: float, causal: bool = False, partitions: int = 0, out=None,
                     out_dtype=None, workspace=None, status=None, checked: bool = False,
                     stream=None, merge_kernel: bool = False):
    """A decode step with slot patching (pa_decode_positions): new row j of
    sequence b is bound for cache slot positions[b, j] (physical block * BLOCK
    + offset, or -1).  Stores the new rows at their slots in ``k_cache`` /
    ``v_cache`` and attends over the updated cache, so that a cached key whose
    slot a new row of its sequence is bound for reads that row (the last such
    row wins).  ``positions``: int32 [B, NQ] on the device.  Other arguments
    as ``decode``; returns ``out``."""
    plan = Plan(q, k_cache, v_cache, block_table, seq_lens, k_new, v_new, scale=scale,
                causal=causal, partitions=partitions, out=out, out_dtype=out_dtype,
                workspace=workspace, status=status, checked=checked, merge_kernel=merge_kernel)
    B, _, NQ, _ = q.shape
    if positions.dtype != torch.int32 or tuple(positions.shape) != (B, NQ):
        raise ValueError("positions must be an int32 [B, NQ] tensor")
    if not (positions.is_cuda and positions.is_contiguous()):
        raise ValueError("positions must be a contiguous CUDA tensor")
    args = plan._args[:7] + [_ptr(positions)] + plan._args[7:]
    with torch.cuda.device(plan.device):
        rc = LIB.pa_decode_positions(*args, _stream_handle(stream))
    if rc != 0:
        raise PagedAttentionError(rc)
    return plan.out


class PrefillPlan:
    """One prepared prefill call (pa_prefill) on fixed device tensors: NQ new
    rows per sequence after ``seq_lens`` cached tokens, causal, any NQ up to
    PA_MAX_PREFILL.  ``run`` stores the new rows in the caches at the slots
    the block table gives tokens seq_lens[b] + j and writes the attention
    output into ``out``; the workspace is allocated (zeroed) here."""

    def __init__(self, q, k_cache, v_cache, block_table, seq_lens, k_new, v_new, *,
                 scale: float, partitions: int = 0, out=None, out_dtype=None, status=None,
                 checked: bool = False):
        B, H, NQ, D = q.shape
        NB, BLOCK, KV, D2 = k_cache.shape
        if (D2 != D or tuple(v_cache.shape) != tuple(k_cache.shape)
                or tuple(k_new.shape) != (B, KV, NQ, D) or tuple(v_new.shape) != (B, KV, NQ, D)):
            raise ValueError("inconsistent q / cache / new-row shapes")
        if block_table.ndim != 2 or block_table.shape[0] != B or tuple(seq_lens.shape) != (B,):
            raise ValueError("block_table must be [B, max_blocks] and seq_lens [B]")
        if block_table.dtype != torch.int32 or seq_lens.dtype != torch.int32:
            raise TypeError("block_table and seq_lens must be int32")
        dt = q.dtype
        if dt not in _DT or any(t.dtype != dt for t in (k_cache, v_cache, k_new, v_new)):
            raise TypeError("q, caches and new rows must share one supported dtype")
        tensors = (q, k_cache, v_cache, block_table, seq_lens, k_new, v_new)
        for t in tensors:
            if not (t.is_cuda and t.is_contiguous()):
                raise ValueError("all tensors must be contiguous CUDA tensors")
        odt = dt if out_dtype is None else out_dtype
        if out is None:
            out = torch.empty((B, H, NQ, D), dtype=odt, device=q.device)
        elif tuple(out.shape) != (B, H, NQ, D) or not out.is_contiguous() or out.dtype != odt:
            raise ValueError("out must be a contiguous [B, H, NQ, D] tensor of the output dtype")
        need = int(LIB.pa_prefill_workspace_bytes(B, H, KV, D, NQ, int(partitions), _DT[dt],
                                                  _DT[odt]))
        if need == 0 and B > 0:
            raise ValueError("unsupported sizes")
        self.workspace = torch.zeros(max(need, 1), dtype=torch.uint8, device=q.device)
        self.tensors, self.out, self.status, self.device = tensors, out, status, q.device
        self.opts = PaOpts(
            batch=B, max_blocks=int(block_table.shape[1]), num_blocks=NB, dtype=_DT[dt],
            out_dtype=_DT[odt], partitions=int(partitions), checked=int(bool(checked)),
            workspace=self.workspace.data_ptr(), workspace_bytes=need,
            status=None if status is None else status.data_ptr(), trace_begin=None,
            trace_split=None, merge_kernel=0)
        self._args = [_ptr(t) for t in tensors] + [_ptr(out), ctypes.c_float(scale), H, KV, D,
                                                   BLOCK, NQ, ctypes.byref(self.opts)]

    def run(self, stream=None):
        with torch.cuda.device(self.device):
            rc = LIB.pa_prefill(*self._args, _stream_handle(stream))
        if rc != 0:
            raise PagedAttentionError(rc)
        return self.out


def prefill(q, k_cache, v_cache, block_table, seq_lens, k_new, v_new, *, scale: float,
            partitions: int = 0, out=None, out_dtype=None, status=None, checked: bool = False,
            stream=None):
    """Causal prefill (pa_prefill): new row j of sequence b is token
    seq_lens[b] + j; output row r attends to keys 0 .. seq_lens[b] + r.  The
    new rows are stored in ``k_cache`` / ``v_cache`` at the slots the block
    table gives their tokens (the table must hold blocks for them).  q
    [B, H, NQ, D], new rows [B, KV, NQ, D]; returns ``out``."""
    return PrefillPlan(q, k_cache, v_cache, block_table, seq_lens, k_new, v_new, scale=scale,
                       partitions=partitions, out=out, out_dtype=out_dtype, status=status,
                       checked=checked).run(stream)


class HostPlan:
    """A prepared host-buffer decode (pa_decode_host) for fixed sizes.

    The device-resident KV cache and a device workspace (the split workspace
    plus staging for the step's inputs and output, zero-filled once here) are
    fixed; each ``run`` takes the step's host tensors (pinned for asynchronous
    copies) and enqueues their copies, the decode and the copy of the output
    into ``out`` (host)."""

    def __init__(self, k_cache, v_cache, *, B: int, H: int, NQ: int, max_blocks: int,
                 scale: float, causal: bool = False, partitions: int = 0, out_dtype=None):
        NB, BLOCK, KV, D = k_cache.shape
        dt = k_cache.dtype
        if dt not in _DT or v_cache.dtype != dt or tuple(v_cache.shape) != tuple(k_cache.shape):
            raise TypeError("k_cache and v_cache must share one supported dtype and shape")
        if not (k_cache.is_cuda and k_cache.is_contiguous() and v_cache.is_contiguous()):
            raise ValueError("the caches must be contiguous CUDA tensors")
        odt = dt if out_dtype is None else out_dtype
        need = int(LIB.pa_host_workspace_bytes(B, max_blocks, H, KV, D, NQ, int(partitions),
                                               _DT[dt], _DT[odt]))
        if need == 0 and B > 0:
            raise ValueError("unsupported sizes")
        self.workspace = torch.zeros(max(need, 1), dtype=torch.uint8, device=k_cache.device)
        self.caches = (k_cache, v_cache)
        self.device = k_cache.device
        self.shape = dict(B=B, H=H, KV=KV, D=D, NQ=NQ, max_blocks=max_blocks)
        self.dtype, self.out_dtype = dt, odt
        self.opts = PaOpts(batch=B, max_blocks=max_blocks, num_blocks=NB, dtype=_DT[dt],
                           out_dtype=_DT[odt], partitions=int(partitions), checked=0,
                           workspace=self.workspace.data_ptr(), workspace_bytes=need,
                           status=None, trace_begin=None, trace_split=None, merge_kernel=0)
        self._fixed = (ctypes.c_float(scale), H, KV, D, BLOCK, NQ, int(bool(causal)),
                       ctypes.byref(self.opts))
        self._kc, self._vc = _ptr(k_cache), _ptr(v_cache)

    def register(self, *tensors):
        """Declare pinned host tensors to the library (pa_host_register): their
        device addresses are then not looked up on every step, and an ``out``
        among them is written by the kernels in place.  The plan keeps them
        alive and releases the records in ``close``."""
        if not hasattr(self, "_registered"):
            self._registered = []
        for x in tensors:
            if x.is_cuda or not x.is_contiguous():
                raise ValueError("only contiguous host tensors can be registered")
            rc = LIB.pa_host_register(ctypes.c_void_p(x.data_ptr()), x.numel() * x.element_size())
            if rc != 0:
                raise PagedAttentionError(rc)
            self._registered.append(x)

    def close(self):
        """Release the records of the registered tensors (before freeing them)."""
        for x in getattr(self, "_registered", []):
            LIB.pa_host_unregister(ctypes.c_void_p(x.data_ptr()))
        self._registered = []

    def __del__(self):
        try:
            self.close()
        except Exception:  # interpreter shutdown: the library may be gone
            pass

    def bind(self, q, block_table, seq_lens, k_new, v_new, out, stream=None):
        """Check the step's host tensors once and fix them and the stream for
        ``run_bound`` (a loop that refills the same pinned buffers each step)."""
        self._check(q, block_table, seq_lens, k_new, v_new, out)
        self._bound = (_ptr(q), self._kc, self._vc, _ptr(block_table), _ptr(seq_lens), _ptr(k_new),
                       _ptr(v_new), _ptr(out), *self._fixed, _stream_handle(stream))
        self._bound_out = out

    def run_bound(self):
        """One step on the tensors fixed by ``bind``: one foreign call."""
        rc = LIB.pa_decode_host(*self._bound)
        if rc != 0:
            raise PagedAttentionError(rc)
        return self._bound_out

    def _check(self, q, block_table, seq_lens, k_new, v_new, out):
        s = self.shape
        if (tuple(q.shape) != (s["B"], s["H"], s["NQ"], s["D"]) or
                tuple(block_table.shape) != (s["B"], s["max_blocks"]) or
                tuple(seq_lens.shape) != (s["B"],) or tuple(out.shape) != tuple(q.shape) or
                tuple(k_new.shape) != (s["B"], s["KV"], s["NQ"], s["D"]) or
                tuple(v_new.shape) != tuple(k_new.shape)):
            raise ValueError("step tensors do not match the plan's sizes")
        for x in (q, block_table, seq_lens, k_new, v_new, out):
            if x.is_cuda or not x.is_contiguous():
                raise ValueError("step tensors must be contiguous host tensors")
        if q.dtype != self.dtype or k_new.dtype != self.dtype or v_new.dtype != self.dtype:
            raise TypeError("q and the new rows must have the caches' dtype")
        if out.dtype != self.out_dtype:
            raise TypeError("out must have the plan's output dtype")
        if block_table.dtype != torch.int32 or seq_lens.dtype != torch.int32:
            raise TypeError("block_table and seq_lens must be int32")

    def run(self, q, block_table, seq_lens, k_new, v_new, out, stream=None):
        """Enqueue one step on ``stream`` (default: torch's current stream).  All
        six tensors are host tensors; ``out`` holds the result once the stream
        has been synchronised."""
        self._check(q, block_table, seq_lens, k_new, v_new, out)
        args = (_ptr(q), self._kc, self._vc, _ptr(block_table), _ptr(seq_lens), _ptr(k_new),
                _ptr(v_new), _ptr(out), *self._fixed)
        if torch.cuda.current_device() == self.device.index:
            rc = LIB.pa_decode_host(*args, _stream_handle(stream))
        else:
            with torch.cuda.device(self.device):
                rc = LIB.pa_decode_host(*args, _stream_handle(stream))
        if rc != 0:
            raise PagedAttentionError(rc)
        return out


_host_plans = {}


def decode_host(q, block_table, seq_lens, k_new, v_new, *, k_cache, v_cache, scale: float,
                causal: bool = False, partitions: int = 0, out_dtype=None, stream=None):
    """End-to-end decode step from host tensors through pa_decode_host.

    The KV cache (``k_cache``, ``v_cache``) is device-resident state, as a KV
    cache is; the step's inputs -- q, the block table, the lengths and the
    new rows -- are host tensors (pinned for asynchronous copies).  The copies,
    the kernels and the copy of the output back to pinned host memory are
    enqueued by one library call; the device workspace is kept per size.
    Returns the host output tensor after synchronising the stream.
    """
    B, H, NQ, _ = q.shape
    odt = q.dtype if out_dtype is None else out_dtype
    key = (k_cache.data_ptr(), v_cache.data_ptr(), tuple(k_cache.shape), B, H, NQ,
           int(block_table.shape[1]), float(scale), bool(causal), int(partitions), odt)
    plan = _host_plans.get(key)
    if plan is None:
        plan = HostPlan(k_cache, v_cache, B=B, H=H, NQ=NQ, max_blocks=int(block_table.shape[1]),
                        scale=scale, causal=causal, partitions=partitions, out_dtype=out_dtype)
        _host_plans.clear()  # one plan at a time: it owns a device workspace
        _host_plans[key] = plan
    if stream is None:
        stream = torch.cuda.current_stream(k_cache.device)
    out = torch.empty(q.shape, dtype=odt, pin_memory=True)
    plan.run(q, block_table, seq_lens, k_new, v_new, out, stream)
    stream.synchronize()
    return out


def cache_append(k_cache, v_cache, k_new, v_new, slot_mapping, *, status=None, stream=None):
    """Writes the new rows into the paged cache (pa_cache_append): for every
    sequence b, new row j and KV head kh with s = slot_mapping[b, j] >= 0,
    k_cache[s // BLOCK, s % BLOCK, kh] = k_new[b, kh, j] (and the same for V).
    All tensors on one CUDA device: caches [num_blocks, BLOCK, KV, D], new rows
    [B, KV, NQ, D] of the caches' dtype, slot_mapping int32 [B, NQ], status an
    optional int32 device scalar for PA_STATUS_BAD_SLOT.  Enqueued on ``stream``
    (default: torch's current stream)."""
    NB, BLOCK, KV, D = k_cache.shape
    B, kv2, NQ, d2 = k_new.shape
    dt = k_cache.dtype
    if dt not in _DT or v_cache.dtype != dt or k_new.dtype != dt or v_new.dtype != dt:
        raise TypeError("caches and new rows must share one supported dtype")
    if (tuple(v_cache.shape) != tuple(k_cache.shape) or tuple(v_new.shape) != tuple(k_new.shape)
            or kv2 != KV or d2 != D or tuple(slot_mapping.shape) != (B, NQ)):
        raise ValueError("shapes: caches [NB, BLOCK, KV, D], new rows [B, KV, NQ, D], slots [B, NQ]")
    if slot_mapping.dtype != torch.int32:
        raise TypeError("slot_mapping must be int32")
    for x in (k_cache, v_cache, k_new, v_new, slot_mapping):
        if not (x.is_cuda and x.is_contiguous()):
            raise ValueError("all tensors must be contiguous CUDA tensors")
    args = (_ptr(k_cache), _ptr(v_cache), _ptr(k_new), _ptr(v_new), _ptr(slot_mapping), B, KV, D,
            NQ, BLOCK, NB, _DT[dt], _ptr(status))
    if torch.cuda.current_device() == k_cache.device.index:
        rc = LIB.pa_cache_append(*args, _stream_handle(stream))
    else:
        with torch.cuda.device(k_cache.device):
            rc = LIB.pa_cache_append(*args, _stream_handle(stream))
    if rc != 0:
        raise PagedAttentionError(rc)


PA_VJP_MASK_NONE, PA_VJP_MASK_BOOL, PA_VJP_MASK_ADD = 0, 1, 2


def vjp_workspace_bytes(B: int, HQ: int, SQ: int, D: int, dtype=torch.bfloat16,
                        out_dtype=None) -> int:
    odt = -1 if out_dtype is None else _DT[out_dtype]
    return int(LIB.pa_attention_vjp_workspace_bytes(B, HQ, SQ, D, _DT[dtype], odt))


class VjpPlan:
    """One prepared attention backward (pa_attention_vjp) on fixed device
    tensors: q, y, g [B, HQ, SQ, D] and k, v [B, HK, SK, D] of one dtype, an
    optional mask (uint8 = boolean, float32 = additive) of dims [MB, MH, MQ, W]
    broadcasting against the scores [B, HQ, SQ, SK].  ``run()`` enqueues the
    kernels and returns (dq, dk, dv); the outputs and the workspace are
    allocated once, here (or given as ``out``)."""

    def __init__(self, q, k, v, y, g, mask=None, *, scale: float, causal: bool = False,
                 out_dtype=None, kernel: int = 0, status=None, wait_limit_ns: int = 0, out=None):
        B, HQ, SQ, D = q.shape
        b2, HK, SK, d2 = k.shape
        dt = q.dtype
        if dt not in _DT or any(t.dtype != dt for t in (k, v, y, g)):
            raise TypeError("q, k, v, y, g must share one supported dtype")
        if (b2 != B or d2 != D or tuple(v.shape) != tuple(k.shape) or tuple(y.shape) != tuple(q.shape)
                or tuple(g.shape) != tuple(q.shape)):
            raise ValueError("shapes: q, y, g [B, HQ, SQ, D]; k, v [B, HK, SK, D]")
        for x in (q, k, v, y, g) + (() if mask is None else (mask,)):
            if not (x.is_cuda and x.is_contiguous()):
                raise ValueError("all tensors must be contiguous CUDA tensors")
        o = VjpOpts()
        o.dtype = _DT[dt]
        odt = dt if out_dtype is None else out_dtype
        o.out_dtype = -1 if out_dtype is None else _DT[out_dtype]
        o.causal = int(bool(causal))
        if mask is None:
            o.mask_kind = PA_VJP_MASK_NONE
        else:
            if mask.dim() != 4:
                raise ValueError("mask must have 4 dims [MB, MH, MQ, W]")
            if mask.dtype == torch.uint8 or mask.dtype == torch.bool:
                mask = mask.to(torch.uint8)
                o.mask_kind = PA_VJP_MASK_BOOL
            elif mask.dtype == torch.float32:
                o.mask_kind = PA_VJP_MASK_ADD
            else:
                raise TypeError("mask must be uint8/bool (boolean) or float32 (additive)")
            for e in range(4):
                o.mask_dims[e] = int(mask.shape[e])
        dev = q.device
        if out is None:
            out = tuple(torch.empty(t.shape, dtype=odt, device=dev) for t in (q, k, k))
        self.dq, self.dk, self.dv = out
        for t, ref in zip(out, (q, k, k)):
            if t.dtype != odt or tuple(t.shape) != tuple(ref.shape) or not t.is_contiguous():
                raise ValueError("out: dq like q, dk and dv like k, of the output dtype")
        need = int(LIB.pa_attention_vjp_workspace_bytes(B, HQ, SQ, D, o.dtype, o.out_dtype))
        self.workspace = torch.empty(max(need, 256), dtype=torch.uint8, device=dev)
        o.workspace = _ptr(self.workspace)
        o.workspace_bytes = int(self.workspace.numel())
        o.status = _ptr(status)
        o.kernel = int(kernel)
        o.wait_limit_ns = int(wait_limit_ns)
        self.opts = o
        self._keep = (q, k, v, y, g, mask, status)
        self.device = dev
        self._args = (_ptr(q), _ptr(k), _ptr(v), _ptr(y), _ptr(g), _ptr(mask), _ptr(self.dq),
                      _ptr(self.dk), _ptr(self.dv), ctypes.c_float(scale), B, HQ, HK, SQ, SK, D,
                      ctypes.byref(self.opts))

    def run(self, stream=None):
        if torch.cuda.current_device() == self.device.index:
            rc = LIB.pa_attention_vjp(*self._args, _stream_handle(stream))
        else:
            with torch.cuda.device(self.device):
                rc = LIB.pa_attention_vjp(*self._args, _stream_handle(stream))
        if rc != 0:
            raise PagedAttentionError(rc)
        return self.dq, self.dk, self.dv


def attention_vjp(q, k, v, y, g, mask=None, *, scale: float, causal: bool = False,
                  out_dtype=None, kernel: int = 0, status=None, stream=None, out=None):
    """dq, dk, dv of attention (pa_attention_vjp): see ``VjpPlan``."""
    return VjpPlan(q, k, v, y, g, mask, scale=scale, causal=causal, out_dtype=out_dtype,
                   kernel=kernel, status=status, out=out).run(stream)
