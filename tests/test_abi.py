"""The C-ABI library loads, exports what include/*.h declares, and rejects
invalid arguments on the host before any CUDA call (runs without a GPU)."""
import ctypes
import math
import re
from pathlib import Path

import pytest

ROOT = Path(__file__).resolve().parent.parent


@pytest.fixture(scope="module")
def lib():
    from paged_kv_cache_182_gb300 import _build

    _build.build()
    from paged_kv_cache_182_gb300 import binding

    return binding


def declared_functions():
    names = set()
    for header in sorted((ROOT / "include").glob("*.h")):
        text = re.sub(r"/\*.*?\*/", "", header.read_text(), flags=re.S)
        names.update(re.findall(r"\b(pa_[a-z0-9_]+)\s*\(", text))
    return sorted(names)


def test_header_declares_entry_points():
    names = declared_functions()
    for required in ("pa_decode", "pa_workspace_bytes", "pa_strerror", "pa_version"):
        assert required in names


def test_every_declared_symbol_is_exported(lib):
    raw = ctypes.CDLL(str(lib.LIBRARY))
    for name in declared_functions():
        assert hasattr(raw, name), f"{name} declared in include/ but not exported"


def test_version_and_messages(lib):
    assert lib.LIB.pa_version() >= 100
    msgs = {c: lib.strerror(c) for c in range(-7, 1)}
    assert len(set(msgs.values())) == len(msgs)
    for c in range(-7, 0):
        assert "verify" in msgs[c]


def test_workspace_bytes(lib):
    ws = lib.workspace_bytes
    assert ws(8, 32, 8, 128, 1, 1) == 0
    assert ws(8, 32, 7, 128, 1, 0) == 0  # H % KV != 0
    assert ws(8, 32, 8, 96, 1, 0) == 0   # unsupported D
    assert ws(8, 32, 8, 128, 1, 0) > 0
    assert ws(1, 32, 8, 128, 1, 32) < ws(1, 32, 8, 128, 1, 64)
    # one float32 (max, sum, D accumulators) state per row and key range
    assert ws(1, 32, 8, 128, 1, 32) >= 32 * 8 * 4 * (128 + 2) * 4
    zb = lib.workspace_zero_bytes
    assert zb(8, 32, 8, 128, 1, 1) == 0
    assert zb(8, 32, 8, 128, 1, 4) == 0  # fixed partitions: the merge kernel, no counters
    assert 0 < zb(8, 32, 8, 128, 1, 0) < ws(8, 32, 8, 128, 1, 0)
    assert zb(8, 32, 8, 128, 1, 0) >= 8 * 8 * 4  # one counter per (sequence, KV head)


class Fake:
    """16-byte aligned fake device addresses: validation must fail before any use."""

    q = ctypes.c_void_p(0x10000)
    kc = ctypes.c_void_p(0x20000)
    vc = ctypes.c_void_p(0x30000)
    table = ctypes.c_void_p(0x40000)
    lens = ctypes.c_void_p(0x50000)
    kn = ctypes.c_void_p(0x60000)
    vn = ctypes.c_void_p(0x70000)
    out = ctypes.c_void_p(0x80000)


def call(lib, *, H=8, KV=2, D=64, BLOCK=16, NQ=1, scale=0.125, opts=None, q=Fake.q, **ov):
    o = lib.PaOpts(batch=2, max_blocks=4, num_blocks=8, dtype=lib.PA_F16, out_dtype=-1,
                   partitions=1, checked=0, workspace=None, workspace_bytes=0, status=None,
                   trace_begin=None, trace_split=None)
    for k, v in ov.items():
        setattr(o, k, v)
    ref = None if opts == "null" else ctypes.byref(o)
    return lib.LIB.pa_decode(q, Fake.kc, Fake.vc, Fake.table, Fake.lens, Fake.kn, Fake.vn,
                             Fake.out, ctypes.c_float(scale), H, KV, D, BLOCK, NQ, 0, ref, None)


def test_rejects_invalid_arguments(lib):
    assert call(lib, opts="null") == -1
    assert call(lib, H=8, KV=3) == -2
    assert call(lib, batch=-1) == -2
    assert call(lib, max_blocks=0) == -2
    assert call(lib, scale=math.nan) == -2
    assert call(lib, num_blocks=1 << 28) == -2
    assert call(lib, D=96) == -3
    assert call(lib, BLOCK=12) == -3
    assert call(lib, NQ=0) == -3
    assert call(lib, NQ=17) == -3
    assert call(lib, dtype=7) == -3
    assert call(lib, dtype=lib.PA_BF16, out_dtype=lib.PA_F16) == -3
    assert call(lib, q=None) == -1
    assert call(lib, q=ctypes.c_void_p(0x10008)) == -4
    assert call(lib, partitions=0) == -5
    assert call(lib, partitions=0, workspace=0x100010, workspace_bytes=1 << 30) == -4
    assert call(lib, kernel=2) == -3
    assert call(lib, kernel=-1, batch=0) == -3  # checked before the empty-batch return


def test_batch_limit_is_unsupported_not_a_workspace_limit(lib):
    """Above 4096 sequences the size queries return 0 (as for every argument
    pa_decode rejects), so the static-scratch entry reports the batch limit
    (PA_ERR_UNSUPPORTED), not PA_ERR_STATIC_LIMIT: fewer partitions cannot fix
    such a call."""
    assert lib.workspace_bytes(4096, 32, 8, 128, 1, 0) > 0
    assert lib.workspace_bytes(4097, 32, 8, 128, 1, 0) == 0
    assert lib.workspace_bytes(4097, 32, 8, 128, 1, 32) == 0
    assert lib.workspace_zero_bytes(4097, 32, 8, 128, 1, 0) == 0
    assert call(lib, batch=4097, partitions=0) == -3
    o = lib.PaOpts(batch=4097, max_blocks=4, num_blocks=8, dtype=lib.PA_F16, out_dtype=-1,
                   partitions=32, checked=0, workspace=None, workspace_bytes=0, status=None,
                   trace_begin=None, trace_split=None)
    before = lib.kernel_launches()
    rc = lib.LIB.pa_decode_static_workspace(Fake.q, Fake.kc, Fake.vc, Fake.table, Fake.lens,
                                            Fake.kn, Fake.vn, Fake.out, ctypes.c_float(0.1), 32,
                                            8, 128, 16, 1, 0, ctypes.byref(o), None)
    assert rc == -3
    assert lib.kernel_launches() == before


def test_static_entry_without_a_device_fails_cleanly(lib):
    """The static-scratch entry looks its array up under the current CUDA
    context; with no device at all that lookup fails with PA_ERR_CUDA instead
    of handing a kernel a host-side stand-in address."""
    import torch

    if torch.cuda.is_available():
        pytest.skip("needs a machine without a CUDA device")
    o = lib.PaOpts(batch=2, max_blocks=4, num_blocks=8, dtype=lib.PA_F16, out_dtype=-1,
                   partitions=0, checked=0, workspace=None, workspace_bytes=0, status=None,
                   trace_begin=None, trace_split=None)
    before = lib.kernel_launches()
    rc = lib.LIB.pa_decode_static_workspace(Fake.q, Fake.kc, Fake.vc, Fake.table, Fake.lens,
                                            Fake.kn, Fake.vn, Fake.out, ctypes.c_float(0.1), 8,
                                            2, 64, 16, 1, 0, ctypes.byref(o), None)
    assert rc == -6
    assert lib.kernel_launches() == before


def test_empty_batch_is_a_no_op(lib):
    before = lib.kernel_launches()
    assert call(lib, batch=0) == 0
    assert lib.kernel_launches() == before


def test_host_workspace_bytes_covers_split_workspace_and_staging(lib):
    hw = lib.LIB.pa_host_workspace_bytes
    split = lib.workspace_bytes(8, 32, 8, 128, 1, 0)
    # q + out (8*32*128*2 B each), table (8*257*4), lengths, new rows (2 * 8*8*128*2)
    staging = 2 * 8 * 32 * 128 * 2 + 8 * 257 * 4 + 8 * 4 + 2 * 8 * 8 * 128 * 2
    need = hw(8, 257, 32, 8, 128, 1, 0, lib.PA_F16, -1)
    assert need >= split + staging
    assert need < split + staging + 7 * 256  # six staging regions, 256-byte aligned
    assert hw(8, 257, 32, 8, 128, 1, 0, lib.PA_F16, lib.PA_F32) > need  # float32 output
    assert hw(8, 0, 32, 8, 128, 1, 0, lib.PA_F16, -1) == 0
    assert hw(8, 257, 32, 8, 96, 1, 0, lib.PA_F16, -1) == 0


def test_host_entry_point_rejects_before_copying(lib):
    """Argument checks of pa_decode_host return before any copy is enqueued
    (these calls run without a GPU)."""
    f = lib.LIB.pa_decode_host
    host = [ctypes.c_void_p(0x10000 * (i + 1)) for i in range(8)]

    def go(opts, **kw):
        a = dict(zip(("q", "kc", "vc", "table", "lens", "kn", "vn", "out"), host))
        a.update(kw)
        return f(a["q"], a["kc"], a["vc"], a["table"], a["lens"], a["kn"], a["vn"], a["out"],
                 ctypes.c_float(0.1), 32, 8, 128, 16, 1, 0, opts, None)

    def opts(**kw):
        o = dict(batch=8, max_blocks=257, num_blocks=2048, dtype=lib.PA_F16, out_dtype=-1,
                 partitions=0, checked=0, workspace=None, workspace_bytes=0, status=None,
                 trace_begin=None, trace_split=None, merge_kernel=0)
        o.update(kw)
        return ctypes.byref(lib.PaOpts(**o))

    need = lib.LIB.pa_host_workspace_bytes(8, 257, 32, 8, 128, 1, 0, lib.PA_F16, -1)
    assert f(*host, ctypes.c_float(0.1), 32, 8, 128, 16, 1, 0, None, None) == -1
    assert go(opts(batch=0)) == 0
    assert go(opts(workspace=0x100000, workspace_bytes=need), q=None) == -1
    assert go(opts()) == -1  # no workspace
    assert go(opts(workspace=0x100000, workspace_bytes=need - 1)) == -5
    assert go(opts(workspace=0x100010, workspace_bytes=need)) == -4
    assert go(opts(workspace=0x100000, workspace_bytes=need, dtype=9)) == -3


def test_cache_append_rejects_before_launching(lib):
    """pa_cache_append's argument checks (these calls run without a GPU)."""
    f = lib.LIB.pa_cache_append
    a = [ctypes.c_void_p(0x10000 * (i + 1)) for i in range(5)]

    def go(*ptrs, B=2, KV=2, D=64, NQ=1, BLOCK=16, NB=4, dt=lib.PA_F16):
        p = list(ptrs) if ptrs else a
        return f(*p, B, KV, D, NQ, BLOCK, NB, dt, None, None)

    launches = lib.kernel_launches()
    assert go(B=0) == 0  # nothing to do
    assert go(B=-1) == -2
    assert go(NQ=0) == -2
    assert go(dt=7) == -3
    assert go(D=4) == -3  # D * 2 bytes is not a multiple of 16
    assert go(None, *a[1:]) == -1
    assert go(a[0], ctypes.c_void_p(0x20008), *a[2:]) == -4
    assert go(*a[:4], ctypes.c_void_p(0x50002)) == -4  # slot_mapping 4-byte aligned
    assert lib.kernel_launches() == launches


def test_decode_positions_rejects_before_launching(lib):
    """pa_decode_positions checks every argument, its own and pa_decode's,
    before it enqueues the append (these calls run without a GPU)."""
    f = lib.LIB.pa_decode_positions
    ptrs = [ctypes.c_void_p(0x10000 * (i + 1)) for i in range(9)]

    def go(opts, **kw):
        names = ("q", "kc", "vc", "table", "lens", "kn", "vn", "pos", "out")
        a = dict(zip(names, ptrs))
        a.update(kw)
        return f(*(a[n] for n in names), ctypes.c_float(0.1), 32, 8, 128, 16, 1, 0, opts, None)

    def opts(**kw):
        o = dict(batch=8, max_blocks=257, num_blocks=2048, dtype=lib.PA_F16, out_dtype=-1,
                 partitions=1, checked=0, workspace=None, workspace_bytes=0, status=None,
                 trace_begin=None, trace_split=None, merge_kernel=0)
        o.update(kw)
        return ctypes.byref(lib.PaOpts(**o))

    launches = lib.kernel_launches()
    assert go(None) == -1
    assert go(opts(batch=0)) == 0
    assert go(opts(), kc=None) == -1
    assert go(opts(), pos=ctypes.c_void_p(0x80002)) == -4  # positions 4-byte aligned
    assert go(opts(dtype=9)) == -3
    assert go(opts(partitions=0)) == -5  # the decode's workspace is checked first
    assert lib.kernel_launches() == launches


def test_prefill_rejects_before_launching(lib):
    """pa_prefill's own checks and those of its chunk decodes come before any
    launch (these calls run without a GPU)."""
    f = lib.LIB.pa_prefill
    ptrs = [ctypes.c_void_p(0x10000 * (i + 1)) for i in range(8)]

    def go(opts, NQ=100, D=128, **kw):
        names = ("q", "kc", "vc", "table", "lens", "kn", "vn", "out")
        a = dict(zip(names, ptrs))
        a.update(kw)
        return f(*(a[n] for n in names), ctypes.c_float(0.1), 32, 8, D, 16, NQ, opts, None)

    def opts(**kw):
        o = dict(batch=4, max_blocks=96, num_blocks=384, dtype=lib.PA_F16, out_dtype=-1,
                 partitions=0, checked=0, workspace=None, workspace_bytes=0, status=None,
                 trace_begin=None, trace_split=None, merge_kernel=0)
        o.update(kw)
        return ctypes.byref(lib.PaOpts(**o))

    need = lib.LIB.pa_prefill_workspace_bytes(4, 32, 8, 128, 100, 0, lib.PA_F16, -1)
    launches = lib.kernel_launches()
    assert go(None) == -1
    assert go(opts(), NQ=0) == -2
    assert go(opts(), NQ=65537) == -3
    assert go(opts(), D=96) == -3
    assert go(opts(batch=0)) == 0
    assert go(opts(), q=None) == -1
    assert go(opts()) == -5  # no workspace
    assert go(opts(workspace=0x100000, workspace_bytes=need - 1)) == -5
    assert go(opts(workspace=0x100010, workspace_bytes=need)) == -4
    assert go(opts(workspace=0x100000, workspace_bytes=need), kn=ctypes.c_void_p(0x70008)) == -4
    assert go(opts(workspace=0x100000, workspace_bytes=need, out_dtype=lib.PA_BF16)) == -3
    assert lib.kernel_launches() == launches


def test_prefill_workspace_sizes(lib):
    pb = lib.LIB.pa_prefill_workspace_bytes
    pz = lib.LIB.pa_prefill_workspace_zero_bytes
    B, H, KV, D = 4, 32, 8, 128
    staging = B * H * 16 * D * 2 * 2 + 2 * B * KV * 16 * D * 2 + B * 4  # q, out, k/v new, lens
    split = max(lib.LIB.pa_workspace_bytes(B, H, KV, D, n, 0) for n in range(1, 17))
    assert pb(B, H, KV, D, 512, 0, lib.PA_F16, -1) >= split + staging
    assert pb(B, H, KV, D, 512, 0, lib.PA_F16, -1) < split + staging + 6 * 256
    assert pz(B, H, KV, D, 512, 0, lib.PA_F16, -1) == max(
        lib.LIB.pa_workspace_zero_bytes(B, H, KV, D, n, 0) for n in range(1, 17))
    assert pb(B, H, KV, D, 8, 0, lib.PA_F16, -1) >= lib.LIB.pa_workspace_bytes(B, H, KV, D, 8, 0)
    assert pz(B, H, KV, D, 512, 1, lib.PA_F16, -1) == 0
    assert pb(B, H, KV, D, 0, 0, lib.PA_F16, -1) == 0
    assert pb(B, H, KV, D, 65537, 0, lib.PA_F16, -1) == 0
    assert pb(B, H, KV, 96, 512, 0, lib.PA_F16, -1) == 0
    assert pb(B, H, KV, D, 512, 0, 7, -1) == 0


def test_binding_constants_match_the_header(lib):
    """Every #define of include/pa_decode.h that the binding mirrors has the
    header's value."""
    text = (ROOT / "include" / "pa_decode.h").read_text()
    defines = {}
    for name, value in re.findall(r"#define\s+(PA_[A-Z0-9_]+)\s+\(?(-?\d+)\)?", text):
        defines[name] = int(value)
    mirrored = [n for n in defines if hasattr(lib, n)]
    assert {"PA_F32", "PA_F16", "PA_BF16", "PA_MAX_NQ", "PA_MAX_PREFILL",
            "PA_STATUS_BAD_SLOT"} <= set(mirrored)
    for name in mirrored:
        assert getattr(lib, name) == defines[name], name


def _brute_force_split(lens, max_len, U, TT, V, grid):
    """The automatic split by its definition: segments of ceil((len + NQ) / TT)
    units each, laid end to end with V virtual units charged before each
    segment; G CTAs take part (each at least 4 stages of cost unless there are
    more segments than that, at most C); CTA k of G owns the cost positions
    [ceil(k C / G), ceil((k + 1) C / G)); a segment's pieces are the CTAs its
    real units fall in (NQ = 1 here).  When the segments are no more than G
    and the longest is at most W / G + 4 stages (W: all real units; 4: what a
    merge costs), every CTA takes one whole segment instead."""
    units = [(min(max(n, 0), max_len) + 1 + TT - 1) // TT for n in lens]
    C = sum(u * U for u in units) + V * len(lens) * U
    # every CTA at least 4 stages of cost, unless the segments are more; never more than C
    G = min(grid, min(C, max(len(units) * U, -(-C // 4))))
    W = sum(u * U for u in units)
    if len(units) * U <= G and max(units) * G <= W + 4 * G:
        return [1] * (len(units) * U), len(units) * U
    starts = [-(-k * C // G) for k in range(G + 1)]  # ceil(k C / G)

    def owner(c):
        k = 0
        while starts[k + 1] <= c:
            k += 1
        return k

    counts = []
    x0 = g = 0
    for u in units:
        for _ in range(U):
            c0 = x0 + V * (g + 1)
            counts.append(len({owner(c) for c in range(c0, c0 + u)}))
            x0 += u
            g += 1
    return counts, G


def test_choose_partitions_matches_its_definition(lib):
    """pa_choose_partitions against a brute-force walk of the cost positions
    (16-bit caches, D = 128, 4 query rows per KV head: 128-token stages, one
    charged unit per segment), on random length mixes and SM counts."""
    import random

    import torch

    rng = random.Random(5)
    whole = 0
    for trial in range(40):
        B = rng.randint(1, 40)
        KV = rng.choice([1, 2, 8])
        lens = [rng.choice([0, 1, rng.randint(0, 300), rng.randint(0, 20000)]) for _ in range(B)]
        max_len = rng.choice([4096, 16384, 32768])
        sms = rng.choice([1, 7, 148, 152, 300])
        plan = lib.choose_partitions(lens, max_len, 4 * KV, KV, 128, 16, 1, torch.float16, sms=sms)
        bound = B * KV * ((max_len + 1 + 127) // 128 + 1)  # pa_decode's launch: no idle CTAs
        counts, G = _brute_force_split(lens, max_len, KV, 128, 1, min(sms, 1024, bound))
        whole += all(n == 1 for n in counts) and G == len(counts)
        assert plan.active == G and plan.grid == min(sms, 1024, bound)
        assert plan.segments == len(counts)
        assert plan.pieces == sum(counts)
        assert plan.split_segments == sum(1 for n in counts if n > 1)
        assert plan.records == sum(n for n in counts if n > 1)
        assert plan.max_pieces == max(counts)
    assert whole > 0  # the whole-segment rule was taken
    # 128 equal segments on 152 SMs (the causal-append shape): whole segments
    eq = lib.choose_partitions([2048] * 16, 2048, 64, 8, 128, 32, 4, torch.float16, sms=152)
    assert (eq.active, eq.pieces, eq.records, eq.max_pieces) == (128, 128, 0, 1)
    # no lengths: every sequence holds max_len tokens
    a = lib.choose_partitions(None, 32768, 32, 8, 128, 16, 1, torch.bfloat16, sms=152, batch=1)
    b = lib.choose_partitions([32768], 32768, 32, 8, 128, 16, 1, torch.bfloat16, sms=152)
    assert (a.pieces, a.max_pieces) == (b.pieces, b.max_pieces) == (152, 19)
    short = lib.choose_partitions([10] * 1000, 4096, 32, 8, 128, 16, 1, torch.float16, sms=152)
    assert short.max_pieces == 1 and short.records == 0
    with pytest.raises(lib.PagedAttentionError):
        lib.choose_partitions([5], 100, 32, 7, 128, 16, 1, torch.float16, sms=152)


def test_failure_test_switches_are_off_by_default(lib):
    """A zero-filled pa_opts (what the binding builds) leaves the wait limit at
    its default, withholds no stage and reads no input early; the binding's
    structure lists the header's members in the header's order."""
    o = lib.PaOpts()
    assert o.wait_limit_ns == 0 and o.debug_withhold_stage == 0 and o.inputs_unchanged == 0
    header = (ROOT / "include" / "pa_decode.h").read_text()
    body = header[header.index("typedef struct pa_opts {"):header.index("} pa_opts;")]
    body = re.sub(r"/\*.*?\*/", "", body, flags=re.S)
    members = re.findall(r"\b(\w+)\s*;", body)
    assert members == [f[0] for f in lib.PaOpts._fields_]
    assert "unsigned long long wait_limit_ns;" in header
    assert "int debug_withhold_stage;" in header
    assert "int inputs_unchanged;" in header
    assert o.kernel == 0 and "int kernel;" in body


def test_host_register_rejects_memory_that_is_not_page_locked(lib):
    """pa_host_register accepts only page-locked host memory (here: a plain
    Python buffer, which is not), and unregistering an unknown pointer is an
    error; nothing is enqueued either way."""
    buf = ctypes.create_string_buffer(4096)
    before = lib.kernel_launches()
    assert lib.LIB.pa_host_register(ctypes.addressof(buf), 4096) == -9
    assert lib.LIB.pa_host_register(None, 4096) == -1
    assert lib.LIB.pa_host_unregister(ctypes.addressof(buf)) == -1
    assert "page-locked" in lib.strerror(-9)
    assert lib.kernel_launches() == before


def test_vjp_rejects_before_launching(lib):
    """pa_attention_vjp checks every argument before its first launch (these
    calls run without a GPU)."""
    f = lib.LIB.pa_attention_vjp
    ptrs = [ctypes.c_void_p(0x10000 * (i + 1)) for i in range(9)]
    names = ("q", "k", "v", "y", "g", "mask", "dq", "dk", "dv")

    def go(opts, B=2, HQ=8, HK=2, SQ=64, SK=80, D=128, scale=0.1, **kw):
        a = dict(zip(names, ptrs))
        a.update(kw)
        return f(*(a[n] for n in names), ctypes.c_float(scale), B, HQ, HK, SQ, SK, D, opts, None)

    def opts(**kw):
        o = dict(dtype=lib.PA_BF16, out_dtype=-1, causal=0, mask_kind=0, workspace=None,
                 workspace_bytes=0, status=None, kernel=0, wait_limit_ns=0)
        dims = kw.pop("mask_dims", (1, 1, 1, 1))
        o.update(kw)
        s = lib.VjpOpts(**o)
        for e in range(4):
            s.mask_dims[e] = dims[e]
        return ctypes.byref(s)

    need = lib.LIB.pa_attention_vjp_workspace_bytes(2, 8, 64, 128, lib.PA_BF16, -1)
    ok = dict(workspace=0x100000, workspace_bytes=need)
    launches = lib.kernel_launches()
    assert go(None) == -1
    assert go(opts(**ok), q=None) == -1
    assert go(opts(**ok), dv=None) == -1
    assert go(opts(**ok, mask_kind=1, mask_dims=(1, 1, 1, 80)), mask=None) == -1
    assert go(opts(**ok), HQ=6, HK=4) == -2
    assert go(opts(**ok), HK=0) == -2
    assert go(opts(**ok), SQ=-1) == -2
    assert go(opts(**ok), scale=0.0) == -2
    assert go(opts(**ok), scale=-0.5) == -2
    assert go(opts(**ok), scale=math.inf) == -2
    assert go(opts(**ok, mask_kind=3)) == -2
    assert go(opts(**ok, mask_kind=1, mask_dims=(3, 1, 1, 80))) == -2   # MB not 1 or B
    assert go(opts(**ok, mask_kind=1, mask_dims=(1, 4, 1, 80))) == -2   # MH not 1 or HQ
    assert go(opts(**ok, mask_kind=1, mask_dims=(1, 1, 63, 80))) == -2  # MQ not 1 or SQ
    assert go(opts(**ok, mask_kind=2, mask_dims=(2, 8, 64, 81))) == -2  # wider than SK
    assert go(opts(**ok, mask_kind=2, mask_dims=(2, 8, 64, 0))) == -2
    assert go(opts(**ok), D=257) == -3
    assert go(opts(**ok, dtype=7)) == -3
    assert go(opts(**ok, out_dtype=lib.PA_F16)) == -3  # bf16 inputs, f16 outputs
    assert go(opts(**ok), B=70000, SQ=1, SK=1, D=8, HQ=2, HK=1) == -3
    assert go(opts(**ok), k=ctypes.c_void_p(0x20008)) == -4
    assert go(opts(workspace=0x100010, workspace_bytes=need)) == -4
    assert go(opts()) == -1  # no workspace
    assert go(opts(workspace=0x100000, workspace_bytes=need - 1)) == -5
    assert go(opts(**ok), B=0) == 0
    assert go(opts(**ok), SQ=0, SK=0) == 0
    assert lib.kernel_launches() == launches


def test_vjp_workspace_bytes(lib):
    wb = lib.LIB.pa_attention_vjp_workspace_bytes
    rows = 2 * 8 * 128  # B * HQ * SQ rounded up to 128 rows
    assert wb(2, 8, 100, 64, lib.PA_F32, -1) == 2 * rows * 4  # lse2 and delta only
    assert wb(2, 8, 100, 64, lib.PA_BF16, lib.PA_F32) == 2 * rows * 4
    acc = -(-2 * 8 * 100 * 64 * 4 // 256) * 256
    assert wb(2, 8, 100, 64, lib.PA_BF16, -1) == 2 * rows * 4 + acc  # + float32 dq accumulator
    assert wb(2, 8, 100, 64, 9, -1) == 0
    assert wb(2, 8, 100, 64, lib.PA_BF16, lib.PA_F16) == 0
    assert wb(-1, 8, 100, 64, lib.PA_BF16, -1) == 0
