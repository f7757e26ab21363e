"""The C-ABI library on the host: it builds, loads, exports every declared symbol, rejects
bad arguments before touching CUDA, and its planner obeys its invariants (CPU only)."""
import ctypes
import os
import re

import pytest
import torch

import bf16_attention_forward_gb300 as attn
from bf16_attention_forward_gb300 import build as libbuild

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "bf16_attn.h")
NO_GPU = not torch.cuda.is_available()
# Tests that call the library's compute entry points with fake device pointers.  They expect
# every call to stop at argument validation or at the device query (no device here); where a
# GPU is visible a call that passes validation would launch kernels on those addresses, so
# they run only where none is.
fake_pointers = pytest.mark.skipif(not NO_GPU, reason="fake device pointers: only where no GPU is visible")


@pytest.fixture(scope="module")
def lib():
    libbuild.build()
    return attn.load()


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(attn_[a-z_]+)\s*\(", text)))


def test_exports_every_declared_symbol(lib):
    names = declared_functions()
    assert "attn_fwd" in names and "attn_fwd_ws" in names
    for n in names:
        assert hasattr(lib, n), n
    assert set(attn.EXPORTS) <= set(names)


def test_version_and_status_strings(lib):
    assert lib.attn_version() >= 100
    for code in range(9):
        assert attn.status_string(code)
    assert "unknown" in attn.status_string(99)


P = 0x10000   # fake, aligned, never dereferenced: every call below fails validation first


def call(lib, q=P, k=2 * P, v=3 * P, o=4 * P, B=1, H=1, Sq=8, Skv=8, d=128, layout=0, mode=0):
    return lib.attn_fwd(q, k, v, o, B, H, Sq, Skv, d, layout, mode, None)


@fake_pointers
def test_argument_errors(lib):
    assert call(lib, q=0) == 1
    assert call(lib, o=0) == 1
    for kw in ({"B": 0}, {"H": -1}, {"Sq": 0}, {"Skv": 0}, {"layout": 2}, {"mode": 3},
               {"mode": -1}):
        assert call(lib, **kw) == 1, kw
    assert call(lib, d=32) == 2
    assert call(lib, d=256) == 2
    assert call(lib, Sq=(1 << 30) + 1) == 2
    assert call(lib, q=P + 8) == 3
    assert call(lib, o=P + 2) == 3
    # o overlapping q: q occupies [P, P + 8*128*2)
    assert call(lib, o=P + 1024) == 4
    assert call(lib, o=2 * P, k=2 * P + 1024) == 4


@fake_pointers
def test_ws_entry_validates_too(lib):
    f = lib.attn_fwd_ws
    assert f(0, P, P, P, 1, 1, 8, 8, 128, 0, 0, None, None, 0, None) == 1
    assert f(P, 2 * P, 3 * P, 4 * P, 1, 1, 8, 8, 96, 0, 0, None, None, 0, None) == 2


@fake_pointers
def test_valid_args_without_gpu_report_no_device(lib):
    assert call(lib) == 5
    assert call(lib, d=64) == 5
    assert lib.attn_fwd_workspace_size(1, 1, 8, 8, 128) == 0


PLAN_SHAPES = [(1, 2, 128, 128), (4, 16, 2048, 2048), (2, 24, 4096, 300),
               (1, 12, 32760, 32760), (1, 8, 128, 65536), (3, 5, 1000, 7), (1, 1, 1, 1),
               (7, 3, 511, 4097), (1, 1, 256, 1 << 20)]


@pytest.mark.parametrize("shape", PLAN_SHAPES)
@pytest.mark.parametrize("sms", [1, 7, 148, 152])
def test_planner_invariants(lib, shape, sms):
    B, H, Sq, Skv = shape
    p = attn.plan(B, H, Sq, Skv, 128, sms)
    units = B * H * -(-Sq // 256)
    nkv = -(-Skv // 128)
    assert p["units"] == units and p["kv_tiles"] == nkv
    assert p["full_items"] + p["split_units"] == units
    assert p["items"] == p["full_items"] + p["split_units"] * p["splits"]
    assert 1 <= p["grid"] <= min(sms, p["items"])
    if p["split_units"]:
        assert 2 <= p["splits"] <= nkv and nkv // p["splits"] >= 4
        # the split tail fills at most one round, after whole rounds of full units
        assert p["split_units"] * p["splits"] <= sms
        assert p["full_items"] % sms == 0
        assert p["workspace_bytes"] == p["split_units"] * p["splits"] * 256 * (128 * 4 + 4)
    else:
        assert p["splits"] == 1 and p["workspace_bytes"] == 0
    assert attn.plan(B, H, Sq, Skv, 128, sms) == p          # pure function of its inputs


def test_planner_forced_options(lib):
    p = attn.plan(1, 2, 300, 1100, 128, 152, force_splits=3)
    assert p["split_units"] == p["units"] and p["splits"] == 3 and p["full_items"] == 0
    p = attn.plan(1, 2, 300, 300, 128, 152, force_splits=50)
    assert p["splits"] == 3                                   # capped at the key tiles
    p = attn.plan(4, 16, 2048, 2048, 128, 152, max_ctas=5)
    assert p["grid"] == 5
    with pytest.raises(attn.AttnError):
        attn.plan(1, 1, 1, 1, 32)


def ex_args(q=P, k=2 * P, v=3 * P, o=4 * P, lse=0, B=1, H=2, Hkv=2, Sq=8, Skv=8, d=128, layout=0,
            mode=0, causal=0, reserved=0):
    a = attn.Args()
    a.q, a.k, a.v, a.o, a.lse = q, k, v, o, (lse or None)
    a.B, a.H, a.Hkv, a.Sq, a.Skv, a.d = B, H, Hkv, Sq, Skv, d
    a.layout, a.round_mode, a.causal, a.reserved = layout, mode, causal, reserved
    return a


def call_ex(lib, opts=None, **kw):
    return lib.attn_fwd_ex(ctypes.byref(ex_args(**kw)), ctypes.byref(opts) if opts else None,
                           None, 0, None)


@fake_pointers
def test_ex_argument_errors(lib):
    assert lib.attn_fwd_ex(None, None, None, 0, None) == 1
    assert call_ex(lib, q=0) == 1
    for kw in ({"Hkv": 0}, {"Hkv": 3, "H": 4}, {"Hkv": 4, "H": 2}, {"causal": 2},
               {"causal": -1}, {"reserved": 1}, {"layout": 5}, {"mode": 7}):
        assert call_ex(lib, **kw) == 1, kw
    assert call_ex(lib, d=48) == 2
    # causal with a forced key split is refused: the causal planner never splits
    assert call_ex(lib, causal=1, opts=attn.Options(3, 0, 0, 0)) == 2
    assert call_ex(lib, lse=5 * P + 2) == 3
    # lse [B*H*Sq] fp32 = 64 bytes: overlapping o, q or v is an alias
    assert call_ex(lib, lse=4 * P + 16) == 4
    assert call_ex(lib, lse=P + 2044) == 4
    assert call_ex(lib, lse=3 * P - 32) == 4
    # k, v hold B*Hkv*Skv*d elements: with Hkv=1 they end earlier, so o right after k fits
    assert call_ex(lib, H=2, Hkv=1, o=2 * P + 8 * 128 * 2, q=6 * P) != 4


@fake_pointers
def test_ex_valid_args_without_gpu_report_no_device(lib):
    assert call_ex(lib) == 5
    W = 1 << 24   # far apart: no overlap at this size
    assert call_ex(lib, q=W, k=2 * W, v=3 * W, o=4 * W, lse=5 * W, H=8, Hkv=1, causal=1, Sq=100,
                   Skv=300, layout=1, mode=2) == 5
    assert lib.attn_fwd_ex_workspace_size(ctypes.byref(ex_args()), None) == 0


@pytest.mark.parametrize("shape", PLAN_SHAPES)
def test_planner_ex_matches_plain_and_causal_never_splits(lib, shape):
    B, H, Sq, Skv = shape
    assert attn.plan_ex(B, H, Sq, Skv) == attn.plan(B, H, Sq, Skv)
    # grouped heads do not change the work split: units are query-head row tiles
    if H % 2 == 0:
        assert attn.plan_ex(B, H, Sq, Skv, Hkv=H // 2) == attn.plan(B, H, Sq, Skv)
    p = attn.plan_ex(B, H, Sq, Skv, causal=True)
    assert p["split_units"] == 0 and p["splits"] == 1 and p["workspace_bytes"] == 0
    assert p["full_items"] == p["units"] == B * H * -(-Sq // 256)
    assert 1 <= p["grid"] <= min(152, p["units"])
    with pytest.raises(attn.AttnError):
        attn.plan_ex(B, H, Sq, Skv, causal=True, force_splits=2)


@pytest.mark.parametrize("shape", PLAN_SHAPES)
def test_planner_head_dim_64(lib, shape):
    B, H, Sq, Skv = shape
    p128, p64 = attn.plan(B, H, Sq, Skv, 128), attn.plan(B, H, Sq, Skv, 64)
    # the work split does not depend on d; the split partials are d fp32 + 1 LSE per row
    assert {k: v for k, v in p64.items() if k != "workspace_bytes"} == \
           {k: v for k, v in p128.items() if k != "workspace_bytes"}
    assert p64["workspace_bytes"] == p64["split_units"] * p64["splits"] * 256 * (64 * 4 + 4)


@fake_pointers
def test_test_hooks_and_bwd_wait_limit_are_validated(lib):
    """The forward's test_hooks accepts 0 or ATTN_TEST_WITHHOLD_O_READY only; the backward's
    wait_limit_ms must be >= 0 and its test_hooks 0 or 1 (checked before any device call)."""
    pl = attn.Plan()
    o = attn.Options(0, 0, 0, 2)
    assert lib.attn_plan(1, 1, 8, 8, 128, 152, ctypes.byref(o), ctypes.byref(pl)) == 1
    o.test_hooks = 1
    assert lib.attn_plan(1, 1, 8, 8, 128, 152, ctypes.byref(o), ctypes.byref(pl)) == 0
    a = attn.BwdArgs()
    for i, n in enumerate(("q", "k", "v", "o", "dout", "lse", "dq", "dk", "dv")):
        setattr(a, n, (i + 1) * P)
    a.B, a.H, a.Hkv, a.Sq, a.Skv, a.d = 1, 1, 1, 8, 8, 128
    ws = 16 * P
    for bad in ({"wait_limit_ms": -1}, {"test_hooks": 2}, {"test_hooks": -1}, {"deterministic": 2},
                {"deterministic": -1}):
        a.wait_limit_ms, a.test_hooks, a.deterministic = 0, 0, 0
        for k_, v_ in bad.items():
            setattr(a, k_, v_)
        assert lib.attn_bwd(ctypes.byref(a), ws, 1 << 20, None) == 1, bad
        assert lib.attn_bwd_workspace_size(ctypes.byref(a)) == 0, bad
    a.wait_limit_ms, a.test_hooks, a.deterministic = 50, 1, 1
    assert lib.attn_bwd_workspace_size(ctypes.byref(a)) > 0


def test_bwd_workspace_size_deterministic(lib):
    """The deterministic backward holds one fp32 dQ slice per 128-key tile where the default
    mode holds one accumulator; the per-row statistics are the same.  (No device here, so no
    tail split and no dK/dV partials.)"""
    a = attn.BwdArgs()
    a.B, a.H, a.Hkv, a.Sq, a.Skv, a.d = 2, 4, 2, 300, 700, 128
    rows_pad = 2 * 4 * 384
    dq = 2 * 4 * 300 * 128 * 4
    assert lib.attn_bwd_workspace_size(ctypes.byref(a)) == dq + 2 * rows_pad * 4
    a.deterministic = 1
    assert lib.attn_bwd_workspace_size(ctypes.byref(a)) == 6 * dq + 2 * rows_pad * 4
    a.Skv, a.d = 128, 64
    assert lib.attn_bwd_workspace_size(ctypes.byref(a)) == dq // 2 + 2 * rows_pad * 4


def varlen_args(**kw):
    a = attn.VarlenArgs()
    a.q, a.k, a.v, a.o = P, 2 * P, 3 * P, 4 * P
    a.cu_seqlens_q, a.cu_seqlens_k = 5 * P, 6 * P
    a.B, a.H, a.Hkv, a.total_q, a.total_k, a.max_seqlen_q, a.d = 2, 2, 1, 16, 16, 0, 128
    for k_, v_ in kw.items():
        setattr(a, k_, v_)
    return a


@fake_pointers
def test_varlen_argument_errors(lib):
    """attn_fwd_varlen checks its arguments before any device call: bad sizes or enums are
    ATTN_ERR_INVALID_ARG, d not 64/128, a key split or int32 overflow ATTN_ERR_UNSUPPORTED,
    unaligned pointers ATTN_ERR_MISALIGNED and an output overlapping an input ATTN_ERR_ALIAS;
    valid arguments get as far as the device query (no GPU here: ATTN_ERR_NO_DEVICE)."""
    def run(opts=None, **kw):
        return lib.attn_fwd_varlen(ctypes.byref(varlen_args(**kw)), ctypes.byref(opts) if opts else None,
                                   None, 0, None)
    assert lib.attn_fwd_varlen(None, None, None, 0, None) == 1
    assert run() == 5
    assert run(B=3, total_q=0, total_k=0, max_seqlen_q=7, d=64) == 5
    for bad in ({"B": 0}, {"Hkv": 3}, {"total_q": -1}, {"total_k": -1}, {"max_seqlen_q": -1},
                {"round_mode": 3}, {"causal": 2}, {"max_splits": -1}, {"pack_heads": 2},
                {"cu_seqlens_q": 0}, {"cu_seqlens_k": 0}, {"q": 0}, {"o": 0}):
        assert run(**bad) == 1, bad
    assert run(d=96) == 2
    assert run(total_q=(1 << 30) + 1) == 2
    # packed heads: H / Hkv a power of two of at most 32
    assert run(pack_heads=1) == 5
    assert run(pack_heads=1, H=32, Hkv=1) == 5
    assert run(pack_heads=1, H=6, Hkv=2) == 2
    assert run(pack_heads=1, H=64, Hkv=1) == 2
    # key splits: any count >= 0 (0 and 1: none)
    for n in (0, 1, 2, 64, 1 << 20):
        assert run(max_splits=n) == 5, n
    assert run(opts=attn.Options(2, 0, 0, 0)) == 2
    assert run(opts=attn.Options(1, 0, 0, 0)) == 5
    assert run(opts=attn.Options(0, 0, 0, 1)) == 1
    assert run(q=P + 8) == 3
    assert run(cu_seqlens_k=6 * P + 2) == 3
    assert run(lse=7 * P + 2) == 3
    assert run(o=P) == 4
    assert run(lse=4 * P + 64) == 4


def test_varlen_workspace_size(lib):
    """Per-sequence tensor maps (4 x 128 bytes), the item count (16 bytes) and room for every
    (sequence, 256-row query block) pair (16 bytes each, at most total_q / 256 + B of them),
    plus alignment room.  With key splits the size depends on the device's SM count: with no
    device it is 0."""
    for B, total_q in ((1, 16), (2, 16), (7, 5000), (1000, 1 << 20)):
        a = varlen_args(B=B, total_q=total_q)
        want = 128 + B * 512 + 16 + (total_q // 256 + B) * 16
        assert lib.attn_fwd_varlen_workspace_size(ctypes.byref(a)) == want, B
    assert lib.attn_fwd_varlen_workspace_size(ctypes.byref(varlen_args(B=0))) == 0
    assert lib.attn_fwd_varlen_workspace_size(None) == 0
    # with packed heads (here 2 per K/V head) a block holds 128 tokens: room for more pairs
    a = varlen_args(B=7, total_q=5000, pack_heads=1)
    assert lib.attn_fwd_varlen_workspace_size(ctypes.byref(a)) == 128 + 7 * 512 + 16 + (5000 // 128 + 7) * 16
    a = varlen_args(B=7, total_q=5000, max_splits=1)
    assert lib.attn_fwd_varlen_workspace_size(ctypes.byref(a)) == 128 + 7 * 512 + 16 + (5000 // 256 + 7) * 16
    a = varlen_args(B=7, total_q=5000, max_splits=2)
    got = lib.attn_fwd_varlen_workspace_size(ctypes.byref(a))
    if torch.cuda.is_available():
        sms = torch.cuda.get_device_properties(0).multi_processor_count
        base = 128 + 7 * 512 + 16 + max(5000 // 256 + 7, 2 * sms) * 16
        assert got == -(-base // 256) * 256 + 2 * sms * 256 * 129 * 4
    else:
        assert got == 0


PG = 1 << 24   # fake pointers for the paged calls, far enough apart for their cache sizes


def paged_args(**kw):
    a = attn.PagedArgs()
    a.q, a.k_cache, a.v_cache, a.o = PG, 2 * PG, 3 * PG, 4 * PG
    a.cu_seqlens_q, a.seqlens_k, a.block_table = 5 * PG, 6 * PG, 7 * PG
    a.B, a.H, a.Hkv, a.total_q, a.num_pages, a.page_size, a.max_pages, a.max_seqlen_q, a.d = \
        2, 2, 1, 16, 4, 128, 2, 0, 128
    for k_, v_ in kw.items():
        setattr(a, k_, v_)
    return a


@fake_pointers
def test_paged_argument_errors(lib):
    """attn_fwd_paged checks its arguments before any device call, as attn_fwd_varlen does,
    plus the cache geometry: at least one page, a page size that is a positive multiple of 128,
    at least one page per sequence in the table, and int32-safe sizes."""
    def run(**kw):
        return lib.attn_fwd_paged(ctypes.byref(paged_args(**kw)), None, None, 0, None)
    assert lib.attn_fwd_paged(None, None, None, 0, None) == 1
    assert run() == 5
    assert run(page_size=256, d=64, causal=1) == 5
    for bad in ({"num_pages": 0}, {"page_size": 0}, {"page_size": 64}, {"page_size": 200}, {"max_pages": 0},
                {"seqlens_k": 0}, {"block_table": 0}, {"cu_seqlens_q": 0}, {"k_cache": 0}, {"B": 0},
                {"Hkv": 3}, {"max_splits": -1}):
        assert run(**bad) == 1, bad
    assert run(max_pages=(1 << 23) + 1) == 2
    assert run(num_pages=(1 << 23) + 1) == 2
    assert run(block_table=7 * PG + 2) == 3
    assert run(o=2 * PG + 4096) == 4     # o overlaps the K cache


def test_paged_workspace_size(lib):
    a = paged_args(B=3, total_q=1000)
    assert lib.attn_fwd_paged_workspace_size(ctypes.byref(a)) == 128 + 3 * 512 + 16 + (1000 // 256 + 3) * 16
    assert lib.attn_fwd_paged_workspace_size(ctypes.byref(paged_args(page_size=100))) == 0


def bwd_varlen_args(**kw):
    a = attn.BwdVarlenArgs()
    for i, n in enumerate(("q", "k", "v", "o", "dout", "lse", "dq", "dk", "dv", "cu_seqlens_q", "cu_seqlens_k")):
        setattr(a, n, (i + 1) * PG)
    a.B, a.H, a.Hkv, a.total_q, a.total_k, a.d = 3, 4, 2, 1000, 900, 128
    for k_, v_ in kw.items():
        setattr(a, k_, v_)
    return a


@fake_pointers
def test_bwd_varlen_argument_errors_and_workspace(lib):
    """attn_bwd_varlen checks its arguments before any device call; its workspace holds the
    fp32 dQ accumulator [H][total_q][d], the padded row statistics (two fp32 per head and
    padded row, rows rounded up per sequence: total_q + 127 B, to a multiple of 128), seven
    tensor maps per sequence (128-byte aligned), the unit count and padded offsets, and one
    16-byte unit per (K/V head, key tile) it can hold."""
    ws = 20 * PG
    def run(**kw):
        return lib.attn_bwd_varlen(ctypes.byref(bwd_varlen_args(**kw)), ws, 1 << 30, None)
    assert lib.attn_bwd_varlen(None, ws, 1 << 30, None) == 1
    assert run() == 5
    for bad in ({"B": 0}, {"Hkv": 3}, {"total_q": -1}, {"total_k": -1}, {"causal": 2}, {"wait_limit_ms": -1},
                {"reserved": 1}, {"reserved2": 1}, {"q": 0}, {"lse": 0}, {"cu_seqlens_k": 0}, {"dk": 0}):
        assert run(**bad) == 1, bad
    assert run(d=96) == 2
    assert run(total_q=(1 << 30) + 1) == 2
    assert run(q=PG + 8) == 3
    assert run(cu_seqlens_q=10 * PG + 2) == 3
    assert run(dq=PG + 4096) == 4
    assert lib.attn_bwd_varlen(ctypes.byref(bwd_varlen_args()), ws, 16, None) == 6
    a = bwd_varlen_args()
    sp = -(-(1000 + 127 * 3) // 128) * 128
    maps = -(-(4 * 1000 * 128 * 4 + 2 * 4 * sp * 4) // 128) * 128
    misc = maps + 7 * 3 * 128
    units = misc + -(-(3 + 2) // 4) * 16
    assert lib.attn_bwd_varlen_workspace_size(ctypes.byref(a)) == units + 2 * (900 // 128 + 3) * 16
    assert lib.attn_bwd_varlen_workspace_size(ctypes.byref(bwd_varlen_args(d=32))) == 0
