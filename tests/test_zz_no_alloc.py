"""attn_fwd_noalloc (the entry point for callers that cannot allocate device memory) gives
the same results as attn_fwd, through the C ABI, on two calls in a row.

Callers that cannot let a library allocate -- code recording a CUDA graph, programs whose
device memory all belongs to their own allocator or a fixed budget -- use attn_fwd_noalloc,
which keeps the split path's partial results in a scratch array compiled into the library.
The shapes below make the planner split keys, so the scratch is really used; the second call
runs on the scratch the first call left behind.  This file is collected last on purpose.
"""
import ctypes

import numpy as np
import pytest
import torch

from workloads import make_qkv

pytestmark = pytest.mark.gpu

LAYOUT = {"bshd": 0, "bhsd": 1}
MODE = {"rtne": 0, "rtna": 1, "rtz": 2}


@pytest.fixture(scope="module")
def lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from bf16_attention_forward_gb300 import build as libbuild
    libbuild.build()
    import bf16_attention_forward_gb300 as attn
    return attn.load()


def _dims(q, k, layout):
    if layout == "bshd":
        return q.shape[0], q.shape[2], q.shape[1], k.shape[1], q.shape[3]
    return q.shape[0], q.shape[1], q.shape[2], k.shape[2], q.shape[3]


def _call(fn, q, k, v, o, layout, mode):
    B, H, Sq, Skv, d = _dims(q, k, layout)
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    return fn(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), B, H, Sq, Skv, d,
              LAYOUT[layout], MODE[mode], stream)


def _bits(o):
    return o.detach().cpu().contiguous().view(torch.int16).numpy().view(np.uint16).reshape(-1)


@pytest.mark.parametrize("shape,layout,mode", [
    ((1, 2, 300, 5000), "bhsd", "rtne"),      # 4 units on 152 SMs: keys split 10 ways
    ((1, 8, 128, 20000), "bshd", "rtz"),
    ((2, 3, 700, 3000), "bshd", "rtna"),
])
def test_noalloc_matches_attn_fwd_twice(lib, shape, layout, mode):
    """Same plan and kernels as attn_fwd, and the forward is deterministic: the bits must be
    identical.  The output also meets the parity criteria against the oracle, and free device
    memory does not move across the two calls (after a warm-up call that may look up the
    scratch array's device address)."""
    import bf16_attention_forward_gb300 as attn
    import oracle
    from tests import parity
    B, H, Sq, Skv = shape
    plan = attn.plan(B, H, Sq, Skv, 128, torch.cuda.get_device_properties(0).multi_processor_count)
    assert plan["split_units"] > 0, plan                     # the scratch is exercised
    q, k, v = make_qkv(B, H, Sq, Skv, 128, layout, seed=sum(shape))
    qd, kd, vd = (t.cuda() for t in (q, k, v))
    ref = torch.empty_like(qd)
    outs = [torch.empty_like(qd) for _ in range(2)]
    assert _call(lib.attn_fwd, qd, kd, vd, ref, layout, mode) == 0
    assert _call(lib.attn_fwd_noalloc, qd, kd, vd, outs[0], layout, mode) == 0   # warm-up
    for o in outs:
        o.fill_(float("nan"))
    torch.cuda.synchronize()
    free_before = torch.cuda.mem_get_info()[0]
    for o in outs:
        assert _call(lib.attn_fwd_noalloc, qd, kd, vd, o, layout, mode) == 0
    torch.cuda.synchronize()
    assert torch.cuda.mem_get_info()[0] == free_before
    st = ctypes.c_int32(0)
    assert lib.attn_get_device_status(ctypes.c_void_p(torch.cuda.current_stream().cuda_stream),
                                      ctypes.byref(st)) == 0
    r = _bits(ref)
    for o in outs:
        assert np.array_equal(_bits(o), r)
    want = oracle.attention(q, k, v, layout, mode, want_a=True)
    res = parity.compare(parity.gpu_rows_bits(outs[1], layout), want["o_bits"], want["a"])
    assert res["ok"], res


def test_noalloc_rejects_bad_arguments(lib):
    q, k, v = (t.cuda() for t in make_qkv(1, 1, 8, 8, 128, "bhsd", seed=1))
    o = torch.empty_like(q)
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    assert lib.attn_fwd_noalloc(None, k.data_ptr(), v.data_ptr(), o.data_ptr(), 1, 1, 8, 8, 128,
                                1, 0, stream) == 1
    assert lib.attn_fwd_noalloc(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), 1, 1, 8,
                                8, 96, 1, 0, stream) == 2
    assert lib.attn_fwd_noalloc(q.data_ptr(), k.data_ptr(), v.data_ptr(), q.data_ptr(), 1, 1, 8,
                                8, 128, 1, 0, stream) == 4
