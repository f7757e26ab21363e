"""Stream order across calls (needs a GB300).

Every kernel of a call is launched as a programmatic dependent of the kernel before it in the
stream: it may start while that kernel is still running and waits for its memory before it
reads or writes global memory.  The attention kernel lets its dependents launch as soon as
its CTAs start, so the next call's kernels really do run early.  These tests chain calls
back to back on one stream, each reading what the previous one wrote (as Q, K, V, O, dO or the
LSE), with no synchronisation in between, and then check every output bit for bit against
the same call re-run once its inputs have settled.  The forward, the backward's dK and dV, and
the deterministic backward's dQ are reproducible bit for bit, so any read of a stale or
half-written input shows up as a mismatch.
"""
import pytest
import torch

from workloads import make_qkv

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def attn():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import bf16_attention_forward_gb300 as a
    a.load()
    return a


def bits(t):
    return t.view(torch.int16)


def check_status(attn):
    torch.cuda.synchronize()
    st, site = attn.device_status()
    assert st == 0, (st, site)


# (B, H, S, d, layout): the split path with its combine kernel, the plain persistent path, the
# short-query kernel, and head dimension 64
SHAPES = [(1, 5, 1024, 128, "bhsd"), (2, 8, 512, 128, "bshd"), (2, 8, 128, 128, "bshd"),
          (2, 8, 512, 64, "bhsd")]


@pytest.mark.parametrize("shape", SHAPES, ids=lambda s: "B%dH%dS%dd%d%s" % s)
def test_forward_chain_reads_settled_inputs(attn, shape):
    B, H, S, d, layout = shape
    q, k, v = (t.cuda() for t in make_qkv(B, H, S, S, d, layout, seed=4100 + S + d))
    n = 9
    outs = [torch.empty_like(q) for _ in range(n)]
    ins = []
    x = q
    for i in range(n):
        # the previous output becomes Q, K or V of the next call, in turn
        args = (x, k, v) if i % 3 == 0 else (q, x, v) if i % 3 == 1 else (q, k, x)
        attn.attn_fwd(*args, o=outs[i], layout=layout)
        ins.append(args)
        x = outs[i]
    check_status(attn)
    for i in range(n):
        again = attn.attn_fwd(*ins[i], layout=layout)
        torch.cuda.synchronize()
        assert torch.equal(bits(again), bits(outs[i])), "call %d read an unsettled input" % i


def test_forward_writes_do_not_overtake_readers(attn):
    # a call whose output buffer the previous call still reads (its V): the later call must
    # not write O before the earlier one is done with it
    B, H, S, d, layout = 2, 8, 512, 128, "bshd"
    q, k, v = (t.cuda() for t in make_qkv(B, H, S, S, d, layout, seed=4200))
    buf = v.clone()
    first = torch.empty_like(q)
    attn.attn_fwd(q, k, buf, o=first, layout=layout)      # reads buf as V
    attn.attn_fwd(k, q, v, o=buf, layout=layout)          # overwrites buf
    check_status(attn)
    want_first = attn.attn_fwd(q, k, v, layout=layout)
    want_second = attn.attn_fwd(k, q, v, layout=layout)
    torch.cuda.synchronize()
    assert torch.equal(bits(first), bits(want_first))
    assert torch.equal(bits(buf), bits(want_second))


@pytest.mark.parametrize("det", [False, True], ids=["acc", "det"])
@pytest.mark.parametrize("d", [128, 64])
def test_backward_between_forward_calls(attn, d, det):
    # forward -> backward (its O, LSE and dO come from the forward calls just before) ->
    # forward on the backward's dK (as Q) and dQ (as V)
    B, H, S, layout = 1, 4, 640, "bshd"
    q, k, v = (t.cuda() for t in make_qkv(B, H, S, S, d, layout, seed=4300 + d))
    q2 = make_qkv(B, H, S, S, d, layout, seed=4400 + d)[0].cuda()
    o, lse = attn.attn_fwd_ex(q, k, v, layout=layout, return_lse=True)
    g = attn.attn_fwd(q2, k, v, layout=layout)
    dq, dk, dv = attn.attn_bwd(q, k, v, o, g, lse, layout=layout, deterministic=det)
    o3 = attn.attn_fwd(dk, k, v, layout=layout)
    o4 = attn.attn_fwd(q, k, dq, layout=layout)
    check_status(attn)
    assert attn.bwd_device_status() == (0, 0)
    o_ref, lse_ref = attn.attn_fwd_ex(q, k, v, layout=layout, return_lse=True)
    g_ref = attn.attn_fwd(q2, k, v, layout=layout)
    torch.cuda.synchronize()
    assert torch.equal(bits(o), bits(o_ref)) and torch.equal(bits(g), bits(g_ref))
    assert torch.equal(lse.view(torch.int32), lse_ref.view(torch.int32))
    dq_ref, dk_ref, dv_ref = attn.attn_bwd(q, k, v, o, g, lse, layout=layout, deterministic=det)
    torch.cuda.synchronize()
    assert torch.equal(bits(dk), bits(dk_ref)) and torch.equal(bits(dv), bits(dv_ref))
    if det:
        assert torch.equal(bits(dq), bits(dq_ref)), "deterministic dQ read an unsettled input"
    o3_ref = attn.attn_fwd(dk, k, v, layout=layout)
    o4_ref = attn.attn_fwd(q, k, dq, layout=layout)
    torch.cuda.synchronize()
    assert torch.equal(bits(o3), bits(o3_ref)), "forward read dK before the backward finished"
    assert torch.equal(bits(o4), bits(o4_ref)), "forward read dQ before the backward finished"


def test_varlen_calls_chained_on_one_workspace(attn):
    # back-to-back variable-length calls with different offsets on one workspace: each call's
    # preprocessing rewrites the tensor maps and the work list that the previous call's
    # attention kernel reads (it waits for that kernel first), and each call reads the
    # previous call's output as its Q
    import ctypes
    import numpy as np
    H, d, T = 4, 128, 1300
    mixes = [[300, 129, 700], [1, 1000, 64, 200], [512, 512], [77, 900, 3, 5, 250, 1]]
    q, k, v = (t[0].contiguous().cuda() for t in make_qkv(1, H, T, T, d, "bshd", seed=4500))
    a = attn.VarlenArgs()
    a.B, a.H, a.Hkv, a.total_q, a.total_k, a.d = max(len(m) for m in mixes), H, H, T, T, d
    ws = torch.empty(int(attn.load().attn_fwd_varlen_workspace_size(ctypes.byref(a))), dtype=torch.uint8,
                     device="cuda")
    cus = [torch.as_tensor(np.cumsum([0] + m).astype(np.int32)).cuda() for m in mixes]
    outs, ins = [], []
    x = q
    for i, cu in enumerate(cus):
        o = torch.zeros_like(q)
        attn.attn_fwd_varlen(x, k, v, cu, cu, o=o, causal=bool(i & 1), workspace=ws)
        outs.append(o)
        ins.append(x)
        x = o
    check_status(attn)
    for i, cu in enumerate(cus):
        o = torch.zeros_like(q)
        attn.attn_fwd_varlen(ins[i], k, v, cu, cu, o=o, causal=bool(i & 1))
        torch.cuda.synchronize()
        assert torch.equal(bits(o), bits(outs[i])), "call %d read a stale map, list or input" % i
