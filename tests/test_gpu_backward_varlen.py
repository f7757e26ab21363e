"""GPU parity of the variable-length backward (attn_bwd_varlen) against the fp64 oracle
(needs a GB300).

Each sequence's gradients are those of its own attention problem; the criteria are the dense
backward's (|gpu - oracle| <= 2^-7 * A + ulp per element).  The backward kernel runs each
sequence's units with tensor maps narrowed to its rows, so dK and dV of a sequence are bit for
bit those of the dense backward on that sequence alone (same tiles, same step order), and
nothing in other sequences, non-finite values included, can reach them.
"""
import ctypes

import numpy as np
import pytest
import torch

import oracle
from tests import parity
from tests.test_gpu_canaries import guarded, guards_intact
from tests.test_gpu_varlen import offsets, packed

pytestmark = pytest.mark.gpu

BF16_SENTINEL = 0x7BAD
SITE_SEQLENS = 16


@pytest.fixture(scope="module")
def attn():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import bf16_attention_forward_gb300 as a
    a.load()
    return a


def forward(attn, q, k, v, cq, ck, causal):
    o, lse = attn.attn_fwd_varlen(q, k, v, cq, ck, causal=causal, return_lse=True)
    return o, lse


def run_bwd(attn, q, k, v, g, cu_q, cu_k, causal, sentinel=True):
    qd, kd, vd, gd = (t.cuda() for t in (q, k, v, g))
    cq, ck = (torch.as_tensor(np.asarray(c, dtype=np.int32)).cuda() for c in (cu_q, cu_k))
    o, lse = forward(attn, qd, kd, vd, cq, ck, causal)
    outs = [torch.empty_like(t) for t in (qd, kd, vd)]
    if sentinel:
        for t in outs:
            t.view(torch.int16).fill_(BF16_SENTINEL)
    attn.attn_bwd_varlen(qd, kd, vd, o, gd, lse, cq, ck, causal=causal, dq=outs[0], dk=outs[1], dv=outs[2])
    torch.cuda.synchronize()
    return outs


def status_ok(attn):
    assert attn.device_status()[0] == 0
    st, site = attn.bwd_device_status()
    assert st == 0, "backward device status %d at site %d" % (st, site)


def _bits(t):
    return t.cpu().view(torch.int16).numpy().view(np.uint16)


def check(attn, q, k, v, g, cu_q, cu_k, causal=False):
    dq, dk, dv = run_bwd(attn, q, k, v, g, cu_q, cu_k, causal)
    status_ok(attn)
    ref = oracle.backward_varlen(q, k, v, g, cu_q, cu_k, causal=causal, want_a=True)
    for name, got, cov in (("dq", dq, ref["covered_q"]), ("dk", dk, ref["covered_k"]), ("dv", dv, ref["covered_k"])):
        gb = _bits(got)
        assert (gb[~cov] == BF16_SENTINEL).all(), name + ": a row outside every sequence was written"
        gb = gb[cov].reshape(-1)
        r = ref[name][cov].reshape(-1)
        a = ref[name + "_a"][cov].reshape(-1)
        rb = ref[name + "_bits"][cov].reshape(-1).astype(np.uint16)
        err = np.abs(parity.bits_to_f64(gb) - r)
        tol = 2.0 ** -7 * a + parity.bf16_ulp(rb)
        bad = ~(err <= tol)
        assert not bad.any(), (name, int(bad.sum()))
    return dq, dk, dv


MIXES = [  # (lens_q, lens_k, H, Hkv, d, causal)
    ([300, 1, 128, 129], None, 4, 2, 128, False),
    ([300, 1, 128, 129], None, 4, 2, 128, True),
    ([257, 64, 500], [513, 1, 200], 2, 2, 64, True),
    ([100, 0, 70, 200], [130, 90, 0, 256], 2, 1, 128, False),     # no queries / no keys
]


@pytest.mark.parametrize("mix", MIXES, ids=lambda m: "n%d_H%dKV%d_d%d%s" % (len(m[0]), m[2], m[3], m[4],
                                                                             "_causal" if m[5] else ""))
def test_varlen_backward_matches_oracle(attn, mix):
    lq, lk, H, Hkv, d, causal = mix
    lk = lq if lk is None else lk
    q, k, v = packed(sum(lq), sum(lk), H, Hkv, d, seed=9500 + sum(lq))
    g = packed(sum(lq), 1, H, H, d, seed=9501)[0]
    check(attn, q, k, v, g, offsets(lq), offsets(lk), causal)


@pytest.mark.parametrize("causal", [False, True])
def test_varlen_backward_dk_dv_equal_dense_per_sequence(attn, causal):
    # 6 query steps or fewer per unit, so the dense call on one sequence does not split units
    lq = [300, 129, 384, 200]
    lk = lq if causal else [200, 700, 131, 1000]
    H, Hkv, d = 4, 2, 128
    q, k, v = packed(sum(lq), sum(lk), H, Hkv, d, seed=9600 + causal)
    g = packed(sum(lq), 1, H, H, d, seed=9601)[0]
    cu_q, cu_k = offsets(lq), offsets(lk)
    dq, dk, dv = run_bwd(attn, q, k, v, g, cu_q, cu_k, causal)
    status_ok(attn)
    for b in range(len(lq)):
        qs, ks, vs, gs = (t[c[b]:c[b + 1]][None].cuda() for t, c in ((q, cu_q), (k, cu_k), (v, cu_k), (g, cu_q)))
        o, lse = attn.attn_fwd_ex(qs, ks, vs, layout="bshd", causal=causal, return_lse=True, force_splits=1)
        _, dk1, dv1 = attn.attn_bwd(qs, ks, vs, o, gs, lse, layout="bshd", causal=causal)
        torch.cuda.synchronize()
        assert torch.equal(dk[cu_k[b]:cu_k[b + 1]].view(torch.int16), dk1[0].view(torch.int16)), b
        assert torch.equal(dv[cu_k[b]:cu_k[b + 1]].view(torch.int16), dv1[0].view(torch.int16)), b


def test_varlen_backward_neighbours_do_not_leak(attn):
    lq, lk = [200, 150, 260], [250, 129, 300]
    H, d = 2, 128
    q, k, v = packed(sum(lq), sum(lk), H, H, d, seed=9700)
    g = packed(sum(lq), 1, H, H, d, seed=9701)[0]
    cu_q, cu_k = offsets(lq), offsets(lk)
    _, dk0, dv0 = run_bwd(attn, q, k, v, g, cu_q, cu_k, True)
    status_ok(attn)
    q2, k2, v2, g2 = q.clone(), k.clone(), v.clone(), g.clone()
    for t, cu in ((q2, cu_q), (k2, cu_k), (v2, cu_k), (g2, cu_q)):
        rows = t[cu[1]:cu[3]]
        rows.view(torch.int16)[::2] = 0x7F80
        rows.view(torch.int16)[1::3] = 0x7FC1
    _, dk1, dv1 = run_bwd(attn, q2, k2, v2, g2, cu_q, cu_k, True)
    status_ok(attn)
    r = slice(cu_k[0], cu_k[1])
    assert torch.equal(dk1[r].view(torch.int16), dk0[r].view(torch.int16))
    assert torch.equal(dv1[r].view(torch.int16), dv0[r].view(torch.int16))


def test_varlen_backward_writes_stay_in_bounds(attn):
    lq, lk, H, d = [130, 1, 77], [200, 5, 129], 2, 64
    q, k, v = packed(sum(lq), sum(lk), H, H, d, seed=9800)
    g = packed(sum(lq), 1, H, H, d, seed=9801)[0]
    qd, kd, vd, gd = (t.cuda() for t in (q, k, v, g))
    cq, ck = (torch.as_tensor(offsets(x)).cuda() for x in (lq, lk))
    o, lse = forward(attn, qd, kd, vd, cq, ck, False)
    bufs = [guarded(t.numel(), "bf16") for t in (qd, kd, vd)]
    a = attn.BwdVarlenArgs()
    a.B, a.H, a.Hkv, a.total_q, a.total_k, a.d = len(lq), H, H, q.shape[0], k.shape[0], d
    wbytes = int(attn.load().attn_bwd_varlen_workspace_size(ctypes.byref(a)))
    wbuf, ws = guarded(wbytes, "ws")
    attn.attn_bwd_varlen(qd, kd, vd, o, gd, lse, cq, ck, dq=bufs[0][1].view(q.shape), dk=bufs[1][1].view(k.shape),
                         dv=bufs[2][1].view(v.shape), workspace=ws)
    torch.cuda.synchronize()
    status_ok(attn)
    for buf, view in bufs:
        assert guards_intact(buf, "bf16")
        assert not (view.view(torch.int16) == 0x7BAD).any()
    assert guards_intact(wbuf, "ws")


def test_varlen_backward_bad_offsets_are_reported_and_write_nothing(attn):
    lq = [100, 60, 140]
    q, k, v = packed(sum(lq), sum(lq), 2, 2, 128, seed=9900)
    g = packed(sum(lq), 1, 2, 2, 128, seed=9901)[0]
    qd, kd, vd, gd = (t.cuda() for t in (q, k, v, g))
    cu = torch.as_tensor(offsets(lq)).cuda()
    o, lse = forward(attn, qd, kd, vd, cu, cu, False)
    bad = cu.clone()
    bad[2] = bad[1] - 1
    outs = [torch.empty_like(t) for t in (qd, kd, vd)]
    for t in outs:
        t.view(torch.int16).fill_(BF16_SENTINEL)
    attn.attn_bwd_varlen(qd, kd, vd, o, gd, lse, bad, cu, dq=outs[0], dk=outs[1], dv=outs[2])
    torch.cuda.synchronize()
    assert attn.bwd_device_status() == (1, SITE_SEQLENS)
    for t in outs:
        assert (t.view(torch.int16) == BF16_SENTINEL).all()
    check(attn, q, k, v, g, offsets(lq), offsets(lq))
