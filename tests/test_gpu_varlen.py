"""GPU parity of the variable-length forward (attn_fwd_varlen) against the fp64 oracle
(needs a GB300).

B sequences packed along the token axis, each an attention problem of its own (the MoonMath
page's limitations paragraph names variable-length batching).  Every covered output element
must meet the forward's criteria (within 2 bf16 ULP of the oracle or its forward-error bound,
non-finite values bitwise equal) and the LSE the extended forward's tolerance; rows outside
every sequence, and every byte around the outputs, must stay unwritten.  The kernel gives
each sequence tensor maps of its own, so a tile at a sequence's end reads zeros, not the next
sequence: a sequence's outputs are bit for bit those of the dense kernel on the sequence
alone, and non-finite values in its neighbours cannot reach it.
"""
import ctypes

import numpy as np
import pytest
import torch

import oracle
from tests import parity
from tests.test_gpu_canaries import guarded, guards_intact
from tests.test_gpu_causal_gqa import abs_logit_scale, check_lse
from workloads import make_qkv

pytestmark = pytest.mark.gpu

BF16_SENTINEL = 0x7BAD
F32_SENTINEL = 0x7F7BAD01
SITE_SEQLENS = 13


@pytest.fixture(scope="module")
def attn():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import bf16_attention_forward_gb300 as a
    a.load()
    return a


def packed(Tq, Tk, H, Hkv, d, seed, sigma=1.0):
    q, k, v = make_qkv(1, H, Tq, Tk, d, "bshd", seed=seed, sigma=sigma, Hkv=Hkv)
    return q[0].contiguous(), k[0].contiguous(), v[0].contiguous()


def offsets(lens, start=0):
    return np.cumsum([start] + list(lens)).astype(np.int32)


def run_varlen(attn, q, k, v, cu_q, cu_k, mode="rtne", causal=False, **kw):
    qd, kd, vd = (t.cuda() for t in (q, k, v))
    o = torch.empty_like(qd)
    o.view(torch.int16).fill_(BF16_SENTINEL)
    lse = torch.empty((q.shape[1], q.shape[0]), dtype=torch.float32, device="cuda")
    lse.view(torch.int32).fill_(F32_SENTINEL)
    cq = torch.as_tensor(np.asarray(cu_q, dtype=np.int32)).cuda()
    ck = torch.as_tensor(np.asarray(cu_k, dtype=np.int32)).cuda()
    attn.attn_fwd_varlen(qd, kd, vd, cq, ck, o=o, lse=lse, round=mode, causal=causal, **kw)
    torch.cuda.synchronize()
    return o, lse


def status_ok(attn):
    st, site = attn.device_status()
    assert st == 0, "device status %d at site %d" % (st, site)


def lse_scale(q, k, cu_q, cu_k):
    """A_i per [H, Tq] row: the largest |q_i|.|k_j| sum over the sequence's keys / sqrt(d)."""
    H, Tq = q.shape[1], q.shape[0]
    out = np.zeros((H, Tq))
    for b in range(len(cu_q) - 1):
        q0, q1, k0, k1 = (int(x) for x in (cu_q[b], cu_q[b + 1], cu_k[b], cu_k[b + 1]))
        if q1 > q0 and k1 > k0:
            out[:, q0:q1] = abs_logit_scale(q[None, q0:q1], k[None, k0:k1], "bshd").reshape(H, q1 - q0)
    return out


def check_varlen(attn, q, k, v, cu_q, cu_k, mode="rtne", causal=False, **kw):
    o, lse = run_varlen(attn, q, k, v, cu_q, cu_k, mode, causal, **kw)
    status_ok(attn)
    ref = oracle.attention_varlen(q, k, v, cu_q, cu_k, mode, causal=causal, want_a=True, want_lse=True)
    cov = ref["covered"]
    ob = o.cpu().view(torch.int16).numpy().view(np.uint16)
    res = parity.compare(ob[cov].reshape(-1, q.shape[2]), ref["o_bits"][cov].reshape(-1, q.shape[2]),
                         ref["a"][cov].reshape(-1, q.shape[2]))
    assert res["ok"], res
    assert (ob[~cov] == BF16_SENTINEL).all(), "a row outside every sequence was written"
    lg = lse.cpu().numpy()
    assert (lg[:, ~cov].view(np.int32) == F32_SENTINEL).all(), "an LSE row outside every sequence was written"
    check_lse(lg[:, cov].reshape(-1), ref["lse"][:, cov].reshape(-1), lse_scale(q, k, cu_q, cu_k)[:, cov].reshape(-1))
    return o, lse


MIXES = [  # (lens_q, lens_k, H, Hkv, d, mode, causal)
    ([300, 1, 128, 129, 700], None, 4, 2, 128, "rtne", False),
    ([300, 1, 128, 129, 700], None, 4, 2, 128, "rtne", True),
    ([257, 64, 1000], [513, 1, 200], 2, 2, 64, "rtna", True),
    ([257, 64, 1000], [513, 1, 200], 2, 2, 64, "rtz", False),
    ([5, 255, 256, 511], [600, 3, 256, 90], 3, 1, 128, "rtz", True),
]


@pytest.mark.parametrize("mix", MIXES, ids=lambda m: "n%d_H%dKV%d_d%d_%s%s" % (len(m[0]), m[2], m[3], m[4], m[5],
                                                                                "_causal" if m[6] else ""))
def test_varlen_matches_oracle(attn, mix):
    lq, lk, H, Hkv, d, mode, causal = mix
    lk = lq if lk is None else lk
    q, k, v = packed(sum(lq), sum(lk), H, Hkv, d, seed=8000 + sum(lq) + d)
    check_varlen(attn, q, k, v, offsets(lq), offsets(lk), mode, causal)


@pytest.mark.parametrize("causal", [False, True])
def test_varlen_random_lengths(attn, causal):
    rng = np.random.default_rng(8100 + causal)
    B = 12
    lq = rng.integers(1, 700, B).tolist()
    lk = lq if causal else rng.integers(1, 900, B).tolist()
    q, k, v = packed(sum(lq), sum(lk), 3, 1, 128, seed=8101 + causal, sigma=2.0)
    check_varlen(attn, q, k, v, offsets(lq), offsets(lk), "rtne", causal, max_seqlen_q=max(lq))


def test_varlen_empty_sequences_keyless_rows_and_gaps(attn):
    # rows 0..2 before the first sequence and 5 rows after the last belong to none; an empty
    # sequence, a sequence with queries but no keys (NaN rows, LSE -inf), empty keys at the end
    lq, lk = [0, 50, 200, 0, 129], [10, 0, 300, 4, 0]
    Tq, Tk = 3 + sum(lq) + 5, sum(lk) + 7
    q, k, v = packed(Tq, Tk, 2, 2, 128, seed=8200)
    cu_q, cu_k = offsets(lq, start=3), offsets(lk, start=2)
    o, lse = check_varlen(attn, q, k, v, cu_q, cu_k, "rtna")
    ob = o.cpu().view(torch.int16).numpy().view(np.uint16)
    assert (ob[3:53] == 0x7FC0).all() and (ob[253:382] == 0x7FC0).all()
    assert np.isneginf(lse.cpu().numpy()[:, 3:53]).all()


@pytest.mark.parametrize("causal", [False, True])
def test_varlen_equals_dense_kernel_per_sequence(attn, causal):
    # the same tiles, masks and arithmetic as the dense kernel on the sequence alone (without
    # key splits; sequences of more than 128 queries, which the dense path runs on this kernel)
    lq = [300, 129, 1000, 257]
    lk = lq if causal else [200, 700, 131, 1024]
    q, k, v = packed(sum(lq), sum(lk), 4, 2, 128, seed=8300 + causal)
    cu_q, cu_k = offsets(lq), offsets(lk)
    o, lse = run_varlen(attn, q, k, v, cu_q, cu_k, "rtne", causal)
    status_ok(attn)
    for b in range(len(lq)):
        qs, ks, vs = (t[c[b]:c[b + 1]][None].cuda() for t, c in ((q, cu_q), (k, cu_k), (v, cu_k)))
        od, ld = attn.attn_fwd_ex(qs, ks, vs, layout="bshd", causal=causal, return_lse=True, force_splits=1)
        torch.cuda.synchronize()
        assert torch.equal(o[cu_q[b]:cu_q[b + 1]].view(torch.int16), od[0].view(torch.int16)), b
        assert torch.equal(lse[:, cu_q[b]:cu_q[b + 1]].view(torch.int32), ld[0].view(torch.int32)), b


def test_varlen_neighbours_nonfinite_values_do_not_leak(attn):
    lq, lk = [300, 200, 260], [250, 130, 129]
    q, k, v = packed(sum(lq), sum(lk), 2, 1, 128, seed=8400)
    cu_q, cu_k = offsets(lq), offsets(lk)
    base, base_lse = run_varlen(attn, q, k, v, cu_q, cu_k)
    status_ok(attn)
    for b in range(3):
        q2, k2, v2 = q.clone(), k.clone(), v.clone()
        for o_ in range(3):
            if o_ == b:
                continue
            for t, cu in ((q2, cu_q), (k2, cu_k), (v2, cu_k)):
                rows = t[cu[o_]:cu[o_ + 1]]
                rows.view(torch.int16)[::2] = 0x7F80      # +inf
                rows.view(torch.int16)[1::3] = 0x7FC1     # NaN
        o2, lse2 = run_varlen(attn, q2, k2, v2, cu_q, cu_k)
        status_ok(attn)
        r = slice(cu_q[b], cu_q[b + 1])
        assert torch.equal(o2[r].view(torch.int16), base[r].view(torch.int16)), b
        assert torch.equal(lse2[:, r].view(torch.int32), base_lse[:, r].view(torch.int32)), b


def test_varlen_grid_size_does_not_change_results(attn):
    lq, lk = [700, 33, 450, 1], [512, 900, 17, 300]
    q, k, v = packed(sum(lq), sum(lk), 4, 4, 64, seed=8500)
    cu_q, cu_k = offsets(lq), offsets(lk)
    ref, ref_lse = run_varlen(attn, q, k, v, cu_q, cu_k, causal=True)
    for kw in ({"max_seqlen_q": 700}, {"max_seqlen_q": 1}, {"max_ctas": 3}, {"max_ctas": 1}):
        o, lse = run_varlen(attn, q, k, v, cu_q, cu_k, causal=True, **kw)
        status_ok(attn)
        assert torch.equal(o.view(torch.int16), ref.view(torch.int16)), kw
        assert torch.equal(lse.view(torch.int32), ref_lse.view(torch.int32)), kw


def test_varlen_writes_stay_in_bounds(attn):
    lq, lk = [130, 1, 77], [200, 5, 129]
    H, d = 2, 128
    q, k, v = packed(sum(lq), sum(lk), H, H, d, seed=8600)
    qd, kd, vd = (t.cuda() for t in (q, k, v))
    obuf, o = guarded(q.numel(), "bf16")
    lbuf, lse = guarded(H * q.shape[0], "f32")
    a = attn.VarlenArgs()
    a.B, a.H, a.Hkv, a.total_q, a.total_k, a.d = len(lq), H, H, q.shape[0], k.shape[0], d
    wbytes = int(attn.load().attn_fwd_varlen_workspace_size(ctypes.byref(a)))
    assert wbytes > 0
    wbuf, ws = guarded(wbytes, "ws")
    cq, ck = (torch.as_tensor(offsets(x)).cuda() for x in (lq, lk))
    attn.attn_fwd_varlen(qd, kd, vd, cq, ck, o=o.view(q.shape), lse=lse.view(H, -1), workspace=ws)
    torch.cuda.synchronize()
    status_ok(attn)
    assert guards_intact(obuf, "bf16") and guards_intact(lbuf, "f32") and guards_intact(wbuf, "ws")
    assert not (o.view(torch.int16) == 0x7BAD).any() and not (lse.view(torch.int32) == 0x7F7BAD01).any()


@pytest.mark.parametrize("bad", ["decreasing", "past_end", "negative_start"])
def test_varlen_bad_offsets_are_reported_and_write_nothing(attn, bad):
    lq = [100, 60, 140]
    q, k, v = packed(sum(lq), sum(lq), 2, 2, 128, seed=8700)
    cu = offsets(lq)
    cu_bad = cu.copy()
    if bad == "decreasing":
        cu_bad[2] = cu_bad[1] - 1
    elif bad == "past_end":
        cu_bad[3] = sum(lq) + 1
    else:
        cu_bad[0] = -1
    o, lse = run_varlen(attn, q, k, v, cu_bad, cu)
    assert attn.device_status() == (1, SITE_SEQLENS)
    assert (o.view(torch.int16) == BF16_SENTINEL).all() and (lse.view(torch.int32) == F32_SENTINEL).all()
    # the device stays usable and the status word was cleared by reading it
    check_varlen(attn, q, k, v, cu, cu)


PACK = [  # (lens_q, lens_k, H, Hkv, d, causal): decoding-sized and prefill-sized chunks
    ([1, 1, 1, 1, 1], [700, 129, 1, 300, 2000], 8, 2, 128, True),
    ([1, 4, 16, 3], [5000, 64, 300, 128], 32, 8, 128, True),
    ([7, 1, 33], [900, 1000, 33], 16, 2, 64, False),
    ([300, 129, 700, 0], [300, 700, 700, 5], 8, 1, 128, True),
    ([257, 64], [513, 64], 4, 4, 128, False),       # one head per K/V head: packing is a no-op
    ([2, 130], [4000, 600], 64, 2, 64, True),       # 32 heads per K/V head
]


@pytest.mark.parametrize("case", PACK, ids=lambda c: "n%d_H%dKV%d_d%d%s" % (len(c[0]), c[2], c[3], c[4],
                                                                             "_causal" if c[5] else ""))
def test_packed_heads_are_bitwise_the_unpacked_result(attn, case):
    # packing the query heads of a K/V head into one tile changes which rows share a tile,
    # not any row's arithmetic: outputs and LSE must be the same bits, and meet the oracle
    lq, lk, H, Hkv, d, causal = case
    q, k, v = packed(sum(lq), sum(lk), H, Hkv, d, seed=8800 + H + d)
    cu_q, cu_k = offsets(lq), offsets(lk)
    o0, l0 = run_varlen(attn, q, k, v, cu_q, cu_k, "rtne", causal)
    o1, l1 = run_varlen(attn, q, k, v, cu_q, cu_k, "rtne", causal, pack_heads=True, max_seqlen_q=max(lq))
    status_ok(attn)
    assert torch.equal(o1.view(torch.int16), o0.view(torch.int16))
    assert torch.equal(l1.view(torch.int32), l0.view(torch.int32))
    check_varlen(attn, q, k, v, cu_q, cu_k, "rtne", causal, pack_heads=True)


def test_packed_heads_writes_stay_in_bounds(attn):
    lq, lk, H, Hkv, d = [1, 3, 77, 130], [200, 5, 129, 400], 8, 2, 128
    q, k, v = packed(sum(lq), sum(lk), H, Hkv, d, seed=8900)
    qd, kd, vd = (t.cuda() for t in (q, k, v))
    obuf, o = guarded(q.numel(), "bf16")
    lbuf, lse = guarded(H * q.shape[0], "f32")
    a = attn.VarlenArgs()
    a.B, a.H, a.Hkv, a.total_q, a.total_k, a.d, a.pack_heads = len(lq), H, Hkv, q.shape[0], k.shape[0], d, 1
    wbytes = int(attn.load().attn_fwd_varlen_workspace_size(ctypes.byref(a)))
    wbuf, ws = guarded(wbytes, "ws")
    cq, ck = (torch.as_tensor(offsets(x)).cuda() for x in (lq, lk))
    attn.attn_fwd_varlen(qd, kd, vd, cq, ck, o=o.view(q.shape), lse=lse.view(H, -1), workspace=ws, causal=True,
                         pack_heads=True)
    torch.cuda.synchronize()
    status_ok(attn)
    assert guards_intact(obuf, "bf16") and guards_intact(lbuf, "f32") and guards_intact(wbuf, "ws")
    assert not (o.view(torch.int16) == 0x7BAD).any() and not (lse.view(torch.int32) == 0x7F7BAD01).any()
