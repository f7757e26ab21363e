"""GPU parity of the attention backward (attn_bwd, d = 128 and 64) against the fp64 backward
oracle.

The GPU path recomputes P from the forward's fp32 log-sum-exp, rounds P and dS to bf16
before the tensor-core products, and forms D from the forward's bf16 output, so an element
of dQ, dK or dV passes when |gpu - oracle| <= 2^-7 * A + ulp(oracle), with A the oracle's
sum of term magnitudes (dV: sum_i p |dO|; dQ, dK: c sum p (|dP| + |D|) |k| or |q|, where
|D| = sum |dO| |O| also covers D formed from the rounded O).  2^-7 is four times bf16's unit
roundoff: P (or dS) rounding, the rounding of O inside D, and the final bf16 store.  The
oracle itself is pinned against numerical differentiation of the forward.  By default dQ is
summed with reductions in L2 across key tiles in no fixed order, so its last bits may differ
between runs; in the deterministic mode each key tile's terms are stored to a slice of their
own and added in key-tile order.  dK and dV are accumulated in a fixed order and are bitwise
reproducible in both modes.
"""
import numpy as np
import pytest
import torch

import oracle
from tests import parity
from workloads import make_qkv

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def attn():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import bf16_attention_forward_gb300 as a
    a.load()
    return a


def _bits(t):
    return t.detach().cpu().contiguous().view(torch.int16).numpy().view(np.uint16)


def run_bwd(attn, q, k, v, g, layout, causal, deterministic=False):
    qd, kd, vd, gd = (t.cuda() for t in (q, k, v, g))
    o, lse = attn.attn_fwd_ex(qd, kd, vd, layout=layout, causal=causal, return_lse=True)
    dq, dk, dv = attn.attn_bwd(qd, kd, vd, o, gd, lse, layout=layout, causal=causal,
                               deterministic=deterministic)
    torch.cuda.synchronize()
    assert attn.device_status()[0] == 0
    st, site = attn.bwd_device_status()
    assert st == 0, "backward device status %d at wait site %d" % (st, site)
    return dq, dk, dv


def check_bwd(attn, q, k, v, g, layout, causal=False, deterministic=False):
    dq, dk, dv = run_bwd(attn, q, k, v, g, layout, causal, deterministic)
    ref = oracle.backward(q, k, v, g, layout, causal=causal, want_a=True)
    worst = {}
    for name, got in (("dq", dq), ("dk", dk), ("dv", dv)):
        gb = _bits(got).astype(np.uint16).reshape(-1)
        r = ref[name].reshape(-1)
        a = ref[name + "_a"].reshape(-1)
        gf = parity.bits_to_f64(gb)
        rb = ref[name + "_bits"].reshape(-1).astype(np.uint16)
        err = np.abs(gf - r)
        tol = 2.0 ** -7 * a + parity.bf16_ulp(rb)
        bad = ~(err <= tol)
        assert not bad.any(), (name, int(bad.sum()), float((err / np.maximum(a, 1e-30))[bad].max()))
        worst[name] = float(np.max(err / np.maximum(a, 1e-30)))
    return worst, (dq, dk, dv)


SHAPES = [  # (B, H, Hkv, Sq, Skv)
    (1, 1, 1, 128, 128), (1, 2, 2, 300, 200), (2, 2, 1, 129, 257), (1, 4, 2, 256, 384),
    (1, 1, 1, 1, 1), (1, 2, 1, 77, 1000),
]


@pytest.mark.parametrize("shape", SHAPES, ids=lambda s: "B%dH%dHkv%dSq%dSkv%d" % s)
@pytest.mark.parametrize("layout", ["bshd", "bhsd"])
def test_backward_matches_oracle(attn, shape, layout):
    B, H, Hkv, Sq, Skv = shape
    q, k, v = make_qkv(B, H, Sq, Skv, 128, layout, seed=5000 + sum(shape), Hkv=Hkv)
    g = make_qkv(B, H, Sq, 1, 128, layout, seed=5100 + sum(shape))[0]
    check_bwd(attn, q, k, v, g, layout)


@pytest.mark.parametrize("Sq,Skv", [(300, 300), (200, 456), (456, 200), (640, 640), (300, 200)])
def test_backward_causal(attn, Sq, Skv):
    q, k, v = make_qkv(1, 4, Sq, Skv, 128, "bshd", seed=5200 + Sq, Hkv=2)
    g = make_qkv(1, 4, Sq, 1, 128, "bshd", seed=5300 + Skv)[0]
    check_bwd(attn, q, k, v, g, "bshd", causal=True)


def test_backward_dk_dv_reproducible_and_large_logits(attn):
    q, k, v = make_qkv(1, 2, 384, 512, 128, "bhsd", seed=5400, sigma=2.0)
    g = make_qkv(1, 2, 384, 1, 128, "bhsd", seed=5401)[0]
    _, (dq1, dk1, dv1) = check_bwd(attn, q, k, v, g, "bhsd")
    dq2, dk2, dv2 = run_bwd(attn, q, k, v, g, "bhsd", False)
    assert torch.equal(dk1.view(torch.int16), dk2.view(torch.int16))
    assert torch.equal(dv1.view(torch.int16), dv2.view(torch.int16))


def test_backward_argument_errors(attn):
    q, k, v = (t.cuda() for t in make_qkv(1, 1, 8, 8, 128, "bshd", seed=1))
    o, lse = attn.attn_fwd_ex(q, k, v, return_lse=True)
    with pytest.raises(ValueError):
        attn.attn_bwd(q, k, v, o, o, lse[:, :, :4].contiguous())
    with pytest.raises(attn.AttnError):           # the gradient may not alias an input
        attn.attn_bwd(q, k, v, o, o, lse, dq=q)
    q96, k96, v96 = (t.cuda() for t in make_qkv(1, 1, 8, 8, 96, "bshd", seed=2))
    l96 = torch.zeros(8, device="cuda")
    with pytest.raises(attn.AttnError):           # head dimension 96 is not supported
        attn.attn_bwd(q96, k96, v96, q96, q96, l96)


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("layout", ["bshd", "bhsd"])
def test_backward_head_dim_64(attn, causal, layout):
    for (B, H, Hkv, Sq, Skv) in ((1, 2, 2, 300, 200), (2, 4, 1, 129, 257)):
        q, k, v = make_qkv(B, H, Sq, Skv, 64, layout, seed=5500 + Sq, Hkv=Hkv)
        g = make_qkv(B, H, Sq, 1, 64, layout, seed=5600 + Skv)[0]
        check_bwd(attn, q, k, v, g, layout, causal=causal)


@pytest.mark.parametrize("causal", [False, True])
def test_backward_many_units_per_cta(attn, causal):
    # more (b, K/V head, key tile) units than SMs: CTAs run several units in turn, so the dK/dV
    # hand-off between units and the Q/dO ring across unit boundaries are exercised
    if causal:
        B, H, Hkv, Sq, Skv = 2, 16, 8, 300, 1300      # 2 * 8 * 11 = 176 units
    else:
        B, H, Hkv, Sq, Skv = 4, 16, 16, 130, 1280     # 4 * 16 * 10 = 640 units
    q, k, v = make_qkv(B, H, Sq, Skv, 128, "bshd", seed=5700 + causal, Hkv=Hkv)
    g = make_qkv(B, H, Sq, 1, 128, "bshd", seed=5800 + causal)[0]
    check_bwd(attn, q, k, v, g, "bshd", causal=causal)


def test_backward_square_workload_sampled_heads(attn):
    """The square workload's shape (B4 H16 Sq=Skv=2048, d = 128, BHSD) at full size on the GPU;
    without grouped heads every (b, h) is an independent problem, so the oracle runs on three
    sampled (b, h) slices (first, last and a middle one) and their dQ, dK and dV must meet the
    criteria element by element."""
    from workloads import WORKLOADS
    w = WORKLOADS["square"]
    q, k, v = make_qkv(w.B, w.H, w.Sq, w.Skv, w.d, w.layout, seed=w.seed)
    g = make_qkv(w.B, w.H, w.Sq, 1, w.d, w.layout, seed=w.seed + 77)[0]
    dq, dk, dv = run_bwd(attn, q, k, v, g, w.layout, False)
    heads = ((0, 0), (w.B - 1, w.H - 1), (1, 7))
    pick = lambda t: torch.cat([t[b:b + 1, h:h + 1] for b, h in heads], dim=0)   # a batch of 3 heads
    ref = oracle.backward(pick(q), pick(k), pick(v), pick(g), w.layout, want_a=True)
    for name, got in (("dq", dq), ("dk", dk), ("dv", dv)):
        gf = parity.bits_to_f64(_bits(pick(got.cpu())).reshape(-1))
        r = ref[name].reshape(-1)
        tol = 2.0 ** -7 * ref[name + "_a"].reshape(-1) + parity.bf16_ulp(ref[name + "_bits"].reshape(-1))
        bad = ~(np.abs(gf - r) <= tol)
        assert not bad.any(), (name, int(bad.sum()))


@pytest.mark.parametrize("shape", [(2, 32, 16, 1280, 1280, "bshd"), (1, 40, 40, 700, 1000, "bhsd")],
                         ids=lambda s: "B%dH%dHkv%dSq%dSkv%d%s" % s)
def test_backward_causal_paired_schedule(attn, shape):
    # at least two causal units per SM: the backward then runs its paired schedule (key tiles
    # jt and n-1-jt of one (b, K/V head) on the same CTA, two positions per round)
    B, H, Hkv, Sq, Skv, layout = shape
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    assert B * Hkv * -(-Skv // 128) >= 2 * sms, "shape too small for the paired schedule"
    q, k, v = make_qkv(B, H, Sq, Skv, 128, layout, seed=5900 + Sq, Hkv=Hkv)
    g = make_qkv(B, H, Sq, 1, 128, layout, seed=5950 + Skv)[0]
    check_bwd(attn, q, k, v, g, layout, causal=True)


@pytest.mark.parametrize("shape", [(1, 5, 5, 1024, 1024, 128, "bshd"), (2, 8, 2, 512, 640, 128, "bhsd"),
                                   (1, 3, 3, 1000, 700, 64, "bhsd")],
                         ids=lambda s: "B%dH%dHkv%dSq%dSkv%dd%d%s" % s)
def test_backward_split_tail_units(attn, shape):
    # fewer units than SMs with enough query steps each: every unit is split into query-range
    # parts whose dK/dV partials the final kernel adds in part order (dQ is unaffected)
    B, H, Hkv, Sq, Skv, d, layout = shape
    q, k, v = make_qkv(B, H, Sq, Skv, d, layout, seed=6100 + Sq, Hkv=Hkv)
    g = make_qkv(B, H, Sq, 1, d, layout, seed=6150 + Skv)[0]
    _, (dq, dk, dv) = check_bwd(attn, q, k, v, g, layout)
    # the split plan is deterministic: a second call gives the same dK and dV bits
    _, (dq2, dk2, dv2) = check_bwd(attn, q, k, v, g, layout)
    assert torch.equal(dk.view(torch.int16), dk2.view(torch.int16))
    assert torch.equal(dv.view(torch.int16), dv2.view(torch.int16))


DET = [  # (B, H, Hkv, Sq, Skv, d, layout, causal)
    (1, 2, 2, 300, 200, 128, "bshd", False),
    (2, 4, 2, 257, 640, 128, "bhsd", False),
    (1, 4, 2, 456, 200, 128, "bshd", True),     # Sq > Skv: rows that see no key
    (1, 4, 4, 300, 777, 64, "bhsd", True),
    (1, 5, 5, 1024, 1024, 128, "bshd", False),  # split tail units
    (1, 3, 3, 1000, 700, 64, "bhsd", False),
]


@pytest.mark.parametrize("case", DET, ids=lambda c: "B%dH%dHkv%dSq%dSkv%dd%d%s" % c[:7] + ("c" if c[7] else ""))
def test_backward_deterministic_dq(attn, case):
    # the deterministic mode meets the same criteria, its dQ is bit-for-bit the same on a
    # second call, and its dK and dV are those of the default mode (the same path)
    B, H, Hkv, Sq, Skv, d, layout, causal = case
    q, k, v = make_qkv(B, H, Sq, Skv, d, layout, seed=6300 + Sq + Skv, Hkv=Hkv)
    g = make_qkv(B, H, Sq, 1, d, layout, seed=6350 + Sq)[0]
    _, (dq, dk, dv) = check_bwd(attn, q, k, v, g, layout, causal=causal, deterministic=True)
    dq2, dk2, dv2 = run_bwd(attn, q, k, v, g, layout, causal, deterministic=True)
    assert torch.equal(dq.view(torch.int16), dq2.view(torch.int16)), "deterministic dQ changed between calls"
    _, dk0, dv0 = run_bwd(attn, q, k, v, g, layout, causal)
    assert torch.equal(dk.view(torch.int16), dk0.view(torch.int16))
    assert torch.equal(dv.view(torch.int16), dv0.view(torch.int16))
