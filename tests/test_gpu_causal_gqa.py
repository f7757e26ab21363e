"""GPU parity of the extended forward (attn_fwd_ex): causal mask, grouped K/V heads and the
row log-sum-exp, against the fp64 oracle (needs a GB300).

The causal mask is aligned at the last query and key (key j visible to query i iff
j <= i + Skv - Sq), so Sq > Skv leaves leading rows with no visible key: their outputs are
NaN and their log-sum-exp is -inf.  Grouped heads (GQA, MQA when K/V carry one head): query
head h reads K/V head h // (H // Hkv).

LSE tolerance, derived from the arithmetic: the kernel forms each logit as an fp32
tensor-core sum of d exact bf16 products, off by at most d * 2^-24 * A_i with
A_i = max_j sum_x |q_ix k_jx| / sqrt(d); the log-sum-exp moves by at most that (its gradient
in the logits is the softmax row, which sums to 1).  The fp32 weights (ex2.approx, ~2^-22
relative), their fp32 running sum over at most a few thousand key tiles and the final
log2 / ln 2 conversion add well under 2^-14 * (1 + |lse|).  So
|gpu - oracle| <= 2^-14 * (1 + |lse|) + 2^-17 * A_i.
"""
import numpy as np
import pytest
import torch

import oracle
from tests import parity
from workloads import WORKLOADS, make_qkv, make_workload, sample_rows

pytestmark = pytest.mark.gpu

MODES = ("rtne", "rtna", "rtz")


@pytest.fixture(scope="module")
def attn():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import bf16_attention_forward_gb300 as a
    a.load()
    return a


def run_ex(attn, q, k, v, layout, mode, causal=False, **kw):
    qd, kd, vd = (t.cuda() for t in (q, k, v))
    o, lse = attn.attn_fwd_ex(qd, kd, vd, layout=layout, round=mode, causal=causal,
                              return_lse=True, **kw)
    torch.cuda.synchronize()
    st, site = attn.device_status()
    assert st == 0, "device status %d at wait site %d" % (st, site)
    return o, lse.cpu().numpy().reshape(-1).astype(np.float64)


def abs_logit_scale(q, k, layout, rows=None):
    """A_i = max over keys of sum_x |q_ix k_jx| / sqrt(d), per flat row (b*H + h)*Sq + i
    (over all keys: an upper bound for the visible ones)."""
    qf, kf = q.double().abs(), k.double().abs()
    if layout == "bshd":
        qf, kf = qf.permute(0, 2, 1, 3), kf.permute(0, 2, 1, 3)
    B, H, Sq, d = qf.shape
    group = H // kf.shape[1]
    rows = np.arange(B * H * Sq) if rows is None else np.asarray(rows)
    out = np.empty(len(rows))
    bh = rows // Sq
    for u in np.unique(bh):
        sel = np.nonzero(bh == u)[0]
        b, h = divmod(int(u), H)
        qr = qf[b, h, torch.as_tensor(rows[sel] % Sq)]
        out[sel] = (qr @ kf[b, h // group].T).amax(dim=-1).numpy() / d ** 0.5
    return out


def check_lse(gpu, ref, a_scale):
    gpu = np.asarray(gpu, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    fin = np.isfinite(ref)
    # non-finite: same class (NaN, +inf, -inf)
    assert np.array_equal(np.isnan(gpu[~fin]), np.isnan(ref[~fin]))
    nn = ~fin & ~np.isnan(ref)
    assert np.array_equal(gpu[nn], ref[nn])
    assert np.all(np.isfinite(gpu[fin]))
    tol = 2.0 ** -14 * (1 + np.abs(ref[fin])) + 2.0 ** -17 * a_scale[fin]
    err = np.abs(gpu[fin] - ref[fin])
    assert np.all(err <= tol), (float(np.max(err - tol)), int(np.argmax(err - tol)))
    return float(np.max(err)) if err.size else 0.0


def check_ex(attn, q, k, v, layout, mode, causal=False, rows=None, **kw):
    o, lse = run_ex(attn, q, k, v, layout, mode, causal, **kw)
    ref = oracle.attention(q, k, v, layout, mode, rows=rows, want_a=True, want_lse=True,
                           causal=causal)
    g = parity.gpu_rows_bits(o, layout, rows)
    res = parity.compare(g, ref["o_bits"], ref["a"])
    assert res["ok"], res
    lse_ref = ref["lse"].reshape(-1)
    lse_gpu = lse if rows is None else lse[np.asarray(rows)]
    check_lse(lse_gpu, lse_ref, abs_logit_scale(q, k, layout, rows))
    return res, o, lse


CAUSAL = [  # (B, H, Sq, Skv)
    (1, 1, 1, 1), (1, 2, 128, 128), (1, 1, 300, 300), (2, 3, 257, 513), (1, 2, 513, 257),
    (1, 1, 1, 1000), (1, 1, 1000, 1), (2, 1, 640, 640), (1, 1, 129, 2000),
]


@pytest.mark.parametrize("shape", CAUSAL, ids=lambda s: "B%dH%dSq%dSkv%d" % s)
@pytest.mark.parametrize("layout", ["bshd", "bhsd"])
def test_causal_small_shapes(attn, shape, layout):
    B, H, Sq, Skv = shape
    q, k, v = make_qkv(B, H, Sq, Skv, 128, layout, seed=1000 + sum(shape))
    for mode in MODES:
        check_ex(attn, q, k, v, layout, mode, causal=True)


def test_causal_rows_without_keys_are_nan_with_minus_inf_lse(attn):
    # Sq - Skv = 200 leading rows see no key at all
    q, k, v = make_qkv(1, 2, 456, 256, 128, "bshd", seed=31)
    _, o, lse = check_ex(attn, q, k, v, "bshd", "rtne", causal=True)
    ob = o.float().permute(0, 2, 1, 3).cpu()
    assert torch.isnan(ob[:, :, :200]).all() and not torch.isnan(ob[:, :, 200:]).any()
    lse = lse.reshape(2, 456)
    assert np.all(lse[:, :200] == -np.inf) and np.all(np.isfinite(lse[:, 200:]))


GROUPED = [  # (B, H, Hkv, Sq, Skv)
    (1, 8, 2, 300, 700), (2, 4, 1, 257, 129), (1, 6, 3, 128, 1000), (1, 16, 16, 130, 130),
]


@pytest.mark.parametrize("shape", GROUPED, ids=lambda s: "B%dH%dHkv%dSq%dSkv%d" % s)
@pytest.mark.parametrize("causal", [False, True])
def test_grouped_heads(attn, shape, causal):
    B, H, Hkv, Sq, Skv = shape
    for layout in ("bshd", "bhsd"):
        q, k, v = make_qkv(B, H, Sq, Skv, 128, layout, seed=2000 + sum(shape), Hkv=Hkv)
        check_ex(attn, q, k, v, layout, "rtne", causal=causal)


@pytest.mark.parametrize("splits", [2, 5])
def test_grouped_heads_and_lse_through_the_split_path(attn, splits):
    q, k, v = make_qkv(1, 8, 260, 1500, 128, "bhsd", seed=41, sigma=2.0, Hkv=2)
    check_ex(attn, q, k, v, "bhsd", "rtna", force_splits=splits)


def test_grouped_equals_repeated_heads_bitwise(attn):
    for causal in (False, True):
        q, k, v = make_qkv(2, 8, 333, 444, 128, "bshd", seed=43, Hkv=2)
        o1, l1 = run_ex(attn, q, k, v, "bshd", "rtne", causal)
        kr, vr = (t.repeat_interleave(4, dim=2) for t in (k, v))
        o2, l2 = run_ex(attn, q, kr, vr, "bshd", "rtne", causal)
        assert torch.equal(o1.view(torch.int16), o2.view(torch.int16))
        assert np.array_equal(l1.view(np.int64), l2.view(np.int64))


def test_causal_last_row_equals_full_attention_bitwise(attn):
    # the last query sees every key, so it must match the unmasked call bit for bit (with
    # the unmasked call kept off the key-split path, which the causal planner never takes)
    q, k, v = make_qkv(1, 4, 640, 900, 128, "bhsd", seed=44)
    oc, lc = run_ex(attn, q, k, v, "bhsd", "rtz", causal=True)
    of, lf = run_ex(attn, q, k, v, "bhsd", "rtz", causal=False, force_splits=1)
    assert torch.equal(oc[:, :, -1].view(torch.int16), of[:, :, -1].view(torch.int16))
    last = np.arange(4) * 640 + 639
    assert np.array_equal(lc[last], lf[last])


def test_causal_deterministic_across_grid_sizes(attn):
    q, k, v = make_qkv(2, 3, 1100, 1100, 128, "bshd", seed=45)
    o0, l0 = run_ex(attn, q, k, v, "bshd", "rtne", causal=True)
    for max_ctas in (1, 7, 0):
        o1, l1 = run_ex(attn, q, k, v, "bshd", "rtne", causal=True, max_ctas=max_ctas)
        assert torch.equal(o0.view(torch.int16), o1.view(torch.int16))
        assert np.array_equal(l0, l1)


def test_lse_plain_and_split_agree_with_oracle(attn):
    q, k, v = make_qkv(2, 3, 300, 2000, 128, "bshd", seed=46, sigma=3.0)
    check_ex(attn, q, k, v, "bshd", "rtne")
    check_ex(attn, q, k, v, "bshd", "rtne", force_splits=4)


def test_lse_nonfinite_rows(attn):
    # one +inf in K: rows with q_i0 > 0 meet a +inf logit (NaN row), q_i0 < 0 a -inf logit
    # (that key drops out), q_i0 = 0 a 0*inf = NaN logit
    for force_splits in (0, 3):
        q, k, v = make_qkv(1, 2, 200, 700, 128, "bhsd", seed=47)
        k[0, 1, 333, 0] = float("inf")
        q[0, 1, 5, 0] = 0.0
        check_ex(attn, q, k, v, "bhsd", "rtne", force_splits=force_splits)


def test_lse_all_minus_inf_rows(attn):
    # K[..., 0] = -inf for every key: head 0's queries get q_i0 = 1, so every logit is -inf
    # (NaN outputs, lse -inf); head 1's get q_i0 = 0, so every logit is 0 * inf = NaN
    q, k, v = make_qkv(1, 2, 130, 260, 128, "bshd", seed=48)
    k[0, :, :, 0] = float("-inf")
    q[0, :, 0, 0] = 1.0
    q[0, :, 1, 0] = 0.0
    _, _, lse = check_ex(attn, q, k, v, "bshd", "rtne")
    lse = lse.reshape(2, 130)
    assert np.all(lse[0] == -np.inf) and np.all(np.isnan(lse[1]))


def test_lse_argument_checks(attn):
    q, k, v = (t.cuda() for t in make_qkv(1, 2, 64, 64, 128, "bshd", seed=49))
    with pytest.raises(ValueError):
        attn.attn_fwd_ex(q, k, v, lse=torch.empty(127, device="cuda"))
    with pytest.raises(ValueError):
        attn.attn_fwd_ex(q, k[:, :, :1].contiguous(), v, causal=True)
    kk, vv = k[:, :, :1].contiguous(), v[:, :, :1].contiguous()
    o = attn.attn_fwd_ex(q, kk, vv)           # MQA
    assert o.shape == q.shape
    with pytest.raises(attn.AttnError):
        attn.attn_fwd_ex(q, k, v, causal=True, force_splits=2)


@pytest.mark.parametrize("name", ["causal_gqa"])
def test_workload_sampled_rows(attn, name):
    w = WORKLOADS[name]
    q, k, v = make_workload(w)
    rows = sample_rows(w.B, w.H, w.Sq, 96, seed=7)
    for mode in w.modes:
        res, _, _ = check_ex(attn, q, k, v, w.layout, mode, causal=w.causal, rows=rows)
        parity.log_result("%s/%s" % (name, mode), res)
        # fraction within 2 bf16 ULP of the oracle, floor just under the measured value
        assert res["literal_frac"] >= 0.935, res
