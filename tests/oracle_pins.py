"""Pins for the fp64 oracle: checks against what the pages and the mathematics fix.

Each ``pin_*`` takes an oracle library handle (so the same checks can be run against a
deliberately broken copy of the oracle) and raises AssertionError on a mismatch.  None of
them re-types the oracle's formula: they use closed forms, invariants, special cases that
reduce to a plain statistic, 50-digit brute force on tiny inputs, torch's own fp32->bf16
conversion and an independent table-based rounding.

Page cited: "MoonMath AI open-sources a HIP attention kernel for AMD MI300X that beats
AITER" -- opening section (softmax(QK^T/sqrt(d))V, head dim 128, BSHD/BHSD, arbitrary
lengths) and its limitations paragraph (three rounding modes, NaN/Inf, determinism).
"""
from __future__ import annotations

import math
from fractions import Fraction

import numpy as np
import torch

import oracle
from tests import bf16_exact as bx
from workloads import make_qkv, shape

MODES = ("rtne", "rtna", "rtz")
D = 128


def _bits(t: torch.Tensor) -> np.ndarray:
    return t.contiguous().view(torch.int16).numpy().view(np.uint16)


def _bf16(a) -> torch.Tensor:
    return torch.as_tensor(np.asarray(a, dtype=np.float32)).to(torch.bfloat16)


# --------------------------------------------------------------------------- rounding
def pin_round_rtne_matches_torch(lib):
    """RTNE of fp32-representable doubles equals torch's fp32 -> bf16 conversion."""
    g = torch.Generator().manual_seed(7)
    raw = torch.randint(0, 2**32, (200000,), generator=g, dtype=torch.int64)
    u = raw.to(torch.int64) & 0xFFFFFFFF
    # keep finite fp32 patterns; include subnormals and huge values
    f = torch.from_numpy(u.numpy().astype(np.uint32).view(np.float32).copy())
    f = f[torch.isfinite(f)]
    # plus exact ties: bf16 value + half quantum, and near-overflow
    ties = torch.from_numpy((np.arange(0, 0x7F7F, 97, dtype=np.uint32) << 16 | 0x8000)
                            .view(np.float32).copy())
    f = torch.cat([f, ties, -ties, torch.tensor([3.3895e38, -3.3895e38, 3.39e38])])
    want = f.to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    got = oracle.round_bf16(f.double().numpy(), "rtne", lib=lib)
    assert np.array_equal(got, want), "RTNE disagrees with torch on %d values" % (
        int((got != want).sum()))


def pin_round_rtz_rtna_bit_rules(lib):
    """On fp32 inputs RTZ keeps the top 16 bits; RTNA equals RTNE except on exact ties,
    where it moves away from zero."""
    g = torch.Generator().manual_seed(8)
    u = torch.randint(0, 2**31 - 1, (100000,), generator=g, dtype=torch.int64).numpy()
    u = u.astype(np.uint32)
    u[::3] = (u[::3] & 0xFFFF0000) | 0x8000            # exact ties
    u[1::7] |= 0x80000000                               # negatives
    f = u.view(np.float32)
    ok = np.isfinite(f)
    f, u = f[ok], u[ok]
    rtz = oracle.round_bf16(f.astype(np.float64), "rtz", lib=lib)
    want_rtz = (u >> 16).astype(np.uint16)
    # values beyond the largest bf16 truncate to it under RTZ, which the plain bit rule gives
    assert np.array_equal(rtz, want_rtz)
    rtne = oracle.round_bf16(f.astype(np.float64), "rtne", lib=lib)
    rtna = oracle.round_bf16(f.astype(np.float64), "rtna", lib=lib)
    tie = (u & 0xFFFF) == 0x8000
    assert np.array_equal(rtna[~tie], rtne[~tie])
    away = ((u[tie] >> 16) + 1).astype(np.uint16)      # magnitude up, sign kept
    assert np.array_equal(rtna[tie], away)


def pin_round_exact_doubles(lib):
    """On doubles that are not fp32 values, all three modes agree with the table-based
    rounding of the exact value, including exact midpoints and the subnormal range."""
    rng = np.random.default_rng(9)
    xs = list(rng.standard_normal(3000) * np.exp2(rng.integers(-140, 128, 3000)))
    for b in range(0x0001, 0x7F7F, 251):                 # midpoints between neighbours
        lo, hi = bx.bits_to_float(b), bx.bits_to_float(b + 1)
        xs += [(lo + hi) / 2, -(lo + hi) / 2, np.nextafter((lo + hi) / 2, 0.0),
               np.nextafter((lo + hi) / 2, np.inf)]
    mx = bx.bits_to_float(0x7F7F)
    xs += [mx + 2.0**119, mx + 2.0**119 - 2.0**80, mx, 1e300, -1e300, 5e-324, 2.0**-133,
           2.0**-134, 3 * 2.0**-135, 0.0, -0.0]
    xs = np.array(xs, dtype=np.float64)
    for mode in MODES:
        got = oracle.round_bf16(xs, mode, lib=lib)
        want = np.array([bx.round_exact(Fraction(float(x)), mode) for x in xs],
                        dtype=np.uint16)
        # -0.0: Fraction loses the sign; the oracle keeps it
        neg0 = (xs == 0) & np.signbit(xs)
        want[neg0] = 0x8000
        bad = np.nonzero(got != want)[0]
        assert bad.size == 0, "%s: %r -> %04x, want %04x" % (
            mode, xs[bad[0]], got[bad[0]], want[bad[0]])


def pin_round_nonfinite(lib):
    xs = np.array([np.nan, -np.nan, np.inf, -np.inf], dtype=np.float64)
    neg_nan = np.frombuffer(np.array([0xFFF8000000000001], dtype=np.uint64).tobytes(),
                            dtype=np.float64)
    xs = np.concatenate([xs, neg_nan])
    for mode in MODES:
        got = oracle.round_bf16(xs, mode, lib=lib)
        assert list(got) == [0x7FC0, 0x7FC0, 0x7F80, 0xFF80, 0x7FC0], (mode, got)


# --------------------------------------------------------------------------- closed forms
def pin_single_key_returns_v(lib):
    """Skv = 1: the only weight is 1, so O is the V row, bit for bit, in every mode."""
    for layout in ("bshd", "bhsd"):
        q, k, v = make_qkv(2, 3, 5, 1, D, layout, seed=11, sigma=3.0)
        for mode in MODES:
            o = oracle.attention(q, k, v, layout, mode, lib=lib)["o_bits"]
            vb = _bits(v if layout == "bhsd" else v.permute(0, 2, 1, 3))  # (B, H, 1, d)
            assert np.array_equal(o, np.broadcast_to(vb, o.shape)), (layout, mode)


def pin_constant_v(lib):
    """V rows all equal to one vector c: O = c exactly (weights sum to 1).  The exact value
    is a bf16 value, so RTNE/RTNA must return c; RTZ sits on its boundary there and may
    return c or its neighbour toward zero, while the unrounded result is c to 1e-15."""
    B, H, Sq, Skv = 1, 2, 7, 37
    q, k, _ = make_qkv(B, H, Sq, Skv, D, "bhsd", seed=12, sigma=2.0)
    c = torch.randn(D, generator=torch.Generator().manual_seed(1)).to(torch.bfloat16)
    v = c.view(1, 1, 1, D).expand(B, H, Skv, D).contiguous()
    cb = np.broadcast_to(_bits(c), (B, H, Sq, D))
    for mode in ("rtne", "rtna"):
        o = oracle.attention(q, k, v, "bhsd", mode, lib=lib)["o_bits"]
        assert np.array_equal(o, cb), mode
    r = oracle.attention(q, k, v, "bhsd", "rtz", want_f64=True, lib=lib)
    cd = c.double().numpy()
    assert np.allclose(r["o_f64"], np.broadcast_to(cd, r["o_f64"].shape), rtol=1e-15, atol=0)
    d = cb.astype(np.int64) - r["o_bits"].astype(np.int64)
    assert np.all((d == 0) | ((d == 1) & (cd != 0)))


def pin_zero_query_is_column_mean(lib):
    """Q = 0 (and separately K = 0): all logits 0, uniform weights, O = mean of V's rows."""
    B, H, Sq, Skv = 1, 2, 3, 29
    q, k, v = make_qkv(B, H, Sq, Skv, D, "bshd", seed=13)
    vv = v.permute(0, 2, 1, 3).double().numpy()                 # (B, H, Skv, d)
    for zq, zk in ((True, False), (False, True)):
        qq = torch.zeros_like(q) if zq else q
        kk = torch.zeros_like(k) if zk else k
        res = oracle.attention(qq, kk, v, "bshd", "rtne", want_f64=True, lib=lib)
        mean = vv.mean(axis=2, keepdims=True)                    # (B, H, 1, d)
        assert np.allclose(res["o_f64"], np.broadcast_to(mean, res["o_f64"].shape),
                           rtol=0, atol=1e-14)
        # exact mean (rational) rounded by the table method
        obits = {m: oracle.attention(qq, kk, v, "bshd", m, lib=lib)["o_bits"] for m in MODES}
        for h in range(H):
            for x in range(0, D, 9):
                exact = sum(Fraction(float(t)) for t in vv[0, h, :, x]) / Skv
                if bx.near_midpoint(exact):
                    continue
                for mode in MODES:
                    assert obits[mode][0, h, 0, x] == bx.round_exact(exact, mode), (h, x, mode)


def pin_two_keys_sigmoid(lib):
    """Two keys: O = sigma(s1 - s2) v1 + sigma(s2 - s1) v2 with s = q.k / sqrt(d)."""
    g = torch.Generator().manual_seed(14)
    q = torch.randn(1, 1, 4, D, generator=g).to(torch.bfloat16)
    k = torch.randn(1, 1, 2, D, generator=g).to(torch.bfloat16)
    v = torch.randn(1, 1, 2, D, generator=g).to(torch.bfloat16)
    res = oracle.attention(q, k, v, "bhsd", "rtne", want_f64=True, lib=lib)
    qd, kd, vd = q.double()[0, 0], k.double()[0, 0], v.double()[0, 0]
    for i in range(4):
        s = [float((qd[i] * kd[j]).sum()) / math.sqrt(D) for j in range(2)]
        a = 1.0 / (1.0 + math.exp(s[1] - s[0]))
        want = a * vd[0].numpy() + (1.0 - a) * vd[1].numpy()
        assert np.allclose(res["o_f64"][0, 0, i], want, rtol=1e-13, atol=1e-14)


def pin_dominant_key(lib):
    """One key with a logit gap above 60 takes all the weight: O equals its V row
    (the others' weights are below e^-60, under half an fp64-scaled bf16 quantum)."""
    B, H, Sq, Skv = 1, 1, 3, 50
    q, k, v = make_qkv(B, H, Sq, Skv, D, "bhsd", seed=15)
    q = torch.zeros_like(q)
    q[..., 0] = 1.0
    k = k.clone()
    k[..., 0] = 0.0
    k[0, 0, 17, 0] = 1024.0                                   # logit 1024/sqrt(128) ~ 90.5
    res = oracle.attention(q, k, v, "bhsd", "rtne", want_f64=True, lib=lib)
    assert np.allclose(res["o_f64"][0, 0], v.double().numpy()[0, 0, 17][None, :],
                       rtol=1e-20, atol=1e-25)
    for mode in ("rtne", "rtna"):   # the exact value is within 1e-38 of a bf16 value
        o = oracle.attention(q, k, v, "bhsd", mode, lib=lib)["o_bits"]
        assert np.array_equal(o[0, 0], np.broadcast_to(_bits(v)[0, 0, 17], (Sq, D)))


def pin_probs_sum_to_one(lib):
    B, H, Sq, Skv = 1, 2, 6, 300
    q, k, v = make_qkv(B, H, Sq, Skv, D, "bshd", seed=16, sigma=4.0)
    res = oracle.attention(q, k, v, "bshd", "rtne", want_probs=True, lib=lib)
    p = res["probs"]
    assert np.all(p >= 0)
    assert np.all(np.abs(p.sum(axis=1) - 1.0) <= 4 * Skv * 2.0**-53)


# --------------------------------------------------------------------------- brute force
def _mp_attention(q, k, v, mode_list, dps=50):
    """50-digit evaluation of softmax(QK^T/sqrt(d))V for finite BHSD inputs (B = H = 1)."""
    import mpmath
    mpmath.mp.dps = dps
    qd = q.double().numpy()[0, 0]
    kd = k.double().numpy()[0, 0]
    vd = v.double().numpy()[0, 0]
    Sq, Skv, d = qd.shape[0], kd.shape[0], qd.shape[1]
    inv = 1 / mpmath.sqrt(d)
    out = {}
    for i in range(Sq):
        s = [mpmath.fsum(mpmath.mpf(float(qd[i, x])) * mpmath.mpf(float(kd[j, x]))
                         for x in range(d)) * inv for j in range(Skv)]
        m = max(s)
        w = [mpmath.exp(sj - m) for sj in s]
        l = mpmath.fsum(w)
        for x in range(d):
            val = mpmath.fsum(w[j] * mpmath.mpf(float(vd[j, x])) for j in range(Skv)) / l
            out[(i, x)] = val
    return out


def pin_brute_force_mpmath(lib):
    """Tiny shapes against 50-digit arithmetic: unrounded O to 1e-13 relative to A, and the
    rounded bits in all modes except within 1e-12 of a rounding boundary."""
    for seed, (Sq, Skv, sigma) in enumerate(((1, 1, 1.0), (2, 3, 1.0), (4, 8, 1.0),
                                             (3, 5, 4.0), (2, 7, 0.25))):
        q, k, v = make_qkv(1, 1, Sq, Skv, D, "bhsd", seed=100 + seed, sigma=sigma)
        ref = _mp_attention(q, k, v, MODES)
        res = {m: oracle.attention(q, k, v, "bhsd", m, want_f64=True, want_a=True, lib=lib)
               for m in MODES}
        for (i, x), val in ref.items():
            f64 = res["rtne"]["o_f64"][0, 0, i, x]
            a = res["rtne"]["a"][0, 0, i, x]
            assert abs(f64 - float(val)) <= 1e-13 * max(a, 1e-300), (seed, i, x, f64, val)
            if bx.near_midpoint(val):
                continue
            for m in MODES:
                assert res[m]["o_bits"][0, 0, i, x] == bx.round_exact(val, m), (seed, i, x, m)


def pin_head_dim_64_brute_force_mpmath(lib):
    """Head dimension 64 (the scale is 1/sqrt(64) = 1/8) against 50-digit arithmetic, and the
    closed form Q = 0 -> column mean at d = 64 in both layouts."""
    for seed, (Sq, Skv, sigma) in enumerate(((1, 1, 1.0), (3, 6, 1.0), (2, 5, 3.0))):
        q, k, v = make_qkv(1, 1, Sq, Skv, 64, "bhsd", seed=300 + seed, sigma=sigma)
        ref = _mp_attention(q, k, v, MODES)
        res = {m: oracle.attention(q, k, v, "bhsd", m, want_f64=True, want_a=True, lib=lib)
               for m in MODES}
        for (i, x), val in ref.items():
            assert abs(res["rtne"]["o_f64"][0, 0, i, x] - float(val)) <= \
                1e-13 * max(res["rtne"]["a"][0, 0, i, x], 1e-300), (seed, i, x)
            if bx.near_midpoint(val):
                continue
            for m in MODES:
                assert res[m]["o_bits"][0, 0, i, x] == bx.round_exact(val, m), (seed, i, x, m)
    g = torch.Generator().manual_seed(310)
    v = torch.randn(2, 9, 3, 64, generator=g).to(torch.bfloat16)          # BSHD, Skv = 9
    k = torch.randn(2, 9, 3, 64, generator=g).to(torch.bfloat16)
    q = torch.zeros(2, 4, 3, 64, dtype=torch.bfloat16)
    o = oracle.attention(q, k, v, "bshd", "rtne", want_f64=True, lib=lib)["o_f64"]
    mean = v.double().mean(dim=1).numpy()                                 # (B, H, d)
    assert np.allclose(o, mean[:, :, None, :], rtol=0, atol=1e-15)


# --------------------------------------------------------------------------- structure
def pin_layouts_agree(lib):
    """The same logical tensors in BSHD and BHSD give the same output."""
    B, H, Sq, Skv = 2, 3, 9, 21
    q, k, v = make_qkv(B, H, Sq, Skv, D, "bshd", seed=17)
    a = oracle.attention(q, k, v, "bshd", "rtna", lib=lib)["o_bits"]
    t = lambda x: x.permute(0, 2, 1, 3).contiguous()
    b = oracle.attention(t(q), t(k), t(v), "bhsd", "rtna", lib=lib)["o_bits"]
    assert np.array_equal(a, b)
    # a per-head check that each (b, h) reads its own slice: swap heads 0 and 2 in BSHD
    perm = [2, 1, 0]
    c = oracle.attention(q[:, :, perm], k[:, :, perm], v[:, :, perm], "bshd", "rtna",
                         lib=lib)["o_bits"]
    assert np.array_equal(c[:, perm], a)


def pin_key_permutation_and_rows(lib):
    """Permuting K and V rows together changes nothing beyond fp64 summation order; the
    row-subset entry point agrees with the full evaluation."""
    B, H, Sq, Skv = 1, 2, 11, 64
    q, k, v = make_qkv(B, H, Sq, Skv, D, "bhsd", seed=18)
    full = oracle.attention(q, k, v, "bhsd", "rtne", want_f64=True, want_a=True, lib=lib)
    perm = torch.randperm(Skv, generator=torch.Generator().manual_seed(3))
    pk = oracle.attention(q, k[:, :, perm], v[:, :, perm], "bhsd", "rtne", want_f64=True,
                          lib=lib)
    assert np.all(np.abs(full["o_f64"] - pk["o_f64"]) <= 1e-14 * full["a"] + 1e-300)
    rows = [0, 5, 10, 11, 21]
    sub = oracle.attention(q, k, v, "bhsd", "rtne", rows=rows, lib=lib)["o_bits"]
    assert np.array_equal(sub, full["o_bits"].reshape(-1, D)[rows])


def pin_softmax_shift_and_scale(lib):
    """Adding one vector c to every key row shifts each row's logits by the constant
    q_i.c/sqrt(d), which leaves O unchanged (c = 3 e_0 on integer-valued column 0, so the
    shifted keys are exact in bf16).  And the scale is exactly 1/sqrt(128): with two keys of
    raw dot products 8 and 0 the first weight is sigmoid(8/sqrt(128))."""
    B, H, Sq, Skv = 1, 1, 4, 16
    q, k, v = make_qkv(B, H, Sq, Skv, D, "bhsd", seed=19)
    k = k.clone()
    g = torch.Generator().manual_seed(5)
    k[..., 0] = torch.randint(-8, 9, (B, H, Skv), generator=g).to(torch.bfloat16)
    k2 = k.clone()
    k2[..., 0] = k2[..., 0] + 3.0
    a = oracle.attention(q, k, v, "bhsd", "rtne", want_f64=True, want_a=True, lib=lib)
    b = oracle.attention(q, k2, v, "bhsd", "rtne", want_f64=True, lib=lib)
    assert np.all(np.abs(a["o_f64"] - b["o_f64"]) <= 1e-13 * a["a"] + 1e-300)
    qq = torch.zeros(1, 1, 1, D, dtype=torch.bfloat16)
    qq[..., 0] = 4.0
    kk = torch.zeros(1, 1, 2, D, dtype=torch.bfloat16)
    kk[0, 0, 0, 0] = 2.0                                      # raw dot 8 -> logit 8/sqrt(128)
    vv = torch.zeros(1, 1, 2, D, dtype=torch.bfloat16)
    vv[0, 0, 0, :] = 1.0
    r = oracle.attention(qq, kk, vv, "bhsd", "rtne", want_f64=True, lib=lib)["o_f64"]
    t = 8.0 / math.sqrt(128.0)
    assert abs(r[0, 0, 0, 0] - 1.0 / (1.0 + math.exp(-t))) < 1e-15


# --------------------------------------------------------------------------- non-finite
def _nf_base(seed=20, Sq=4, Skv=12):
    q, k, v = make_qkv(1, 1, Sq, Skv, D, "bhsd", seed=seed)
    return q.clone(), k.clone(), v.clone()


def pin_nan_in_q_poisons_only_its_row(lib):
    q, k, v = _nf_base()
    q[0, 0, 1, 5] = float("nan")
    o = oracle.attention(q, k, v, "bhsd", "rtne", lib=lib)["o_bits"][0, 0]
    assert np.all(o[1] == 0x7FC0)
    assert np.all(bx.is_finite_bits(o[[0, 2, 3]]))


def pin_nan_in_k_poisons_every_row(lib):
    q, k, v = _nf_base()
    k[0, 0, 3, 77] = float("nan")
    o = oracle.attention(q, k, v, "bhsd", "rtz", lib=lib)["o_bits"]
    assert np.all(o == 0x7FC0)


def pin_inf_key_sign_rules(lib):
    """k_j,x = +inf: rows with q_x > 0 get logit +inf (row NaN); rows with q_x < 0 get
    logit -inf, i.e. key j drops out: equal to attention without key j -- except columns
    where v_j is not finite, which become NaN (0 * inf); rows with q_x = 0 get NaN."""
    q, k, v = _nf_base(Sq=3)
    j, x = 4, 9
    q[0, 0, 0, x] = 1.0
    q[0, 0, 1, x] = -1.0
    q[0, 0, 2, x] = 0.0
    k[0, 0, j, x] = float("inf")
    v[0, 0, j, 30] = float("inf")
    for mode in MODES:
        o = oracle.attention(q, k, v, "bhsd", mode, lib=lib)["o_bits"][0, 0]
        assert np.all(o[0] == 0x7FC0) and np.all(o[2] == 0x7FC0)
        keep = [t for t in range(k.shape[2]) if t != j]
        ref = oracle.attention(q, k[:, :, keep], v[:, :, keep], "bhsd", mode,
                               lib=lib)["o_bits"][0, 0]
        want = ref[1].copy()
        want[30] = 0x7FC0
        assert np.array_equal(o[1], want), mode


def pin_inf_in_v_rules(lib):
    """Finite logits: +inf in a V column gives +inf there; +inf and -inf in one column
    give NaN; a weight that underflows in fp64 still carries the infinity (its exact value
    is positive)."""
    q, k, v = _nf_base(Sq=2, Skv=6)
    v[0, 0, 2, 3] = float("inf")
    v[0, 0, 1, 4] = float("inf")
    v[0, 0, 5, 4] = float("-inf")
    o = oracle.attention(q, k, v, "bhsd", "rtne", lib=lib)["o_bits"][0, 0]
    assert np.all(o[:, 3] == 0x7F80)
    assert np.all(o[:, 4] == 0x7FC0)
    finite_cols = [c for c in range(D) if c not in (3, 4)]
    assert np.all(bx.is_finite_bits(o[:, finite_cols]))
    # underflow: key 0 logit ~ -1000 below the max
    q2 = torch.zeros(1, 1, 1, D, dtype=torch.bfloat16)
    q2[..., 0] = 128.0
    k2 = torch.zeros(1, 1, 3, D, dtype=torch.bfloat16)
    k2[0, 0, 1, 0] = 96.0                 # logit 128*96/sqrt(128) ~ 1086
    v2 = torch.ones(1, 1, 3, D, dtype=torch.bfloat16)
    v2[0, 0, 0, 7] = float("-inf")        # key 0 (logit 0): weight e^-1086 underflows
    o2 = oracle.attention(q2, k2, v2, "bhsd", "rtne", lib=lib)["o_bits"][0, 0, 0]
    assert o2[7] == 0xFF80
    assert np.all(np.delete(o2, 7) == 0x3F80)


def pin_all_neginf_row_is_nan(lib):
    q = torch.zeros(1, 1, 2, D, dtype=torch.bfloat16)
    q[0, 0, 0, 0] = 1.0
    q[0, 0, 1, 0] = -1.0
    k = torch.zeros(1, 1, 3, D, dtype=torch.bfloat16)
    k[0, 0, :, 0] = float("-inf")        # row 0: every logit -inf; row 1: every logit +inf
    v = torch.ones(1, 1, 3, D, dtype=torch.bfloat16)
    o = oracle.attention(q, k, v, "bhsd", "rtna", lib=lib)["o_bits"]
    assert np.all(o == 0x7FC0)


# --------------------------------------------------------------------------- causal / GQA / LSE
def pin_causal_rows_are_prefix_attention(lib):
    """Causal row i (Sq = Skv) is plain attention over keys 0..i; with Skv = Sq + off it is
    attention over keys 0..i+off; rows with no visible key are NaN with LSE -inf."""
    for (Sq, Skv) in ((7, 7), (4, 9), (9, 4)):
        q, k, v = make_qkv(1, 2, Sq, Skv, D, "bhsd", seed=200 + Sq * 10 + Skv)
        for mode in ("rtne", "rtz"):
            c = oracle.attention(q, k, v, "bhsd", mode, causal=True, want_lse=True, lib=lib)
            for i in range(Sq):
                nvis = min(Skv, i + (Skv - Sq) + 1)
                if nvis <= 0:
                    assert np.all(c["o_bits"][:, :, i] == 0x7FC0)
                    assert np.all(np.isneginf(c["lse"][:, :, i]))
                    continue
                ref = oracle.attention(q[:, :, i:i + 1], k[:, :, :nvis], v[:, :, :nvis], "bhsd",
                                       mode, want_lse=True, lib=lib)
                assert np.array_equal(c["o_bits"][:, :, i], ref["o_bits"][:, :, 0]), (Sq, Skv, i)
                assert np.array_equal(c["lse"][:, :, i], ref["lse"][:, :, 0])


def pin_causal_first_row_is_first_value(lib):
    """Sq = Skv: query 0 sees only key 0, so its output is V row 0 in every mode."""
    q, k, v = make_qkv(2, 3, 6, 6, D, "bshd", seed=210, sigma=3.0)
    for mode in MODES:
        o = oracle.attention(q, k, v, "bshd", mode, causal=True, lib=lib)["o_bits"]
        vb = _bits(v.permute(0, 2, 1, 3).contiguous())          # (B, H, S, d)
        assert np.array_equal(o[:, :, 0], vb[:, :, 0]), mode


def pin_grouped_heads_equal_repeated_heads(lib):
    """K/V with Hkv heads (query head h reads K/V head h // (H/Hkv)) equal plain attention
    with each K/V head repeated H/Hkv times; Hkv = 1 is multi-query attention."""
    B, H, Sq, Skv = 2, 6, 5, 11
    for Hkv in (1, 2, 3, 6):
        for layout in ("bshd", "bhsd"):
            g = torch.Generator().manual_seed(220 + Hkv)
            q = torch.randn(shape(layout, B, H, Sq, D), generator=g).to(torch.bfloat16)
            k = torch.randn(shape(layout, B, Hkv, Skv, D), generator=g).to(torch.bfloat16)
            v = torch.randn(shape(layout, B, Hkv, Skv, D), generator=g).to(torch.bfloat16)
            ax = 2 if layout == "bshd" else 1
            kr = k.repeat_interleave(H // Hkv, dim=ax).contiguous()
            vr = v.repeat_interleave(H // Hkv, dim=ax).contiguous()
            for causal in (False, True):
                a = oracle.attention(q, k, v, layout, "rtna", causal=causal, lib=lib)["o_bits"]
                b = oracle.attention(q, kr, vr, layout, "rtna", causal=causal, lib=lib)["o_bits"]
                assert np.array_equal(a, b), (Hkv, layout, causal)


def pin_lse_closed_forms(lib):
    """LSE = log sum_j exp(s_j): two keys give log(e^s1 + e^s2); Q = 0 gives log(Skv);
    NaN rows give NaN; an all -inf row gives -inf."""
    g = torch.Generator().manual_seed(230)
    q = torch.randn(1, 1, 3, D, generator=g).to(torch.bfloat16)
    k = torch.randn(1, 1, 2, D, generator=g).to(torch.bfloat16)
    v = torch.randn(1, 1, 2, D, generator=g).to(torch.bfloat16)
    lse = oracle.attention(q, k, v, "bhsd", "rtne", want_lse=True, lib=lib)["lse"][0, 0]
    qd, kd = q.double()[0, 0], k.double()[0, 0]
    for i in range(3):
        s = [float((qd[i] * kd[j]).sum()) / math.sqrt(D) for j in range(2)]
        mx = max(s)
        assert abs(lse[i] - (mx + math.log(sum(math.exp(x - mx) for x in s)))) < 1e-13
    q0 = torch.zeros(1, 2, 4, D, dtype=torch.bfloat16)
    kk = torch.randn(1, 2, 37, D, generator=g).to(torch.bfloat16)
    vv = torch.randn(1, 2, 37, D, generator=g).to(torch.bfloat16)
    l0 = oracle.attention(q0, kk, vv, "bhsd", "rtne", want_lse=True, lib=lib)["lse"]
    assert np.allclose(l0, math.log(37), rtol=0, atol=1e-14)
    qn = q.clone()
    qn[0, 0, 1, 0] = float("nan")
    ln = oracle.attention(qn, k, v, "bhsd", "rtne", want_lse=True, lib=lib)["lse"][0, 0]
    assert math.isnan(ln[1]) and math.isfinite(ln[0])
    qi = torch.zeros(1, 1, 1, D, dtype=torch.bfloat16)
    qi[..., 0] = 1.0
    ki = torch.zeros(1, 1, 3, D, dtype=torch.bfloat16)
    ki[..., 0] = float("-inf")
    li = oracle.attention(qi, ki, v[:, :, :1].expand(1, 1, 3, D).contiguous(), "bhsd", "rtne",
                          want_lse=True, lib=lib)["lse"]
    assert np.isneginf(li).all()


def pin_brute_force_causal_lse_mpmath(lib):
    """Causal, grouped heads and LSE on tiny shapes against 50-digit arithmetic."""
    import mpmath
    mpmath.mp.dps = 50
    B, H, Hkv, Sq, Skv = 1, 2, 1, 3, 5
    g = torch.Generator().manual_seed(240)
    q = torch.randn(B, H, Sq, D, generator=g).to(torch.bfloat16)
    k = torch.randn(B, Hkv, Skv, D, generator=g).to(torch.bfloat16)
    v = torch.randn(B, Hkv, Skv, D, generator=g).to(torch.bfloat16)
    res = oracle.attention(q, k, v, "bhsd", "rtne", causal=True, want_f64=True, want_lse=True,
                           want_a=True, lib=lib)
    inv = 1 / mpmath.sqrt(D)
    for h in range(H):
        qd, kd, vd = q.double().numpy()[0, h], k.double().numpy()[0, 0], v.double().numpy()[0, 0]
        for i in range(Sq):
            nvis = i + (Skv - Sq) + 1
            s = [mpmath.fsum(mpmath.mpf(float(qd[i, x])) * mpmath.mpf(float(kd[j, x]))
                             for x in range(D)) * inv for j in range(nvis)]
            m = max(s)
            w = [mpmath.exp(sj - m) for sj in s]
            l = mpmath.fsum(w)
            assert abs(res["lse"][0, h, i] - float(m + mpmath.log(l))) < 1e-13
            for x in range(0, D, 7):
                val = mpmath.fsum(w[j] * mpmath.mpf(float(vd[j, x])) for j in range(nvis)) / l
                assert abs(res["o_f64"][0, h, i, x] - float(val)) <= 1e-13 * res["a"][0, h, i, x]
                if not bx.near_midpoint(val):
                    assert res["o_bits"][0, h, i, x] == bx.round_exact(val, "rtne")


# --------------------------------------------------------------------------- error scales
# A = sum_j w_j |v_jx| / l is the forward-error scale of output column x: the parity
# criterion accepts |gpu - O| <= 2^-8 A + ulp(O) where the literal 2-ULP rule cannot hold.
# A too large would silently widen every GPU check, so its value is pinned here on its own.
def pin_error_scale_nonnegative_v_is_output(lib):
    """V >= 0: every term w_j v_jx is non-negative, so A equals O itself (the same sums)."""
    for layout in ("bshd", "bhsd"):
        q, k, v = make_qkv(1, 2, 5, 70, D, layout, seed=500, sigma=2.0)
        v = v.abs()
        res = oracle.attention(q, k, v, layout, "rtne", want_f64=True, want_a=True, lib=lib)
        assert np.all(res["o_f64"] > 0)
        assert np.allclose(res["a"], res["o_f64"], rtol=1e-14, atol=0), layout


def pin_error_scale_uniform_weights(lib):
    """Q = 0: every logit is 0, every weight 1 and l = Skv, so A is the column mean of |V|
    (and |O| <= A, with equality only where a column has one sign)."""
    q, k, v = make_qkv(1, 2, 3, 41, D, "bshd", seed=501)
    q = torch.zeros_like(q)
    res = oracle.attention(q, k, v, "bshd", "rtne", want_f64=True, want_a=True, lib=lib)
    vv = v.permute(0, 2, 1, 3).double().numpy()                  # (B, H, Skv, d)
    mean_abs = np.abs(vv).mean(axis=2, keepdims=True)
    assert np.allclose(res["a"], np.broadcast_to(mean_abs, res["a"].shape), rtol=1e-14, atol=0)
    assert np.all(np.abs(res["o_f64"]) <= res["a"] * (1 + 1e-14))
    assert np.any(np.abs(res["o_f64"]) < 0.5 * res["a"])          # cancellation is present


def pin_error_scale_two_keys(lib):
    """Two keys: A = sigma(s1 - s2) |v1| + sigma(s2 - s1) |v2| with s = q.k / sqrt(d)."""
    g = torch.Generator().manual_seed(502)
    q = torch.randn(1, 1, 6, D, generator=g).to(torch.bfloat16)
    k = torch.randn(1, 1, 2, D, generator=g).to(torch.bfloat16)
    v = torch.randn(1, 1, 2, D, generator=g).to(torch.bfloat16)
    res = oracle.attention(q, k, v, "bhsd", "rtne", want_a=True, lib=lib)
    qd, kd, vd = q.double()[0, 0], k.double()[0, 0], v.double()[0, 0].abs().numpy()
    for i in range(6):
        s = [float((qd[i] * kd[j]).sum()) / math.sqrt(D) for j in range(2)]
        a = 1.0 / (1.0 + math.exp(s[1] - s[0]))
        want = a * vd[0] + (1.0 - a) * vd[1]
        assert np.allclose(res["a"][0, 0, i], want, rtol=1e-13, atol=0), i


def pin_error_scale_brute_force_mpmath(lib):
    """A against 50-digit arithmetic on tiny shapes (d = 128 and 64), to 1e-13 relative."""
    import mpmath
    mpmath.mp.dps = 50
    for seed, (Sq, Skv, d, sigma) in enumerate(((2, 3, D, 1.0), (3, 6, D, 4.0), (2, 5, 64, 2.0))):
        q, k, v = make_qkv(1, 1, Sq, Skv, d, "bhsd", seed=510 + seed, sigma=sigma)
        res = oracle.attention(q, k, v, "bhsd", "rtne", want_a=True, lib=lib)
        qd, kd, vd = (t.double().numpy()[0, 0] for t in (q, k, v))
        inv = 1 / mpmath.sqrt(d)
        for i in range(Sq):
            s = [mpmath.fsum(mpmath.mpf(float(qd[i, x])) * mpmath.mpf(float(kd[j, x]))
                             for x in range(d)) * inv for j in range(Skv)]
            m = max(s)
            w = [mpmath.exp(sj - m) for sj in s]
            l = mpmath.fsum(w)
            for x in range(d):
                want = mpmath.fsum(w[j] * abs(mpmath.mpf(float(vd[j, x]))) for j in range(Skv)) / l
                got = res["a"][0, 0, i, x]
                assert abs(got - float(want)) <= 1e-13 * float(want), (seed, i, x, got, want)


def pin_bwd_error_scales_single_key(lib):
    """One key: p = 1 for every row, so with dP_i = dO_i.v and |D|_i = sum_x |dO_ix| |v_x|
    (O_i = v):  dV_a = sum over the rows and query heads of |dO_i|,
    dQ_a[i, x] = c (|dP_i| + |D|_i) |k_x|,  dK_a[x] = c sum_i (|dP_i| + |D|_i) |q_ix|."""
    g0 = torch.Generator().manual_seed(520)
    H, Hkv, Sq, d = 4, 2, 5, 32
    q = torch.randn(1, H, Sq, d, generator=g0).to(torch.bfloat16)
    k = torch.randn(1, Hkv, 1, d, generator=g0).to(torch.bfloat16)
    v = torch.randn(1, Hkv, 1, d, generator=g0).to(torch.bfloat16)
    g = torch.randn(1, H, Sq, d, generator=g0).to(torch.bfloat16)
    res = oracle.backward(q, k, v, g, "bhsd", want_a=True, lib=lib)
    c = 1.0 / math.sqrt(d)
    qd, kd, vd, gd = (t.double().numpy()[0] for t in (q, k, v, g))
    grp = H // Hkv
    for kh in range(Hkv):
        heads = range(kh * grp, (kh + 1) * grp)
        dv_a = sum(np.abs(gd[h]).sum(axis=0) for h in heads)
        assert np.allclose(res["dv_a"][0, kh, 0], dv_a, rtol=1e-14, atol=0), kh
        dk_a = np.zeros(d)
        for h in heads:
            dp = gd[h] @ vd[kh, 0]                                  # (Sq,)
            dabs = np.abs(gd[h]) @ np.abs(vd[kh, 0])                # (Sq,)
            coef = np.abs(dp) + dabs
            want_dq = c * coef[:, None] * np.abs(kd[kh, 0])[None, :]
            assert np.allclose(res["dq_a"][0, h], want_dq, rtol=1e-13, atol=0), h
            dk_a += c * (coef[:, None] * np.abs(qd[h])).sum(axis=0)
        assert np.allclose(res["dk_a"][0, kh, 0], dk_a, rtol=1e-13, atol=0), kh


def pin_bwd_error_scales_brute_force_mpmath(lib):
    """dQ_a, dK_a and dV_a against 50-digit sums of the term magnitudes on a 2 x 3 case:
    dV_a[j] = sum_i p_ij |dO_i|, dQ_a[i] = c sum_j p_ij (|dP_ij| + |D|_i) |k_j| and
    dK_a[j] = c sum_i p_ij (|dP_ij| + |D|_i) |q_i|, with |D|_i = sum_x |dO_ix| |O_ix|."""
    import mpmath
    mpmath.mp.dps = 50
    g0 = torch.Generator().manual_seed(530)
    Sq, Skv, d = 2, 3, 16
    q, k, v, g = (torch.randn(1, 1, n, d, generator=g0).to(torch.bfloat16)
                  for n in (Sq, Skv, Skv, Sq))
    res = oracle.backward(q, k, v, g, "bhsd", want_a=True, lib=lib)
    mp = lambda t: [[mpmath.mpf(float(x)) for x in row] for row in t.double().numpy()[0, 0]]
    Q, K, V, G = mp(q), mp(k), mp(v), mp(g)
    c = 1 / mpmath.sqrt(d)
    dot = lambda a, b: mpmath.fsum(x * y for x, y in zip(a, b))
    P, coef = [], []
    for i in range(Sq):
        s = [c * dot(Q[i], K[j]) for j in range(Skv)]
        m = max(s)
        w = [mpmath.exp(t - m) for t in s]
        l = mpmath.fsum(w)
        p = [t / l for t in w]
        o = [mpmath.fsum(p[j] * V[j][x] for j in range(Skv)) for x in range(d)]
        dabs = mpmath.fsum(abs(G[i][x]) * abs(o[x]) for x in range(d))
        P.append(p)
        coef.append([p[j] * (abs(dot(G[i], V[j])) + dabs) for j in range(Skv)])
    for x in range(d):
        for i in range(Sq):
            want = c * mpmath.fsum(coef[i][j] * abs(K[j][x]) for j in range(Skv))
            assert abs(res["dq_a"][0, 0, i, x] - float(want)) <= 1e-13 * float(want), (i, x)
        for j in range(Skv):
            want_k = c * mpmath.fsum(coef[i][j] * abs(Q[i][x]) for i in range(Sq))
            want_v = mpmath.fsum(P[i][j] * abs(G[i][x]) for i in range(Sq))
            assert abs(res["dk_a"][0, 0, j, x] - float(want_k)) <= 1e-13 * float(want_k), (j, x)
            assert abs(res["dv_a"][0, 0, j, x] - float(want_v)) <= 1e-13 * float(want_v), (j, x)


# --------------------------------------------------------------------------- backward
def _fd_gradients(q, k, v, g, layout, causal, lib, h=1e-6):
    """Central differences of L = sum(dO * O) through the fp64 forward, for every element of
    q, k and v (tiny shapes only)."""
    base = [np.ascontiguousarray(t.double().numpy()) for t in (q, k, v)]
    gd = g.double().numpy()
    out = []
    for which in range(3):
        grad = np.empty_like(base[which])
        flat = grad.reshape(-1)
        for idx in range(flat.size):
            vals = []
            for sgn in (1.0, -1.0):
                ts = [b.copy() for b in base]
                ts[which].reshape(-1)[idx] += sgn * h
                o = oracle.forward_f64(*ts, layout=layout, causal=causal, lib=lib)
                vals.append(float((o * gd).sum()))
            flat[idx] = (vals[0] - vals[1]) / (2 * h)
        out.append(grad)
    return out


def pin_bwd_matches_finite_differences(lib):
    """dQ, dK, dV equal the numerical derivative of sum(dO * O) through the fp64 forward, with
    and without the causal mask and with grouped K/V heads (2 query heads per K/V head)."""
    g0 = torch.Generator().manual_seed(400)
    for causal, (Sq, Skv), layout in ((False, (3, 5), "bshd"), (True, (4, 4), "bhsd"),
                                      (True, (2, 5), "bshd")):
        shp_q = shape(layout, 1, 2, Sq, 16)
        shp_k = shape(layout, 1, 1, Skv, 16)
        q = torch.randn(shp_q, generator=g0).to(torch.bfloat16)
        k = torch.randn(shp_k, generator=g0).to(torch.bfloat16)
        v = torch.randn(shp_k, generator=g0).to(torch.bfloat16)
        g = torch.randn(shp_q, generator=g0).to(torch.bfloat16)
        res = oracle.backward(q, k, v, g, layout, causal=causal, lib=lib)
        fd = _fd_gradients(q, k, v, g, layout, causal, lib)
        for name, num in zip(("dq", "dk", "dv"), fd):
            err = np.abs(res[name] - num)
            assert np.all(err <= 1e-7 * (1 + np.abs(num))), (causal, name, float(err.max()))


def pin_bwd_forward_f64_equals_forward(lib):
    """The fp64-input forward used for the derivative equals the bf16 oracle's unrounded
    output on bf16-representable inputs."""
    q, k, v = make_qkv(2, 4, 9, 13, 32, "bshd", seed=410, Hkv=2)
    for causal in (False, True):
        o64 = oracle.forward_f64(q.double().numpy(), k.double().numpy(), v.double().numpy(),
                                 "bshd", causal=causal, lib=lib)
        ref = oracle.attention(q, k, v, "bshd", "rtne", want_f64=True, causal=causal,
                               lib=lib)["o_f64"]                    # (B, H, Sq, d)
        assert np.allclose(o64.transpose(0, 2, 1, 3), ref, rtol=1e-14, atol=1e-15)


def pin_bwd_single_key_and_delta(lib):
    """One key: every weight is 1, so dS = 0 (dQ = dK = 0) and dV is the sum of dO over the
    rows and query heads that read it; D_i equals dO_i . O_i from the forward."""
    g0 = torch.Generator().manual_seed(420)
    q = torch.randn(1, 4, 6, 32, generator=g0).to(torch.bfloat16)
    k = torch.randn(1, 2, 1, 32, generator=g0).to(torch.bfloat16)
    v = torch.randn(1, 2, 1, 32, generator=g0).to(torch.bfloat16)
    g = torch.randn(1, 4, 6, 32, generator=g0).to(torch.bfloat16)
    res = oracle.backward(q, k, v, g, "bhsd", want_delta=True, lib=lib)
    assert np.all(res["dq"] == 0) and np.all(res["dk"] == 0)
    gd = g.double().numpy()
    want = np.stack([gd[0, 0:2].sum(axis=(0, 1)), gd[0, 2:4].sum(axis=(0, 1))])[None, :, None, :]
    assert np.allclose(res["dv"], want, rtol=1e-14, atol=1e-13)
    q, k, v = make_qkv(1, 2, 7, 11, 32, "bhsd", seed=421)
    g = torch.randn(1, 2, 7, 32, generator=g0).to(torch.bfloat16)
    res = oracle.backward(q, k, v, g, "bhsd", want_delta=True, lib=lib)
    o = oracle.attention(q, k, v, "bhsd", "rtne", want_f64=True, lib=lib)["o_f64"]
    assert np.allclose(res["delta"], (g.double().numpy() * o).sum(axis=-1), rtol=1e-13, atol=1e-14)


ALL_PINS = [v for k_, v in sorted(globals().items()) if k_.startswith("pin_")]
