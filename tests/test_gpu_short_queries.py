"""GPU parity of the short-query path (Sq <= 128: one 128-row query tile per (b, h), where
the forward runs attn_fwd_short_kernel) against the fp64 oracle (needs a GB300).

That kernel splits every 128-key tile between two softmax warpgroups (keys 0-63 and 64-127),
each with its own running max, row sum and accumulator, and merges the halves at the end with
weights 2^((m_h - m) c), kept >= 2^-125 for a finite m_h.  The tests cover the features of
the forward (layouts, head dimensions, grouped heads, causal mask, key splits, rounding
modes, the log-sum-exp) on that path, plus the cases the merge decides: a half with no
visible key, and a finite weight far below the other half's maximum meeting an infinite V.
Tolerances are the forward's (see tests/parity.py and tests/test_gpu_causal_gqa.py).
"""
import pytest
import torch

from tests.test_gpu_causal_gqa import MODES, attn, check_ex  # noqa: F401  (fixture)
from workloads import make_qkv

pytestmark = pytest.mark.gpu

SHAPES = [  # (B, H, Hkv, Sq, Skv, d)
    (1, 4, 4, 1, 1000, 128), (2, 8, 2, 77, 3000, 128), (1, 2, 2, 128, 129, 128),
    (1, 3, 3, 100, 257, 64), (2, 4, 1, 128, 700, 64), (1, 1, 1, 5, 5, 128),
]


@pytest.mark.parametrize("shape", SHAPES, ids=lambda s: "B%dH%dHkv%dSq%dSkv%dd%d" % s)
@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("layout", ["bshd", "bhsd"])
def test_short_queries_match_oracle(attn, shape, causal, layout):
    B, H, Hkv, Sq, Skv, d = shape
    q, k, v = make_qkv(B, H, Sq, Skv, d, layout, seed=3000 + sum(shape), Hkv=Hkv)
    check_ex(attn, q, k, v, layout, "rtne", causal=causal)


@pytest.mark.parametrize("splits", [0, 3, 7])
def test_short_queries_all_modes_and_key_splits(attn, splits):
    q, k, v = make_qkv(1, 4, 128, 2000, 128, "bhsd", seed=3100, sigma=3.0, Hkv=2)
    for mode in MODES:
        check_ex(attn, q, k, v, "bhsd", mode, force_splits=splits)


def test_short_queries_nonfinite_inputs(attn):
    # +inf in K (NaN rows for q_i0 > 0, a dropped key for q_i0 < 0), 0 * inf logits, and
    # infinities in V, on the plain and the split path
    for splits in (0, 4):
        q, k, v = make_qkv(1, 2, 128, 900, 128, "bshd", seed=3200)
        k[0, 333, 1, 0] = float("inf")
        q[0, 5, 1, 0] = 0.0
        v[0, 10, 0, 7] = float("inf")
        v[0, 700, 0, 9] = float("-inf")
        for mode in MODES:
            check_ex(attn, q, k, v, "bshd", mode, force_splits=splits)


def test_merge_keeps_a_tiny_weight_against_an_infinite_value(attn):
    # One query, one tile: keys 0-63 have logit 0, keys 64-127 logit 1400 / sqrt(128)
    # (about 178 in base 2 above), and V holds +inf in key 3 (first half).  The exact result
    # is +inf in that column (a positive weight times +inf), finite elsewhere; the merge must
    # not let the first half's weight underflow to 0 (0 * inf would give NaN).
    q, k, v = make_qkv(1, 1, 1, 128, 128, "bhsd", seed=3300)
    q.zero_()
    q[0, 0, 0, 0] = 1.0
    k.zero_()
    k[0, 0, 64:, 0] = 1400.0
    v[0, 0, 3, 5] = float("inf")
    _, o, _ = check_ex(attn, q, k, v, "bhsd", "rtne")
    o = o.float().cpu()
    assert torch.isinf(o[0, 0, 0, 5]) and o[0, 0, 0, 5] > 0
    assert torch.isfinite(o[0, 0, 0, :5]).all() and torch.isfinite(o[0, 0, 0, 6:]).all()


def test_half_without_visible_keys(attn):
    # causal, Sq = Skv = 128: rows 0-63 see no key of the tile's second half
    for d in (128, 64):
        q, k, v = make_qkv(1, 2, 128, 128, d, "bshd", seed=3400 + d)
        for mode in MODES:
            check_ex(attn, q, k, v, "bshd", mode, causal=True)


@pytest.mark.parametrize("max_ctas", [0, 7, 1])
def test_short_queries_many_units_per_cta(attn, max_ctas):
    # B*H = 320 units of one query tile each, 3 key tiles per unit (an odd count, so the two S
    # buffers alternate across unit boundaries); max_ctas caps the grid so each CTA runs up to
    # all 320 units in turn (query double buffer, per-unit statistics, O hand-off)
    q, k, v = make_qkv(4, 80, 64, 300, 128, "bshd", seed=3500, Hkv=20)
    check_ex(attn, q, k, v, "bshd", "rtne", max_ctas=max_ctas)


@pytest.mark.parametrize("d", [128, 64])
def test_short_queries_many_units_causal_and_splits(attn, d):
    q, k, v = make_qkv(2, 100, 100, 400, d, "bhsd", seed=3600 + d)
    check_ex(attn, q, k, v, "bhsd", "rtna", causal=True, max_ctas=19)
    check_ex(attn, q, k, v, "bhsd", "rtz", force_splits=2, max_ctas=23)


@pytest.mark.parametrize("case", ["skv_le_128", "one_tile_splits", "causal_one_tile"])
def test_short_queries_one_tile_units_many_per_cta(attn, case):
    # units (or key splits) of a single key tile, many per CTA: the softmax warpgroups can then
    # finish a unit two ahead of the epilogue, and the per-unit statistics hand-off must hold
    if case == "skv_le_128":
        q, k, v = make_qkv(4, 100, 32, 100, 128, "bshd", seed=3700)
        check_ex(attn, q, k, v, "bshd", "rtne", max_ctas=3)
    elif case == "one_tile_splits":
        q, k, v = make_qkv(1, 8, 64, 512, 128, "bhsd", seed=3701)
        check_ex(attn, q, k, v, "bhsd", "rtz", force_splits=4, max_ctas=2)
    else:
        q, k, v = make_qkv(2, 200, 100, 100, 64, "bhsd", seed=3702)
        check_ex(attn, q, k, v, "bhsd", "rtna", causal=True, max_ctas=5)
