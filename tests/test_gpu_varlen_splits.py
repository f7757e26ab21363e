"""GPU parity of key splits in the variable-length and paged forwards (max_splits >= 2)
against the fp64 oracle (needs a GB300).

With fewer (sequence, query block, head) items than CTAs, the preprocessing kernel splits each
block's key tiles into up to max_splits contiguous parts, more for costlier blocks; the
attention kernel runs each part into an fp32 slot and a merge kernel combines the parts with
log-sum-exp weights ([MoonMath] "Data placement and the 16x16x16 choice": the key split of the
tail, here on the variable-length work list).  The result must meet the forward's criteria and
the LSE tolerance, be the same bits on every run whatever the workspace held before, write
nothing outside its outputs, and the schedule must be the one the header's rule gives (read
back from the work list, which sits in the caller's workspace after the per-sequence tensor
maps and the item count).
"""
import ctypes

import numpy as np
import pytest
import torch

import oracle
from tests import parity
from tests.test_gpu_canaries import guarded, guards_intact
from tests.test_gpu_causal_gqa import check_lse
from tests.test_gpu_paged import build_cache
from tests.test_gpu_varlen import BF16_SENTINEL, F32_SENTINEL, lse_scale, offsets, packed

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def attn():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import bf16_attention_forward_gb300 as a
    a.load()
    return a


def cdiv(a, b):
    return -(-a // b)


def pack_shift(H, Hkv, pack):
    return (H // Hkv).bit_length() - 1 if pack else 0


def grid_for(lq, H, Hkv, pack, max_splits, max_ctas=0, max_seqlen_q=0):
    """The attention kernel's CTA count: one per SM, at most max_ctas, and (max_seqlen_q > 0)
    no more than B * (H >> shift) * ceil(max_seqlen_q / tokens per block) items, times
    max_splits when that bound is below the SM count."""
    G = torch.cuda.get_device_properties(0).multi_processor_count
    if 0 < max_ctas < G:
        G = max_ctas
    sh = pack_shift(H, Hkv, pack)
    if max_seqlen_q > 0:
        cap = len(lq) * (H >> sh) * cdiv(max_seqlen_q, 256 >> sh)
        if max_splits > 1:
            cap = G if cap > G else cap * max_splits
        G = min(G, cap)
    return max(G, 1)


ITEM_OVERHEAD_TILES = 2


def busiest(costs, M, cap, per, grid):
    """The busiest CTA's modelled work: pairs heaviest first, each as min(cap, ceil(c / M))
    near-equal parts in a row, per items an entry, item k on the CTA the alternating
    round-robin gives it, an item costing its tiles plus ITEM_OVERHEAD_TILES."""
    load = [0] * grid
    k = 0
    for c in sorted(costs, reverse=True):
        n = min(cap, cdiv(c, M))
        for i in range(n):
            t = c // n + (1 if i < c % n else 0)
            for _ in range(per):
                r, col = divmod(k, grid)
                load[grid - 1 - col if r & 1 else col] += t + ITEM_OVERHEAD_TILES
                k += 1
    return max(load)


def expected_schedule(lq, lk, H, Hkv, causal, pack, grid, max_splits):
    """Entries (b, qb, part, parts) and costs by the stated rule.  With P pairs and Gp = grid //
    (H >> shift) entry places (max_splits >= 2, Gp > P), a pair of cost c gets n(c) =
    min(max_splits, Gp, ceil(c / M)) parts, M the smallest with sum n(c) <= Gp; or, when
    2 P (H >> shift) >= grid, the smallest with sum n(c) <= 2 Gp if its busiest CTA has less
    work (searches by brute force here)."""
    sh = pack_shift(H, Hkv, pack)
    tb = 256 >> sh
    pairs = []
    for b, (sq, skv) in enumerate(zip(lq, lk)):
        if sq <= 0 or skv <= 0:
            continue
        for qb in range(cdiv(sq, tb)):
            tiles = cdiv(skv, 128)
            if causal:
                last = (((qb + 1) * 256) >> sh) - 1 + skv - sq
                tiles = min(tiles, 1 if last < 0 else last // 128 + 1)
            pairs.append((b, qb, min(tiles, 4095)))
    per = H >> sh
    P, gp = len(pairs), grid // per
    cap = min(max_splits, gp)
    costs = [p[2] for p in pairs]
    M = 0
    if max_splits > 1 and P > 0 and gp > P and grid <= 1024:
        def smallest(places):
            return next(m for m in range(1, max(costs) + 1)
                        if sum(min(cap, cdiv(c, m)) for c in costs) <= places)
        M = smallest(gp)
        if 2 * P * per >= grid:
            m2 = smallest(2 * gp)
            if busiest(costs, m2, cap, per, grid) < busiest(costs, M, cap, per, grid):
                M = m2
    entries, cost = [], {}
    for b, qb, c in pairs:
        n = min(cap, cdiv(c, M)) if M else 1
        cost[(b, qb)] = c
        entries += [(b, qb, i, n) for i in range(n)]
    return entries, cost


def read_schedule(ws, B):
    """(item count, entries in list order) from the workspace after a call."""
    base = ws.data_ptr()
    off = ((base + 127) & ~127) - base + B * 4 * 128
    n_items = int(ws[off:off + 4].cpu().view(torch.int32)[0])
    return n_items, off + 16


def check_schedule(ws, lq, lk, H, Hkv, causal, pack, grid, max_splits):
    entries, cost = expected_schedule(lq, lk, H, Hkv, causal, pack, grid, max_splits)
    per = H >> pack_shift(H, Hkv, pack)
    n_items, off = read_schedule(ws, len(lq))
    assert n_items == len(entries) * per
    raw = ws[off:off + 16 * len(entries)].cpu().view(torch.int32).numpy().reshape(-1, 4)
    got = [tuple(int(x) for x in e) for e in raw]
    assert sorted(got) == sorted(entries)
    # heaviest first, each pair's parts consecutive and in order
    costs = [cost[(b, qb)] for b, qb, _, _ in got]
    assert all(x >= y for x, y in zip(costs, costs[1:]))
    for i, (b, qb, part, n) in enumerate(got):
        if part > 0:
            assert got[i - 1] == (b, qb, part - 1, n)
    if any(n > 1 for *_, n in entries):
        assert n_items <= 2 * grid, "more split items than slots"
    return entries


def varlen_ws_bytes(attn, lq, lk, H, Hkv, d, pack, max_splits, total_q):
    a = attn.VarlenArgs()
    a.B, a.H, a.Hkv, a.total_q, a.total_k, a.d = len(lq), H, Hkv, total_q, sum(lk), d
    a.pack_heads, a.max_splits = int(pack), max_splits
    n = int(attn.load().attn_fwd_varlen_workspace_size(ctypes.byref(a)))
    assert n > 0
    return n


def run(attn, q, k, v, cu_q, cu_k, ws, mode, causal, **kw):
    qd, kd, vd = (t.cuda() for t in (q, k, v))
    obuf, o = guarded(q.numel(), "bf16")
    lbuf, lse = guarded(q.shape[0] * q.shape[1], "f32")
    o.view(torch.int16).fill_(BF16_SENTINEL)
    lse.view(torch.int32).fill_(F32_SENTINEL)
    cq = torch.as_tensor(np.asarray(cu_q, dtype=np.int32)).cuda()
    ck = torch.as_tensor(np.asarray(cu_k, dtype=np.int32)).cuda()
    attn.attn_fwd_varlen(qd, kd, vd, cq, ck, o=o.view(q.shape), lse=lse.view(q.shape[1], -1), round=mode,
                         causal=causal, workspace=ws, **kw)
    torch.cuda.synchronize()
    st, site = attn.device_status()
    assert st == 0, "device status %d at site %d" % (st, site)
    assert guards_intact(obuf, "bf16") and guards_intact(lbuf, "f32")
    return o.view(q.shape), lse.view(q.shape[1], -1)


CASES = [  # (lens_q, lens_k, H, Hkv, d, mode, causal, pack, max_splits, max_ctas, max_seqlen_q)
    ([1, 1, 1, 1], [5000, 300, 1, 2000], 16, 2, 128, "rtne", True, True, 8, 0, 1),     # packed decode
    ([1, 1, 1], [3000, 4100, 129], 4, 2, 128, "rtne", True, False, 16, 0, 0),           # decode, one head a tile
    ([700], [3000], 2, 1, 64, "rtna", False, False, 4, 0, 0),                           # one long prefill chunk
    ([300, 40], [200, 1000], 2, 2, 128, "rtz", True, False, 16, 0, 0),                  # rows with no visible key
    ([129, 1], [900, 4000], 4, 1, 128, "rtne", False, False, 3, 20, 0),                 # few CTAs: uneven parts
    ([3, 2], [700, 260], 8, 1, 64, "rtz", True, True, 8, 0, 0),                         # speculative tokens, packed
    ([1] * 12, [2870, 2837, 6945, 5115, 7500, 2250, 4000, 6000, 4500, 8000, 3500, 5500],
     32, 8, 128, "rtne", True, True, 16, 0, 1),                                         # 12 caches: two waves
]


@pytest.mark.parametrize("case", CASES, ids=lambda c: "n%d_H%dKV%d_d%d_%s%s%s_s%d_g%d" % (
    len(c[0]), c[2], c[3], c[4], c[5], "_causal" if c[6] else "", "_pack" if c[7] else "", c[8], c[9]))
def test_varlen_key_splits(attn, case):
    lq, lk, H, Hkv, d, mode, causal, pack, ms, max_ctas, msq = case
    q, k, v = packed(sum(lq), sum(lk), H, Hkv, d, seed=10000 + sum(lk) + d)
    cu_q, cu_k = offsets(lq), offsets(lk)
    nbytes = varlen_ws_bytes(attn, lq, lk, H, Hkv, d, pack, ms, q.shape[0])
    wbuf, ws = guarded(nbytes, "ws")           # a workspace full of stale bytes
    kw = dict(pack_heads=pack, max_splits=ms, max_ctas=max_ctas, max_seqlen_q=msq)
    o, lse = run(attn, q, k, v, cu_q, cu_k, ws, mode, causal, **kw)
    assert guards_intact(wbuf, "ws")
    entries = check_schedule(ws, lq, lk, H, Hkv, causal, pack, grid_for(lq, H, Hkv, pack, ms, max_ctas, msq), ms)
    assert any(n > 1 for *_, n in entries), "the case was meant to split"
    ref = oracle.attention_varlen(q, k, v, cu_q, cu_k, mode, causal=causal, want_a=True, want_lse=True)
    ob = o.cpu().view(torch.int16).numpy().view(np.uint16)
    res = parity.compare(ob.reshape(-1, d), ref["o_bits"].reshape(-1, d), ref["a"].reshape(-1, d))
    assert res["ok"], res
    check_lse(lse.cpu().numpy().reshape(-1), ref["lse"].reshape(-1), lse_scale(q, k, cu_q, cu_k).reshape(-1))
    # the same bits again, from a workspace of 0xFF bytes (NaN in every fp32 slot)
    ws.fill_(0xFF)
    o2, lse2 = run(attn, q, k, v, cu_q, cu_k, ws, mode, causal, **kw)
    assert torch.equal(o2.view(torch.int16), o.view(torch.int16))
    assert torch.equal(lse2.view(torch.int32), lse.view(torch.int32))
    assert guards_intact(wbuf, "ws")


def test_varlen_key_splits_unused_when_items_fill_the_grid(attn):
    # 80 sequences x 2 blocks x 2 heads = 320 items, more than the CTAs: nothing is split and
    # the result is bit for bit the unsplit one
    lq, lk, H, Hkv, d = [300] * 80, [500] * 80, 2, 1, 128
    q, k, v = packed(sum(lq), sum(lk), H, Hkv, d, seed=10100)
    cu_q, cu_k = offsets(lq), offsets(lk)
    ws = torch.empty(varlen_ws_bytes(attn, lq, lk, H, Hkv, d, False, 4, q.shape[0]), dtype=torch.uint8,
                     device="cuda")
    o, lse = run(attn, q, k, v, cu_q, cu_k, ws, "rtne", True, max_splits=4)
    entries = check_schedule(ws, lq, lk, H, Hkv, True, False, grid_for(lq, H, Hkv, False, 4), 4)
    assert all(n == 1 for *_, n in entries)
    o0, lse0 = run(attn, q, k, v, cu_q, cu_k, None, "rtne", True)
    assert torch.equal(o.view(torch.int16), o0.view(torch.int16))
    assert torch.equal(lse.view(torch.int32), lse0.view(torch.int32))


def test_varlen_key_splits_empty_and_keyless_sequences(attn):
    # an empty sequence, one with queries but no keys (NaN rows, -inf LSE, written by the
    # preprocessing kernel) and a long one that splits; rows outside every sequence untouched
    lq, lk, H, d = [0, 5, 1, 0], [10, 0, 6000, 0], 2, 128
    Tq = 2 + sum(lq) + 3
    q, k, v = packed(Tq, sum(lk), H, H, d, seed=10200)
    cu_q, cu_k = offsets(lq, start=2), offsets(lk)
    ws = torch.empty(varlen_ws_bytes(attn, lq, lk, H, H, d, False, 8, Tq), dtype=torch.uint8, device="cuda")
    o, lse = run(attn, q, k, v, cu_q, cu_k, ws, "rtna", False, max_splits=8)
    check_schedule(ws, lq, lk, H, H, False, False, grid_for(lq, H, H, False, 8), 8)
    ref = oracle.attention_varlen(q, k, v, cu_q, cu_k, "rtna", want_a=True, want_lse=True)
    cov = ref["covered"]
    ob = o.cpu().view(torch.int16).numpy().view(np.uint16)
    res = parity.compare(ob[cov].reshape(-1, d), ref["o_bits"][cov].reshape(-1, d), ref["a"][cov].reshape(-1, d))
    assert res["ok"], res
    assert (ob[~cov] == BF16_SENTINEL).all()
    assert (ob[2:7] == 0x7FC0).all() and np.isneginf(lse.cpu().numpy()[:, 2:7]).all()
    assert (lse.cpu().numpy()[:, ~cov].view(np.int32) == F32_SENTINEL).all()


def test_paged_decode_key_splits(attn):
    # decoding over a paged cache with packed heads and key splits: the oracle's criteria, and
    # the bits of the variable-length call with splits on the keys gathered in order (same
    # schedule, same tiles)
    lq, lk, P, H, Hkv, d = [1] * 5, [6000, 1, 1300, 257, 3100], 256, 8, 2, 128
    q, k, v = packed(sum(lq), sum(lk), H, Hkv, d, seed=10300)
    kc, vc, table = build_cache(k, v, lk, P, seed=10301)
    cu_q = offsets(lq)
    a = attn.PagedArgs()
    a.B, a.H, a.Hkv, a.total_q, a.num_pages, a.page_size, a.max_pages, a.d = \
        len(lq), H, Hkv, q.shape[0], kc.shape[0], P, table.shape[1], d
    a.pack_heads, a.max_splits = 1, 8
    wbuf, ws = guarded(int(attn.load().attn_fwd_paged_workspace_size(ctypes.byref(a))), "ws")
    obuf, o = guarded(q.numel(), "bf16")
    lbuf, lse = guarded(H * q.shape[0], "f32")
    attn.attn_fwd_paged(q.cuda(), kc.cuda(), vc.cuda(), torch.as_tensor(cu_q).cuda(),
                        torch.as_tensor(np.asarray(lk, dtype=np.int32)).cuda(), torch.as_tensor(table).cuda(),
                        max_seqlen_q=1, o=o.view(q.shape), lse=lse.view(H, -1), causal=True, workspace=ws,
                        pack_heads=True, max_splits=8)
    torch.cuda.synchronize()
    st, site = attn.device_status()
    assert st == 0, (st, site)
    assert guards_intact(obuf, "bf16") and guards_intact(lbuf, "f32") and guards_intact(wbuf, "ws")
    entries = check_schedule(ws, lq, lk, H, Hkv, True, True, grid_for(lq, H, Hkv, True, 8, 0, 1), 8)
    assert any(n > 1 for *_, n in entries)
    ref = oracle.attention_paged(q, kc, vc, cu_q, lk, table, "rtne", causal=True, want_a=True, want_lse=True)
    ob = o.cpu().view(torch.int16).numpy().view(np.uint16)
    res = parity.compare(ob.reshape(-1, d), ref["o_bits"].reshape(-1, d), ref["a"].reshape(-1, d))
    assert res["ok"], res
    check_lse(lse.cpu().numpy().reshape(-1), ref["lse"].reshape(-1),
              lse_scale(q, k, cu_q, offsets(lk)).reshape(-1))
    ov, lv = attn.attn_fwd_varlen(q.cuda(), k.cuda(), v.cuda(), torch.as_tensor(cu_q).cuda(),
                                  torch.as_tensor(offsets(lk)).cuda(), max_seqlen_q=1, causal=True,
                                  return_lse=True, pack_heads=True, max_splits=8)
    torch.cuda.synchronize()
    assert torch.equal(o.view(q.shape).view(torch.int16), ov.view(torch.int16))
    assert torch.equal(lse.view(H, -1).view(torch.int32), lv.view(torch.int32))


def test_varlen_key_split_schedule_random(attn):
    # the preprocessing kernel's search for the longest part against brute force, over seeded
    # random batches, head layouts, part caps (some above the entry places) and CTA counts
    rng = np.random.default_rng(10400)
    for trial in range(32):
        B = int(rng.integers(1, 24))
        lq = rng.integers(0, 600, B)
        lq[rng.random(B) < 0.5] = 1
        lk = rng.integers(0, 30000, B)
        lq, lk = [int(x) for x in lq], [int(x) for x in lk]
        Hkv, grp = int(rng.choice([1, 2, 4])), int(rng.choice([1, 2, 4, 8]))
        H, d = Hkv * grp, int(rng.choice([64, 128]))
        pack, causal = bool(rng.integers(0, 2)), bool(rng.integers(0, 2))
        ms, max_ctas = int(rng.choice([2, 3, 8, 64, 1000])), int(rng.choice([0, 7, 40, 151]))
        msq = max(lq) if rng.random() < 0.5 else 0
        Tq, Tk = max(sum(lq), 1), max(sum(lk), 1)
        q = torch.randn((Tq, H, d), device="cuda").to(torch.bfloat16)
        k = torch.randn((Tk, Hkv, d), device="cuda").to(torch.bfloat16)
        v = torch.randn((Tk, Hkv, d), device="cuda").to(torch.bfloat16)
        ws = torch.empty(varlen_ws_bytes(attn, lq, lk, H, Hkv, d, pack, ms, Tq), dtype=torch.uint8, device="cuda")
        attn.attn_fwd_varlen(q, k, v, torch.as_tensor(offsets(lq)).cuda(), torch.as_tensor(offsets(lk)).cuda(),
                             max_seqlen_q=msq, causal=causal, workspace=ws, pack_heads=pack, max_splits=ms,
                             max_ctas=max_ctas)
        torch.cuda.synchronize()
        st, site = attn.device_status()
        assert st == 0, (trial, st, site)
        check_schedule(ws, lq, lk, H, Hkv, causal, pack, grid_for(lq, H, Hkv, pack, ms, max_ctas, msq), ms)


def test_varlen_key_splits_nonfinite_values(attn):
    # +inf in one key of one cache (a +inf or -inf logit, by the sign of the query's element)
    # and NaN in one value of another, both inside a part of a split: the merge must give the
    # oracle's NaN rows and NaN or finite LSE, bit for bit where non-finite
    lq, lk, H, Hkv, d = [1, 1, 1, 1], [3000, 2000, 5000, 900], 8, 2, 128
    q, k, v = packed(sum(lq), sum(lk), H, Hkv, d, seed=10500)
    cu_q, cu_k = offsets(lq), offsets(lk)
    k.view(torch.int16)[cu_k[1] + 700, 0, 5] = 0x7F80        # +inf
    v.view(torch.int16)[cu_k[2] + 4000, 1, 17] = 0x7FC1      # NaN
    ws = torch.empty(varlen_ws_bytes(attn, lq, lk, H, Hkv, d, True, 8, q.shape[0]), dtype=torch.uint8, device="cuda")
    o, lse = run(attn, q, k, v, cu_q, cu_k, ws, "rtne", True, pack_heads=True, max_splits=8, max_seqlen_q=1)
    entries = check_schedule(ws, lq, lk, H, Hkv, True, True, grid_for(lq, H, Hkv, True, 8, 0, 1), 8)
    assert any(n > 1 for *_, n in entries)
    ref = oracle.attention_varlen(q, k, v, cu_q, cu_k, "rtne", causal=True, want_a=True, want_lse=True)
    ob = o.cpu().view(torch.int16).numpy().view(np.uint16)
    res = parity.compare(ob.reshape(-1, d), ref["o_bits"].reshape(-1, d), ref["a"].reshape(-1, d))
    assert res["ok"], res
    assert res["n_nonfinite"] > 0, "the planted values reach no row"
    # the LSE's error scale from finite keys (the planted +inf would make it inf or NaN)
    k_fin = k.clone()
    k_fin.view(torch.int16)[cu_k[1] + 700, 0, 5] = 0
    check_lse(lse.cpu().numpy().reshape(-1), ref["lse"].reshape(-1), lse_scale(q, k_fin, cu_q, cu_k).reshape(-1))
