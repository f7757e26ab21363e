"""GPU parity of attention over a paged K/V cache (attn_fwd_paged) against the fp64 oracle
(needs a GB300).

Queries are packed as in the variable-length forward; each sequence's keys and values sit in
fixed-size pages of a cache, found through a block table ([FlyDSL] page: a paged KV cache is
among the layouts an attention kernel has to take).  Full pages load through one map over
the whole cache and a sequence's last page through a map narrowed to its used slots, so the
result must be bit for bit that of attn_fwd_varlen on the keys gathered in order, whatever
the page order, and whatever the cache holds outside the used slots (+-inf and NaN included).
"""
import ctypes

import numpy as np
import pytest
import torch

import oracle
from tests import parity
from tests.test_gpu_canaries import guarded, guards_intact
from tests.test_gpu_varlen import BF16_SENTINEL, F32_SENTINEL, SITE_SEQLENS, lse_scale, offsets, packed
from tests.test_gpu_causal_gqa import check_lse

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def attn():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import bf16_attention_forward_gb300 as a
    a.load()
    return a


def build_cache(k, v, lens, P, seed, spare=3, stale=True):
    """A paged cache holding each sequence's keys (k, v packed [sum(lens), Hkv, d]) in a
    seeded random page order, `spare` extra pages, and (stale=True) +inf / NaN / large values
    in every slot no key uses.  Returns (k_cache, v_cache, block_table [B, max_pages])."""
    rng = np.random.default_rng(seed)
    Hkv, d = k.shape[1], k.shape[2]
    need = [-(-n // P) for n in lens]
    n_pages = sum(need) + spare
    order = rng.permutation(n_pages)
    kc = torch.empty((n_pages, P, Hkv, d), dtype=torch.bfloat16)
    vc = torch.empty_like(kc)
    if stale:
        junk = torch.tensor([0x7F80, 0x7FC1, -0x80, 0x7F00], dtype=torch.int16)   # +inf, NaN, -inf, 2^127
        idx = torch.as_tensor(rng.integers(0, 4, kc.numel()))
        kc.view(torch.int16).view(-1)[:] = junk[idx]
        vc.view(torch.int16).view(-1)[:] = junk[torch.as_tensor(rng.integers(0, 4, vc.numel()))]
    else:
        kc.zero_()
        vc.zero_()
    maxp = max(1, max(need))
    table = np.zeros((len(lens), maxp), dtype=np.int32)
    row, nxt = 0, 0
    for b, n in enumerate(lens):
        for pg in range(need[b]):
            phys = int(order[nxt])
            nxt += 1
            m = min(P, n - pg * P)
            kc[phys, :m] = k[row + pg * P: row + pg * P + m]
            vc[phys, :m] = v[row + pg * P: row + pg * P + m]
            table[b, pg] = phys
        row += n
    return kc, vc, table


def run_paged(attn, q, kc, vc, cu_q, lens_k, table, mode="rtne", causal=False, **kw):
    qd = q.cuda()
    o = torch.empty_like(qd)
    o.view(torch.int16).fill_(BF16_SENTINEL)
    lse = torch.empty((q.shape[1], q.shape[0]), dtype=torch.float32, device="cuda")
    lse.view(torch.int32).fill_(F32_SENTINEL)
    attn.attn_fwd_paged(qd, kc.cuda(), vc.cuda(), torch.as_tensor(np.asarray(cu_q, dtype=np.int32)).cuda(),
                        torch.as_tensor(np.asarray(lens_k, dtype=np.int32)).cuda(),
                        torch.as_tensor(np.asarray(table, dtype=np.int32)).cuda(), o=o, lse=lse, round=mode,
                        causal=causal, **kw)
    torch.cuda.synchronize()
    return o, lse


def status_ok(attn):
    st, site = attn.device_status()
    assert st == 0, "device status %d at site %d" % (st, site)


CASES = [  # (lens_q, lens_k, H, Hkv, d, page_size, mode, causal)
    ([300, 1, 128], [300, 700, 128], 4, 2, 128, 128, "rtne", False),
    ([64, 512, 1], [1000, 512, 129], 4, 2, 128, 256, "rtne", True),    # chunked prefill
    ([200, 17], [1023, 17], 2, 2, 64, 512, "rtna", True),
    ([129, 255], [384, 257], 3, 1, 128, 128, "rtz", False),
]


@pytest.mark.parametrize("case", CASES, ids=lambda c: "n%d_H%dKV%d_d%d_P%d_%s%s" % (
    len(c[0]), c[2], c[3], c[4], c[5], c[6], "_causal" if c[7] else ""))
def test_paged_matches_oracle_and_varlen(attn, case):
    lq, lk, H, Hkv, d, P, mode, causal = case
    q, k, v = packed(sum(lq), sum(lk), H, Hkv, d, seed=9000 + P + d)
    kc, vc, table = build_cache(k, v, lk, P, seed=9001)
    cu_q = offsets(lq)
    o, lse = run_paged(attn, q, kc, vc, cu_q, lk, table, mode, causal)
    status_ok(attn)
    ref = oracle.attention_paged(q, kc, vc, cu_q, lk, table, mode, causal=causal, want_a=True, want_lse=True)
    ob = o.cpu().view(torch.int16).numpy().view(np.uint16)
    res = parity.compare(ob.reshape(-1, d), ref["o_bits"].reshape(-1, d), ref["a"].reshape(-1, d))
    assert res["ok"], res
    check_lse(lse.cpu().numpy().reshape(-1), ref["lse"].reshape(-1),
              lse_scale(q, k, cu_q, offsets(lk)).reshape(-1))
    # the same keys gathered in order, through the variable-length path: the same bits
    ov, lv = attn.attn_fwd_varlen(q.cuda(), k.cuda(), v.cuda(), torch.as_tensor(cu_q).cuda(),
                                  torch.as_tensor(offsets(lk)).cuda(), round=mode, causal=causal, return_lse=True)
    torch.cuda.synchronize()
    assert torch.equal(o.view(torch.int16), ov.view(torch.int16))
    assert torch.equal(lse.view(torch.int32), lv.view(torch.int32))


def test_paged_page_order_and_stale_slots_change_nothing(attn):
    lq, lk, P = [300, 90], [1100, 300], 256
    q, k, v = packed(sum(lq), sum(lk), 2, 1, 128, seed=9100)
    cu_q = offsets(lq)
    kc0, vc0, t0 = build_cache(k, v, lk, P, seed=1, spare=0, stale=False)
    base, base_lse = run_paged(attn, q, kc0, vc0, cu_q, lk, t0, causal=True)
    status_ok(attn)
    for seed in (2, 3):
        kc, vc, t = build_cache(k, v, lk, P, seed=seed, spare=4, stale=True)
        o, lse = run_paged(attn, q, kc, vc, cu_q, lk, t, causal=True)
        status_ok(attn)
        assert torch.equal(o.view(torch.int16), base.view(torch.int16)), seed
        assert torch.equal(lse.view(torch.int32), base_lse.view(torch.int32)), seed


def test_paged_shared_prefix_pages(attn):
    # three sequences on one 640-key prefix (five 128-slot pages): the whole prefix, its first
    # 300 keys, and the prefix plus one page of their own
    P, H, d = 128, 2, 128
    q, k, v = packed(3 * 64, 768, H, H, d, seed=9200)
    kc, vc, t = build_cache(k, v, [768], P, seed=4, spare=1)
    row = t[0]
    table = np.stack([row, row, row])
    lk = [640, 300, 768]
    cu_q = offsets([64, 64, 64])
    o, _ = run_paged(attn, q, kc, vc, cu_q, lk, table, causal=True)
    status_ok(attn)
    ref = oracle.attention_paged(q, kc, vc, cu_q, lk, table, causal=True, want_a=True)
    ob = o.cpu().view(torch.int16).numpy().view(np.uint16)
    res = parity.compare(ob.reshape(-1, d), ref["o_bits"].reshape(-1, d), ref["a"].reshape(-1, d))
    assert res["ok"], res


def test_paged_writes_stay_in_bounds(attn):
    lq, lk, P, H, d = [130, 1, 77], [200, 5, 384], 128, 2, 64
    q, k, v = packed(sum(lq), sum(lk), H, H, d, seed=9300)
    kc, vc, table = build_cache(k, v, lk, P, seed=5)
    qd = q.cuda()
    obuf, o = guarded(q.numel(), "bf16")
    lbuf, lse = guarded(H * q.shape[0], "f32")
    a = attn.PagedArgs()
    a.B, a.H, a.Hkv, a.total_q, a.num_pages, a.page_size, a.max_pages, a.d = \
        len(lq), H, H, q.shape[0], kc.shape[0], P, table.shape[1], d
    wbytes = int(attn.load().attn_fwd_paged_workspace_size(ctypes.byref(a)))
    assert wbytes > 0
    wbuf, ws = guarded(wbytes, "ws")
    attn.attn_fwd_paged(qd, kc.cuda(), vc.cuda(), torch.as_tensor(offsets(lq)).cuda(),
                        torch.as_tensor(np.asarray(lk, dtype=np.int32)).cuda(), torch.as_tensor(table).cuda(),
                        o=o.view(q.shape), lse=lse.view(H, -1), workspace=ws)
    torch.cuda.synchronize()
    status_ok(attn)
    assert guards_intact(obuf, "bf16") and guards_intact(lbuf, "f32") and guards_intact(wbuf, "ws")
    assert not (o.view(torch.int16) == BF16_SENTINEL).any() and not (lse.view(torch.int32) == F32_SENTINEL).any()


@pytest.mark.parametrize("bad", ["page_past_end", "negative_page", "too_many_keys"])
def test_paged_bad_tables_are_reported_and_write_nothing(attn, bad):
    lq, lk, P = [100, 60], [300, 128], 128
    q, k, v = packed(sum(lq), sum(lk), 2, 2, 128, seed=9400)
    kc, vc, table = build_cache(k, v, lk, P, seed=6, spare=0)
    table, lens = table.copy(), list(lk)
    if bad == "page_past_end":
        table[0, 2] = kc.shape[0]
    elif bad == "negative_page":
        table[1, 0] = -1
    else:
        lens[1] = table.shape[1] * P + 1
    o, lse = run_paged(attn, q, kc, vc, offsets(lq), lens, table)
    assert attn.device_status() == (1, SITE_SEQLENS)
    assert (o.view(torch.int16) == BF16_SENTINEL).all() and (lse.view(torch.int32) == F32_SENTINEL).all()
    o, _ = run_paged(attn, q, kc, vc, offsets(lq), lk, build_cache(k, v, lk, P, seed=6, spare=0)[2])
    status_ok(attn)


def test_paged_decode_with_packed_heads(attn):
    # one query per sequence over long paged caches, query heads packed per K/V head: the
    # same bits as without packing, and the oracle's criteria
    lq, lk, P, H, Hkv, d = [1] * 6, [3000, 1, 257, 1024, 700, 129], 256, 16, 4, 128
    q, k, v = packed(sum(lq), sum(lk), H, Hkv, d, seed=9950)
    kc, vc, table = build_cache(k, v, lk, P, seed=9951)
    cu_q = offsets(lq)
    o0, l0 = run_paged(attn, q, kc, vc, cu_q, lk, table, "rtne", True)
    o1, l1 = run_paged(attn, q, kc, vc, cu_q, lk, table, "rtne", True, pack_heads=True, max_seqlen_q=1)
    status_ok(attn)
    assert torch.equal(o1.view(torch.int16), o0.view(torch.int16))
    assert torch.equal(l1.view(torch.int32), l0.view(torch.int32))
    ref = oracle.attention_paged(q, kc, vc, cu_q, lk, table, "rtne", causal=True, want_a=True)
    ob = o1.cpu().view(torch.int16).numpy().view(np.uint16)
    res = parity.compare(ob.reshape(-1, d), ref["o_bits"].reshape(-1, d), ref["a"].reshape(-1, d))
    assert res["ok"], res
