"""Pins for the oracle's variable-length batches (``oracle.attention_varlen``).

The page "MoonMath AI open-sources a HIP attention kernel for AMD MI300X that beats AITER"
lists variable-length batching among its kernel's limitations.  The reading taken: each
sequence of the packed batch is an attention problem of its own.  These checks pin the
oracle's composition to things other than itself:
  * a batch of equal-length sequences equals the dense batched oracle on the same data
    reshaped to [B, S, H, d] (the C oracle's own batch indexing, not the slicing);
  * sequences do not see each other: rewriting every other sequence's rows (with values
    including +-inf and NaN) leaves a sequence's outputs bit for bit unchanged, and
    reordering the sequences reorders the outputs;
  * a lone sequence equals the dense oracle, and the edge rules hold: empty sequences cover
    no rows, a sequence with no keys gets NaN (0x7FC0) outputs and LSE -inf, rows outside
    every sequence stay uncovered.
"""
import numpy as np
import pytest
import torch

import oracle
from workloads import make_qkv


def _packed(Tq, Tk, H, Hkv, d, seed, sigma=1.0):
    q, k, v = make_qkv(1, H, Tq, Tk, d, "bshd", seed=seed, sigma=sigma, Hkv=Hkv)
    return q[0], k[0], v[0]


def _bits(t):
    return t.contiguous().view(torch.int16).numpy().view(np.uint16)


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("mode", ["rtne", "rtz"])
def test_equal_lengths_match_the_dense_batch(mode, causal):
    B, Sq, Skv, H, Hkv, d = 3, 37, 53, 4, 2, 64
    q, k, v = _packed(B * Sq, B * Skv, H, Hkv, d, seed=11)
    cu_q = np.arange(B + 1) * Sq
    cu_k = np.arange(B + 1) * Skv
    r = oracle.attention_varlen(q, k, v, cu_q, cu_k, mode, causal=causal, want_a=True, want_lse=True)
    dense = oracle.attention(q.reshape(B, Sq, H, d), k.reshape(B, Skv, Hkv, d), v.reshape(B, Skv, Hkv, d),
                             "bshd", mode, want_a=True, want_lse=True, causal=causal)
    # dense is (B, H, Sq, d); the packed rows are token-major
    assert np.array_equal(r["o_bits"], dense["o_bits"].transpose(0, 2, 1, 3).reshape(B * Sq, H, d))
    assert np.array_equal(r["a"], dense["a"].transpose(0, 2, 1, 3).reshape(B * Sq, H, d))
    assert np.array_equal(r["lse"], dense["lse"].transpose(1, 0, 2).reshape(H, B * Sq))
    assert r["covered"].all()


def test_sequences_do_not_see_each_other():
    H, Hkv, d = 2, 1, 128
    lq, lk = [130, 1, 57], [70, 300, 5]
    cu_q, cu_k = np.cumsum([0] + lq), np.cumsum([0] + lk)
    q, k, v = _packed(sum(lq), sum(lk), H, Hkv, d, seed=12)
    base = oracle.attention_varlen(q, k, v, cu_q, cu_k, "rtna", want_lse=True)
    g = torch.Generator().manual_seed(3)
    for b in range(3):
        q2, k2, v2 = q.clone(), k.clone(), v.clone()
        for o in range(3):
            if o == b:
                continue
            for t, cu in ((q2, cu_q), (k2, cu_k), (v2, cu_k)):
                rows = slice(cu[o], cu[o + 1])
                x = torch.randn(t[rows].shape, generator=g) * 50
                x.view(-1)[::7] = float("inf")
                x.view(-1)[3::11] = float("nan")
                t[rows] = x.to(torch.bfloat16)
        r = oracle.attention_varlen(q2, k2, v2, cu_q, cu_k, "rtna", want_lse=True)
        rows = slice(cu_q[b], cu_q[b + 1])
        assert np.array_equal(r["o_bits"][rows], base["o_bits"][rows]), b
        assert np.array_equal(r["lse"][:, rows], base["lse"][:, rows]), b


def test_reordering_sequences_reorders_outputs():
    H, d = 2, 64
    lq, lk = [40, 9, 23], [17, 64, 3]
    q, k, v = _packed(sum(lq), sum(lk), H, H, d, seed=13)
    cu_q, cu_k = np.cumsum([0] + lq), np.cumsum([0] + lk)
    base = oracle.attention_varlen(q, k, v, cu_q, cu_k, causal=True)
    perm = [2, 0, 1]

    def gather(t, cu):
        return torch.cat([t[cu[b]:cu[b + 1]] for b in perm])

    cu_q2 = np.cumsum([0] + [lq[b] for b in perm])
    cu_k2 = np.cumsum([0] + [lk[b] for b in perm])
    r = oracle.attention_varlen(gather(q, cu_q), gather(k, cu_k), gather(v, cu_k), cu_q2, cu_k2, causal=True)
    want = np.concatenate([base["o_bits"][cu_q[b]:cu_q[b + 1]] for b in perm])
    assert np.array_equal(r["o_bits"], want)


def test_single_sequence_and_edge_rules():
    H, Hkv, d = 4, 2, 128
    q, k, v = _packed(20, 12, H, Hkv, d, seed=14)
    # one sequence over rows 2..16 and keys 1..10; rows 0, 1 and 17.. belong to none
    r = oracle.attention_varlen(q, k, v, [2, 17], [1, 11], want_lse=True)
    dense = oracle.attention(q[None, 2:17], k[None, 1:11], v[None, 1:11], "bshd", want_lse=True)
    assert np.array_equal(r["o_bits"][2:17], dense["o_bits"][0].transpose(1, 0, 2))
    assert np.array_equal(r["lse"][:, 2:17], dense["lse"][0])
    assert r["covered"].tolist() == [False] * 2 + [True] * 15 + [False] * 3
    assert not r["o_bits"][:2].any() and not r["o_bits"][17:].any()
    # an empty sequence, a sequence with queries but no keys, then a normal one
    r = oracle.attention_varlen(q, k, v, [0, 0, 5, 20], [0, 4, 4, 12], want_lse=True)
    assert (r["o_bits"][0:5] == 0x7FC0).all()
    assert np.isneginf(r["lse"][:, 0:5]).all()
    dense = oracle.attention(q[None, 5:20], k[None, 4:12], v[None, 4:12], "bshd", want_lse=True)
    assert np.array_equal(r["o_bits"][5:20], dense["o_bits"][0].transpose(1, 0, 2))
    assert r["covered"].all()


def test_rejects_bad_offsets():
    q, k, v = _packed(8, 8, 1, 1, 64, seed=15)
    for cu_q, cu_k in (([0, 5, 3], [0, 4, 8]), ([0, 9], [0, 8]), ([0, 8], [-1, 8])):
        with pytest.raises(ValueError):
            oracle.attention_varlen(q, k, v, cu_q, cu_k)


# --------------------------------------------------------------------------- paged K/V
# oracle.attention_paged gathers each sequence's keys from the cache pages and runs the
# varlen oracle; pinned by: pages laid out in order equal the contiguous keys, a permutation
# of the physical pages (with the table following it) changes nothing, values outside the
# used slots cannot matter, and shared pages behave as copies.

def _paged_from_contiguous(k, v, lens, P, perm=None, fill=None):
    """Cache pages holding each sequence's keys in order (sequence after sequence, each
    starting a new page), physical pages renumbered by `perm`; unused slots set to `fill`."""
    Hkv, d = k.shape[1], k.shape[2]
    pages, table, row = [], [], 0
    maxp = max(1, max(-(-n // P) for n in lens))
    for n in lens:
        ids = []
        for p0 in range(0, n, P):
            page = torch.zeros((P, Hkv, d), dtype=torch.bfloat16)
            if fill is not None:
                page.view(torch.int16).fill_(fill)
            m = min(P, n - p0)
            page[:m] = k[row + p0: row + p0 + m]
            vpage = page.clone()
            vpage[:m] = v[row + p0: row + p0 + m]
            ids.append(len(pages))
            pages.append((page, vpage))
        row += n
        table.append(ids + [0] * (maxp - len(ids)))
    order = list(range(len(pages))) if perm is None else perm
    inv = {old: new for new, old in enumerate(order)}
    kc = torch.stack([pages[o][0] for o in order])
    vc = torch.stack([pages[o][1] for o in order])
    table = [[inv[i] if j < -(-lens[b] // P) else 0 for j, i in enumerate(t)] for b, t in enumerate(table)]
    return kc, vc, np.asarray(table, dtype=np.int32)


@pytest.mark.parametrize("causal", [False, True])
def test_paged_in_order_equals_contiguous(causal):
    H, Hkv, d, P = 2, 1, 64, 128
    lq, lk = [40, 7, 130], [300, 128, 129]
    q, k, v = _packed(sum(lq), sum(lk), H, Hkv, d, seed=21)
    kc, vc, table = _paged_from_contiguous(k, v, lk, P)
    cu_q, cu_k = np.cumsum([0] + lq), np.cumsum([0] + lk)
    r = oracle.attention_paged(q, kc, vc, cu_q, lk, table, causal=causal, want_lse=True)
    want = oracle.attention_varlen(q, k, v, cu_q, cu_k, causal=causal, want_lse=True)
    assert np.array_equal(r["o_bits"], want["o_bits"]) and np.array_equal(r["lse"], want["lse"])


def test_paged_page_permutation_and_stale_slots_change_nothing():
    H, d, P = 2, 128, 256
    lq, lk = [100, 33], [600, 257]
    q, k, v = _packed(sum(lq), sum(lk), H, H, d, seed=22)
    cu_q = np.cumsum([0] + lq)
    kc, vc, table = _paged_from_contiguous(k, v, lk, P)
    base = oracle.attention_paged(q, kc, vc, cu_q, lk, table)
    n = kc.shape[0]
    perm = list(np.random.default_rng(5).permutation(n))
    kc2, vc2, table2 = _paged_from_contiguous(k, v, lk, P, perm=perm, fill=0x7F80)   # +inf past the keys
    assert not np.array_equal(table, table2)
    r = oracle.attention_paged(q, kc2, vc2, cu_q, lk, table2)
    assert np.array_equal(r["o_bits"], base["o_bits"])


def test_paged_shared_pages_act_as_copies():
    H, d, P = 1, 64, 128
    q, k, v = _packed(20, 256, H, H, d, seed=23)
    kc, vc, table = _paged_from_contiguous(k, v, [256], P)
    # two sequences reading the same two pages, the second one only its first 130 keys
    tbl = np.asarray([[0, 1], [0, 1]], dtype=np.int32)
    r = oracle.attention_paged(q, kc, vc, [0, 12, 20], [256, 130], tbl)
    want = oracle.attention_varlen(q, torch.cat([k, k[:130]]), torch.cat([v, v[:130]]), [0, 12, 20], [0, 256, 386])
    assert np.array_equal(r["o_bits"], want["o_bits"])


def test_paged_rejects_pages_out_of_range():
    q, k, v = _packed(8, 128, 1, 1, 64, seed=24)
    kc, vc, table = _paged_from_contiguous(k, v, [128], 128)
    with pytest.raises(ValueError):
        oracle.attention_paged(q, kc, vc, [0, 8], [128], np.asarray([[1]], dtype=np.int32))


# --------------------------------------------------------------------------- varlen backward
@pytest.mark.parametrize("causal", [False, True])
def test_backward_equal_lengths_match_the_dense_batch(causal):
    # the same batch through the dense backward oracle (its own batch indexing)
    B, Sq, Skv, H, Hkv, d = 2, 21, 34, 4, 2, 64
    q, k, v = _packed(B * Sq, B * Skv, H, Hkv, d, seed=31)
    g = _packed(B * Sq, 1, H, H, d, seed=32)[0]
    r = oracle.backward_varlen(q, k, v, g, np.arange(B + 1) * Sq, np.arange(B + 1) * Skv, causal=causal,
                               want_a=True)
    dense = oracle.backward(q.reshape(B, Sq, H, d), k.reshape(B, Skv, Hkv, d), v.reshape(B, Skv, Hkv, d),
                            g.reshape(B, Sq, H, d), "bshd", causal=causal, want_a=True)
    for n, rows in (("dq", B * Sq), ("dk", B * Skv), ("dv", B * Skv)):
        assert np.array_equal(r[n], dense[n].reshape(rows, -1, d)), n
        assert np.array_equal(r[n + "_a"], dense[n + "_a"].reshape(rows, -1, d)), n


def test_backward_sequences_do_not_see_each_other_and_edge_rules():
    H, d = 2, 64
    lq, lk = [30, 0, 17, 9], [25, 12, 0, 40]     # sequence 1 has no queries, sequence 2 no keys
    cu_q, cu_k = np.cumsum([0] + lq), np.cumsum([0] + lk)
    q, k, v = _packed(sum(lq) + 3, sum(lk) + 2, H, H, d, seed=33)   # trailing rows belong to none
    g = _packed(sum(lq) + 3, 1, H, H, d, seed=34)[0]
    base = oracle.backward_varlen(q, k, v, g, cu_q, cu_k)
    assert not base["dk"][cu_k[1]:cu_k[2]].any() and not base["dv"][cu_k[1]:cu_k[2]].any()
    assert not base["dq"][cu_q[2]:cu_q[3]].any()
    assert not base["covered_q"][-3:].any() and not base["covered_k"][-2:].any()
    # rewriting sequence 3's rows leaves sequence 0 alone
    q2, k2, v2, g2 = q.clone(), k.clone(), v.clone(), g.clone()
    for t, cu in ((q2, cu_q), (k2, cu_k), (v2, cu_k), (g2, cu_q)):
        t[cu[3]:cu[4]] = (torch.randn(t[cu[3]:cu[4]].shape) * 30).to(torch.bfloat16)
    r = oracle.backward_varlen(q2, k2, v2, g2, cu_q, cu_k)
    for n, cu in (("dq", cu_q), ("dk", cu_k), ("dv", cu_k)):
        assert np.array_equal(r[n][cu[0]:cu[1]], base[n][cu[0]:cu[1]]), n
