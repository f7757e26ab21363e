"""Seeded random shapes against the fp64 oracle (needs a GB300).

A fixed-seed draw over the options the fixed-shape tests cover one at a time: batch, query and
K/V heads (grouped or not), query and key lengths around and away from the 128-row tile and
256-row unit edges (1, 127-129, 255-257, ...), head dimension 64 or 128, both layouts, the
three rounding modes, the causal mask, forced key splits and the logit scale.  Every output
element (and the LSE) must meet the same criteria as everywhere else: within 2 bf16 ULP of
the oracle or its forward-error bound, non-finite values bitwise equal.  The backward draws
smaller shapes and checks dQ, dK and dV element by element.  Variable-length batches draw
sequence lengths from 0, 1, 2 and the tile edges up to 700 (empty and key-less sequences
included); each goes through attn_fwd_varlen against the oracle, through attn_fwd_paged with
its keys in shuffled cache pages (bit for bit the varlen result), and through the varlen
backward.
"""
import random

import pytest
import torch

from tests.test_gpu_backward import check_bwd
from tests.test_gpu_causal_gqa import check_ex
from workloads import make_qkv

pytestmark = pytest.mark.gpu

SQ = (1, 2, 63, 127, 128, 129, 200, 255, 256, 257, 384, 511, 700)
SKV = (1, 5, 64, 127, 128, 129, 300, 500, 777, 1024, 1500)


@pytest.fixture(scope="module")
def attn():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import bf16_attention_forward_gb300 as a
    a.load()
    return a


def _forward_cases(n=64, seed=20261203):
    rng = random.Random(seed)
    out = []
    for i in range(n):
        Hkv = rng.choice((1, 2, 3))
        H = Hkv * rng.choice((1, 1, 2, 4))
        causal = rng.random() < 0.35
        splits = 0 if causal or rng.random() < 0.7 else rng.choice((2, 3, 5))
        out.append(dict(B=rng.choice((1, 2)), H=H, Hkv=Hkv, Sq=rng.choice(SQ), Skv=rng.choice(SKV),
                        d=rng.choice((128, 128, 64)), layout=rng.choice(("bshd", "bhsd")),
                        mode=rng.choice(("rtne", "rtna", "rtz")), causal=causal, splits=splits,
                        sigma=rng.choice((0.5, 1.0, 2.0, 4.0)), seed=5000 + i))
    return out


def _backward_cases(n=16, seed=20261204):
    rng = random.Random(seed)
    out = []
    for i in range(n):
        Hkv = rng.choice((1, 2))
        out.append(dict(B=rng.choice((1, 2)), H=Hkv * rng.choice((1, 2)), Hkv=Hkv,
                        Sq=rng.choice((1, 100, 128, 129, 257, 300)),
                        Skv=rng.choice((1, 64, 128, 200, 385)), d=rng.choice((128, 64)),
                        layout=rng.choice(("bshd", "bhsd")), causal=rng.random() < 0.4,
                        seed=6000 + i))
    return out


def _id(c):
    return "B%(B)dH%(H)dKV%(Hkv)dSq%(Sq)dSkv%(Skv)dd%(d)d" % c + ("c" if c["causal"] else "")


@pytest.mark.parametrize("case", _forward_cases(), ids=_id)
def test_forward_random_shape(attn, case):
    c = case
    q, k, v = make_qkv(c["B"], c["H"], c["Sq"], c["Skv"], c["d"], c["layout"], seed=c["seed"],
                       sigma=c["sigma"], Hkv=c["Hkv"])
    kw = {"force_splits": c["splits"]} if c["splits"] else {}
    check_ex(attn, q, k, v, c["layout"], c["mode"], causal=c["causal"], **kw)


@pytest.mark.parametrize("case", _backward_cases(), ids=_id)
def test_backward_random_shape(attn, case):
    c = case
    q, k, v = make_qkv(c["B"], c["H"], c["Sq"], c["Skv"], c["d"], c["layout"], seed=c["seed"],
                       Hkv=c["Hkv"])
    g = make_qkv(c["B"], c["H"], c["Sq"], 1, c["d"], c["layout"], seed=c["seed"] + 1)[0]
    check_bwd(attn, q, k, v, g, c["layout"], causal=c["causal"])


LEN = (0, 1, 2, 63, 127, 128, 129, 255, 256, 257, 300, 511, 700)


def _varlen_cases(n=12, seed=20261205):
    rng = random.Random(seed)
    out = []
    for i in range(n):
        Hkv = rng.choice((1, 2))
        B = rng.choice((1, 2, 3, 5))
        causal = rng.random() < 0.5
        lq = [rng.choice(LEN) for _ in range(B)]
        lk = lq if causal and rng.random() < 0.5 else [rng.choice(LEN) for _ in range(B)]
        out.append(dict(lq=lq, lk=lk, H=Hkv * rng.choice((1, 2, 4)), Hkv=Hkv, d=rng.choice((128, 64)),
                        mode=rng.choice(("rtne", "rtna", "rtz")), causal=causal, P=rng.choice((128, 256)),
                        seed=7000 + i))
    return out


def _vid(c):
    return "B%dH%dKV%dd%d%s" % (len(c["lq"]), c["H"], c["Hkv"], c["d"], "c" if c["causal"] else "")


@pytest.mark.parametrize("case", _varlen_cases(), ids=_vid)
def test_varlen_paged_random(attn, case):
    # the same random batch through attn_fwd_varlen (against the oracle) and through
    # attn_fwd_paged with its keys in shuffled cache pages (bit for bit the varlen result)
    from tests.test_gpu_paged import build_cache, run_paged
    from tests.test_gpu_varlen import check_varlen, offsets, packed
    c = case
    if sum(c["lq"]) == 0:
        c["lq"][0] = 1
    q, k, v = packed(sum(c["lq"]), max(sum(c["lk"]), 1), c["H"], c["Hkv"], c["d"], seed=c["seed"])
    cu_q, cu_k = offsets(c["lq"]), offsets(c["lk"])
    o, lse = check_varlen(attn, q, k, v, cu_q, cu_k, c["mode"], c["causal"])
    kc, vc, table = build_cache(k, v, c["lk"], c["P"], seed=c["seed"])
    op, lp = run_paged(attn, q, kc, vc, cu_q, c["lk"], table, c["mode"], c["causal"])
    assert attn.device_status()[0] == 0
    assert torch.equal(op.view(torch.int16), o.view(torch.int16))
    assert torch.equal(lp.view(torch.int32), lse.view(torch.int32))


@pytest.mark.parametrize("case", _varlen_cases(n=6, seed=20261206), ids=_vid)
def test_varlen_backward_random(attn, case):
    from tests.test_gpu_backward_varlen import check
    from tests.test_gpu_varlen import offsets, packed
    c = case
    if sum(c["lq"]) == 0:
        c["lq"][0] = 1
    q, k, v = packed(sum(c["lq"]), max(sum(c["lk"]), 1), c["H"], c["Hkv"], c["d"], seed=c["seed"])
    g = packed(sum(c["lq"]), 1, c["H"], c["H"], c["d"], seed=c["seed"] + 1)[0]
    check(attn, q, k, v, g, offsets(c["lq"]), offsets(c["lk"]), c["causal"])
