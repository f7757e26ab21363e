"""The bounded-wait path on the GPU: a wait that runs out is reported, and the device stays
usable (needs a GB300).

Every wait inside the kernels gives up after a time limit: the kernel then records
ATTN_ERR_DEVICE_TIMEOUT and the wait's site in a status word, raises its CTA's abort flag,
lets its in-flight copies and matrix products finish (with bounded waits) and returns.  The
test hook ATTN_TEST_WITHHOLD_O_READY makes the first CTA skip one signal that exactly one
wait depends on (its first unit's output-ready signal), so that wait expires under a 50 ms
limit.  Nothing faults, traps or spins without a bound; afterwards a normal call on the same
device must still match the oracle.
"""
import numpy as np
import pytest
import torch

import oracle
from tests import parity
from workloads import make_qkv

pytestmark = pytest.mark.gpu

WITHHOLD = 1            # ATTN_TEST_WITHHOLD_O_READY
SITE_O_READY = 7        # ATTN_SITE_O_READY
SITE_DKV_READY = 9      # ATTN_BWD_SITE_DKV_READY
TIMEOUT = 8             # ATTN_ERR_DEVICE_TIMEOUT


@pytest.fixture(scope="module")
def attn():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import bf16_attention_forward_gb300 as a
    a.load()
    return a


# Sq > 128 runs attn_fwd_kernel, Sq <= 128 the short-query kernel; one unit each (one CTA)
@pytest.mark.parametrize("Sq", [200, 100])
def test_forward_wait_expires_and_device_recovers(attn, Sq):
    q, k, v = make_qkv(1, 1, Sq, 300, 128, "bhsd", seed=60 + Sq)
    qd, kd, vd = (t.cuda() for t in (q, k, v))
    assert attn.device_status() == (0, 0)
    attn.attn_fwd(qd, kd, vd, layout="bhsd", wait_limit_ms=50, test_hooks=WITHHOLD)
    assert attn.device_status() == (TIMEOUT, SITE_O_READY)
    assert attn.device_status() == (0, 0)                  # read and cleared
    o = attn.attn_fwd(qd, kd, vd, layout="bhsd")
    assert attn.device_status() == (0, 0)
    ref = oracle.attention(q, k, v, "bhsd", "rtne", want_a=True)
    res = parity.compare(parity.gpu_rows_bits(o, "bhsd"), ref["o_bits"], ref["a"])
    assert res["ok"], res


def test_backward_wait_expires_and_device_recovers(attn):
    q, k, v = make_qkv(1, 1, 200, 100, 128, "bhsd", seed=70)      # one key tile: one unit
    g = make_qkv(1, 1, 200, 1, 128, "bhsd", seed=71)[0]
    qd, kd, vd, gd = (t.cuda() for t in (q, k, v, g))
    o, lse = attn.attn_fwd_ex(qd, kd, vd, layout="bhsd", return_lse=True)
    assert attn.bwd_device_status() == (0, 0)
    attn.attn_bwd(qd, kd, vd, o, gd, lse, layout="bhsd", wait_limit_ms=50, test_hooks=WITHHOLD)
    assert attn.bwd_device_status() == (TIMEOUT, SITE_DKV_READY)
    assert attn.bwd_device_status() == (0, 0)
    dq, dk, dv = attn.attn_bwd(qd, kd, vd, o, gd, lse, layout="bhsd")
    assert attn.bwd_device_status() == (0, 0) and attn.device_status() == (0, 0)
    ref = oracle.backward(q, k, v, g, "bhsd", want_a=True)
    for name, got in (("dq", dq), ("dk", dk), ("dv", dv)):
        err = np.abs(got.float().cpu().double().numpy() - ref[name])
        tol = 2.0 ** -7 * ref[name + "_a"] + parity.bf16_ulp(ref[name + "_bits"])
        assert np.all(err <= tol), (name, float((err - tol).max()))
