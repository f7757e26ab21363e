"""Guard canaries around every buffer the kernels write (needs a GB300).

Each output (O, the log-sum-exp, dQ, dK, dV) and each workspace is a view into a larger buffer
whose bytes are first filled with a canary pattern.  After the call the guard regions on both
sides must still hold the pattern (no write strayed out of bounds: TMA stores and reductions on
ragged tiles, the split partials, the combine), and every output element must have been written
(no canary left inside).  Shapes are ragged on purpose, and cover the forward kernel, the
short-query kernel, the key-split path with its combine, the causal mask and the backward.
"""
import ctypes

import pytest
import torch

from workloads import make_qkv

pytestmark = pytest.mark.gpu

G = 4096                     # guard elements on each side (a multiple of 16 bytes for any dtype)
BF16_CANARY = 0x7BAD         # a finite bf16 near 2^119, which no output here can equal
F32_CANARY = 0x7F7BAD01      # a finite fp32 near 3.3e38
WS_CANARY = 0xA5


@pytest.fixture(scope="module")
def attn():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import bf16_attention_forward_gb300 as a
    a.load()
    return a


def guarded(n, kind):
    """(whole buffer, payload view of n elements) with the canary in every byte."""
    if kind == "bf16":
        buf = torch.empty(n + 2 * G, dtype=torch.bfloat16, device="cuda")
        buf.view(torch.int16).fill_(BF16_CANARY)
    elif kind == "f32":
        buf = torch.empty(n + 2 * G, dtype=torch.float32, device="cuda")
        buf.view(torch.int32).fill_(F32_CANARY)
    else:
        buf = torch.empty(n + 2 * G, dtype=torch.uint8, device="cuda")
        buf.fill_(WS_CANARY)
    return buf, buf[G:G + n]


def guards_intact(buf, kind):
    raw = {"bf16": buf.view(torch.int16), "f32": buf.view(torch.int32), "ws": buf}[kind]
    pat = {"bf16": BF16_CANARY, "f32": F32_CANARY, "ws": WS_CANARY}[kind]
    return bool((raw[:G] == pat).all()) and bool((raw[-G:] == pat).all())


def fully_written(view, kind):
    raw = view.view(torch.int16) if kind == "bf16" else view.view(torch.int32)
    pat = BF16_CANARY if kind == "bf16" else F32_CANARY
    return not bool((raw == pat).any())


FWD = [  # (B, H, Hkv, Sq, Skv, d, layout, causal, force_splits)
    (2, 3, 3, 130, 200, 128, "bshd", False, 3),      # forward kernel, ragged, key split
    (1, 4, 2, 77, 300, 128, "bhsd", False, 2),       # short-query kernel, grouped, key split
    (1, 2, 2, 300, 200, 128, "bshd", True, 0),       # causal, leading rows without keys
    (2, 2, 1, 129, 513, 64, "bhsd", False, 0),       # head dimension 64, ragged
    (1, 8, 8, 1, 1000, 128, "bshd", False, 4),       # one query row, split
]


@pytest.mark.parametrize("case", FWD, ids=lambda c: "B%dH%dHkv%dSq%dSkv%dd%d_%s%s_fs%d" % (c[:6] + (c[6], "_causal" if c[7] else "", c[8])))
def test_forward_writes_stay_in_bounds(attn, case):
    B, H, Hkv, Sq, Skv, d, layout, causal, fs = case
    q, k, v = (t.cuda() for t in make_qkv(B, H, Sq, Skv, d, layout, seed=7000 + Sq, Hkv=Hkv))
    obuf, o = guarded(q.numel(), "bf16")
    o = o.view(q.shape)
    lbuf, lse = guarded(B * H * Sq, "f32")
    need = attn.workspace_size_ex(q, k, v, layout=layout, causal=causal, force_splits=fs)
    wbuf, ws = guarded(max(need, 16), "ws")
    attn.attn_fwd_ex(q, k, v, o, lse, layout=layout, causal=causal, workspace=ws, force_splits=fs)
    torch.cuda.synchronize()
    assert attn.device_status()[0] == 0
    assert guards_intact(obuf, "bf16"), "O written out of bounds"
    assert guards_intact(lbuf, "f32"), "LSE written out of bounds"
    assert guards_intact(wbuf, "ws"), "workspace written out of bounds"
    assert fully_written(o, "bf16"), "O element left unwritten"
    assert fully_written(lse, "f32"), "LSE element left unwritten"


BWD = [  # (B, H, Hkv, Sq, Skv, d, layout, causal)
    (1, 2, 2, 130, 200, 128, "bshd", False),
    (2, 4, 2, 300, 129, 128, "bhsd", True),
    (1, 2, 1, 77, 1000, 64, "bshd", False),
]


@pytest.mark.parametrize("det", [False, True], ids=["acc", "det"])
@pytest.mark.parametrize("case", BWD, ids=lambda c: "B%dH%dHkv%dSq%dSkv%dd%d_%s%s" % (c[:6] + (c[6], "_causal" if c[7] else "")))
def test_backward_writes_stay_in_bounds(attn, case, det):
    B, H, Hkv, Sq, Skv, d, layout, causal = case
    q, k, v = (t.cuda() for t in make_qkv(B, H, Sq, Skv, d, layout, seed=7100 + Sq, Hkv=Hkv))
    g = make_qkv(B, H, Sq, 1, d, layout, seed=7200 + Sq)[0].cuda()
    o, lse = attn.attn_fwd_ex(q, k, v, layout=layout, causal=causal, return_lse=True)
    outs = []
    for ref in (q, k, v):
        buf, view = guarded(ref.numel(), "bf16")
        outs.append((buf, view.view(ref.shape)))
    a = attn.BwdArgs()
    a.B, a.H, a.Hkv, a.Sq, a.Skv, a.d = B, H, Hkv, Sq, Skv, d
    a.layout, a.causal, a.wait_limit_ms, a.test_hooks = attn.LAYOUTS[layout], int(causal), 0, 0
    a.deterministic = int(det)
    need = int(attn.load().attn_bwd_workspace_size(ctypes.byref(a)))
    assert need > 0
    wbuf, ws = guarded(need, "ws")
    attn.attn_bwd(q, k, v, o, g, lse, layout=layout, causal=causal, dq=outs[0][1], dk=outs[1][1],
                  dv=outs[2][1], workspace=ws, deterministic=det)
    torch.cuda.synchronize()
    assert attn.bwd_device_status()[0] == 0
    for name, (buf, view) in zip(("dQ", "dK", "dV"), outs):
        assert guards_intact(buf, "bf16"), name + " written out of bounds"
        assert fully_written(view, "bf16"), name + " element left unwritten"
    assert guards_intact(wbuf, "ws"), "workspace written out of bounds"
