"""fp64 CPU oracle for the bf16 attention forward.  TEST INFRASTRUCTURE ONLY.

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline / reference leg of
``bench.py`` may import this package.  The product library never loads it and shares no
code with it.  The arithmetic lives in ``attn_oracle.c`` (plain C, fp64, OpenMP over rows)
and, for the backward, ``attn_oracle_bwd.c``; this module compiles them with gcc and
marshals numpy arrays through ``ctypes``.

What it computes is stated in the C file's header: softmax(Q K^T / sqrt(d)) V per row, in
fp64, two passes, rounded once to bf16 in the requested mode, following the page
"MoonMath AI open-sources a HIP attention kernel for AMD MI300X that beats AITER"
(opening section: definition and contract; limitations paragraph: rounding modes, NaN/Inf).
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "attn_oracle.c")
_SRC_BWD = os.path.join(_HERE, "attn_oracle_bwd.c")
_BUILD_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD_DIR, "libattn_oracle.so")

LAYOUTS = {"bshd": 0, "bhsd": 1}
MODES = {"rtne": 0, "rtna": 1, "rtz": 2}

_lock = threading.Lock()
_lib = None


def build(force: bool = False, src: str = _SRC, out: str = _LIB_PATH,
          bwd_src: str = _SRC_BWD) -> str:
    """Compile the oracle (``src``, the forward, and ``bwd_src``, the backward) into a shared
    object (gcc, -O2, OpenMP, no fast-math)."""
    srcs = [src, bwd_src]
    if not force and os.path.exists(out) and \
            all(os.path.getmtime(out) >= os.path.getmtime(f) for f in srcs):
        return out
    os.makedirs(os.path.dirname(out), exist_ok=True)
    tmp = out + ".tmp%d" % os.getpid()
    cmd = ["gcc", "-O2", "-fopenmp", "-fPIC", "-shared", "-std=c11", "-fno-fast-math",
           *srcs, "-o", tmp, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, out)
    return out


def _bind(lib):
    u16p = ctypes.POINTER(ctypes.c_uint16)
    f64p = ctypes.POINTER(ctypes.c_double)
    i64p = ctypes.POINTER(ctypes.c_int64)
    lib.attn_oracle.restype = ctypes.c_int
    lib.attn_oracle.argtypes = [u16p, u16p, u16p] + [ctypes.c_int64] * 5 + [
        ctypes.c_int, ctypes.c_int, i64p, ctypes.c_int64, u16p, f64p, f64p, f64p, f64p,
        ctypes.c_int]
    lib.attn_oracle_ex.restype = ctypes.c_int
    lib.attn_oracle_ex.argtypes = [u16p, u16p, u16p] + [ctypes.c_int64] * 6 + [
        ctypes.c_int, ctypes.c_int, ctypes.c_int, i64p, ctypes.c_int64, u16p, f64p, f64p,
        f64p, f64p, ctypes.c_int]
    lib.oracle_round_bf16_array.restype = None
    lib.oracle_round_bf16_array.argtypes = [f64p, ctypes.c_int64, ctypes.c_int, u16p]
    lib.oracle_max_threads.restype = ctypes.c_int
    lib.oracle_max_threads.argtypes = []
    lib.attn_oracle_f64_forward.restype = ctypes.c_int
    lib.attn_oracle_f64_forward.argtypes = [f64p, f64p, f64p] + [ctypes.c_int64] * 6 + [
        ctypes.c_int, ctypes.c_int, f64p]
    lib.attn_oracle_bwd.restype = ctypes.c_int
    lib.attn_oracle_bwd.argtypes = [u16p, u16p, u16p, u16p] + [ctypes.c_int64] * 6 + [
        ctypes.c_int, ctypes.c_int] + [f64p] * 7 + [ctypes.c_int]
    return lib


def load(path: str | None = None):
    """Load (building first if needed) the oracle library."""
    global _lib
    with _lock:
        if path is not None:
            return _bind(ctypes.CDLL(path))
        if _lib is None:
            _lib = _bind(ctypes.CDLL(build()))
        return _lib


def _ptr(a, ctype):
    return a.ctypes.data_as(ctypes.POINTER(ctype)) if a is not None else None


def _as_bits(t) -> np.ndarray:
    """Accept a torch bf16 tensor (CPU) or a uint16/int16 numpy array of bf16 bits."""
    if isinstance(t, np.ndarray):
        a = t
    else:  # torch tensor
        import torch
        a = t.detach().cpu().contiguous().view(torch.int16).numpy()
    return np.ascontiguousarray(a).view(np.uint16)


def dims(q_shape, k_shape, layout: str):
    """(B, H, Sq, Skv, d) from BSHD (B, S, H, d) or BHSD (B, H, S, d) shapes."""
    if layout == "bshd":
        B, Sq, H, d = q_shape
        Skv = k_shape[1]
    else:
        B, H, Sq, d = q_shape
        Skv = k_shape[2]
    return B, H, Sq, Skv, d


def kv_heads(k_shape, layout: str) -> int:
    return k_shape[2] if layout == "bshd" else k_shape[1]


def attention(q, k, v, layout: str = "bshd", mode: str = "rtne", rows=None,
              want_f64: bool = False, want_a: bool = False, want_lse: bool = False,
              want_probs: bool = False, threads: int | None = None, lib=None,
              causal: bool = False) -> dict:
    """Oracle attention.  Returns a dict of numpy arrays.

    K and V may have fewer heads than Q (grouped heads: query head h reads K/V head
    h // (H // Hkv)); ``causal`` makes key j visible to query i iff j <= i + (Skv - Sq).

    ``o_bits``: uint16 bf16 patterns.  With ``rows=None`` shaped (B, H, Sq, d) (BHSD order,
    whatever the input layout); with ``rows`` (flat indices (b*H + h)*Sq + i) shaped
    (len(rows), d).  Optional: ``o_f64``, ``a`` (forward-error scale A), ``lse`` (natural
    log), ``probs`` (softmax weights, rows x Skv).
    """
    lib = lib or load()
    qb, kb, vb = _as_bits(q), _as_bits(k), _as_bits(v)
    B, H, Sq, Skv, d = dims(qb.shape, kb.shape, layout)
    if rows is None:
        n = B * H * Sq
        rows_arr = None
    else:
        rows_arr = np.ascontiguousarray(np.asarray(rows, dtype=np.int64))
        n = rows_arr.shape[0]
    o_bits = np.empty((n, d), dtype=np.uint16)
    o_f64 = np.empty((n, d), dtype=np.float64) if want_f64 else None
    a_b = np.empty((n, d), dtype=np.float64) if want_a else None
    lse = np.empty((n,), dtype=np.float64) if want_lse else None
    probs = np.empty((n, Skv), dtype=np.float64) if want_probs else None
    Hkv = kv_heads(kb.shape, layout)
    rc = lib.attn_oracle_ex(_ptr(qb, ctypes.c_uint16), _ptr(kb, ctypes.c_uint16),
                         _ptr(vb, ctypes.c_uint16), B, H, Hkv, Sq, Skv, d, LAYOUTS[layout],
                         MODES[mode], 1 if causal else 0, _ptr(rows_arr, ctypes.c_int64),
                         0 if rows_arr is None else n, _ptr(o_bits, ctypes.c_uint16),
                         _ptr(o_f64, ctypes.c_double), _ptr(a_b, ctypes.c_double),
                         _ptr(lse, ctypes.c_double), _ptr(probs, ctypes.c_double),
                         int(threads or 0))
    if rc != 0:
        raise ValueError("oracle rejected its arguments (rc=%d)" % rc)
    out = {"o_bits": o_bits}
    if o_f64 is not None:
        out["o_f64"] = o_f64
    if a_b is not None:
        out["a"] = a_b
    if lse is not None:
        out["lse"] = lse
    if probs is not None:
        out["probs"] = probs
    if rows is None:
        for key in ("o_bits", "o_f64", "a"):
            if key in out:
                out[key] = out[key].reshape(B, H, Sq, d)
        if "lse" in out:
            out["lse"] = out["lse"].reshape(B, H, Sq)
    return out


def attention_varlen(q, k, v, cu_q, cu_k, mode: str = "rtne", causal: bool = False,
                     want_a: bool = False, want_lse: bool = False, lib=None) -> dict:
    """Oracle attention over a variable-length batch packed along the token axis.

    The page "MoonMath AI open-sources a HIP attention kernel for AMD MI300X that beats AITER"
    lists variable-length batching among its kernel's limitations; the plain reading of the
    feature is that each sequence is an attention problem of its own.  So sequence b (query
    rows cu_q[b] .. cu_q[b+1]-1, key rows cu_k[b] .. cu_k[b+1]-1 of q [Tq, H, d] and
    k, v [Tk, Hkv, d]) is passed alone to :func:`attention` as a one-batch BSHD problem, and
    its rows are put back in place.  A sequence with queries but no keys has no visible key
    for any query: 0/0, so NaN outputs (0x7FC0) and LSE -inf, as for a causal row that sees
    no key.

    Returns ``o_bits`` [Tq, H, d] (uint16), ``covered`` [Tq] (rows that belong to a
    sequence; the others are left 0), and optionally ``a`` [Tq, H, d] and ``lse`` [H, Tq]
    (natural log).
    """
    qb, kb, vb = _as_bits(q), _as_bits(k), _as_bits(v)
    Tq, H, d = qb.shape
    cu_q = [int(x) for x in np.asarray(cu_q).reshape(-1)]
    cu_k = [int(x) for x in np.asarray(cu_k).reshape(-1)]
    if len(cu_q) != len(cu_k) or len(cu_q) < 2:
        raise ValueError("cu_q and cu_k must both hold B + 1 >= 2 offsets")
    o_bits = np.zeros((Tq, H, d), dtype=np.uint16)
    covered = np.zeros((Tq,), dtype=bool)
    a = np.zeros((Tq, H, d), dtype=np.float64) if want_a else None
    lse = np.zeros((H, Tq), dtype=np.float64) if want_lse else None
    for b in range(len(cu_q) - 1):
        q0, q1, k0, k1 = cu_q[b], cu_q[b + 1], cu_k[b], cu_k[b + 1]
        if not (0 <= q0 <= q1 <= Tq and 0 <= k0 <= k1 <= kb.shape[0]):
            raise ValueError("sequence %d: offsets out of order or out of range" % b)
        if q1 == q0:
            continue
        covered[q0:q1] = True
        if k1 == k0:
            o_bits[q0:q1] = 0x7FC0
            if a is not None:
                a[q0:q1] = np.nan
            if lse is not None:
                lse[:, q0:q1] = -np.inf
            continue
        r = attention(qb[None, q0:q1], kb[None, k0:k1], vb[None, k0:k1], "bshd", mode,
                      want_a=want_a, want_lse=want_lse, lib=lib, causal=causal)
        o_bits[q0:q1] = r["o_bits"][0].transpose(1, 0, 2)
        if a is not None:
            a[q0:q1] = r["a"][0].transpose(1, 0, 2)
        if lse is not None:
            lse[:, q0:q1] = r["lse"][0]
    out = {"o_bits": o_bits, "covered": covered}
    if a is not None:
        out["a"] = a
    if lse is not None:
        out["lse"] = lse
    return out


def backward_varlen(q, k, v, dout, cu_q, cu_k, causal: bool = False, want_a: bool = False,
                    lib=None) -> dict:
    """fp64 gradients of the variable-length attention (:func:`attention_varlen`): each
    sequence's gradients are :func:`backward` of that sequence alone, put back in place.  A
    sequence without keys has no term in any gradient (dq 0); keys of a sequence without
    queries get dk = dv = 0.  Returns ``dq``, ``dk``, ``dv`` (float64, packed like the inputs),
    their RTNE ``*_bits``, ``covered_q``/``covered_k`` (rows that belong to a sequence) and,
    with ``want_a``, the error scales ``*_a``."""
    qb, kb, vb, gb = _as_bits(q), _as_bits(k), _as_bits(v), _as_bits(dout)
    cu_q = [int(x) for x in np.asarray(cu_q).reshape(-1)]
    cu_k = [int(x) for x in np.asarray(cu_k).reshape(-1)]
    if len(cu_q) != len(cu_k) or len(cu_q) < 2:
        raise ValueError("cu_q and cu_k must both hold B + 1 >= 2 offsets")
    out = {n: np.zeros(t.shape, dtype=np.float64) for n, t in (("dq", qb), ("dk", kb), ("dv", kb))}
    if want_a:
        out.update({n + "_a": np.zeros_like(out[n]) for n in ("dq", "dk", "dv")})
    cov_q = np.zeros((qb.shape[0],), dtype=bool)
    cov_k = np.zeros((kb.shape[0],), dtype=bool)
    for b in range(len(cu_q) - 1):
        q0, q1, k0, k1 = cu_q[b], cu_q[b + 1], cu_k[b], cu_k[b + 1]
        if not (0 <= q0 <= q1 <= qb.shape[0] and 0 <= k0 <= k1 <= kb.shape[0]):
            raise ValueError("sequence %d: offsets out of order or out of range" % b)
        cov_q[q0:q1] = True
        cov_k[k0:k1] = True
        if q1 == q0 or k1 == k0:
            continue
        r = backward(qb[None, q0:q1], kb[None, k0:k1], vb[None, k0:k1], gb[None, q0:q1], "bshd",
                     causal=causal, want_a=want_a, lib=lib)
        for n, (a0, a1) in (("dq", (q0, q1)), ("dk", (k0, k1)), ("dv", (k0, k1))):
            out[n][a0:a1] = r[n][0]
            if want_a:
                out[n + "_a"][a0:a1] = r[n + "_a"][0]
    for n in ("dq", "dk", "dv"):
        out[n + "_bits"] = round_bf16(out[n], "rtne", lib=lib)
    out["covered_q"], out["covered_k"] = cov_q, cov_k
    return out


def gather_pages(k_cache, v_cache, seqlens_k, block_table):
    """The keys and values of a paged cache, gathered in order: sequence b's key j is slot
    j % page_size of page block_table[b][j // page_size] of the [num_pages, page_size, Hkv,
    d] caches.  Returns (k, v) packed [sum(seqlens_k), Hkv, d] and the key offsets cu_k."""
    kb, vb = _as_bits(k_cache), _as_bits(v_cache)
    P = kb.shape[1]
    table = np.asarray(block_table)
    ks, vs, cu_k = [], [], [0]
    for b, n in enumerate(int(x) for x in np.asarray(seqlens_k).reshape(-1)):
        for j in range(n):
            page = int(table[b][j // P])
            if not 0 <= page < kb.shape[0]:
                raise ValueError("sequence %d: page index %d out of range" % (b, page))
            ks.append(kb[page, j % P])
            vs.append(vb[page, j % P])
        cu_k.append(cu_k[-1] + n)
    shape = (0,) + kb.shape[2:]
    k = np.stack(ks) if ks else np.zeros(shape, dtype=np.uint16)
    v = np.stack(vs) if vs else np.zeros(shape, dtype=np.uint16)
    return k, v, np.asarray(cu_k)


def attention_paged(q, k_cache, v_cache, cu_q, seqlens_k, block_table, mode: str = "rtne",
                    causal: bool = False, want_a: bool = False, want_lse: bool = False, lib=None) -> dict:
    """Oracle attention of packed queries over a paged K/V cache.

    "AMD zverejnilo postup pre custom diffusion attention kernel vo FlyDSL na ROCm" (section
    on what AMD describes) names a paged KV cache among the layouts an attention kernel has to
    take.  The plain reading: the cache only says where each key and value lives, so the
    result is :func:`attention_varlen` over the keys gathered in order (:func:`gather_pages`).
    """
    k, v, cu_k = gather_pages(k_cache, v_cache, seqlens_k, block_table)
    return attention_varlen(q, k, v, cu_q, cu_k, mode, causal=causal, want_a=want_a,
                            want_lse=want_lse, lib=lib)


def round_bf16(x, mode: str = "rtne", lib=None) -> np.ndarray:
    """Round float64 values to bf16 bit patterns with the oracle's rounding rule."""
    lib = lib or load()
    xa = np.ascontiguousarray(np.asarray(x, dtype=np.float64))
    out = np.empty(xa.shape, dtype=np.uint16)
    lib.oracle_round_bf16_array(_ptr(xa, ctypes.c_double), xa.size, MODES[mode],
                                _ptr(out, ctypes.c_uint16))
    return out


def max_threads(lib=None) -> int:
    lib = lib or load()
    return int(lib.oracle_max_threads())


def forward_f64(q, k, v, layout: str = "bshd", causal: bool = False, lib=None) -> np.ndarray:
    """softmax(Q K^T / sqrt(d)) V on float64 arrays (no rounding): the function whose
    derivative :func:`backward` computes.  Shapes as for :func:`attention`."""
    lib = lib or load()
    qa, ka, va = (np.ascontiguousarray(np.asarray(t, dtype=np.float64)) for t in (q, k, v))
    B, H, Sq, Skv, d = dims(qa.shape, ka.shape, layout)
    o = np.empty_like(qa)
    rc = lib.attn_oracle_f64_forward(_ptr(qa, ctypes.c_double), _ptr(ka, ctypes.c_double),
                                     _ptr(va, ctypes.c_double), B, H, kv_heads(ka.shape, layout),
                                     Sq, Skv, d, LAYOUTS[layout], 1 if causal else 0,
                                     _ptr(o, ctypes.c_double))
    if rc != 0:
        raise ValueError("oracle rejected its arguments (rc=%d)" % rc)
    return o


def backward(q, k, v, dout, layout: str = "bshd", causal: bool = False, want_a: bool = False,
             want_delta: bool = False, threads: int | None = None, lib=None) -> dict:
    """fp64 gradients of softmax(Q K^T / sqrt(d)) V for bf16 q, k, v and upstream gradient
    dout (shaped like q).  Returns ``dq``, ``dk``, ``dv`` (float64, in the input layouts),
    their ``*_bits`` (bf16, RTNE), optionally forward-error scales ``dq_a``, ``dk_a``,
    ``dv_a`` and ``delta`` (D_i = dO_i . O_i, [B][H][Sq])."""
    lib = lib or load()
    qb, kb, vb, gb = _as_bits(q), _as_bits(k), _as_bits(v), _as_bits(dout)
    B, H, Sq, Skv, d = dims(qb.shape, kb.shape, layout)
    Hkv = kv_heads(kb.shape, layout)
    dq = np.empty(qb.shape, dtype=np.float64)
    dk = np.empty(kb.shape, dtype=np.float64)
    dv = np.empty(kb.shape, dtype=np.float64)
    dq_a = np.empty_like(dq) if want_a else None
    dk_a = np.empty_like(dk) if want_a else None
    dv_a = np.empty_like(dv) if want_a else None
    delta = np.empty((B, H, Sq), dtype=np.float64) if want_delta else None
    rc = lib.attn_oracle_bwd(_ptr(qb, ctypes.c_uint16), _ptr(kb, ctypes.c_uint16),
                             _ptr(vb, ctypes.c_uint16), _ptr(gb, ctypes.c_uint16), B, H, Hkv,
                             Sq, Skv, d, LAYOUTS[layout], 1 if causal else 0,
                             *(_ptr(a, ctypes.c_double) for a in (dq, dk, dv, dq_a, dk_a, dv_a,
                                                                   delta)),
                             int(threads or 0))
    if rc != 0:
        raise ValueError("oracle rejected its arguments (rc=%d)" % rc)
    out = {"dq": dq, "dk": dk, "dv": dv}
    for key in ("dq", "dk", "dv"):
        out[key + "_bits"] = round_bf16(out[key], "rtne", lib=lib)
    if want_a:
        out.update(dq_a=dq_a, dk_a=dk_a, dv_a=dv_a)
    if want_delta:
        out["delta"] = delta
    return out
