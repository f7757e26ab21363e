"""Compare GPU bf16 outputs with the oracle under the parity criteria.

Criteria (per element, the oracle's value O, its fp64 forward-error scale A):
  * non-finite oracle or GPU value: the bf16 bit patterns must be identical;
  * finite: ordinal bf16 distance <= 2 ("literal"), or, where the literal rule cannot hold
    because bf16-rounded softmax weights cancel, |gpu - O| <= 2^-8 * A + ulp(O) ("A-bound").
The fraction that meets the literal rule is reported next to the pass/fail verdict.
"""
from __future__ import annotations

import json
import os

import numpy as np

from tests import bf16_exact as bx

A_FACTOR = 2.0 ** -8


def bits_to_f64(bits: np.ndarray) -> np.ndarray:
    u = (bits.astype(np.uint32) & 0xFFFF) << 16
    return u.view(np.float32).astype(np.float64)


def bf16_ulp(bits: np.ndarray) -> np.ndarray:
    """Spacing of bf16 values at each (finite) pattern's magnitude."""
    mag = bits.astype(np.int64) & 0x7FFF
    exp = np.maximum(mag >> 7, 1)
    return np.exp2(exp.astype(np.float64) - 127 - 7)


def log_result(tag: str, res: dict) -> None:
    """Append one comparison's summary to the JSON-lines file named by PARITY_LOG, if set."""
    path = os.environ.get("PARITY_LOG")
    if path:
        with open(path, "a") as f:
            f.write(json.dumps(dict(res, tag=tag)) + "\n")


def compare(gpu_bits: np.ndarray, ref_bits: np.ndarray, ref_a: np.ndarray) -> dict:
    g = gpu_bits.reshape(-1).astype(np.uint16)
    r = ref_bits.reshape(-1).astype(np.uint16)
    a = ref_a.reshape(-1)
    fin = bx.is_finite_bits(r) & bx.is_finite_bits(g)
    nonfin = ~fin
    nonfin_ok = np.all(g[nonfin] == r[nonfin])
    n_nonfin_bad = int(np.sum(g[nonfin] != r[nonfin]))
    dist = bx.ulp_distance(g[fin], r[fin])
    literal = dist <= 2
    err = np.abs(bits_to_f64(g[fin]) - bits_to_f64(r[fin]))
    abound = err <= A_FACTOR * a[fin] + bf16_ulp(r[fin])
    ok_fin = literal | abound
    n = g.size
    return {
        "n": n,
        "n_finite": int(fin.sum()),
        "n_nonfinite": int(nonfin.sum()),
        "nonfinite_mismatch": n_nonfin_bad,
        "finite_fail": int((~ok_fin).sum()),
        "literal_frac": float(literal.mean()) if literal.size else 1.0,
        "max_ulp": int(dist.max()) if dist.size else 0,
        "max_err_over_a": float(np.max(err / np.maximum(a[fin], 1e-300))) if err.size else 0.0,
        "ok": bool(nonfin_ok and ok_fin.all()),
    }


def gpu_rows_bits(o, layout: str, rows=None) -> np.ndarray:
    """GPU output tensor -> uint16 bits in BHSD row order ([rows, d] when rows given)."""
    import torch
    t = o.detach()
    if layout == "bshd":
        t = t.permute(0, 2, 1, 3)
    t = t.contiguous().cpu()
    d = t.shape[-1]
    bits = t.view(torch.int16).numpy().view(np.uint16).reshape(-1, d)
    if rows is not None:
        bits = bits[np.asarray(rows, dtype=np.int64)]
    return bits
