"""Exact helpers for the oracle's pins, independent of the oracle's own code.

* ``round_exact``: rounds an exact rational (``fractions.Fraction``) or an ``mpmath.mpf`` to
  a bf16 bit pattern by bisecting the sorted table of every finite bf16 value.  It shares
  nothing with the oracle's frexp/floor rounding.
* ``bits_to_float`` / ``float_to_bits``: bf16 bit patterns <-> Python floats.
* ``ulp_distance``: ordinal distance between bf16 patterns (+0 and -0 are the same point).
"""
from __future__ import annotations

import bisect
import struct
from fractions import Fraction

import numpy as np

BF16_MAX_BITS = 0x7F7F
NAN_BITS = 0x7FC0
INF_BITS = 0x7F80


def bits_to_float(b: int) -> float:
    return struct.unpack("<f", struct.pack("<I", (b & 0xFFFF) << 16))[0]


def float_to_bits_trunc(x: float) -> int:
    return struct.unpack("<I", struct.pack("<f", x))[0] >> 16


# every non-negative finite bf16 value, increasing with the bit pattern
_POS = [Fraction(bits_to_float(b)) for b in range(0, BF16_MAX_BITS + 1)]
_MAX = _POS[-1]
_TOP_QUANTUM = Fraction(2) ** (127 - 7)


def _to_fraction(x) -> Fraction:
    if isinstance(x, Fraction):
        return x
    if isinstance(x, (int,)):
        return Fraction(x)
    if isinstance(x, float):
        return Fraction(x)
    # mpmath.mpf: exact binary value (-1)**sign * man * 2**exp
    import mpmath
    sign, man, exp, _ = mpmath.mpf(x)._mpf_
    f = Fraction(int(man)) * (Fraction(2) ** exp)
    return -f if sign else f


def round_exact(x, mode: str) -> int:
    """Round a finite exact value to bf16 bits (RTNE ties-to-even pattern, RTNA ties away,
    RTZ toward zero).  Non-finite floats map to the canonical patterns."""
    if isinstance(x, float) and x != x:
        return NAN_BITS
    if isinstance(x, float) and x in (float("inf"), float("-inf")):
        return INF_BITS | (0x8000 if x < 0 else 0)
    fx = _to_fraction(x)
    sign = 0x8000 if fx < 0 else 0
    ax = abs(fx)
    if ax > _MAX:
        if mode == "rtz":
            return sign | BF16_MAX_BITS
        mid = _MAX + _TOP_QUANTUM / 2
        if ax < mid:
            return sign | BF16_MAX_BITS
        return sign | INF_BITS        # at the tie the max pattern is odd: both modes go up
    idx = bisect.bisect_right(_POS, ax) - 1
    lo = _POS[idx]
    if ax == lo:
        return sign | idx
    hi = _POS[idx + 1]
    mid = (lo + hi) / 2
    if mode == "rtz":
        r = idx
    elif mode == "rtna":
        r = idx + 1 if ax >= mid else idx
    else:
        if ax < mid:
            r = idx
        elif ax > mid:
            r = idx + 1
        else:
            r = idx if idx % 2 == 0 else idx + 1
    return sign | r


def near_midpoint(x, rel: float = 1e-12) -> bool:
    """True when x lies within rel*|x| of a bf16 rounding midpoint or of a bf16 value
    (where RTZ and the nearest modes are sensitive to the last bits)."""
    fx = abs(_to_fraction(x))
    if fx == 0 or fx > _MAX:
        return False
    idx = bisect.bisect_right(_POS, fx) - 1
    lo = _POS[idx]
    hi = _POS[idx + 1] if idx + 1 < len(_POS) else _MAX + _TOP_QUANTUM
    tol = fx * Fraction(rel)
    return min(abs(fx - (lo + hi) / 2), abs(fx - lo), abs(hi - fx)) <= tol


def ordinal(bits: np.ndarray) -> np.ndarray:
    """Monotone integer image of bf16 patterns: sign-magnitude -> two's complement."""
    b = bits.astype(np.int64) & 0xFFFF
    mag = b & 0x7FFF
    return np.where(b & 0x8000, -mag, mag)


def ulp_distance(a: np.ndarray, b: np.ndarray) -> np.ndarray:
    return np.abs(ordinal(a) - ordinal(b))


def is_nan_bits(b: np.ndarray) -> np.ndarray:
    b = b.astype(np.int64) & 0xFFFF
    return ((b & 0x7F80) == 0x7F80) & ((b & 0x007F) != 0)


def is_finite_bits(b: np.ndarray) -> np.ndarray:
    b = b.astype(np.int64) & 0xFFFF
    return (b & 0x7F80) != 0x7F80
