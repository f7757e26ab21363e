"""Write the oracle regression fixture ``oracle_small.txt`` (calls only ``oracle/``).

The pages print no worked example of the attention forward (their figures are speedup
ratios), so nothing here comes from them.  This fixture freezes the oracle's own output on
small seeded inputs, so that a later change to the oracle's arithmetic shows up as a diff.
Run from the repository root:  python tests/golden/make_golden.py
"""
import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
sys.path.insert(0, ROOT)

import oracle  # noqa: E402
from workloads import make_qkv  # noqa: E402

CASES = [  # (B, H, Sq, Skv, layout, seed, sigma, mode)
    (1, 1, 3, 5, "bhsd", 1, 1.0, "rtne"),
    (1, 2, 2, 7, "bshd", 2, 4.0, "rtna"),
    (2, 1, 2, 3, "bhsd", 3, 0.5, "rtz"),
]


def lines():
    out = []
    for (B, H, Sq, Skv, layout, seed, sigma, mode) in CASES:
        q, k, v = make_qkv(B, H, Sq, Skv, 128, layout, seed=seed, sigma=sigma)
        o = oracle.attention(q, k, v, layout, mode)["o_bits"].reshape(-1)
        out.append("case %d %d %d %d %s %d %g %s" % (B, H, Sq, Skv, layout, seed, sigma, mode))
        out.append(" ".join("%04x" % int(b) for b in o))
    return out


if __name__ == "__main__":
    path = os.path.join(os.path.dirname(os.path.abspath(__file__)), "oracle_small.txt")
    with open(path, "w") as f:
        f.write("# oracle regression fixture, written by tests/golden/make_golden.py\n")
        f.write("\n".join(lines()) + "\n")
