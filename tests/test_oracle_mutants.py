"""Planted mistakes in a private copy of the oracle must each fail at least one pin.

Each mutation is a plausible slip (a dropped term, a wrong sign or index, a transposed
operand, a mis-rounded tie).  The copy is compiled into a temporary directory on the CPU;
the committed oracle is never touched.
"""
import os
import shutil
import subprocess
import tempfile

import pytest

import oracle
from tests import oracle_pins

SRC = os.path.join(os.path.dirname(oracle.__file__), "attn_oracle.c")
SRC_BWD = os.path.join(os.path.dirname(oracle.__file__), "attn_oracle_bwd.c")

MUTANTS = {
    "no_scale": ("s[j] = acc * scale;", "s[j] = acc;"),
    "scale_fixed_at_d128": ("const double scale = 1.0 / sqrt((double)d);",
                            "const double scale = 1.0 / sqrt(128.0);"),
    "kv_stride_uses_Sq": ("elem_offset(layout, b, j, kvh, 0, Skv, Hkv, d)",
                          "elem_offset(layout, b, j, kvh, 0, Sq, Hkv, d)"),
    "exp_sign": ("exp(s[j] - m)", "exp(m - s[j])"),
    "ties_to_odd": ("fmod(n, 2.0) != 0.0", "fmod(n, 2.0) == 0.0"),
    "rtna_as_rtne": ("if (rem >= half) r = a + q;", "if (rem > half) r = a + q;"),
    "neginf_key_drops_nan": ("term = 0.0 * vj;", "term = 0.0;"),
    "underflow_kills_inf": ("term = vj;                       /* positive weight times +-inf */",
                            "term = w[j] * vj;"),
    "nan_not_canonical": ("if (isnan(x)) return 0x7FC0;", "if (isnan(x)) return 0xFFC0;"),
    "bshd_as_bhsd": ("if (layout == ORACLE_LAYOUT_BSHD) return ((b * S + s) * H + h) * d + x;",
                     "if (layout == ORACLE_LAYOUT_BSHD) return ((b * H + h) * S + s) * d + x;"),
    "sum_skips_first_key": ("l += w[j];", "if (j > 0) l += w[j];"),
    "v_transposed": ("v[elem_offset(layout, b, j, kvh, x, Skv, Hkv, d)]",
                     "v[elem_offset(layout, b, x % Skv, kvh, j % d, Skv, Hkv, d)]"),
    "causal_off_by_one": ("nvis = last < 0 ? 0 : (last + 1 < Skv ? last + 1 : Skv);",
                          "nvis = last < 0 ? 0 : (last < Skv ? last : Skv);"),
    "gqa_head_interleaved": ("const int64_t kvh = h / (H / Hkv);", "const int64_t kvh = h % Hkv;"),
    "lse_drops_max": ("if (lse) lse[slot] = m + log(l);", "if (lse) lse[slot] = log(l);"),
    "posinf_logit_ignored": ("if (isnan(s[j]) || (isinf(s[j]) && s[j] > 0)) any_nan_or_posinf = 1;",
                             "if (isnan(s[j])) any_nan_or_posinf = 1;"),
    # the forward-error scale A, which sets the parity tolerance
    "a_not_divided_by_l": ("isfinite(ox) ? absnum / l : NAN", "isfinite(ox) ? absnum : NAN"),
    "a_divided_by_l_twice": ("isfinite(ox) ? absnum / l : NAN", "isfinite(ox) ? absnum / l / l : NAN"),
    "a_unweighted": ("absnum += w[j] * fabs(vj);", "absnum += fabs(vj);"),
    "a_signed": ("absnum += w[j] * fabs(vj);", "absnum += w[j] * vj;"),
}

# planted mistakes in the backward source
MUTANTS_BWD = {
    "bwd_ds_drops_delta": ("const double ds = p[j] * (dp[j] - Di);", "const double ds = p[j] * dp[j];"),
    "bwd_dk_unscaled": ("dk[off] += c * ds * qi[x];", "dk[off] += ds * qi[x];"),
    "bwd_dv_uses_ds": ("dv[off] += p[j] * gi[x];", "dv[off] += (p[j] - Di * 0.0 + dp[j] * p[j]) * gi[x];"),
    "bwd_dq_sign": ("acc += p[j] * (dp[j] - Di) * kjx;", "acc += p[j] * (Di - dp[j]) * kjx;"),
    "bwd_causal_sees_all": ("if (!causal) return Skv;", "return Skv;"),
    # the backward's error scales
    "bwd_dabs_is_abs_delta": ("(fabs(dp[j]) + Dabs)", "(fabs(dp[j]) + fabs(Di))"),
    "bwd_dv_a_unweighted": ("dv_a[off] += p[j] * fabs(gi[x]);", "dv_a[off] += fabs(gi[x]);"),
    "bwd_dq_a_unscaled": ("if (dq_a) dq_a[off] = c * mag;", "if (dq_a) dq_a[off] = mag;"),
    "bwd_dk_a_drops_dp": ("const double dsa = p[j] * (fabs(dp[j]) + Dabs);",
                          "const double dsa = p[j] * Dabs;"),
}


@pytest.fixture(scope="module")
def workdir():
    d = tempfile.mkdtemp(prefix="oracle_mut_")
    yield d
    shutil.rmtree(d, ignore_errors=True)


@pytest.mark.parametrize("name", sorted(MUTANTS) + sorted(MUTANTS_BWD))
def test_mutant_is_caught(name, workdir):
    bwd = name in MUTANTS_BWD
    old, new = (MUTANTS_BWD if bwd else MUTANTS)[name]
    text = open(SRC_BWD if bwd else SRC).read()
    assert text.count(old) >= 1, "mutation site vanished: %s" % name
    src = os.path.join(workdir, name + ".c")
    with open(src, "w") as f:
        f.write(text.replace(old, new))
    so = os.path.join(workdir, "lib%s.so" % name)
    if bwd:
        oracle.build(force=True, out=so, bwd_src=src)
    else:
        oracle.build(force=True, src=src, out=so)
    lib = oracle.load(so)
    failed = []
    for pin in oracle_pins.ALL_PINS:
        try:
            pin(lib)
        except (AssertionError, ValueError):
            failed.append(pin.__name__)
    assert failed, "no pin caught the planted mistake %r" % name
