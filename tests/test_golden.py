"""The oracle still reproduces its frozen regression fixture (CPU only)."""
import os

from tests.golden import make_golden


def test_oracle_matches_fixture():
    path = os.path.join(os.path.dirname(make_golden.__file__), "oracle_small.txt")
    stored = [ln.rstrip("\n") for ln in open(path) if not ln.startswith("#")]
    assert stored == make_golden.lines()
