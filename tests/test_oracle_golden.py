"""The oracle built on this machine reproduces the stored digests (which were
written on another machine by tests/golden/make_golden.py)."""
import os

import pytest

from tests.golden import make_golden

HERE = os.path.dirname(os.path.abspath(__file__))


def _stored():
    out = {}
    with open(os.path.join(HERE, "golden", "oracle_digests.txt")) as f:
        for line in f:
            if line.startswith("#") or not line.strip():
                continue
            name, label, h = line.split()
            out.setdefault(name, {})[label] = h
    return out


@pytest.mark.parametrize("case", make_golden.CASES, ids=[c[0] for c in make_golden.CASES])
def test_oracle_digests_are_stable(oracle_mod, case):
    assert make_golden.digests(*case) == _stored()[case[0]]


@pytest.mark.parametrize("case", make_golden.RMS_CASES, ids=[c[0] for c in make_golden.RMS_CASES])
def test_oracle_rmsnorm_digests_are_stable(oracle_mod, case):
    assert make_golden.rms_digests(*case) == _stored()[case[0]]
