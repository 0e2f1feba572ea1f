"""The oracle still computes what it computed when its digests were written.

The digests in ``tests/golden/oracle_*.txt`` come from
``tests/golden/make_golden.py``, which calls only the oracle. A mismatch means
the oracle's arithmetic changed; the change must name its reason.
"""
import math
import os

import pytest

HERE = os.path.join(os.path.dirname(__file__), "golden")

import tests.golden.make_golden as G  # noqa: E402


@pytest.mark.parametrize("name", list(G.CASES))
def test_oracle_digest_unchanged(name):
    want = {}
    with open(os.path.join(HERE, f"oracle_{name}.txt")) as f:
        for line in f:
            if line.startswith("#"):
                continue
            b, key, val = line.split()
            want[(b, key)] = float(val)
    got = {}
    for line in G.digest(G.CASES[name]):
        b, key, val = line.split()
        got[(b, key)] = float(val)
    assert got.keys() == want.keys()
    for k, v in want.items():
        if math.isnan(v):
            assert math.isnan(got[k]), k
        else:
            assert got[k] == pytest.approx(v, rel=1e-12, abs=1e-14), k
