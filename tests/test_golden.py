"""The oracle still gives the results stored in tests/golden/oracle_tiny.json
(written by tests/golden/make_golden.py from the oracle itself on seeded
inputs). Integers must match exactly and floating-point values to 1e-12: a
change to the oracle's arithmetic shows up here and must be justified by
the passage it follows. CPU only."""
import json
import os
import sys

import numpy as np

HERE = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, os.path.join(HERE, "golden"))

import make_golden  # noqa: E402


def _same(a, b, path=""):
    if isinstance(a, dict):
        assert set(a) == set(b), path
        for k in a:
            _same(a[k], b[k], f"{path}.{k}")
    elif isinstance(a, list):
        assert len(a) == len(b), path
        for i, (x, y) in enumerate(zip(a, b)):
            _same(x, y, f"{path}[{i}]")
    elif isinstance(a, float) or isinstance(b, float):
        if a is None or b is None:
            assert a is None and b is None, path
        elif np.isinf(a) or np.isinf(b):
            assert a == b, path
        else:
            assert abs(a - b) <= 1e-12 * max(1.0, abs(b)), f"{path}: {a} vs {b}"
    else:
        assert a == b, f"{path}: {a} vs {b}"


def test_oracle_matches_the_stored_fixture():
    with open(os.path.join(HERE, "golden", "oracle_tiny.json")) as f:
        stored = json.load(f)
    _same(json.loads(json.dumps(make_golden.compute())), stored)
