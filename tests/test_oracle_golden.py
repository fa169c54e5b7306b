"""The oracle still returns what it returned when the regression fixture was written."""
import os

import numpy as np

from tests.golden import make_golden


def _read(path):
    out = {}
    with open(path) as f:
        lines = [l for l in f.read().splitlines() if not l.startswith("#")]
    for head, body in zip(lines[0::2], lines[1::2]):
        name, *shape = head.split()
        out[name] = np.array([float(v) for v in body.split()]).reshape([int(s) for s in shape])
    return out


def test_oracle_matches_regression_fixture():
    stored = _read(os.path.join(os.path.dirname(make_golden.__file__), "oracle_small_case.txt"))
    live = make_golden.compute()
    assert set(stored) == set(live)
    for name, arr in live.items():
        np.testing.assert_allclose(arr, stored[name], rtol=1e-12, atol=1e-14, err_msg=name)
