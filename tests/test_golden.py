"""The oracle still reproduces its recorded small cases (regression pin)."""

import json
import os

import numpy as np

from .golden import make_golden

HERE = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def _walk(a, b, path):
    if isinstance(b, dict):
        assert set(a) == set(b), path
        for k in b:
            _walk(a[k], b[k], f"{path}.{k}")
    elif b is None:
        assert a is None, path
    else:
        np.testing.assert_allclose(np.asarray(a, np.float64),
                                   np.asarray(b, np.float64),
                                   rtol=1e-13, atol=1e-13, err_msg=path)


def test_oracle_matches_recorded_small_cases():
    with open(os.path.join(HERE, "oracle_small.json")) as fh:
        stored = json.load(fh)
    fresh = json.loads(json.dumps(make_golden.compute()))
    _walk(fresh, stored, "golden")
