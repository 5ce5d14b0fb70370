"""The oracle still reproduces its frozen outputs in tests/golden/oracle_tiny.json."""
import json
import os

import numpy as np

from golden import make_golden

HERE = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def test_oracle_matches_frozen_outputs():
    data = json.load(open(os.path.join(HERE, "oracle_tiny.json")))
    assert len(data["cases"]) == len(make_golden.CASES)
    for entry in data["cases"]:
        o, lse = make_golden.compute(tuple(entry["case"]))
        want_o = np.array([float(x) for x in entry["o"]])
        want_l = np.array([float(x) for x in entry["lse"]])
        assert np.array_equal(o.ravel(), want_o)
        assert np.array_equal(lse.ravel(), want_l)
