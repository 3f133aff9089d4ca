"""The oracle against hand-worked examples stored in tests/golden/."""
import json
import os

import numpy as np
import pytest

import oracle
from oracle import Conv

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "worked_examples.json")
EXAMPLES = json.load(open(GOLDEN))["examples"]


@pytest.mark.parametrize("ex", EXAMPLES, ids=lambda e: e["name"])
def test_worked_example(ex):
    cv = Conv(**ex["conv"])
    x = np.array(ex["x"], dtype=np.float64)
    w = np.array(ex["w"], dtype=np.float64)
    b = None if ex["bias"] is None else np.array(ex["bias"], dtype=np.float64)
    assert np.array_equal(oracle.fwd(cv, x, w, b), np.array(ex["y"], dtype=np.float64))
    if "gy_ones_gx" in ex:
        g = np.ones((cv.N, cv.OC, cv.Ho, cv.Wo))
        assert np.array_equal(oracle.bwd_data(cv, g, w), np.array(ex["gy_ones_gx"], dtype=np.float64))
        gw, gb = oracle.bwd_weight(cv, x, g, want_b=True)
        assert np.array_equal(gw, np.array(ex["gy_ones_gw"], dtype=np.float64))
        assert np.array_equal(gb, np.array(ex["gy_ones_gb"], dtype=np.float64))
