"""Regression pin: the oracle still reproduces the fixture written by
tests/golden/make_golden.py (oracle-only script) on the seeded tiny workload."""
import json
import os

import numpy as np

from tests.golden.make_golden import compute

HERE = os.path.dirname(os.path.abspath(__file__))


def test_oracle_matches_golden_fixture():
    with open(os.path.join(HERE, "golden", "tiny_oracle.json")) as f:
        gold = json.load(f)
    now = compute()
    assert now["counts"] == gold["counts"]
    assert now["row2slot_head"] == gold["row2slot_head"]
    for key in ("y", "dx", "dw", "dW1", "dW2"):
        for k, v in gold[key].items():
            np.testing.assert_allclose(now[key][k], v, rtol=1e-12, atol=1e-14)
    np.testing.assert_allclose(now["y_abs_sum"], gold["y_abs_sum"], rtol=1e-12)
    np.testing.assert_allclose(now["dW1_abs_sum"], gold["dW1_abs_sum"], rtol=1e-12)
