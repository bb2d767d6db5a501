"""The oracle reproduces the stored formula-input case (regression pin written by tests/golden/make_golden.py)."""

import json
import os

import numpy as np

from tests.golden import make_golden as mg

HERE = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def test_formula_case_matches_stored():
    with open(os.path.join(HERE, "formula_case.json")) as f:
        gold = json.load(f)
    raw, pooled, idx = mg.expected()
    np.testing.assert_allclose(raw, gold["raw"], rtol=1e-13)
    np.testing.assert_allclose(pooled, gold["pooled"], rtol=1e-13)
    np.testing.assert_array_equal(idx, gold["idx"])
    # column mass of a group is bounded by G * W
    assert np.all(np.asarray(gold["raw"]).sum(axis=1) <= 2 * 4 + 1e-9)
