"""Regression anchor: the oracle still reproduces the stored tiny-step values
(written by tests/golden/make_golden.py from the oracle alone)."""

import json
import os

import numpy as np

HERE = os.path.dirname(os.path.abspath(__file__))


def test_tiny_step_matches_stored_values():
    from tests.golden.make_golden import tiny_case
    stored = json.load(open(os.path.join(HERE, "golden", "tiny_step.json")))
    now = tiny_case()
    for key in ("root_token", "parents", "tokens", "depth", "mask", "path", "n_accepted", "bonus"):
        assert now[key] == stored[key], key
    np.testing.assert_allclose(now["values"], stored["values"], rtol=0, atol=1e-12)
    np.testing.assert_allclose(now["attn_row_sums"], stored["attn_row_sums"], rtol=0, atol=1e-10)
    assert stored["near_ties"] == ""
