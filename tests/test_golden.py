"""Oracle regression fixture (CPU): the tiny workload's first greedy steps."""
import json
import os

import numpy as np

from tests.golden.make_golden import tiny_greedy

HERE = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def test_tiny_greedy_matches_fixture():
    ref = json.load(open(os.path.join(HERE, "tiny_oracle_greedy.json")))["steps"]
    got = tiny_greedy(len(ref))
    for r, g in zip(ref, got):
        assert r["token_in"] == g["token_in"] and r["argmax"] == g["argmax"]
        np.testing.assert_allclose(g["logits_head"], r["logits_head"], rtol=1e-12, atol=1e-14)
        np.testing.assert_allclose(g["logits_sum"], r["logits_sum"], rtol=1e-10, atol=1e-12)
