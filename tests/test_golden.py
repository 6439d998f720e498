"""Regression pin: the oracle's 'tiny' rows equal the stored fixture."""
import json
import os

import numpy as np

import oracle
import rpa_inputs as ri
from golden.make_golden import digest

HERE = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def test_tiny_fixture():
    with open(os.path.join(HERE, "tiny_oracle.json")) as f:
        g = json.load(f)
    p = ri.workload("tiny")
    assert digest(p) == g["input_sha256"], "input generator changed"
    o = oracle.forward(p)
    for r in g["rows"]:
        np.testing.assert_allclose(o[r["token"], r["q_head"]], r["o"], rtol=0, atol=1e-12)
    np.testing.assert_allclose(o.sum(axis=(1, 2)), g["row_sums"], rtol=0, atol=1e-10)
