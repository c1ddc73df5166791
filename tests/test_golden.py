"""Regression pin: the oracle still reproduces the stored closed-form fixture
(written by tests/golden/make_golden.py, which calls only the oracle)."""
import json
import os

import numpy as np

from activated_mlp_gemms_gb300.workloads import closed_form_inputs, to_f64
from oracle import mlp_backward, mlp_forward

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "closed_form_small.json")


def load_golden():
    with open(GOLDEN) as f:
        return json.load(f)["cases"]


def test_inputs_are_exact_in_bf16():
    t = closed_form_inputs(4, 8, 16, "swiglu")
    for k, v in t.items():
        assert np.array_equal(to_f64(v), to_f64(v.double())), k


def test_oracle_reproduces_golden():
    for c in load_golden():
        t = {k: to_f64(v) for k, v in closed_form_inputs(c["M"], c["H"], c["I"], c["act"]).items()}
        fw = mlp_forward(t["x"], t["Wg"], t["Wu"], t["Wd"], c["act"], c["gate_mult"], c["down_mult"])
        bw = mlp_backward(t["dout"], t["x"], t["Wg"], t["Wu"], t["Wd"], c["act"],
                          c["gate_mult"], c["down_mult"])
        np.testing.assert_allclose(fw["out"], np.array(c["out"]), rtol=1e-12, atol=1e-14)
        for k in ("dx", "dWg", "dWu", "dWd"):
            if c[k] is None:
                assert bw[k] is None
            else:
                np.testing.assert_allclose(bw[k], np.array(c[k]), rtol=1e-12, atol=1e-14)
