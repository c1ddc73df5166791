"""Regression pins: the oracles still reproduce the stored closed-form
fixtures (written by tests/golden/make_golden.py and make_golden_fp8.py,
which call only the oracles)."""
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


FP8_GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "fp8_closed_form.json")


def test_fp8_closed_form_inputs_are_exact():
    from activated_mlp_gemms_gb300.workloads import fp8_closed_form_codes
    from oracle import e4m3
    t = fp8_closed_form_codes(4, 16, 32)
    for k in ("x8", "W1_8", "W2_8"):
        v = t[k].numpy()
        assert np.array_equal(e4m3(v), v), k  # integer codes on the e4m3 grid
    assert np.array_equal(to_f64(t["dout"]), to_f64(t["dout"].double()))


def test_oracle_reproduces_fp8_golden():
    """The FP8 oracle still reproduces the stored fixture (written by
    tests/golden/make_golden_fp8.py, which calls only the oracle)."""
    from activated_mlp_gemms_gb300.workloads import fp8_closed_form_codes
    from oracle import fp8_relu_sq_backward, fp8_relu_sq_forward
    with open(FP8_GOLDEN) as f:
        g = json.load(f)
    sc = g["scales"]
    for c in g["cases"]:
        t = fp8_closed_form_codes(c["M"], c["H"], c["I"])
        x8, W1, W2 = (t[k].numpy() for k in ("x8", "W1_8", "W2_8"))
        fw = fp8_relu_sq_forward(x8, W1, W2, sc["sx"], sc["s1"], sc["s2"], sc["s_post"],
                                 c["gate_mult"], c["down_mult"])
        assert np.array_equal(fw["a8"], np.array(c["a8"]))
        np.testing.assert_allclose(fw["out"], np.array(c["out"]), rtol=1e-12, atol=0)
        bw = fp8_relu_sq_backward(to_f64(t["dout"]), x8, W1, W2, fw["a8"], sc["sx"], sc["s1"],
                                  sc["s2"], sc["s_post"], sc["sg"], c["s_dpre"], c["gate_mult"],
                                  c["down_mult"], pre=np.array(c["pre_bf16"]))
        for k in ("dout8", "dP8"):
            assert np.array_equal(bw[k], np.array(c[k])), k
        for k in ("dx", "dW1", "dW2"):
            np.testing.assert_allclose(bw[k], np.array(c[k]), rtol=1e-12, atol=0)
        assert bw["amax_dpre"] == c["amax_dpre"] and fw["amax_a"] == c["amax_a"]
