"""Writes closed_form_small.json: oracle outputs on the closed-form inputs of
``activated_mlp_gemms_gb300.workloads.closed_form_inputs``.  Calls only the
oracle; run from the repository root: ``python tests/golden/make_golden.py``."""
import json
import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
sys.path.insert(0, ROOT)

from activated_mlp_gemms_gb300.workloads import closed_form_inputs, to_f64  # noqa: E402
from oracle import mlp_backward, mlp_forward  # noqa: E402

CASES = [  # (M, H, I, act, gate_mult, down_mult)
    (4, 8, 16, "swiglu", 1.0, 1.0),
    (4, 8, 16, "swiglu", 1.125, 2.0),
    (4, 8, 16, "relu_sq", 1.0, 1.0),
    (4, 8, 16, "gelu_tanh_approx", 0.5, 1.5),
]


def main():
    out = {"generator": "activated_mlp_gemms_gb300.workloads.closed_form_inputs",
           "writer": "tests/golden/make_golden.py (oracle only)", "cases": []}
    for (M, H, I, act, gm, dm) in CASES:
        t = closed_form_inputs(M, H, I, act)
        a = {k: to_f64(v) for k, v in t.items()}
        fw = mlp_forward(a["x"], a["Wg"], a["Wu"], a["Wd"], act, gm, dm)
        bw = mlp_backward(a["dout"], a["x"], a["Wg"], a["Wu"], a["Wd"], act, gm, dm)
        rec = {"M": M, "H": H, "I": I, "act": act, "gate_mult": gm, "down_mult": dm,
               "out": fw["out"].tolist()}
        for k in ("dx", "dWg", "dWu", "dWd"):
            rec[k] = None if bw[k] is None else bw[k].tolist()
        out["cases"].append(rec)
    path = os.path.join(os.path.dirname(os.path.abspath(__file__)), "closed_form_small.json")
    with open(path, "w") as f:
        json.dump(out, f, indent=0)
    print("wrote", path)


if __name__ == "__main__":
    main()
