"""Writes fp8_closed_form.json: the FP8 oracle's outputs on the closed-form
8-bit inputs of ``activated_mlp_gemms_gb300.workloads.fp8_closed_form_codes``
with power-of-two scales.  Calls only the oracle (and torch's bf16 cast for
the saved preact); run from the repository root:
``python tests/golden/make_golden_fp8.py``."""
import json
import math
import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402
import torch  # noqa: E402

from activated_mlp_gemms_gb300.workloads import fp8_closed_form_codes, to_f64  # noqa: E402
from oracle import E5M2_MAX, fp8_relu_sq_backward, fp8_relu_sq_forward  # noqa: E402

CASES = [  # (M, H, I, gate_mult, down_mult)
    (4, 16, 32, 1.0, 1.0),
    (4, 16, 48, 0.5, 2.0),
]
SX, S1, S2, S_POST, SG = 2.0 ** -4, 2.0 ** -5, 2.0 ** -5, 2.0 ** -15, 2.0 ** -6


def main():
    out = {"generator": "activated_mlp_gemms_gb300.workloads.fp8_closed_form_codes",
           "writer": "tests/golden/make_golden_fp8.py (oracle only)",
           "scales": {"sx": SX, "s1": S1, "s2": S2, "s_post": S_POST, "sg": SG}, "cases": []}
    for (M, H, I, gm, dm) in CASES:
        t = fp8_closed_form_codes(M, H, I)
        x8, W1, W2 = (t[k].numpy() for k in ("x8", "W1_8", "W2_8"))
        dout = to_f64(t["dout"])
        fw = fp8_relu_sq_forward(x8, W1, W2, SX, S1, S2, S_POST, gm, dm)
        pre = (x8 @ W1.T) * (SX * S1)
        pre_bf = to_f64(torch.tensor(pre, dtype=torch.float64).to(torch.bfloat16))
        probe = fp8_relu_sq_backward(dout, x8, W1, W2, fw["a8"], SX, S1, S2, S_POST, SG, 1.0, gm,
                                     dm, pre=pre_bf)
        # a power-of-two delayed dpre scale covering this step's amax
        s_dpre = 2.0 ** math.ceil(math.log2(probe["amax_dpre"] * 1.25 / E5M2_MAX))
        bw = fp8_relu_sq_backward(dout, x8, W1, W2, fw["a8"], SX, S1, S2, S_POST, SG, s_dpre, gm,
                                  dm, pre=pre_bf)
        out["cases"].append({
            "M": M, "H": H, "I": I, "gate_mult": gm, "down_mult": dm, "s_dpre": s_dpre,
            "pre_bf16": pre_bf.tolist(), "out": fw["out"].tolist(), "a8": fw["a8"].tolist(),
            "amax_a": fw["amax_a"], "dout8": bw["dout8"].tolist(), "dP8": bw["dP8"].tolist(),
            "amax_dpre": bw["amax_dpre"], "dx": bw["dx"].tolist(), "dW1": bw["dW1"].tolist(),
            "dW2": bw["dW2"].tolist()})
    path = os.path.join(os.path.dirname(os.path.abspath(__file__)), "fp8_closed_form.json")
    with open(path, "w") as f:
        json.dump(out, f, separators=(",", ":"))
    print("wrote", path, np.round(os.path.getsize(path) / 1024, 1), "KiB")


if __name__ == "__main__":
    main()
