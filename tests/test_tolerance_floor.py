"""Why the small GPU test shapes cannot all meet the 5e-3 bound on
fp32-accumulated weight gradients, and how far above it they may land.

The kernels store G, U (P), the postact and dG, dU (dP) in bf16 between
their GEMMs.  ``bf16_floor.emulated_dw`` repeats the path's arithmetic in
exact fp64 with only those roundings; its distance from the oracle is a
floor no implementation that stores those tensors in bf16 can get under.
These CPU tests pin the emulation to the oracle (with the roundings off it
must give the oracle's values) and show that at the small shapes the floor
itself exceeds 5e-3 in some cases, while staying well under 1e-2.  The GPU
tests hold each fp32-accumulated gradient to max(5e-3, 1.25 x its floor)."""
import numpy as np
import pytest

from activated_mlp_gemms_gb300.workloads import make_inputs, to_f64
from bf16_floor import bf, emulated_dw
from oracle import block_backward, mlp_backward, rel_err, rms_norm

TOL_F32 = 5e-3
SMALL = [(64, 128, 352), (300, 200, 392), (257, 264, 520)]
CASES = [("swiglu", 1.0, 1.0), ("swiglu", 1.125, 2.0), ("relu_sq", 1.0, 1.0),
         ("gelu_tanh_approx", 0.75, 1.5)]


def _inputs(M, H, I, act, seed):
    t = make_inputs(M, H, I, act, seed=seed, dW_prev=True)
    a = {k: to_f64(v) for k, v in t.items()}
    prev = {"dWg": a["dWg_prev"], "dWu": a.get("dWu_prev"), "dWd": a["dWd_prev"]}
    return a, prev


def test_bf16_rounding_is_round_to_nearest_even():
    # 1 + 2^-8 lies halfway between bf16 neighbours 1 and 1 + 2^-7: ties go to even (1)
    assert bf(np.array([1.0 + 2.0 ** -8]))[0] == 1.0
    assert bf(np.array([1.0 + 3 * 2.0 ** -8]))[0] == 1.0 + 2.0 ** -6
    assert bf(np.array([1.0 + 2.0 ** -8 + 2.0 ** -20]))[0] == 1.0 + 2.0 ** -7


@pytest.mark.parametrize("act", ["swiglu", "relu_sq", "gelu_tanh_approx", "reglu", "glu"])
@pytest.mark.parametrize("mode", ["saved", "recompute"])
def test_emulation_without_rounding_is_the_oracle(act, mode):
    M, H, I = 37, 24, 40
    a, prev = _inputs(M, H, I, act, 3)
    got = emulated_dw(a["x"], a["dout"], a["Wg"], a.get("Wu"), a["Wd"], act, 1.125, 2.0, mode,
                      dW_prev=prev, rounding=False)
    ref = mlp_backward(a["dout"], a["x"], a["Wg"], a.get("Wu"), a["Wd"], act, 1.125, 2.0,
                       dW_prev=prev)
    for k in ("dWg", "dWu", "dWd"):
        if ref[k] is not None:
            assert rel_err(got[k], ref[k]) < 1e-12, k


@pytest.mark.parametrize("act", ["swiglu", "relu_sq"])
def test_emulation_without_rounding_is_the_block_oracle(act):
    M, H, I = 37, 24, 40
    a, prev = _inputs(M, H, I, act, 4)
    eps, post = 2.0 ** -7, 0.8
    _, r = rms_norm(a["x"], eps)
    got = emulated_dw(a["x"], a["dout"], a["Wg"], a.get("Wu"), a["Wd"], act, 1.125, 2.0 * post,
                      "saved", dW_prev=prev, rstd=1.0 / r[:, 0], rounding=False)
    ref = block_backward(a["dout"], a["x"], a["Wg"], a.get("Wu"), a["Wd"], act, 1.125, 2.0,
                         resid_lambda=1.1, post_lambda=post, eps=eps, dW_prev=prev)
    for k in ("dWg", "dWu", "dWd"):
        if ref[k] is not None:
            assert rel_err(got[k], ref[k]) < 1e-12, k


def test_rounding_changes_the_result():
    # the emulation does round: a plain planted check that it is not the identity
    M, H, I = 64, 128, 352
    a, prev = _inputs(M, H, I, "swiglu", 1)
    got = emulated_dw(a["x"], a["dout"], a["Wg"], a["Wu"], a["Wd"], "swiglu", 1.0, 1.0)
    ref = mlp_backward(a["dout"], a["x"], a["Wg"], a["Wu"], a["Wd"], "swiglu")
    assert rel_err(got["dWg"], ref["dWg"]) > 1e-4


def floors():
    """The floor of every fp32-accumulated gradient of the small GPU parity
    cases (the inputs of test_small_parity: seed 1)."""
    out = {}
    for M, H, I in SMALL:
        for act, gm, dm in CASES:
            a, prev = _inputs(M, H, I, act, 1)
            ref = mlp_backward(a["dout"], a["x"], a["Wg"], a.get("Wu"), a["Wd"], act, gm, dm,
                               dW_prev=prev)
            for mode in ("saved", "recompute"):
                got = emulated_dw(a["x"], a["dout"], a["Wg"], a.get("Wu"), a["Wd"], act, gm, dm,
                                  mode, dW_prev=prev)
                for k in ("dWg", "dWu", "dWd"):
                    if ref[k] is not None:
                        out[(M, H, I, act, gm, dm, mode, k)] = rel_err(got[k], ref[k])
    return out


def test_small_shapes_floor_exceeds_the_workload_bound():
    f = floors()
    worst = max(f, key=f.get)
    # the bf16 storage alone puts some small cases above 5e-3 ...
    assert f[worst] > TOL_F32, (worst, f[worst])
    over = sorted(k for k, v in f.items() if v > TOL_F32)
    assert over, over
    # ... and every case well below 1e-2
    assert f[worst] < 8e-3, (worst, f[worst])
