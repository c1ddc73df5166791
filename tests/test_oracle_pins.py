"""Pins of the fp64 oracle against facts fixed by the pages and by mathematics.

None of these re-types the oracle's formulas: they check closed-form values,
finite differences, identity/permutation/zero weight cases with hand-derived
results, multiplier scaling, the accumulate and split-M identities, an
independent autograd cross-check, and finally that planted mistakes in the
oracle are caught by at least one of these pins.
"""
import math

import numpy as np
import pytest
import scipy.special as sp

import oracle.mlp_oracle as O

ACTS = list(O.ACTIVATIONS)  # swiglu, relu_sq, gelu_tanh_approx, relu, reglu, geglu, glu


def _rand_problem(rng, M, H, I, act):
    x = rng.standard_normal((M, H))
    Wg = rng.standard_normal((I, H)) / math.sqrt(H)
    Wu = rng.standard_normal((I, H)) / math.sqrt(H) if O.is_gated(act) else None
    Wd = rng.standard_normal((H, I)) / math.sqrt(I)
    dout = rng.standard_normal((M, H))
    return x, Wg, Wu, Wd, dout


# ---------------------------------------------------------------- activations

def check_act_zero(mod):
    for a in ACTS:
        expect = 0.5 if a == "glu" else 0.0  # sigmoid(0) = 1/2; the others vanish at 0
        assert mod.act_fn(a, 0.0) == expect, a
    assert abs(mod.act_grad("swiglu", 0.0) - 0.5) < 1e-15          # sigma(0) = 1/2
    assert abs(mod.act_grad("gelu_tanh_approx", 0.0) - 0.5) < 1e-15  # (1+tanh 0)/2
    assert abs(mod.act_grad("geglu", 0.0) - 0.5) < 1e-15
    assert abs(mod.act_grad("glu", 0.0) - 0.25) < 1e-15             # s (1 - s)
    assert mod.act_grad("relu_sq", 0.0) == 0.0                     # 2 relu(0)
    assert mod.act_grad("relu", 0.0) == 0.0 and mod.act_grad("reglu", 0.0) == 0.0


def test_act_at_zero():
    check_act_zero(O)


def test_silu_closed_form():
    # sigma(ln 3) = 3/4 and sigma(-ln 3) = 1/4 exactly
    L = math.log(3.0)
    assert abs(O.act_fn("swiglu", L) - 0.75 * L) < 1e-15
    assert abs(O.act_fn("swiglu", -L) + 0.25 * L) < 1e-15
    # silu'(z) = sigma(z) (1 + z (1 - sigma(z)))
    assert abs(O.act_grad("swiglu", L) - 0.75 * (1 + 0.25 * L)) < 1e-15
    # limits: silu(z) -> z for z >> 0, -> 0 for z << 0
    assert abs(O.act_fn("swiglu", 40.0) - 40.0) < 1e-12
    assert abs(O.act_fn("swiglu", -40.0)) < 1e-12


def test_sigmoid_and_relu_closed_forms():
    L = math.log(3.0)
    assert abs(O.act_fn("glu", L) - 0.75) < 1e-15 and abs(O.act_fn("glu", -L) - 0.25) < 1e-15
    assert abs(O.act_grad("glu", L) - 0.1875) < 1e-15  # 3/4 * 1/4
    z = np.array([-2.0, -1e-12, 0.0, 0.25, 3.0])
    for a in ("relu", "reglu"):
        np.testing.assert_array_equal(O.act_fn(a, z), [0.0, 0.0, 0.0, 0.25, 3.0])
        np.testing.assert_array_equal(O.act_grad(a, z), [0.0, 0.0, 0.0, 1.0, 1.0])
    # geglu applies the same tanh-approximated GELU as gelu_tanh_approx
    np.testing.assert_array_equal(O.act_fn("geglu", z), O.act_fn("gelu_tanh_approx", z))


def test_relu_sq_closed_form():
    z = np.array([-3.0, -1e-9, 0.0, 0.5, 3.0])
    np.testing.assert_array_equal(O.act_fn("relu_sq", z), [0.0, 0.0, 0.0, 0.25, 9.0])
    np.testing.assert_array_equal(O.act_grad("relu_sq", z), [0.0, 0.0, 0.0, 1.0, 6.0])


def check_gelu_vs_exact(mod):
    # The tanh approximation stays within 4.8e-4 of the exact GELU z*Phi(z)
    # (Phi from scipy's normal CDF, an independent routine).
    z = np.linspace(-8, 8, 40001)
    exact = z * sp.ndtr(z)
    assert np.max(np.abs(mod.act_fn("gelu_tanh_approx", z) - exact)) < 4.8e-4


def test_gelu_tanh_close_to_exact_gelu():
    check_gelu_vs_exact(O)


@pytest.mark.parametrize("act", ["swiglu", "gelu_tanh_approx", "geglu"])
def test_odd_part_identity(act):
    # z*s(z) with s(z)+s(-z)=1  =>  act(z) - act(-z) = z
    z = np.linspace(-6, 6, 1001)
    np.testing.assert_allclose(O.act_fn(act, z) - O.act_fn(act, -z), z, atol=1e-13)


def check_act_grad_fd(mod):
    z = np.linspace(-5, 5, 2001) + 1e-3  # avoid the relu kink exactly at 0
    h = 1e-6
    for a in ACTS:
        fd = (mod.act_fn(a, z + h) - mod.act_fn(a, z - h)) / (2 * h)
        np.testing.assert_allclose(mod.act_grad(a, z), fd, rtol=1e-6, atol=1e-7)


def test_act_grad_matches_finite_difference():
    check_act_grad_fd(O)


# ---------------------------------------------------- whole-MLP finite differences

def check_fd_gradients(mod, act, gm=1.3, dm=0.7, M=3, H=4, I=5, seed=1):
    rng = np.random.default_rng(seed)
    x, Wg, Wu, Wd, dout = _rand_problem(rng, M, H, I, act)
    bw = mod.mlp_backward(dout, x, Wg, Wu, Wd, act, gm, dm)

    def loss(x_, Wg_, Wu_, Wd_):
        return float(np.sum(dout * mod.mlp_forward(x_, Wg_, Wu_, Wd_, act, gm, dm)["out"]))

    params = {"dx": x, "dWg": Wg, "dWd": Wd}
    if Wu is not None:
        params["dWu"] = Wu
    h = 1e-6
    for name, P in params.items():
        fd = np.zeros_like(P)
        for idx in np.ndindex(P.shape):
            old = P[idx]
            P[idx] = old + h
            lp = loss(x, Wg, Wu, Wd)
            P[idx] = old - h
            lm = loss(x, Wg, Wu, Wd)
            P[idx] = old
            fd[idx] = (lp - lm) / (2 * h)
        err = np.max(np.abs(bw[name] - fd)) / max(np.max(np.abs(fd)), 1e-30)
        assert err < 1e-6, (act, name, err)


@pytest.mark.parametrize("act", ACTS)
def test_finite_difference_gradients(act):
    check_fd_gradients(O, act)


# ------------------------------------------------------ structured weight cases

def _gate_closed_form(act, z):
    """The gate function written out independently of the oracle (exact GELU
    for the tanh-approximated one: they agree within 4.8e-4)."""
    name = O.GATE_FN.get(act, act)
    if name == "silu":
        return z / (1 + np.exp(-z))
    if name == "sigmoid":
        return 1 / (1 + np.exp(-z))
    if name == "relu":
        return np.where(z > 0, z, 0.0)
    if name == "relu_sq":
        return np.where(z > 0, z * z, 0.0)
    return z * sp.ndtr(z)


def _tol(act, scale):
    gelu = O.GATE_FN.get(act, act) == "gelu_tanh_approx"
    return 4.8e-4 * scale if gelu else 1e-13


@pytest.mark.parametrize("act", ACTS)
def test_identity_weights(act):
    rng = np.random.default_rng(2)
    M, H = 6, 8
    x = rng.standard_normal((M, H))
    E = np.eye(H)
    gm, dm = 1.125, 2.0
    gated = O.is_gated(act)
    fw = O.mlp_forward(x, E, E if gated else None, E, act, gm, dm)
    expect = gm * dm * _gate_closed_form(act, x) * (x if gated else 1.0)
    tol = _tol(act, gm * dm * (np.abs(x).max() if gated else 1.0))
    np.testing.assert_allclose(fw["out"], expect, atol=tol, rtol=0)


def _perm_matrix(p):
    P = np.zeros((len(p), len(p)))
    P[np.arange(len(p)), p] = 1.0  # P[i, p[i]] = 1
    return P


@pytest.mark.parametrize("act", ACTS)
def test_permutation_weights_forward(act):
    # Wg = P_pi, Wu = P_sigma, Wd = P_tau (P[i, p[i]] = 1), nn.Linear layout:
    # g[m,i] = x[m, pi(i)], u[m,i] = x[m, sigma(i)], out[m,j] = dm*h[m, tau(j)].
    # The cycles are not involutions, so a transposed operand is detected.
    H = 7
    pi = np.array([1, 2, 3, 4, 5, 6, 0])
    sg = np.array([3, 0, 6, 1, 5, 2, 4])
    tau = np.array([2, 5, 1, 6, 0, 3, 4])
    rng = np.random.default_rng(3)
    x = rng.standard_normal((5, H))
    gm, dm = 0.5, 3.0
    gated = O.is_gated(act)
    fw = O.mlp_forward(x, _perm_matrix(pi), _perm_matrix(sg) if gated else None,
                       _perm_matrix(tau), act, gm, dm)
    for m in range(5):
        for j in range(H):
            i = tau[j]
            z = x[m, pi[i]]
            hv = gm * float(_gate_closed_form(act, np.array(z)))
            if gated:
                hv *= x[m, sg[i]]
            tol = _tol(act, gm * dm * (abs(x[m, sg[i]]) if gated else 1.0))
            assert abs(fw["out"][m, j] - dm * hv) <= tol


@pytest.mark.parametrize("act", ACTS)
def test_zero_down_weight(act):
    # zero-initialised c_proj (modded-nanogpt gpt.py): out = 0, dx = 0,
    # dWg = dWu = 0, but dWd = dm * dout^T h != 0.
    rng = np.random.default_rng(4)
    x, Wg, Wu, Wd, dout = _rand_problem(rng, 9, 8, 12, act)
    Wd = np.zeros_like(Wd)
    fw = O.mlp_forward(x, Wg, Wu, Wd, act, 1.5, 0.5)
    bw = O.mlp_backward(dout, x, Wg, Wu, Wd, act, 1.5, 0.5)
    assert np.all(fw["out"] == 0) and np.all(bw["dx"] == 0) and np.all(bw["dWg"] == 0)
    if bw["dWu"] is not None:
        assert np.all(bw["dWu"] == 0)
    assert np.max(np.abs(bw["dWd"])) > 1e-3


def test_zero_gate_weight_swiglu():
    # Wg = 0: g = 0, silu(0) = 0, silu'(0) = 1/2  =>  out = 0, dWd = 0, dWu = 0,
    # dx = 0 (dG Wg = 0, dU = 0) and dWg = 1/2 gm dm ((dout Wd) * u)^T x.
    rng = np.random.default_rng(5)
    x, Wg, Wu, Wd, dout = _rand_problem(rng, 10, 8, 6, "swiglu")
    Wg = np.zeros_like(Wg)
    gm, dm = 1.125, 2.0
    fw = O.mlp_forward(x, Wg, Wu, Wd, "swiglu", gm, dm)
    bw = O.mlp_backward(dout, x, Wg, Wu, Wd, "swiglu", gm, dm)
    assert np.all(fw["out"] == 0)
    assert np.all(bw["dWd"] == 0) and np.all(bw["dWu"] == 0) and np.all(bw["dx"] == 0)
    u = x @ Wu.T
    np.testing.assert_allclose(bw["dWg"], 0.5 * gm * dm * ((dout @ Wd) * u).T @ x,
                               rtol=1e-12, atol=1e-14)


def test_zero_gate_weight_glu():
    # Wg = 0: sigmoid(0) = 1/2, so out = (gm dm / 2) (x Wu^T) Wd^T, and dU = gm/2 dh.
    rng = np.random.default_rng(15)
    x, Wg, Wu, Wd, dout = _rand_problem(rng, 9, 8, 6, "glu")
    Wg = np.zeros_like(Wg)
    gm, dm = 1.125, 2.0
    fw = O.mlp_forward(x, Wg, Wu, Wd, "glu", gm, dm)
    np.testing.assert_allclose(fw["out"], 0.5 * gm * dm * (x @ Wu.T) @ Wd.T, rtol=1e-12,
                               atol=1e-14)
    bw = O.mlp_backward(dout, x, Wg, Wu, Wd, "glu", gm, dm)
    np.testing.assert_allclose(bw["dWu"], (0.5 * gm * dm * (dout @ Wd)).T @ x, rtol=1e-12,
                               atol=1e-14)


def test_zero_fc1_relu_sq():
    rng = np.random.default_rng(6)
    x, Wg, _, Wd, dout = _rand_problem(rng, 7, 8, 16, "relu_sq")
    W1 = np.zeros_like(Wg)
    fw = O.mlp_forward(x, W1, None, Wd, "relu_sq", 1.0, 1.0)
    bw = O.mlp_backward(dout, x, W1, None, Wd, "relu_sq", 1.0, 1.0)
    assert np.all(fw["out"] == 0)
    for k in ("dx", "dWg", "dWd"):
        assert np.all(bw[k] == 0), k


def check_multiplier_scaling(mod, act):
    rng = np.random.default_rng(7)
    x, Wg, Wu, Wd, dout = _rand_problem(rng, 11, 8, 12, act)
    gm, dm = 1.125, 2.0
    f1 = mod.mlp_forward(x, Wg, Wu, Wd, act, 1.0, 1.0)["out"]
    fs = mod.mlp_forward(x, Wg, Wu, Wd, act, gm, dm)["out"]
    np.testing.assert_allclose(fs, gm * dm * f1, rtol=1e-12, atol=1e-14)
    b1 = mod.mlp_backward(dout, x, Wg, Wu, Wd, act, 1.0, 1.0)
    bs = mod.mlp_backward(dout, x, Wg, Wu, Wd, act, gm, dm)
    for k in ("dx", "dWg", "dWu", "dWd"):
        if b1[k] is not None:
            np.testing.assert_allclose(bs[k], gm * dm * b1[k], rtol=1e-12, atol=1e-14)


@pytest.mark.parametrize("act", ACTS)
def test_multiplier_scaling(act):
    check_multiplier_scaling(O, act)


@pytest.mark.parametrize("act", ACTS)
def test_accumulate_identity_and_split_m(act):
    rng = np.random.default_rng(8)
    x, Wg, Wu, Wd, dout = _rand_problem(rng, 20, 8, 12, act)
    plain = O.mlp_backward(dout, x, Wg, Wu, Wd, act, 1.2, 0.9)
    prev = {"dWg": rng.standard_normal(Wg.shape) * 1e-3,
            "dWu": rng.standard_normal(Wg.shape) * 1e-3,
            "dWd": rng.standard_normal(Wd.shape) * 1e-3}
    acc = O.mlp_backward(dout, x, Wg, Wu, Wd, act, 1.2, 0.9, dW_prev=prev)
    for k in ("dWg", "dWu", "dWd"):
        if plain[k] is not None:
            np.testing.assert_allclose(acc[k] - prev[k], plain[k], rtol=1e-12, atol=1e-15)
    # split the tokens in two halves: weight gradients add, dx rows concatenate
    a = O.mlp_backward(dout[:7], x[:7], Wg, Wu, Wd, act, 1.2, 0.9)
    b = O.mlp_backward(dout[7:], x[7:], Wg, Wu, Wd, act, 1.2, 0.9)
    for k in ("dWg", "dWu", "dWd"):
        if plain[k] is not None:
            np.testing.assert_allclose(a[k] + b[k], plain[k], rtol=1e-12, atol=1e-14)
    np.testing.assert_allclose(np.concatenate([a["dx"], b["dx"]]), plain["dx"], rtol=1e-12)


@pytest.mark.parametrize("act", ACTS)
def test_sampled_functions_match_full(act):
    rng = np.random.default_rng(9)
    x, Wg, Wu, Wd, dout = _rand_problem(rng, 33, 16, 24, act)
    gm, dm = 1.125, 2.0
    fw = O.mlp_forward(x, Wg, Wu, Wd, act, gm, dm)
    prev = {"dWg": rng.standard_normal(Wg.shape), "dWu": rng.standard_normal(Wg.shape),
            "dWd": rng.standard_normal(Wd.shape)}
    bw = O.mlp_backward(dout, x, Wg, Wu, Wd, act, gm, dm, dW_prev=prev)
    rows = [0, 5, 32]
    r = O.sampled_token_rows(rows, dout, x, Wg, Wu, Wd, act, gm, dm)
    np.testing.assert_allclose(r["out"], fw["out"][rows], rtol=1e-12, atol=1e-14)
    np.testing.assert_allclose(r["dx"], bw["dx"][rows], rtol=1e-12, atol=1e-14)
    cols = [1, 7, 23]
    c = O.sampled_inter_units(cols, dout, x, Wg, Wu, Wd, act, gm, dm, dW_prev=prev)
    np.testing.assert_allclose(c["dWg"], bw["dWg"][cols], rtol=1e-12, atol=1e-14)
    np.testing.assert_allclose(c["dWd"], bw["dWd"][:, cols], rtol=1e-12, atol=1e-14)
    if O.is_gated(act):
        np.testing.assert_allclose(c["dWu"], bw["dWu"][cols], rtol=1e-12, atol=1e-14)


@pytest.mark.parametrize("act", ACTS)
def test_torch_autograd_cross_check(act):
    # Independent cross-check on the tiny workload's shape: fp64 autograd of
    # the same definition written with torch ops (a library routine, used
    # here only as a second opinion).
    import torch
    M, H, I = 64, 128, 352
    rng = np.random.default_rng(10)
    x, Wg, Wu, Wd, dout = _rand_problem(rng, M, H, I, act)
    gm, dm = 1.125, 2.0
    t = lambda a: torch.tensor(a, dtype=torch.float64, requires_grad=True)  # noqa: E731
    tx, tg, td = t(x), t(Wg), t(Wd)
    tu = t(Wu) if Wu is not None else None
    z = tx @ tg.T
    F = torch.nn.functional
    fn = {"swiglu": F.silu, "relu_sq": lambda v: torch.relu(v) ** 2,
          "gelu_tanh_approx": lambda v: F.gelu(v, approximate="tanh"), "relu": torch.relu,
          "reglu": torch.relu, "geglu": lambda v: F.gelu(v, approximate="tanh"),
          "glu": torch.sigmoid}[act]
    hh = gm * fn(z)
    if tu is not None:
        hh = hh * (tx @ tu.T)
    out = dm * hh @ td.T
    out.backward(torch.tensor(dout))
    fw = O.mlp_forward(x, Wg, Wu, Wd, act, gm, dm)
    bw = O.mlp_backward(dout, x, Wg, Wu, Wd, act, gm, dm)
    assert O.rel_err(fw["out"], out.detach().numpy()) < 1e-12
    assert O.rel_err(bw["dx"], tx.grad.numpy()) < 1e-12
    assert O.rel_err(bw["dWg"], tg.grad.numpy()) < 1e-12
    assert O.rel_err(bw["dWd"], td.grad.numpy()) < 1e-12
    if tu is not None:
        assert O.rel_err(bw["dWu"], tu.grad.numpy()) < 1e-12


def test_rel_err_metric():
    assert O.rel_err([1.0, -2.0], [1.0, -2.0]) == 0.0
    assert O.rel_err([1.1, -2.0], [1.0, -2.0]) == pytest.approx(0.05)
    assert O.rel_err([0.0], [0.0]) == 0.0


def test_flop_counts():
    assert O.flops(2048, 4096, 11008, "swiglu", "fwd") + O.flops(2048, 4096, 11008, "swiglu", "bwd") \
        == pytest.approx(1.662e12, rel=1e-3)
    assert O.flops(49152, 768, 3072, "relu_sq", "bwd_recompute") == pytest.approx(1.160e12, rel=1e-3)


# ----------------------------------------------------- planted mistakes are caught

class _Mut:
    """A copy of the oracle's four entry points with one of them replaced."""

    def __init__(self, **over):
        self.act_fn = over.get("act_fn", O.act_fn)
        self.act_grad = over.get("act_grad", O.act_grad)
        self.mlp_forward = over.get("mlp_forward", O.mlp_forward)
        self.mlp_backward = over.get("mlp_backward", O.mlp_backward)
        self.is_gated = O.is_gated


def _caught(fn):
    try:
        fn()
    except AssertionError:
        return True
    return False


def test_planted_silu_grad_error_is_caught(monkeypatch):
    bad = lambda a, z: (O._sigmoid(np.asarray(z, float)) if a == "swiglu" else O.act_grad(a, z))  # noqa: E731
    monkeypatch.setattr(O, "act_grad", bad)  # dropped the z(1-s) term
    mod = _Mut(act_grad=bad)
    assert _caught(lambda: check_act_grad_fd(mod))
    assert _caught(lambda: check_fd_gradients(O, "swiglu"))


def test_planted_gelu_error_is_caught():
    c = math.sqrt(2 / math.pi)

    def bad(a, z):
        if a == "gelu_tanh_approx":
            z = np.asarray(z, float)
            return 0.5 * z * (1 + np.tanh(c * z))  # dropped the cubic term
        return O.act_fn(a, z)
    assert _caught(lambda: check_gelu_vs_exact(_Mut(act_fn=bad)))


def test_planted_transpose_error_is_caught(monkeypatch):
    orig = O.mlp_backward

    def bad(dout, x, Wg, Wu, Wd, act="swiglu", gate_mult=1.0, down_mult=1.0, dW_prev=None):
        r = orig(dout, x, Wg, Wu, Wd, act, gate_mult, down_mult, dW_prev)
        r["dWd"] = r["dWd"].T if r["dWd"].shape[0] == r["dWd"].shape[1] else r["dWd"] * 1.01
        return r
    assert _caught(lambda: check_fd_gradients(_Mut(mlp_backward=bad), "relu_sq", M=3, H=5, I=5))


def test_planted_multiplier_error_is_caught():
    orig_f = O.mlp_forward

    def bad_f(x, Wg, Wu, Wd, act="swiglu", gate_mult=1.0, down_mult=1.0):
        # gate multiplier moved inside the activation
        fw = orig_f(x, Wg * gate_mult, Wu, Wd, act, 1.0, down_mult)
        return fw
    assert _caught(lambda: check_multiplier_scaling(_Mut(mlp_forward=bad_f), "swiglu"))


def test_planted_missing_down_mult_in_dwd_is_caught():
    orig = O.mlp_backward

    def bad(dout, x, Wg, Wu, Wd, act="swiglu", gate_mult=1.0, down_mult=1.0, dW_prev=None):
        r = orig(dout, x, Wg, Wu, Wd, act, gate_mult, down_mult, dW_prev)
        r["dWd"] = r["dWd"] / down_mult
        return r
    assert _caught(lambda: check_fd_gradients(_Mut(mlp_backward=bad), "swiglu"))
