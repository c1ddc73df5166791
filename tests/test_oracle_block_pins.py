"""Pins of the oracle's MLP block with its neighbours (RMS-normalised input,
scaled residual add; modded-nanogpt gpt.py, "process mlp"), each against
something other than the oracle's own formulas: numerical derivatives, an
independent torch autograd implementation, closed forms and invariances,
and planted mistakes that these must catch."""
import math

import numpy as np
import pytest

import oracle.mlp_oracle as O

BLOCK_ACTS = ["relu_sq", "swiglu", "gelu_tanh_approx"]


def _problem(rng, M, H, I, act, xscale=1.0):
    x = rng.standard_normal((M, H)) * xscale
    Wg = rng.standard_normal((I, H)) / math.sqrt(H)
    Wu = rng.standard_normal((I, H)) / math.sqrt(H) if O.is_gated(act) else None
    Wd = rng.standard_normal((H, I)) / math.sqrt(I)
    dy = rng.standard_normal((M, H))
    return x, Wg, Wu, Wd, dy


KW = dict(gate_mult=1.125, down_mult=0.75, resid_lambda=1.1 ** 0.5, post_lambda=0.8, eps=2.0 ** -7)


@pytest.mark.parametrize("act", BLOCK_ACTS)
def test_block_backward_matches_finite_differences(act):
    # L = sum(dy * y); every gradient entry checked by central differences
    # of the forward alone (independent of the backward's chain rule,
    # including the RMS-norm derivative).
    rng = np.random.default_rng(31)
    M, H, I = 3, 6, 5
    x, Wg, Wu, Wd, dy = _problem(rng, M, H, I, act)
    bw = O.block_backward(dy, x, Wg, Wu, Wd, act, **KW)

    def loss(x_, Wg_, Wu_, Wd_):
        return float(np.sum(dy * O.block_forward(x_, Wg_, Wu_, Wd_, act, **KW)["y"]))

    h = 1e-6
    args = {"x": x, "Wg": Wg, "Wu": Wu, "Wd": Wd}
    names = ["x", "Wg", "Wd"] + (["Wu"] if Wu is not None else [])
    for name in names:
        a = args[name]
        num = np.zeros_like(a)
        for idx in np.ndindex(a.shape):
            old = a[idx]
            a[idx] = old + h
            lp = loss(args["x"], args["Wg"], args["Wu"], args["Wd"])
            a[idx] = old - h
            lm = loss(args["x"], args["Wg"], args["Wu"], args["Wd"])
            a[idx] = old
            num[idx] = (lp - lm) / (2 * h)
        got = bw["dx" if name == "x" else "d" + name]
        assert O.rel_err(got, num) < 1e-6, name


@pytest.mark.parametrize("act", BLOCK_ACTS)
def test_block_torch_autograd_cross_check(act):
    # The same block written with torch ops (F.rms_norm and autograd, fp64),
    # used only as a second opinion.
    import torch
    F = torch.nn.functional
    rng = np.random.default_rng(32)
    M, H, I = 16, 64, 96
    x, Wg, Wu, Wd, dy = _problem(rng, M, H, I, act)
    t = lambda a: torch.tensor(a, dtype=torch.float64, requires_grad=True)  # noqa: E731
    tx, tg, td = t(x), t(Wg), t(Wd)
    tu = t(Wu) if Wu is not None else None
    n = F.rms_norm(tx, (H,), eps=KW["eps"])
    fn = {"relu_sq": lambda v: torch.relu(v) ** 2, "swiglu": F.silu,
          "gelu_tanh_approx": lambda v: F.gelu(v, approximate="tanh")}[act]
    hh = KW["gate_mult"] * fn(n @ tg.T)
    if tu is not None:
        hh = hh * (n @ tu.T)
    y = KW["resid_lambda"] * tx + KW["post_lambda"] * (KW["down_mult"] * hh @ td.T)
    y.backward(torch.tensor(dy))
    fw = O.block_forward(x, Wg, Wu, Wd, act, **KW)
    bw = O.block_backward(dy, x, Wg, Wu, Wd, act, **KW)
    assert O.rel_err(fw["y"], y.detach().numpy()) < 1e-12
    assert O.rel_err(bw["dx"], tx.grad.numpy()) < 1e-12
    assert O.rel_err(bw["dWg"], tg.grad.numpy()) < 1e-12
    assert O.rel_err(bw["dWd"], td.grad.numpy()) < 1e-12
    if tu is not None:
        assert O.rel_err(bw["dWu"], tu.grad.numpy()) < 1e-12


def test_rms_norm_closed_forms():
    rng = np.random.default_rng(33)
    x = rng.standard_normal((7, 10)) * 3.0
    n, r = O.rms_norm(x, 0.0)
    assert np.allclose(np.mean(n * n, axis=-1), 1.0, atol=1e-14)  # unit RMS rows
    # a constant row v normalises to sign(v) / sqrt(1 + eps / v^2)
    v, eps = -0.5, 2.0 ** -7
    n1, r1 = O.rms_norm(np.full((1, 8), v), eps)
    assert np.allclose(n1, np.sign(v) / math.sqrt(1 + eps / v ** 2), atol=1e-15)
    assert abs(r1[0, 0] - math.sqrt(v * v + eps)) < 1e-15


@pytest.mark.parametrize("act", BLOCK_ACTS)
def test_block_scale_invariance_without_eps(act):
    # With eps = 0 the normalised input, hence the MLP branch, ignores a
    # positive per-token scale; with resid_lambda = 0 so does y, and dx
    # scales by 1/c (dy fixed), the weight gradients not at all.
    rng = np.random.default_rng(34)
    x, Wg, Wu, Wd, dy = _problem(rng, 5, 12, 9, act)
    kw = dict(KW, eps=0.0, resid_lambda=0.0)
    c = np.exp(rng.standard_normal((5, 1)))
    y1 = O.block_forward(x, Wg, Wu, Wd, act, **kw)["y"]
    y2 = O.block_forward(c * x, Wg, Wu, Wd, act, **kw)["y"]
    assert O.rel_err(y2, y1) < 1e-13
    b1 = O.block_backward(dy, x, Wg, Wu, Wd, act, **kw)
    b2 = O.block_backward(dy, c * x, Wg, Wu, Wd, act, **kw)
    assert O.rel_err(b2["dx"] * c, b1["dx"]) < 1e-12
    assert O.rel_err(b2["dWg"], b1["dWg"]) < 1e-12


@pytest.mark.parametrize("act", BLOCK_ACTS)
def test_block_without_mlp_branch_is_a_scale(act):
    # post_lambda = 0: y = resid_lambda x, dx = resid_lambda dy, no weight gradient
    rng = np.random.default_rng(35)
    x, Wg, Wu, Wd, dy = _problem(rng, 4, 8, 6, act)
    kw = dict(KW, post_lambda=0.0)
    assert np.array_equal(O.block_forward(x, Wg, Wu, Wd, act, **kw)["y"], kw["resid_lambda"] * x)
    bw = O.block_backward(dy, x, Wg, Wu, Wd, act, **kw)
    assert O.rel_err(bw["dx"], kw["resid_lambda"] * dy) < 1e-15
    assert not np.any(bw["dWg"]) and not np.any(bw["dWd"])


def test_block_with_zero_down_weight_passes_the_residual():
    # gpt.py zero-initialises c_proj: a fresh block is y = resid_lambda x, and
    # its input gradient is resid_lambda dy (the MLP branch has dh = 0)
    rng = np.random.default_rng(36)
    x, Wg, Wu, Wd, dy = _problem(rng, 4, 8, 6, "relu_sq")
    Wd = np.zeros_like(Wd)
    fw = O.block_forward(x, Wg, Wu, Wd, "relu_sq", **KW)
    assert np.array_equal(fw["y"], KW["resid_lambda"] * x)
    bw = O.block_backward(dy, x, Wg, Wu, Wd, "relu_sq", **KW)
    assert O.rel_err(bw["dx"], KW["resid_lambda"] * dy) < 1e-15
    assert not np.any(bw["dWg"]) and np.any(bw["dWd"])  # dWd = dy^T relu(n W1^T)^2 != 0


def test_planted_rms_norm_mistakes_are_caught(monkeypatch):
    # A mean dropped from the RMS-norm derivative (the plausible mistake)
    # fails the finite-difference pin.
    rng = np.random.default_rng(37)
    x, Wg, Wu, Wd, dy = _problem(rng, 2, 5, 4, "relu_sq")
    good = O.block_backward(dy, x, Wg, Wu, Wd, "relu_sq", **KW)["dx"]

    def wrong(dy_, x_, Wg_, Wu_, Wd_, act="relu_sq", gate_mult=1.0, down_mult=1.0,
              resid_lambda=1.0, post_lambda=1.0, eps=0.0, dW_prev=None):
        n, r = O.rms_norm(x_, eps)
        dn = O.mlp_backward(post_lambda * dy_, n, Wg_, Wu_, Wd_, act, gate_mult, down_mult)["dx"]
        return {"dx": resid_lambda * dy_ + dn / r}  # no projection term

    bad = wrong(dy, x, Wg, Wu, Wd, "relu_sq", **KW)["dx"]
    assert O.rel_err(bad, good) > 1e-3


@pytest.mark.parametrize("act", ["swiglu", "relu_sq"])
def test_block_sampled_equals_the_full_definition(act):
    """The sampled block oracle is the full block restricted to the chosen
    token rows and intermediate units."""
    rng = np.random.default_rng(58)
    M, H, I = 9, 6, 7
    x = rng.standard_normal((M, H))
    dy = rng.standard_normal((M, H))
    Wg = rng.standard_normal((I, H))
    Wu = rng.standard_normal((I, H)) if act == "swiglu" else None
    Wd = rng.standard_normal((H, I))
    kw = dict(gate_mult=1.125, down_mult=2.0, resid_lambda=1.1 ** 0.5, post_lambda=0.8, eps=0.01)
    fw = O.block_forward(x, Wg, Wu, Wd, act, **kw)
    bw = O.block_backward(dy, x, Wg, Wu, Wd, act, **kw)
    rows, cols = [0, 4, 8], [1, 6]
    sm = O.block_sampled(rows, cols, dy, x, Wg, Wu, Wd, act, **kw)
    np.testing.assert_allclose(sm["y"], fw["y"][rows], rtol=1e-13, atol=1e-13)
    np.testing.assert_allclose(sm["dx"], bw["dx"][rows], rtol=1e-13, atol=1e-13)
    np.testing.assert_allclose(sm["dWg"], bw["dWg"][cols], rtol=1e-13, atol=1e-13)
    np.testing.assert_allclose(sm["dWd"], bw["dWd"][:, cols], rtol=1e-13, atol=1e-13)
    if act == "swiglu":
        np.testing.assert_allclose(sm["dWu"], bw["dWu"][cols], rtol=1e-13, atol=1e-13)
