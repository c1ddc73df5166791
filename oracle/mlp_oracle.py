"""Plain, slow fp64 CPU oracle of the fused transformer MLP block.

TEST INFRASTRUCTURE ONLY.  Only ``tests/``, ``__graft_entry__.smoke()`` and
``bench.py`` (its ``cpu_baseline`` leg and its ``--impl reference`` arm) may
import this module.  The library (``activated_mlp_gemms_gb300``) never does,
and nothing here imports the library: the two share no code.

What is computed, and where the pages define it
-----------------------------------------------
* flash-swiglu-mlp 0.4.2 README (PyPI METADATA), opening paragraph: the
  computed object is ``down_proj(silu(gate_proj(x)) * up_proj(x))``, with
  ``gate_proj``/``up_proj`` weights ``[intermediate, hidden]`` and
  ``down_proj`` weight ``[hidden, intermediate]`` (section "Module usage",
  nn.Linear layout, no bias).
* Same README, section "Falcon H1 style models": the scaled form
  ``down_multiplier * down_proj(gate_multiplier * silu(gate_proj(x)) *
  up_proj(x))``; both multipliers default to 1.0.
* quack ``mlp.py`` (Tri Dao), ``MLP.forward`` fallback branch: fc1, then the
  activation, then fc2; ``MLPRecomputeFunc.backward``: ``dW2 = dout^T
  postact``, ``dx = dpreact W1``, ``dW1 = dpreact^T x``, and
  ``_compute_weight_grad``: with ``fuse_grad_accum`` the weight gradient is
  added in place into the existing fp32 ``.grad``.
* modded-nanogpt ``track_1_short/model/gpt.py``, the ``ReLUSqrdMLP``
  comment: ``relu(x @ W1.T)^2 @ W2.T`` (the non-gated relu_sq MLP).
* quack ``mlp.py``, the ``Activation`` literal: ``gelu_tanh_approx`` (the
  default activation of ``MLP``).  Its formula is not on the pages; the
  published tanh approximation of GELU (Hendrycks & Gimpel, 2016) is used:
  ``0.5 z (1 + tanh(sqrt(2/pi) (z + 0.044715 z^3)))``.
* The same literal names ``relu`` (non-gated) and the gated ``reglu``,
  ``geglu`` and ``glu`` without formulas.  Plain readings: relu(z) =
  max(z, 0); the gated variants apply relu, the tanh-approximated GELU above,
  and the logistic sigmoid (GLU, Dauphin et al. 2017) to the gate, times the
  up projection, exactly as swiglu applies silu (Shazeer 2020, "GLU variants
  improve Transformer").  ``swiglu_oai`` is left out: nothing on the pages
  defines it.

Readings where the pages are silent (each also listed in the design notes):
* ``gate_multiplier`` multiplies ``act(g)`` outside the activation, exactly
  as the Falcon-H1 formula is written.
* For the non-gated activations the same two multipliers apply with the
  ``* up_proj(x)`` factor dropped: ``h = gm * act(x W1^T)``.
* Inputs are the exact bf16 values widened to fp64; the oracle rounds
  nothing to bf16 on the way (the GPU path stores G, U and the postact in
  bf16; that difference lies inside the parity tolerance).

Every array is a numpy float64 array, row-major, with the shapes
x ``[M,H]``, Wg/Wu ``[I,H]``, Wd ``[H,I]``, dout ``[M,H]``.
For the non-gated activations ``Wu`` is ``None`` and ``Wg`` plays ``W1``.
"""
from __future__ import annotations

import numpy as np

ACTIVATIONS = ("swiglu", "relu_sq", "gelu_tanh_approx", "relu", "reglu", "geglu", "glu")
GATED = ("swiglu", "reglu", "geglu", "glu")
# the function a gated activation applies to the gate
GATE_FN = {"swiglu": "silu", "reglu": "relu", "geglu": "gelu_tanh_approx", "glu": "sigmoid"}

# Hendrycks & Gimpel (2016), tanh approximation of GELU.
_GELU_C = np.sqrt(2.0 / np.pi)
_GELU_A = 0.044715


def is_gated(act: str) -> bool:
    if act not in ACTIVATIONS:
        raise ValueError(f"unknown activation {act!r}")
    return act in GATED


def _sigmoid(z):
    return 1.0 / (1.0 + np.exp(-z))


def _base_fn(name, z):
    if name == "silu":  # z * sigmoid(z)
        return z * _sigmoid(z)
    if name == "sigmoid":
        return _sigmoid(z)
    if name == "relu":
        return np.maximum(z, 0.0)
    if name == "relu_sq":  # relu(z)^2
        r = np.maximum(z, 0.0)
        return r * r
    if name == "gelu_tanh_approx":
        t = np.tanh(_GELU_C * (z + _GELU_A * z ** 3))
        return 0.5 * z * (1.0 + t)
    raise ValueError(f"unknown activation {name!r}")


def _base_grad(name, z):
    if name == "silu":
        s = _sigmoid(z)
        return s * (1.0 + z * (1.0 - s))
    if name == "sigmoid":
        s = _sigmoid(z)
        return s * (1.0 - s)
    if name == "relu":
        return np.where(z > 0.0, 1.0, 0.0)
    if name == "relu_sq":
        return 2.0 * np.maximum(z, 0.0)
    if name == "gelu_tanh_approx":
        t = np.tanh(_GELU_C * (z + _GELU_A * z ** 3))
        dinner = _GELU_C * (1.0 + 3.0 * _GELU_A * z * z)
        return 0.5 * (1.0 + t) + 0.5 * z * (1.0 - t * t) * dinner
    raise ValueError(f"unknown activation {name!r}")


def _fn_name(act):
    if act not in ACTIVATIONS:
        raise ValueError(f"unknown activation {act!r}")
    return GATE_FN.get(act, act)


def act_fn(act: str, z):
    """The activation applied to the gate (gated) or to the preact (non-gated)."""
    return _base_fn(_fn_name(act), np.asarray(z, dtype=np.float64))


def act_grad(act: str, z):
    """d act / dz, differentiated by hand from ``act_fn`` (relu: 0 at z = 0)."""
    return _base_grad(_fn_name(act), np.asarray(z, dtype=np.float64))


def _check(x, Wg, Wu, Wd, act):
    gated = is_gated(act)
    M, H = x.shape
    I = Wg.shape[0]
    assert Wg.shape == (I, H), Wg.shape
    assert Wd.shape == (H, I), Wd.shape
    if gated:
        assert Wu is not None and Wu.shape == (I, H)
    else:
        assert Wu is None, "non-gated activations take a single fc1 weight"
    return gated


def mlp_forward(x, Wg, Wu, Wd, act="swiglu", gate_mult=1.0, down_mult=1.0):
    """Forward pass.  Returns a dict with ``out [M,H]`` and the intermediates
    ``g`` (= gate preact, or the non-gated preact), ``u`` (None if
    non-gated) and ``h`` (the postact ``gm*act(g)*u``, before ``down_mult``).
    """
    gated = _check(x, Wg, Wu, Wd, act)
    g = x @ Wg.T  # gate_proj(x)   [M,I]
    u = x @ Wu.T if gated else None  # up_proj(x)     [M,I]
    h = gate_mult * act_fn(act, g)
    if gated:
        h = h * u
    out = down_mult * (h @ Wd.T)  # down_proj(h)   [M,H]
    return {"out": out, "g": g, "u": u, "h": h}


def mlp_backward(dout, x, Wg, Wu, Wd, act="swiglu", gate_mult=1.0,
                 down_mult=1.0, dW_prev=None):
    """Backward pass of ``mlp_forward`` for the upstream gradient ``dout``.

    Returns ``dx``, ``dWg``, ``dWu`` (None if non-gated) and ``dWd``.
    ``dW_prev``, when given, is a dict ``{"dWg":…, "dWu":…, "dWd":…}`` of
    pre-existing gradients; each returned weight gradient is then
    ``dW_prev + dW`` (the fused fp32 accumulation of quack's
    ``_compute_weight_grad``).
    """
    gated = _check(x, Wg, Wu, Wd, act)
    fw = mlp_forward(x, Wg, Wu, Wd, act, gate_mult, down_mult)
    g, u, h = fw["g"], fw["u"], fw["h"]
    # out = dm * h Wd^T  =>  dL/dh = dm * dout Wd ,  dL/dWd = dm * dout^T h
    dh = down_mult * (dout @ Wd)
    dWd = down_mult * (dout.T @ h)
    if gated:
        # h = gm * act(g) * u
        dG = gate_mult * dh * u * act_grad(act, g)
        dU = gate_mult * dh * act_fn(act, g)
        dx = dG @ Wg + dU @ Wu
        dWg = dG.T @ x
        dWu = dU.T @ x
    else:
        # h = gm * act(g)
        dG = gate_mult * dh * act_grad(act, g)
        dx = dG @ Wg
        dWg = dG.T @ x
        dWu = None
    res = {"dx": dx, "dWg": dWg, "dWu": dWu, "dWd": dWd}
    if dW_prev is not None:
        for k in ("dWg", "dWu", "dWd"):
            if res[k] is not None:
                res[k] = dW_prev[k] + res[k]
    return res


# ---------------------------------------------------------------------------
# Sampled evaluation at full sizes.  Each function is the same definition as
# above, restricted to a subset of output rows or columns; nothing is
# blocked, fused or reordered beyond selecting the rows the subset needs.
# ---------------------------------------------------------------------------

def sampled_token_rows(rows, dout, x, Wg, Wu, Wd, act="swiglu", gate_mult=1.0,
                       down_mult=1.0):
    """``out[rows]`` and ``dx[rows]`` for a list of token indices ``rows``.

    A token's output and input gradient depend only on that token's row of
    ``x`` and ``dout`` (the MLP is applied per token)."""
    rows = np.asarray(rows)
    fw = mlp_forward(x[rows], Wg, Wu, Wd, act, gate_mult, down_mult)
    bw = mlp_backward(dout[rows], x[rows], Wg, Wu, Wd, act, gate_mult, down_mult)
    return {"out": fw["out"], "dx": bw["dx"]}


def sampled_inter_units(cols, dout, x, Wg, Wu, Wd, act="swiglu", gate_mult=1.0,
                        down_mult=1.0, dW_prev=None):
    """For a list of intermediate units ``cols`` (indices into I):
    ``dWg[cols]``, ``dWu[cols]`` (rows of the ``[I,H]`` gradients) and
    ``dWd[:, cols]`` (columns of the ``[H,I]`` gradient), each summed over
    all M tokens.  Unit ``i`` only involves row ``i`` of Wg/Wu and column
    ``i`` of Wd, so this is ``mlp_backward`` on the sub-network of those
    units, whose ``dWd`` columns equal the full network's because ``dWd =
    dm * dout^T h`` is column-separable in ``h``.

    ``dW_prev`` (optional) holds the FULL pre-existing gradients; the
    matching slices are added."""
    cols = np.asarray(cols)
    gated = is_gated(act)
    sub = mlp_backward(dout, x, Wg[cols], Wu[cols] if gated else None,
                       Wd[:, cols], act, gate_mult, down_mult)
    res = {"dWg": sub["dWg"], "dWu": sub["dWu"], "dWd": sub["dWd"]}
    if dW_prev is not None:
        res["dWg"] = dW_prev["dWg"][cols] + res["dWg"]
        if gated:
            res["dWu"] = dW_prev["dWu"][cols] + res["dWu"]
        res["dWd"] = dW_prev["dWd"][:, cols] + res["dWd"]
    return res


# ---------------------------------------------------------------------------
# The MLP block with its neighbours (modded-nanogpt track_1_short/model/gpt.py,
# the "process mlp" step of the layer loop): the input is RMS-normalised,
# ``mlp_in = norm(x)``, and the output joins the residual stream through
# ``x = scale_add(resid_lambdas_mlp[i], x, post_lambdas_mlp[i], mlp_out)``.
# Readings (the pages show the calls, not the bodies): ``norm`` is an RMS
# norm over the last axis with no learned weight, x / sqrt(mean(x^2) + eps);
# ``scale_add(a, x, b, y)`` is a*x + b*y, as the page's other branch
# ``scale(resid_lambdas_mlp[i], x) + mlp_out`` (post-lambda folded) shows.
# ---------------------------------------------------------------------------

def rms_norm(x, eps):
    """``norm(x)`` of the block: ``x / r`` with ``r = sqrt(mean(x^2) + eps)``
    over the last axis (one value per token).  Returns ``(n, r)``."""
    r = np.sqrt(np.mean(x * x, axis=-1, keepdims=True) + eps)
    return x / r, r


def block_forward(x, Wg, Wu, Wd, act="relu_sq", gate_mult=1.0, down_mult=1.0,
                  resid_lambda=1.0, post_lambda=1.0, eps=2.0 ** -7):
    """``y = resid_lambda * x + post_lambda * MLP(norm(x))``.

    Returns ``y``, the normalised input ``n``, ``rstd = 1 / r`` (per token,
    shape ``[M]``) and the MLP output ``mlp_out``."""
    n, r = rms_norm(x, eps)
    fw = mlp_forward(n, Wg, Wu, Wd, act, gate_mult, down_mult)
    y = resid_lambda * x + post_lambda * fw["out"]
    return {"y": y, "n": n, "rstd": 1.0 / r[:, 0], "mlp_out": fw["out"]}


def block_backward(dy, x, Wg, Wu, Wd, act="relu_sq", gate_mult=1.0, down_mult=1.0,
                   resid_lambda=1.0, post_lambda=1.0, eps=2.0 ** -7, dW_prev=None):
    """Backward pass of ``block_forward`` for the upstream gradient ``dy``.

    The MLP sees ``n = norm(x)`` and the gradient ``post_lambda * dy``; its
    input gradient ``dn`` goes back through the RMS norm by the derivative
    of ``n = x / r``, ``dx = (dn - n * mean(dn * n)) / r`` (per token), and
    the residual branch adds ``resid_lambda * dy``."""
    n, r = rms_norm(x, eps)
    bw = mlp_backward(post_lambda * dy, n, Wg, Wu, Wd, act, gate_mult, down_mult,
                      dW_prev=dW_prev)
    dn = bw["dx"]
    dx = resid_lambda * dy + (dn - n * np.mean(dn * n, axis=-1, keepdims=True)) / r
    return {"dx": dx, "dWg": bw["dWg"], "dWu": bw["dWu"], "dWd": bw["dWd"]}


def rel_err(got, ref):
    """The parity metric: max|got - ref| / max|ref| (0 if both are zero)."""
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    num = float(np.max(np.abs(got - ref))) if ref.size else 0.0
    den = float(np.max(np.abs(ref))) if ref.size else 0.0
    if den == 0.0:
        return num
    return num / den


def flops(M, H, I, act, mode):
    """Multiply-add count x2 of the GEMMs a mode executes.

    mode: 'fwd' | 'infer' | 'bwd' | 'bwd_recompute'.  (gated: fwd 6MHI, bwd
    12MHI, +4MHI to recompute; non-gated: fwd 4MHI, bwd 8MHI, +2MHI.)"""
    mhi = float(M) * H * I
    g = is_gated(act)
    if mode in ("fwd", "infer"):
        return (6 if g else 4) * mhi
    if mode == "bwd":
        return (12 if g else 8) * mhi
    if mode == "bwd_recompute":
        return (16 if g else 10) * mhi
    raise ValueError(mode)


def block_sampled(rows, cols, dy, x, Wg, Wu, Wd, act="relu_sq", gate_mult=1.0, down_mult=1.0,
                  resid_lambda=1.0, post_lambda=1.0, eps=2.0 ** -7, dW_prev=None):
    """``block_forward`` / ``block_backward`` restricted to the token rows
    ``rows`` (y, dx) and the intermediate units ``cols`` (rows of dWg/dWu,
    columns of dWd, each summed over all tokens).  The norm is per token, so
    the rows' outputs need only their own rows of ``x`` and ``dy``; the units'
    gradients need every token's normalised input."""
    rows = np.asarray(rows)
    n, r = rms_norm(x, eps)
    tr = sampled_token_rows(rows, post_lambda * dy, n, Wg, Wu, Wd, act, gate_mult, down_mult)
    nr, dn = n[rows], tr["dx"]
    y = resid_lambda * x[rows] + post_lambda * tr["out"]
    dx = resid_lambda * dy[rows] + (dn - nr * np.mean(dn * nr, axis=-1, keepdims=True)) / r[rows]
    cu = sampled_inter_units(cols, post_lambda * dy, n, Wg, Wu, Wd, act, gate_mult, down_mult,
                             dW_prev=dW_prev)
    return {"y": y, "dx": dx, **cu}

