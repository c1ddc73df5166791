"""Plain fp64 CPU oracle of the FP8 forward of the ReLU^2 MLP.

TEST INFRASTRUCTURE ONLY: the same rules as ``oracle.mlp_oracle`` (only
tests, ``__graft_entry__.smoke()`` and ``bench.py`` may use it; it shares no
code with the library).

What is computed, and where the pages define it
-----------------------------------------------
modded-nanogpt ``track_1_short/model/gpt.py`` trains its ReLU^2 MLP in FP8
(the constants block above ``ReLUSqrdMLP`` and the ``_mlp_*`` buffers):
e4m3 operands with dequant scales (a value is its code times the scale):
* the input: static scale ``FP8_MLP_X_SCALE = 2^-4`` (its comment: post-norm
  rows stay below 448 * 2^-4);
* each weight matrix: ``amax / 448`` (``_quantize_mlp_weights_and_scales``,
  the exact branch);
* the GEMM dequant ``up_scales * x_scale`` (``_mlp_up_dequant``);
* the ReLU^2 output: a delayed scale, the last step's amax times
  ``FP8_POST_HEADROOM = 1.03`` over 448, with the kernels recording the new
  amax by atomic max (``_mlp_post_scales``, ``_mlp_post_amax``,
  ``_refresh_delayed_scale``);
* the down projection dequantised by the post scale times the down weight's
  scale.
* the backward: the incoming gradient in e5m2 with the static scale
  ``FP8_GRAD_SCALE = 2^-6``, the preact gradient in e5m2 with a delayed
  scale (last step's amax times ``FP8_DPRE_HEADROOM = 1.25`` over 57344,
  ``_mlp_dpre_scales``, ``_mlp_dpre_amax``), the down projection's backward
  dequantised by ``down_scales * grad_scale`` (``_mlp_dq_bwd``).
Readings where the page is silent (the kernels are not on it):
* quantisation is q = e4m3(v * inv), inv = fp32(1 / scale) computed in fp32,
  v * inv in fp32, then rounded to nearest even on the e4m3 grid with
  saturation at +-448 (e4m3fn has no infinity); e5m2 likewise, saturating
  at +-57344;
* the backward treats the postact's quantisation as the identity (its
  gradient passes straight through) and takes ReLU^2's derivative from the
  preact, recomputed here in full precision unless the saved preact is
  passed in (the GPU path saves it in bf16; its parity tests pass the same
  bf16 preact to both sides);
* the multipliers: ``gate_mult`` scales the ReLU^2 output before it is
  quantised, ``down_mult`` the dequantised output (both 1 on the page).
"""
from __future__ import annotations

import numpy as np

E4M3_MAX = 448.0
E5M2_MAX = 57344.0


def e4m3(v):
    """Round to the e4m3fn grid (1 sign, 4 exponent bits with bias 7, 3
    mantissa bits; subnormals below 2^-6; no infinity), nearest even,
    saturating at +-448."""
    v = np.asarray(v, dtype=np.float64)
    a = np.abs(v)
    _, ex = np.frexp(np.where(a > 0, a, 1.0))   # a = m 2^ex, m in [0.5, 1)
    e = np.maximum(ex - 1, -6)                   # binade, clamped to the subnormal one
    ulp = np.ldexp(1.0, e - 3)                   # 3 mantissa bits
    r = np.round(a / ulp) * ulp                  # np.round: half to even
    r = np.minimum(r, E4M3_MAX)
    return np.where(a > 0, np.sign(v) * r, 0.0 * v)


def e5m2(v):
    """Round to the e5m2 grid (5 exponent bits with bias 15, 2 mantissa bits;
    subnormals below 2^-14), nearest even, saturating at +-57344."""
    v = np.asarray(v, dtype=np.float64)
    a = np.abs(v)
    _, ex = np.frexp(np.where(a > 0, a, 1.0))
    e = np.maximum(ex - 1, -14)
    ulp = np.ldexp(1.0, e - 2)
    r = np.minimum(np.round(a / ulp) * ulp, E5M2_MAX)
    return np.where(a > 0, np.sign(v) * r, 0.0 * v)


def quantize_e5m2(v, scale):
    """e5m2 codes of v with dequant scale `scale` (fp32 product with fp32(1/scale))."""
    inv = np.float32(1.0) / np.float32(scale)
    return e5m2((np.asarray(v, dtype=np.float32) * inv).astype(np.float64))


def quantize(v, scale):
    """Codes (as float64 values) of v with dequant scale `scale`: the fp32
    product v * fp32(1/scale), rounded to e4m3."""
    inv = np.float32(1.0) / np.float32(scale)
    return e4m3((np.asarray(v, dtype=np.float32) * inv).astype(np.float64))


def weight_scale(W):
    """Exact weight scale amax / 448 (the page computes it in the weights' bf16)."""
    return max(float(np.max(np.abs(W))), 1e-12) / E4M3_MAX


def fp8_relu_sq_forward(x8, W1_8, W2_8, sx, s1, s2, s_post, gate_mult=1.0, down_mult=1.0):
    """The forward on e4m3 codes: pre = (x8 W1_8^T) sx s1,
    a = gate_mult relu(pre)^2, a8 = quantize(a, s_post),
    out = down_mult (a8 W2_8^T) s_post s2.  Returns out, a, a8 and amax(|a|)
    (the magnitude a delayed scale must cover; a >= 0 unless gate_mult < 0)."""
    pre = (x8 @ W1_8.T) * (sx * s1)
    a = gate_mult * np.maximum(pre, 0.0) ** 2
    a8 = quantize(a, s_post)
    out = down_mult * (a8 @ W2_8.T) * (s_post * s2)
    return {"out": out, "a": a, "a8": a8, "amax_a": float(np.max(np.abs(a))) if a.size else 0.0}


def fp8_relu_sq_backward(dout, x8, W1_8, W2_8, a8, sx, s1, s2, s_post, sg, s_dpre,
                         gate_mult=1.0, down_mult=1.0, pre=None):
    """The backward of ``fp8_relu_sq_forward`` on codes:
    dout8 = e5m2 codes of dout (scale sg); da = down_mult (dout8 W2_8) sg s2;
    dpre = gate_mult da 2 relu(pre) with pre = (x8 W1_8^T) sx s1 (or the
    saved preact ``pre`` when given);
    dP8 = e5m2 codes of dpre (scale s_dpre);
    dx = (dP8 W1_8) s_dpre s1;  dW1 = (dP8^T x8) s_dpre sx;
    dW2 = down_mult (dout8^T a8) sg s_post.
    Returns those and amax(|dpre|)."""
    dout8 = quantize_e5m2(dout, sg)
    if pre is None:
        pre = (x8 @ W1_8.T) * (sx * s1)
    da = down_mult * (dout8 @ W2_8) * (sg * s2)
    dpre = gate_mult * da * 2.0 * np.maximum(pre, 0.0)
    dP8 = quantize_e5m2(dpre, s_dpre)
    return {"dx": (dP8 @ W1_8) * (s_dpre * s1), "dW1": (dP8.T @ x8) * (s_dpre * sx),
            "dW2": down_mult * (dout8.T @ a8) * (sg * s_post), "dout8": dout8, "dP8": dP8,
            "dpre": dpre, "amax_dpre": float(np.max(np.abs(dpre))) if dpre.size else 0.0}


def fp8_relu_sq_sampled(dout, x8, W1_8, W2_8, sx, s1, s2, s_post, sg, s_dpre, rows, units,
                        gate_mult=1.0, down_mult=1.0, round_pre=None):
    """``fp8_relu_sq_forward`` and ``fp8_relu_sq_backward`` restricted to the
    token rows ``rows`` (out and dx) and the intermediate units ``units``
    (rows of dW1 and columns of dW2, each still reduced over all tokens):
    the same definition, evaluated on the subsets it needs.  The backward's
    saved preact is ``round_pre(pre)`` (the identity when None; the GPU path
    saves it rounded to bf16)."""
    rp = round_pre if round_pre is not None else (lambda v: v)
    dout8 = quantize_e5m2(dout, sg)

    def pre_of(xs, ws):
        return (xs @ ws.T) * (sx * s1)

    def a8_of(pre):
        return quantize(gate_mult * np.maximum(pre, 0.0) ** 2, s_post)

    def dP8_of(dout8_rows, W2_cols, pre):
        da = down_mult * (dout8_rows @ W2_cols) * (sg * s2)
        return quantize_e5m2(gate_mult * da * 2.0 * np.maximum(rp(pre), 0.0), s_dpre)

    # token rows: every unit of these tokens
    pre_r = pre_of(x8[rows], W1_8)
    out = down_mult * (a8_of(pre_r) @ W2_8.T) * (s_post * s2)
    dx = (dP8_of(dout8[rows], W2_8, pre_r) @ W1_8) * (s_dpre * s1)
    # intermediate units: every token of these units
    pre_u = pre_of(x8, W1_8[units])
    dW1 = (dP8_of(dout8, W2_8[:, units], pre_u).T @ x8) * (s_dpre * sx)
    dW2 = down_mult * (dout8.T @ a8_of(pre_u)) * (sg * s_post)
    return {"out": out, "dx": dx, "dW1": dW1, "dW2": dW2}
