"""The error floor that the kernels' bf16 storage of intermediates sets for
the fp32-accumulated weight gradients.

The CUDA path stores the preacts G, U (P), the postact a and the preact
gradients dG, dU (dP) in bf16 between its GEMMs; the weight gradients are
then sums over the tokens of products of those rounded values.  This module
repeats the path's arithmetic in fp64 with exactly those roundings (round to
nearest even, from fp32, at the points the kernels round) and nothing else:
every GEMM is exact fp64, so what it returns differs from the oracle only by
the storage roundings.  max|emulated - oracle| / max|oracle| is then a floor
that no kernel storing those tensors in bf16 can get under, whatever its
accumulation precision.

This is test infrastructure, not the oracle: the oracle (``oracle/``) is the
plain definition, with no rounding; the tests use this module only to state
how far the bf16 storage alone moves the gradients at a given shape.

Rounding points (as the library's epilogues take them):
  gated, forward:        G = bf(g), U = bf(u) from the fp32 accumulators
  gated, backward:       dG = bf(s*dh*U*act'(G)), dU = bf(s*dh*act(G));
                         the postact for dWd: saved mode a = bf(s*act(G)*U)
                         (rebuilt from the stored preacts), recompute mode
                         a = bf(s*act(g)*u) (from the recompute GEMM's fp32
                         accumulators)
  non-gated, saved:      P = bf(p); dP = bf(s*dh*act'(P)); a = bf(s*act(P))
  non-gated, recompute:  a = bf(s*act(p)); d = bf(s*act'(p)); dP = bf(dh*d)
with s = gate_mult * down_mult, dh = dout Wd (fp32 accumulation, exact
here), and the block's row scale r (1/rms of the token's input) multiplying
g, u in the forward and dh in the backward when given.
"""
import numpy as np
import torch

from oracle import act_fn, act_grad, is_gated


def bf(v):
    """Round to bf16 (nearest even) through fp32, as the epilogues do."""
    t = torch.from_numpy(np.ascontiguousarray(v, dtype=np.float64)).to(torch.float32)
    return t.to(torch.bfloat16).to(torch.float64).numpy()


def emulated_dw(x, dout, Wg, Wu, Wd, act, gate_mult, down_mult, mode="saved", dW_prev=None,
                rstd=None, rounding=True):
    """dWg, dWu, dWd as the CUDA path forms them, in fp64 with only the bf16
    storage roundings above (``rounding=False``: none, which must give the
    oracle's values).  x, dout [M,H]; Wg/Wu [I,H]; Wd [H,I]; fp64 arrays.
    rstd: the block's per-token row scale [M] (the block's weight gradients
    then take the un-normalised x, as the library's do)."""
    rnd = bf if rounding else (lambda v: v)
    s = gate_mult * down_mult
    r = np.ones((x.shape[0], 1)) if rstd is None else np.asarray(rstd)[:, None]
    g = r * (x @ Wg.T)
    dh = r * (dout @ Wd)
    if is_gated(act):
        u = r * (x @ Wu.T)
        G, U = rnd(g), rnd(u)
        dG = rnd(s * dh * U * act_grad(act, G))
        dU = rnd(s * dh * act_fn(act, G))
        a = rnd(s * act_fn(act, G) * U) if mode == "saved" else rnd(s * act_fn(act, g) * u)
        res = {"dWg": dG.T @ x, "dWu": dU.T @ x, "dWd": dout.T @ a}
    else:
        if mode == "saved":
            P = rnd(g)
            dP = rnd(s * dh * act_grad(act, P))
            a = rnd(s * act_fn(act, P))
        else:
            a = rnd(s * act_fn(act, g))
            dP = rnd(dh * rnd(s * act_grad(act, g)))
        res = {"dWg": dP.T @ x, "dWu": None, "dWd": dout.T @ a}
    if dW_prev is not None:
        for k in res:
            if res[k] is not None:
                res[k] = res[k] + dW_prev[k]
    return res
