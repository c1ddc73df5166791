"""mlp_func / mlp_block_func: the fused MLP (and the MLP block with its RMS
norm and scaled residual) as differentiable PyTorch functions, on the
library's entry points (quack mlp.py's mlp_func and MLPRecomputeFunc: the
forward saves the preacts, or only x with recompute=True; the backward skips
the gradients autograd does not ask for; fuse_grad_accum adds the weight
gradients in place into fp32 buffers instead of returning them).

Argument marshalling only: the forward is one mlp_fwd call and the backward
one mlp_bwd or mlp_bwd_recompute call; nothing runs outside the library's
kernels.  Tensors are CUDA and bf16: x [..., H], Wg and Wu [I, H] (Wu None
for the non-gated activations), Wd [H, I].

With fuse_grad_accum=True every weight that needs a gradient carries an
fp32 tensor of its own shape as `main_grad`; the backward adds its gradient
there (dW += grad, as quack's _compute_weight_grad adds into the existing
gradient) and returns no gradient for it.

The saved-preact backward writes dG, dU over the saved G, U (the library's
in-place stage), so a graph built with recompute=False can be
differentiated once; recompute=True keeps only x and may be run again.

mlp_block_func is modded-nanogpt gpt.py's "process mlp" step, y =
resid_lambda x + post_lambda MLP(norm(x)), as one mlp_block_fwd and one
mlp_block_bwd call (saved preacts and the per-token 1/rms).
"""
from __future__ import annotations

import torch

from . import (GATED_ACTS, block, mlp_block_bwd, mlp_block_fwd, mlp_bwd, mlp_bwd_recompute,
               mlp_fwd, problem)


def _check_operand(t, name):
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if t.dtype != torch.bfloat16:
        raise ValueError(f"{name} must be bfloat16, got {t.dtype}")


def _grad_buffers(ctx, x2, weights):
    """dx and the three weight-gradient buffers autograd asks for (None where
    it does not): fresh bf16 tensors, or each weight's fp32 main_grad when
    fusing the accumulation."""
    need = ctx.needs_input_grad
    dx = torch.empty_like(x2) if need[0] else None
    bufs = [None, None, None]
    for i, w in enumerate(weights):
        if w is None or not need[i + 1]:
            continue
        if ctx.fuse:
            g = getattr(w, "main_grad", None)
            if (g is None or g.dtype != torch.float32 or g.shape != w.shape
                    or not g.is_contiguous() or g.device != w.device):
                raise ValueError("fuse_grad_accum: each weight needs a contiguous fp32 "
                                 "`main_grad` of its own shape")
            bufs[i] = g
        else:
            bufs[i] = torch.empty_like(w)
    return dx, bufs


def _check_weights(act, Wg, Wu, Wd):
    gated = act in GATED_ACTS
    for t, name in ((Wg, "Wg"), (Wd, "Wd")):
        _check_operand(t, name)
    if gated:
        _check_operand(Wu, "Wu")
    elif Wu is not None:
        raise ValueError(f"{act} is not gated: Wu must be None")
    return gated


class _MlpFunction(torch.autograd.Function):
    @staticmethod
    def forward(ctx, x, Wg, Wu, Wd, act, gate_mult, down_mult, recompute, fuse_grad_accum):
        _check_operand(x, "x")
        gated = _check_weights(act, Wg, Wu, Wd)
        shape = x.shape
        H = shape[-1]
        I = Wd.shape[1]
        x2 = x.reshape(-1, H).contiguous()
        M = x2.shape[0]
        ctx.shape, ctx.recompute, ctx.fuse, ctx.gated = shape, recompute, fuse_grad_accum, gated
        ctx.spent = False
        out = torch.empty((M, H), dtype=torch.bfloat16, device=x.device)
        if M == 0:
            ctx.prob = None
            ctx.save_for_backward(x2, Wg, Wu, Wd, None, None)
            return out.view(shape)
        prob = problem(M, H, I, act, gate_mult, down_mult)
        ctx.prob = prob
        if recompute:
            G = U = None
            mlp_fwd(prob, x2, Wg, Wu, Wd, out)
        else:
            G = torch.empty((M, I), dtype=torch.bfloat16, device=x.device)
            U = torch.empty_like(G) if gated else None
            mlp_fwd(prob, x2, Wg, Wu, Wd, out, G, U)
        ctx.save_for_backward(x2, Wg, Wu, Wd, G, U)
        return out.view(shape)

    @staticmethod
    def backward(ctx, dout):
        x2, Wg, Wu, Wd, G, U = ctx.saved_tensors
        if ctx.spent and not ctx.recompute:
            raise RuntimeError("mlp_func: the saved preacts were overwritten by the first "
                               "backward; use recompute=True to differentiate twice")
        ctx.spent = True
        M, H = x2.shape
        dx, bufs = _grad_buffers(ctx, x2, (Wg, Wu, Wd))
        if M == 0:
            if dx is not None:
                dx = dx.view(ctx.shape)
            grads = [None if ctx.fuse or b is None else b.zero_() for b in bufs]
            return (dx, *grads, None, None, None, None, None)
        dout2 = dout.reshape(-1, H)
        if dout2.dtype != torch.bfloat16:
            dout2 = dout2.to(torch.bfloat16)
        dout2 = dout2.contiguous()
        if any(b is not None for b in bufs) or dx is not None:
            if ctx.recompute:
                mlp_bwd_recompute(ctx.prob, dout2, x2, Wg, Wu, Wd, dx, *bufs,
                                  fuse_grad_accum=ctx.fuse)
            else:
                mlp_bwd(ctx.prob, dout2, x2, Wg, Wu, Wd, G, U, dx, *bufs,
                        fuse_grad_accum=ctx.fuse)
        grads = [None if ctx.fuse else b for b in bufs]
        return (dx.view(ctx.shape) if dx is not None else None, *grads,
                None, None, None, None, None)


def mlp_func(x, Wg, Wu, Wd, activation="swiglu", gate_mult=1.0, down_mult=1.0,
             recompute=False, fuse_grad_accum=False):
    """out = down_mult * Wd (gate_mult * act(x Wg^T) * (x Wu^T)) over the last
    dimension of x, differentiable with respect to x and the weights."""
    return _MlpFunction.apply(x, Wg, Wu, Wd, activation, gate_mult, down_mult, bool(recompute),
                              bool(fuse_grad_accum))


class _MlpBlockFunction(torch.autograd.Function):
    @staticmethod
    def forward(ctx, x, Wg, Wu, Wd, act, gate_mult, down_mult, resid_lambda, post_lambda, eps,
                fuse_grad_accum):
        _check_operand(x, "x")
        gated = _check_weights(act, Wg, Wu, Wd)
        shape = x.shape
        H = shape[-1]
        I = Wd.shape[1]
        x2 = x.reshape(-1, H).contiguous()
        M = x2.shape[0]
        ctx.shape, ctx.fuse = shape, fuse_grad_accum
        ctx.spent = False
        y = torch.empty((M, H), dtype=torch.bfloat16, device=x.device)
        if M == 0:
            ctx.prob = None
            ctx.save_for_backward(x2, Wg, Wu, Wd, None, None, None)
            return y.view(shape)
        prob = problem(M, H, I, act, gate_mult, down_mult)
        blk = block(resid_lambda, post_lambda, eps)
        ctx.prob, ctx.blk = prob, blk
        G = torch.empty((M, I), dtype=torch.bfloat16, device=x.device)
        U = torch.empty_like(G) if gated else None
        rstd, _ = mlp_block_fwd(prob, blk, x2, Wg, Wu, Wd, y, G, U)
        ctx.save_for_backward(x2, Wg, Wu, Wd, G, U, rstd)
        return y.view(shape)

    @staticmethod
    def backward(ctx, dy):
        x2, Wg, Wu, Wd, G, U, rstd = ctx.saved_tensors
        if ctx.spent:
            raise RuntimeError("mlp_block_func: the saved preacts were overwritten by the "
                               "first backward")
        ctx.spent = True
        M, H = x2.shape
        dx, bufs = _grad_buffers(ctx, x2, (Wg, Wu, Wd))
        rest = (None,) * 7
        if M == 0:
            grads = [None if ctx.fuse or b is None else b.zero_() for b in bufs]
            return (dx.view(ctx.shape) if dx is not None else None, *grads, *rest)
        dy2 = dy.reshape(-1, H)
        if dy2.dtype != torch.bfloat16:
            dy2 = dy2.to(torch.bfloat16)
        dy2 = dy2.contiguous()
        if any(b is not None for b in bufs) or dx is not None:
            mlp_block_bwd(ctx.prob, ctx.blk, dy2, x2, Wg, Wu, Wd, G, U, rstd, dx, *bufs,
                          fuse_grad_accum=ctx.fuse)
        grads = [None if ctx.fuse else b for b in bufs]
        return (dx.view(ctx.shape) if dx is not None else None, *grads, *rest)


def mlp_block_func(x, Wg, Wu, Wd, activation="swiglu", gate_mult=1.0, down_mult=1.0,
                   resid_lambda=1.0, post_lambda=1.0, eps=2.0 ** -7, fuse_grad_accum=False):
    """y = resid_lambda x + post_lambda MLP(x / rms(x)) over the last
    dimension of x (rms with eps inside the root), differentiable with
    respect to x and the weights."""
    return _MlpBlockFunction.apply(x, Wg, Wu, Wd, activation, gate_mult, down_mult,
                                   float(resid_lambda), float(post_lambda), float(eps),
                                   bool(fuse_grad_accum))
