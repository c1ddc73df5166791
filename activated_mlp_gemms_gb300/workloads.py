"""Seeded synthetic inputs for the fused-MLP workloads.

This module holds no MLP arithmetic: it only draws random tensors (in fp32,
then rounded to bf16 with round-to-nearest-even) in the shapes and
distributions of the five workloads, so that the CUDA path and the fp64
oracle can be fed identical bytes.

Distributions: x and dout ~ N(0, 1); weights follow nn.Linear's default
Kaiming-uniform initialisation, U(-1/sqrt(fan_in), 1/sqrt(fan_in)), with
fan_in = H for the gate/up (or fc1) weights and I for the down weight, as
the flash-swiglu-mlp README (section "Module usage") states for its three
nn.Linear(bias=False) projections.  The pre-existing fp32 gradients of the
ReLU^2 workload are N(0, 1e-3^2).
"""
from __future__ import annotations

import dataclasses
import math

import torch


# activations with a gate and an up projection (the others take one fc1 weight)
GATED_ACTS = ("swiglu", "reglu", "geglu", "glu")


@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    M: int
    H: int
    I: int
    act: str = "swiglu"          # swiglu | reglu | geglu | glu | relu_sq | gelu_tanh_approx | relu
    gate_mult: float = 1.0
    down_mult: float = 1.0
    recompute: bool = False      # backward recomputes G/U from x
    fuse_grad_accum: bool = False  # fp32 dW += grad
    infer: bool = False          # also exercise the no-grad forward
    seed: int = 0

    @property
    def gated(self) -> bool:
        return self.act in GATED_ACTS


# The five workloads (token count M = batch * sequence).
WORKLOADS = {
    "tiny_swiglu": Workload("tiny_swiglu", M=64, H=128, I=352),
    "llama7b_swiglu": Workload("llama7b_swiglu", M=2 * 1024, H=4096, I=11008),
    "falcon_h1_swiglu": Workload("falcon_h1_swiglu", M=4 * 2048, H=2048, I=4864,
                                 gate_mult=1.125, down_mult=2.0),
    "nanogpt_relu_sq": Workload("nanogpt_relu_sq", M=49152, H=768, I=3072,
                                act="relu_sq", recompute=True,
                                fuse_grad_accum=True),
    "llama3_8b_swiglu": Workload("llama3_8b_swiglu", M=4 * 2048, H=4096, I=14336,
                                 recompute=True, infer=True),
}


def _uniform(gen, shape, bound):
    return (torch.rand(shape, generator=gen, dtype=torch.float32) * 2.0 - 1.0) * bound


def make_inputs(M, H, I, act="swiglu", seed=0, dW_prev=False):
    """Return a dict of CPU tensors: x, Wg, Wu (None if non-gated), Wd, dout
    (all bf16) and, if ``dW_prev``, fp32 pre-existing gradients
    dWg_prev, dWu_prev, dWd_prev."""
    gen = torch.Generator(device="cpu")
    gen.manual_seed(seed)
    gated = act in GATED_ACTS
    bf = torch.bfloat16
    x = torch.randn((M, H), generator=gen, dtype=torch.float32).to(bf)
    Wg = _uniform(gen, (I, H), 1.0 / math.sqrt(H)).to(bf)
    Wu = _uniform(gen, (I, H), 1.0 / math.sqrt(H)).to(bf) if gated else None
    Wd = _uniform(gen, (H, I), 1.0 / math.sqrt(I)).to(bf)
    dout = torch.randn((M, H), generator=gen, dtype=torch.float32).to(bf)
    res = {"x": x, "Wg": Wg, "Wu": Wu, "Wd": Wd, "dout": dout}
    if dW_prev:
        res["dWg_prev"] = torch.randn((I, H), generator=gen, dtype=torch.float32) * 1e-3
        res["dWu_prev"] = (torch.randn((I, H), generator=gen, dtype=torch.float32) * 1e-3
                           if gated else None)
        res["dWd_prev"] = torch.randn((H, I), generator=gen, dtype=torch.float32) * 1e-3
    return res


def workload_inputs(w: Workload):
    return make_inputs(w.M, w.H, w.I, w.act, w.seed, dW_prev=w.fuse_grad_accum)


def to_f64(t):
    """Exact widening of a bf16/fp32 CPU or CUDA tensor to a float64 numpy array."""
    if t is None:
        return None
    return t.detach().to("cpu", torch.float64).numpy()


def closed_form_inputs(M, H, I, act="swiglu"):
    """Deterministic inputs with no RNG, every value exactly representable in
    bf16 (small integers over powers of two), for the stored golden
    fixtures: x[m,h] = ((7m + 3h) mod 33 - 16) / 8, weights
    W[r,c] = ((5r + 11c + k) mod 17 - 8) / 32 with k = 0, 1, 2 for
    Wg, Wu, Wd, and dout[m,h] = ((3m + 5h) mod 13 - 6) / 4."""
    bf = torch.bfloat16
    m = torch.arange(M, dtype=torch.float64)[:, None]
    h = torch.arange(H, dtype=torch.float64)[None, :]
    x = (torch.remainder(7 * m + 3 * h, 33) - 16) / 8
    dout = (torch.remainder(3 * m + 5 * h, 13) - 6) / 4

    def w(rows, cols, k):
        r = torch.arange(rows, dtype=torch.float64)[:, None]
        c = torch.arange(cols, dtype=torch.float64)[None, :]
        return (torch.remainder(5 * r + 11 * c + k, 17) - 8) / 32

    gated = act in GATED_ACTS
    return {"x": x.to(bf), "Wg": w(I, H, 0).to(bf), "Wu": w(I, H, 1).to(bf) if gated else None,
            "Wd": w(H, I, 2).to(bf), "dout": dout.to(bf)}


def fp8_closed_form_codes(M, H, I):
    """Deterministic 8-bit inputs with no RNG for the stored FP8 fixture:
    integer codes (exact in e4m3) x8[m,h] = (3m + 5h + 1) mod 9 - 4,
    W1_8[i,h] = (5i + 3h + 2) mod 7 - 3, W2_8[h,i] = (7h + 2i + 1) mod 5 - 2,
    and dout[m,h] = ((m + 3h) mod 11 - 5) / 8 (exact in bf16).  Returns
    float64 tensors of the codes' values and a bf16 dout."""
    m = torch.arange(M, dtype=torch.float64)[:, None]
    h = torch.arange(H, dtype=torch.float64)[None, :]
    i_r = torch.arange(I, dtype=torch.float64)[:, None]
    h_r = torch.arange(H, dtype=torch.float64)[:, None]
    i_c = torch.arange(I, dtype=torch.float64)[None, :]
    return {"x8": torch.remainder(3 * m + 5 * h + 1, 9) - 4,
            "W1_8": torch.remainder(5 * i_r + 3 * h + 2, 7) - 3,
            "W2_8": torch.remainder(7 * h_r + 2 * i_c + 1, 5) - 2,
            "dout": ((torch.remainder(m + 3 * h, 11) - 5) / 8).to(torch.bfloat16)}
