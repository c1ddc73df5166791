"""GPU parity of the MLP block with its neighbours (mlp_block_fwd /
mlp_block_bwd: RMS-normalised input, scaled residual add; modded-nanogpt
gpt.py, "process mlp") against the fp64 oracle's block_forward /
block_backward, through the C ABI, on seeded inputs."""
import numpy as np
import pytest
import torch

import activated_mlp_gemms_gb300 as m
from activated_mlp_gemms_gb300.workloads import make_inputs, to_f64
from mlp_gpu_helpers import (SAMPLE_ROWS, SAMPLE_UNITS, TOL_BF16, TOL_F32, dw_floor,
                             spread_sample, tol_of)
from oracle import block_backward, block_forward, rel_err, rms_norm

pytestmark = pytest.mark.gpu

LAMBDAS = dict(resid_lambda=1.1 ** 0.5, post_lambda=0.8, eps=2.0 ** -7)


@pytest.fixture
def tile_policy(request):
    m.mlp_set_tile_policy(request.param)
    yield request.param
    m.mlp_set_tile_policy(0)


def _run(t, M, H, I, act, gm, dm, fuse, inplace=False):
    d = {k: (v.cuda() if v is not None else None) for k, v in t.items()}
    gated = act in m.GATED_ACTS
    prob = m.problem(M, H, I, act, gm, dm)
    blk = m.block(**LAMBDAS)
    bf = torch.bfloat16
    G = torch.empty(M, I, dtype=bf, device="cuda")
    U = torch.empty(M, I, dtype=bf, device="cuda") if gated else None
    x_in = d["x"].clone() if inplace else d["x"]
    y = x_in if inplace else torch.full((M, H), float("nan"), dtype=bf, device="cuda")
    rstd, _ = m.mlp_block_fwd(prob, blk, x_in, d["Wg"], d["Wu"], d["Wd"], y, G, U)
    res = {"y": y.clone(), "rstd": rstd.clone()}
    wdt = torch.float32 if fuse else bf
    dx = torch.full((M, H), float("nan"), dtype=bf, device="cuda")
    dW = {}
    for k, shp in (("dWg", (I, H)), ("dWu", (I, H)), ("dWd", (H, I))):
        if k == "dWu" and not gated:
            dW[k] = None
            continue
        dW[k] = (d[k + "_prev"].clone() if fuse else torch.full(shp, float("nan"), dtype=bf,
                                                                  device="cuda"))
    ws = m.mlp_block_bwd(prob, blk, d["dout"], d["x"], d["Wg"], d["Wu"], d["Wd"], G, U, rstd,
                         dx, dW["dWg"], dW["dWu"], dW["dWd"], fuse_grad_accum=fuse)
    torch.cuda.synchronize()
    assert m.mlp_device_status(ws) == 0
    res.update({"dx": dx, **{k: v for k, v in dW.items() if v is not None}})
    return res


def _oracle(t, act, gm, dm, fuse):
    a = {k: to_f64(v) if v is not None else None for k, v in t.items()}
    fw = block_forward(a["x"], a["Wg"], a["Wu"], a["Wd"], act, gm, dm, **LAMBDAS)
    prev = ({"dWg": a["dWg_prev"], "dWu": a.get("dWu_prev"), "dWd": a["dWd_prev"]}
            if fuse else None)
    bw = block_backward(a["dout"], a["x"], a["Wg"], a["Wu"], a["Wd"], act, gm, dm, **LAMBDAS,
                        dW_prev=prev)
    return {"y": fw["y"], "rstd": fw["rstd"], **bw}


def _floor(t, act, gm, dm, ref):
    """The bf16-storage floor of the block's fp32-accumulated gradients: the
    MLP's rounding points with the block's row scale and post_lambda."""
    x = to_f64(t["x"])
    _, r = rms_norm(x, LAMBDAS["eps"])
    prev = {k: t[k] for k in ("dWg_prev", "dWu_prev", "dWd_prev")}
    return dw_floor(t, act, gm, dm * LAMBDAS["post_lambda"], "saved", ref, prev,
                    rstd=1.0 / r[:, 0])


def _compare(got, ref, fuse, floor=None):
    errs = {}
    for k, v in got.items():
        if ref.get(k) is None:
            continue
        g = to_f64(v)
        assert np.all(np.isfinite(g)), k
        errs[k] = rel_err(g, ref[k])
    for k, e in errs.items():
        tol = 1e-5 if k == "rstd" else tol_of(k, fuse, floor)  # rstd: fp32 sums of bf16 squares
        assert e <= tol, f"{k}: rel err {e:.3e} > {tol:.3e} (all: {errs}; floor {floor})"
    return errs


@pytest.mark.parametrize("tile_policy", [1, 2], indirect=True)
@pytest.mark.parametrize("act,gm,dm", [("relu_sq", 1.0, 1.0), ("swiglu", 1.125, 2.0),
                                       ("gelu_tanh_approx", 0.75, 1.5)])
@pytest.mark.parametrize("M,H,I", [(64, 128, 352), (300, 200, 392), (520, 1032, 776)])
@pytest.mark.parametrize("fuse", [False, True])
def test_block_parity(act, gm, dm, M, H, I, fuse, tile_policy):
    t = make_inputs(M, H, I, act, seed=41, dW_prev=fuse)
    got = _run(t, M, H, I, act, gm, dm, fuse)
    ref = _oracle(t, act, gm, dm, fuse)
    _compare(got, ref, fuse, _floor(t, act, gm, dm, ref) if fuse else None)


@pytest.mark.parametrize("act", ["relu_sq", "swiglu"])
@pytest.mark.parametrize("M", [16, 100])
def test_block_decode_sized_split_k(act, M):
    # few tokens: the down projection and dx split K; the residual add moves
    # into the fp32 -> bf16 pass, the norm's projection into its own kernel
    H, I = 512, 2048
    t = make_inputs(M, H, I, act, seed=42)
    got = _run(t, M, H, I, act, 1.0, 1.0, False)
    _compare(got, _oracle(t, act, 1.0, 1.0, False), False)


def test_block_output_over_its_input():
    # y may be x itself: each residual element is read before its tile of y
    # is stored
    M, H, I, act = 300, 264, 392, "relu_sq"
    t = make_inputs(M, H, I, act, seed=43)
    got = _run(t, M, H, I, act, 1.0, 1.0, False, inplace=True)
    ref = _oracle(t, act, 1.0, 1.0, False)
    assert rel_err(to_f64(got["y"]), ref["y"]) <= TOL_BF16


@pytest.mark.parametrize("name", ["llama7b_swiglu", "nanogpt_relu_sq"])
def test_block_full_size_sampled(name):
    """The block at the workloads' full sizes (saved preacts; the ReLU^2
    workload with fp32 gradient accumulation): parity on sampled token rows
    (y, dx) and sampled intermediate units (rows of dWg/dWu, columns of dWd,
    each reduced over all tokens), computed by the oracle."""
    from activated_mlp_gemms_gb300.workloads import WORKLOADS, workload_inputs
    from oracle import block_sampled
    w = WORKLOADS[name]
    t = workload_inputs(w)
    got = _run(t, w.M, w.H, w.I, w.act, w.gate_mult, w.down_mult, w.fuse_grad_accum)
    rows = spread_sample(w.M, SAMPLE_ROWS)
    cols = spread_sample(w.I, SAMPLE_UNITS)
    a = {k: to_f64(v) if v is not None else None for k, v in t.items()}
    prev = ({"dWg": a["dWg_prev"], "dWu": a.get("dWu_prev"), "dWd": a["dWd_prev"]}
            if w.fuse_grad_accum else None)
    ref = block_sampled(rows, cols, a["dout"], a["x"], a["Wg"], a["Wu"], a["Wd"], w.act,
                        w.gate_mult, w.down_mult, **LAMBDAS, dW_prev=prev)
    r_t, c_t = torch.as_tensor(rows), torch.as_tensor(cols)
    errs = {"y": rel_err(to_f64(got["y"][r_t]), ref["y"]),
            "dx": rel_err(to_f64(got["dx"][r_t]), ref["dx"]),
            "dWg": rel_err(to_f64(got["dWg"][c_t]), ref["dWg"]),
            "dWd": rel_err(to_f64(got["dWd"][:, c_t]), ref["dWd"])}
    if w.gated:
        errs["dWu"] = rel_err(to_f64(got["dWu"][c_t]), ref["dWu"])
    tol_w = TOL_F32 if w.fuse_grad_accum else TOL_BF16
    for k, e in errs.items():
        assert e <= (tol_w if k.startswith("dW") else TOL_BF16), (name, errs)
