"""Shared helpers of the GPU parity tests: run the CUDA path through the C
ABI on seeded inputs, run the fp64 oracle on the same bytes, compare."""
import numpy as np
import torch

import activated_mlp_gemms_gb300 as m
from activated_mlp_gemms_gb300.workloads import to_f64
from oracle import mlp_backward, mlp_forward, rel_err, sampled_inter_units, sampled_token_rows

TOL_BF16 = 2e-2   # max|err| / max|ref| for bf16 outputs (out, dx, bf16 dW)
TOL_F32 = 5e-3    # for fp32-accumulated dW (the workloads' sizes)
# Below F32_TOL_MIN_TOKENS tokens the fp32-accumulated weight gradients are
# held to TOL_F32_SMALL instead: there the error floor is set by the bf16
# storage of the intermediates (G, U, dG, dU, postact), not by the
# accumulation.  Emulating exactly those roundings in fp64 gives
# max|err|/max|ref| up to 6.0e-3 (relu_sq dWd, M = 257; SwiGLU dWg 5.1e-3
# at M = 64), and 1.6e-3 .. 4.4e-3 for M >= 1024.
F32_TOL_MIN_TOKENS = 1024
TOL_F32_SMALL = 1e-2
GUARD = 64        # guard elements after every output buffer
SENTINEL = float("nan")


def dev_tensors(t, device="cuda"):
    return {k: (v.to(device) if v is not None else None) for k, v in t.items()}


def guarded(shape, dtype, fill=SENTINEL, device="cuda"):
    """A buffer with GUARD trailing elements; returns (view, full)."""
    n = int(np.prod(shape))
    full = torch.full((n + GUARD,), fill, dtype=dtype, device=device)
    return full[:n].view(*shape), full


def guard_intact(full, fill=SENTINEL):
    tail = full[-GUARD:].float()
    if np.isnan(fill):
        return bool(torch.isnan(tail).all())
    return bool((tail == fill).all())


def run_gpu(t, M, H, I, act, gm, dm, mode="saved", fuse=False, want=("dx", "dWg", "dWu", "dWd"),
            dW_prev=None):
    """Runs mlp_fwd (+ mlp_bwd or mlp_bwd_recompute) on the CUDA tensors `t`.
    Returns a dict of CPU fp64 arrays and a list of guard-band violations."""
    gated = act in m.GATED_ACTS
    prob = m.problem(M, H, I, act, gm, dm)
    bf = torch.bfloat16
    out, out_f = guarded((M, H), bf)
    G, G_f = guarded((M, I), bf)
    U, U_f = guarded((M, I), bf) if gated else (None, None)
    save = mode == "saved"
    ws = m.mlp_fwd(prob, t["x"], t["Wg"], t["Wu"], t["Wd"], out, G if save else None,
                   U if save else None)
    wdt = torch.float32 if fuse else bf
    res = {"out": out}
    fulls = {"out": out_f}
    bufs = {}
    shapes = {"dx": (M, H), "dWg": (I, H), "dWu": (I, H), "dWd": (H, I)}
    for k in ("dx", "dWg", "dWu", "dWd"):
        if k == "dWu" and not gated:
            bufs[k] = None
            continue
        if k not in want:
            bufs[k] = None
            continue
        dt = bf if k == "dx" else wdt
        fill = SENTINEL
        if k != "dx" and fuse:
            fill = 0.0
        view, full = guarded(shapes[k], dt, fill)
        if k != "dx" and fuse and dW_prev is not None:
            view.copy_(dW_prev[k + "_prev"].to(view.device))
        bufs[k] = view
        fulls[k] = full
    if mode == "saved":
        m.mlp_bwd(prob, t["dout"], t["x"], t["Wg"], t["Wu"], t["Wd"], G, U, bufs["dx"], bufs["dWg"],
                  bufs["dWu"], bufs["dWd"], fuse_grad_accum=fuse)
    else:
        m.mlp_bwd_recompute(prob, t["dout"], t["x"], t["Wg"], t["Wu"], t["Wd"], bufs["dx"],
                            bufs["dWg"], bufs["dWu"], bufs["dWd"], fuse_grad_accum=fuse)
    torch.cuda.synchronize()
    status = m.mlp_device_status(ws)
    assert status == 0, m.mlp_status_string(status)
    bad = []
    for k, full in fulls.items():
        fill = 0.0 if (k.startswith("dW") and fuse) else SENTINEL
        if not guard_intact(full, fill):
            bad.append(k)
    for k, v in bufs.items():
        if v is not None:
            res[k] = v
    return {k: v for k, v in res.items()}, bad, {"G": G, "U": U}


def oracle_full(tc, act, gm, dm, dW_prev=None):
    a = {k: to_f64(v) for k, v in tc.items()}
    fw = mlp_forward(a["x"], a["Wg"], a["Wu"], a["Wd"], act, gm, dm)
    prev = None
    if dW_prev is not None:
        prev = {"dWg": to_f64(dW_prev["dWg_prev"]), "dWd": to_f64(dW_prev["dWd_prev"]),
                "dWu": to_f64(dW_prev["dWu_prev"]) if dW_prev.get("dWu_prev") is not None else None}
    bw = mlp_backward(a["dout"], a["x"], a["Wg"], a["Wu"], a["Wd"], act, gm, dm, dW_prev=prev)
    return {"out": fw["out"], **bw}


def compare_full(got, ref, fuse, M=None):
    errs = {}
    for k, v in got.items():
        if v is None or ref.get(k) is None:
            continue
        g = to_f64(v)
        assert np.all(np.isfinite(g)), f"{k}: non-finite values (untouched tile?)"
        errs[k] = rel_err(g, ref[k])
    for k, e in errs.items():
        if fuse and k.startswith("dW"):
            tol = TOL_F32 if (M is None or M >= F32_TOL_MIN_TOKENS) else TOL_F32_SMALL
        else:
            tol = TOL_BF16
        assert e <= tol, f"{k}: rel err {e:.3e} > {tol} (all: {errs})"
    return errs


def oracle_sampled(tc, act, gm, dm, rows, cols, dW_prev=None):
    a = {k: to_f64(v) for k, v in tc.items()}
    r = sampled_token_rows(rows, a["dout"], a["x"], a["Wg"], a["Wu"], a["Wd"], act, gm, dm)
    prev = None
    if dW_prev is not None:
        prev = {"dWg": to_f64(dW_prev["dWg_prev"]), "dWd": to_f64(dW_prev["dWd_prev"]),
                "dWu": to_f64(dW_prev["dWu_prev"]) if dW_prev.get("dWu_prev") is not None else None}
    c = sampled_inter_units(cols, a["dout"], a["x"], a["Wg"], a["Wu"], a["Wd"], act, gm, dm,
                            dW_prev=prev)
    return r, c
