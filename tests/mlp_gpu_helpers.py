"""Shared helpers of the GPU parity tests: run the CUDA path through the C
ABI on seeded inputs, run the fp64 oracle on the same bytes, compare."""
import numpy as np
import torch

import activated_mlp_gemms_gb300 as m
from activated_mlp_gemms_gb300.workloads import to_f64
from bf16_floor import emulated_dw
from oracle import mlp_backward, mlp_forward, rel_err, sampled_inter_units, sampled_token_rows

TOL_BF16 = 2e-2   # max|err| / max|ref| for bf16 outputs (out, dx, bf16 dW)
TOL_F32 = 5e-3    # for fp32-accumulated dW
# Where the bf16 storage of the intermediates (G, U, dG, dU, the postact)
# alone moves an fp32-accumulated gradient by more than TOL_F32 (small test
# shapes; see bf16_floor and test_tolerance_floor), that gradient is held to
# FLOOR_MARGIN times its emulated floor instead.
FLOOR_MARGIN = 1.25
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


def dw_floor(tc, act, gm, dm, mode, ref, dW_prev=None, rstd=None):
    """Per weight gradient, max|emulated - ref| / max|ref| of the kernels'
    bf16 storage roundings alone (bf16_floor.emulated_dw) on the inputs `tc`."""
    a = {k: to_f64(v) for k, v in tc.items() if v is not None}
    prev = None
    if dW_prev is not None:
        prev = {k: to_f64(dW_prev[k + "_prev"]) if dW_prev.get(k + "_prev") is not None else None
                for k in ("dWg", "dWu", "dWd")}
    em = emulated_dw(a["x"], a["dout"], a["Wg"], a.get("Wu"), a["Wd"], act, gm, dm,
                     "saved" if mode == "saved" else "recompute", dW_prev=prev, rstd=rstd)
    return {k: rel_err(em[k], ref[k]) for k in em if em[k] is not None and ref.get(k) is not None}


def tol_of(k, fuse, floor=None):
    """The bound of output k: TOL_BF16 for bf16 outputs; TOL_F32 for
    fp32-accumulated weight gradients, or FLOOR_MARGIN x their bf16-storage
    floor where that is higher."""
    if not (fuse and k.startswith("dW")):
        return TOL_BF16
    if floor is not None and k in floor:
        return max(TOL_F32, FLOOR_MARGIN * floor[k])
    return TOL_F32


def compare_full(got, ref, fuse, floor=None):
    errs = {}
    for k, v in got.items():
        if v is None or ref.get(k) is None:
            continue
        g = to_f64(v)
        assert np.all(np.isfinite(g)), f"{k}: non-finite values (untouched tile?)"
        errs[k] = rel_err(g, ref[k])
    for k, e in errs.items():
        tol = tol_of(k, fuse, floor)
        assert e <= tol, f"{k}: rel err {e:.3e} > {tol:.3e} (all: {errs}; floor {floor})"
    return errs


def spread_sample(n, size, tile=256, seed=0):
    """`size` sorted distinct indices in [0, n): the first and the last, then
    one random index in each `tile`-wide block (blocks in random order) until
    `size` are taken, then random ones.  At the workloads' sizes this puts a
    sampled token row into every 256-row output tile and a sampled
    intermediate unit into every 256-column one."""
    rng = np.random.default_rng(seed)
    size = min(size, n)
    pick = {0, n - 1}
    for b in rng.permutation((n + tile - 1) // tile):
        if len(pick) >= size:
            break
        pick.add(int(rng.integers(b * tile, min(n, (b + 1) * tile))))
    while len(pick) < size:
        pick.add(int(rng.integers(0, n)))
    return np.array(sorted(pick), dtype=np.int64)


SAMPLE_ROWS = 256   # token rows of out / dx checked at full size
SAMPLE_UNITS = 64   # intermediate units (rows of dWg/dWu, columns of dWd) checked at full size


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
