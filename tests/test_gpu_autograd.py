"""mlp_func, the differentiable form of the entry points: its forward and
the gradients autograd gets from it are the bytes the direct mlp_fwd /
mlp_bwd / mlp_bwd_recompute calls write (whose parity with the oracle the
other GPU tests establish), for batched [B, S, H] inputs, partial
gradients, in-place fp32 accumulation and both backward modes.  The shapes
split no reduction across work units, so two runs agree bitwise (the C
header's determinism statement; checked through mlp_plan)."""
import pytest
import torch

import activated_mlp_gemms_gb300 as m
from activated_mlp_gemms_gb300.workloads import make_inputs

BF = torch.bfloat16


def test_mlp_func_rejects_host_tensors():
    x = torch.zeros(2, 8, dtype=BF)
    W = torch.zeros(16, 8, dtype=BF)
    with pytest.raises(ValueError, match="CUDA"):
        m.mlp_func(x, W, W, torch.zeros(8, 16, dtype=BF))


def _inputs(B, S, H, I, act, seed):
    t = make_inputs(B * S, H, I, act, seed=seed)
    d = {k: (v.cuda() if v is not None else None) for k, v in t.items()}
    d["x"] = d["x"].view(B, S, H)
    d["dout"] = d["dout"].view(B, S, H)
    return d


def _direct(d, act, gm, dm, recompute, want=(True, True, True, True), fuse=False, prev=None):
    x = d["x"].reshape(-1, d["x"].shape[-1])
    dout = d["dout"].reshape(x.shape)
    M, H = x.shape
    I = d["Wd"].shape[1]
    gated = act in m.GATED_ACTS
    prob = m.problem(M, H, I, act, gm, dm)
    fwd = m.mlp_plan(prob, m.MODE_FWD)
    bwd = m.mlp_plan(prob, m.MODE_BWD_RECOMPUTE if recompute else m.MODE_BWD, fuse)
    assert fwd["out_split"] == 1 and bwd["out_split"] == 1 and bwd["wgrad_split"] <= 1
    out = torch.empty(M, H, dtype=BF, device="cuda")
    G = U = None
    if not recompute:
        G = torch.empty(M, I, dtype=BF, device="cuda")
        U = torch.empty_like(G) if gated else None
    m.mlp_fwd(prob, x, d["Wg"], d["Wu"], d["Wd"], out, G, U)
    wdt = torch.float32 if fuse else BF
    dx = torch.empty_like(x) if want[0] else None
    ws = []
    for i, (k, shape) in enumerate((("Wg", (I, H)), ("Wu", (I, H)), ("Wd", (H, I)))):
        if not want[i + 1] or d[k] is None:
            ws.append(None)
        elif fuse:
            ws.append(prev[k].clone())
        else:
            ws.append(torch.empty(shape, dtype=wdt, device="cuda"))
    if recompute:
        m.mlp_bwd_recompute(prob, dout, x, d["Wg"], d["Wu"], d["Wd"], dx, *ws, fuse_grad_accum=fuse)
    else:
        m.mlp_bwd(prob, dout, x, d["Wg"], d["Wu"], d["Wd"], G, U, dx, *ws, fuse_grad_accum=fuse)
    torch.cuda.synchronize()
    return out.view(d["x"].shape), dx, ws


def _leaves(d, want):
    x = d["x"].clone().requires_grad_(want[0])
    ws = []
    for i, k in enumerate(("Wg", "Wu", "Wd")):
        w = d[k]
        ws.append(None if w is None else w.clone().requires_grad_(want[i + 1]))
    return x, ws


@pytest.mark.gpu
@pytest.mark.parametrize("act,gm,dm,recompute", [("swiglu", 1.0, 1.0, False),
                                                 ("swiglu", 1.125, 2.0, True),
                                                 ("relu_sq", 1.0, 1.0, True),
                                                 ("geglu", 1.0, 1.0, False)])
def test_mlp_func_equals_the_entry_points(act, gm, dm, recompute):
    d = _inputs(2, 1024, 2048, 2816, act, seed=11)
    ref_out, ref_dx, ref_w = _direct(d, act, gm, dm, recompute)
    x, (Wg, Wu, Wd) = _leaves(d, (True, True, True, True))
    out = m.mlp_func(x, Wg, Wu, Wd, act, gm, dm, recompute=recompute)
    assert out.shape == x.shape and out.dtype == BF
    assert torch.equal(out.detach(), ref_out)
    out.backward(d["dout"])
    assert torch.equal(x.grad.view(-1, x.shape[-1]), ref_dx)
    for w, r in zip((Wg, Wu, Wd), ref_w):
        if w is not None:
            assert torch.equal(w.grad, r)


@pytest.mark.gpu
@pytest.mark.parametrize("want", [(True, False, False, False), (False, True, False, True),
                                  (False, False, False, True)])
def test_mlp_func_computes_only_what_autograd_asks_for(want):
    act = "swiglu"
    d = _inputs(2, 1024, 2048, 2816, act, seed=12)
    _, ref_dx, ref_w = _direct(d, act, 1.0, 1.0, False, want=want)
    x, (Wg, Wu, Wd) = _leaves(d, want)
    out = m.mlp_func(x, Wg, Wu, Wd, act)
    out.backward(d["dout"])
    if want[0]:
        assert torch.equal(x.grad.view(-1, x.shape[-1]), ref_dx)
    else:
        assert x.grad is None
    for w, r, wanted in zip((Wg, Wu, Wd), ref_w, want[1:]):
        if wanted:
            assert torch.equal(w.grad, r)
        else:
            assert w.grad is None


@pytest.mark.gpu
@pytest.mark.parametrize("recompute", [False, True])
def test_mlp_func_accumulates_into_main_grad(recompute):
    act = "swiglu"
    d = _inputs(2, 1024, 2048, 2816, act, seed=13)
    g = torch.Generator(device="cpu").manual_seed(5)
    prev = {k: (1e-3 * torch.randn(d[k].shape, generator=g)).cuda() for k in ("Wg", "Wu", "Wd")}
    _, ref_dx, ref_w = _direct(d, act, 1.0, 1.0, recompute, fuse=True, prev=prev)
    x, ws = _leaves(d, (True, True, True, True))
    for w, k in zip(ws, ("Wg", "Wu", "Wd")):
        w.main_grad = prev[k].clone()
    out = m.mlp_func(x, *ws, act, recompute=recompute, fuse_grad_accum=True)
    out.backward(d["dout"])
    assert torch.equal(x.grad.view(-1, x.shape[-1]), ref_dx)
    for w, r in zip(ws, ref_w):
        assert w.grad is None
        assert torch.equal(w.main_grad, r)


@pytest.mark.gpu
def test_mlp_func_main_grad_is_required_when_fusing():
    d = _inputs(1, 64, 512, 1416, "swiglu", seed=14)
    x, ws = _leaves(d, (True, True, True, True))
    out = m.mlp_func(x, *ws, "swiglu", fuse_grad_accum=True)
    with pytest.raises(ValueError, match="main_grad"):
        out.backward(d["dout"])


@pytest.mark.gpu
def test_mlp_func_second_backward():
    """The saved-preact graph is spent by its backward (dG, dU overwrite G,
    U); the recompute graph can be differentiated again, to the same bytes."""
    d = _inputs(2, 1024, 2048, 2816, "swiglu", seed=15)
    x, ws = _leaves(d, (True, True, True, True))
    out = m.mlp_func(x, *ws, "swiglu")
    out.backward(d["dout"], retain_graph=True)
    with pytest.raises(RuntimeError, match="recompute=True"):
        out.backward(d["dout"])
    x, ws = _leaves(d, (True, False, False, False))
    out = m.mlp_func(x, *ws, "swiglu", recompute=True)
    out.backward(d["dout"], retain_graph=True)
    first = x.grad.clone()
    x.grad = None
    out.backward(d["dout"])
    assert torch.equal(x.grad, first)


@pytest.mark.gpu
def test_mlp_func_empty_batch():
    d = _inputs(1, 8, 512, 1416, "relu_sq", seed=16)
    x = d["x"][:, :0].clone().requires_grad_(True)
    W1 = d["Wg"].clone().requires_grad_(True)
    Wd = d["Wd"].clone().requires_grad_(True)
    out = m.mlp_func(x, W1, None, Wd, "relu_sq")
    assert out.shape == x.shape
    out.backward(torch.empty_like(out))
    assert x.grad.shape == x.shape
    assert torch.count_nonzero(W1.grad) == 0 and torch.count_nonzero(Wd.grad) == 0


@pytest.mark.gpu
@pytest.mark.parametrize("act,gm,dm,fuse", [("swiglu", 1.125, 2.0, False), ("relu_sq", 1.0, 1.0, True)])
def test_mlp_block_func_equals_the_entry_points(act, gm, dm, fuse):
    d = _inputs(2, 1024, 2048, 2816, act, seed=17)
    B, S, H = d["x"].shape
    x2 = d["x"].reshape(-1, H)
    M, I = x2.shape[0], d["Wd"].shape[1]
    gated = act in m.GATED_ACTS
    lam, post, eps = 1.1 ** 0.5, 0.8, 2.0 ** -7
    prob = m.problem(M, H, I, act, gm, dm)
    blk = m.block(lam, post, eps)
    assert m.mlp_plan(prob, m.MODE_FWD)["out_split"] == 1
    bwd = m.mlp_plan(prob, m.MODE_BWD, fuse)
    assert bwd["out_split"] == 1 and bwd["wgrad_split"] <= 1
    g = torch.Generator(device="cpu").manual_seed(6)
    prev = {k: (1e-3 * torch.randn(d[k].shape, generator=g)).cuda()
            for k in ("Wg", "Wu", "Wd") if d[k] is not None}
    y = torch.empty(M, H, dtype=BF, device="cuda")
    G = torch.empty(M, I, dtype=BF, device="cuda")
    U = torch.empty_like(G) if gated else None
    rstd, _ = m.mlp_block_fwd(prob, blk, x2, d["Wg"], d["Wu"], d["Wd"], y, G, U)
    dx = torch.empty_like(x2)
    ref_w = [None if d[k] is None else prev[k].clone() if fuse else torch.empty_like(d[k])
             for k in ("Wg", "Wu", "Wd")]
    m.mlp_block_bwd(prob, blk, d["dout"].reshape(-1, H), x2, d["Wg"], d["Wu"], d["Wd"], G, U,
                    rstd, dx, *ref_w, fuse_grad_accum=fuse)
    torch.cuda.synchronize()

    x, ws = _leaves(d, (True, True, True, True))
    if fuse:
        for w, k in zip(ws, ("Wg", "Wu", "Wd")):
            if w is not None:
                w.main_grad = prev[k].clone()
    out = m.mlp_block_func(x, *ws, act, gm, dm, lam, post, eps, fuse_grad_accum=fuse)
    assert torch.equal(out.detach().view(-1, H), y)
    out.backward(d["dout"])
    assert torch.equal(x.grad.view(-1, H), dx)
    for w, r in zip(ws, ref_w):
        if w is None:
            continue
        assert torch.equal(w.main_grad if fuse else w.grad, r)
        if fuse:
            assert w.grad is None
