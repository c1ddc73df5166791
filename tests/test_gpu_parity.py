"""GPU parity of the CUDA path (through the C ABI) against the fp64 oracle.

Tolerances: max|err|/max|ref| <= 2e-2 for bf16 outputs and <= 5e-3 for
fp32-accumulated weight gradients, per tensor.  Every output buffer carries
a NaN-filled guard band (checked after each call) and starts NaN-filled, so
an untouched tile or an out-of-range store fails the test.
"""
import json
import os

import numpy as np
import pytest
import torch

import activated_mlp_gemms_gb300 as m
from activated_mlp_gemms_gb300.workloads import (WORKLOADS, closed_form_inputs, make_inputs,
                                                 to_f64, workload_inputs)
from mlp_gpu_helpers import (SAMPLE_ROWS, SAMPLE_UNITS, TOL_BF16, TOL_F32, compare_full,
                             dev_tensors, dw_floor, oracle_full, oracle_sampled, run_gpu,
                             spread_sample)
from oracle import rel_err

pytestmark = pytest.mark.gpu


@pytest.fixture
def tile_policy(request):
    """Forces single-CTA (1) or CTA-pair (2) tiles for one test."""
    m.mlp_set_tile_policy(request.param)
    yield request.param
    m.mlp_set_tile_policy(0)

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "closed_form_small.json")


def _golden_cases():
    with open(GOLDEN) as f:
        return json.load(f)["cases"]


@pytest.mark.parametrize("tile_policy", [1, 2], indirect=True)
@pytest.mark.parametrize("mode", ["saved", "recompute"])
def test_golden_closed_form(mode, tile_policy):
    for c in _golden_cases():
        M, H, I, act = c["M"], c["H"], c["I"], c["act"]
        t = dev_tensors(closed_form_inputs(M, H, I, act))
        got, bad, _ = run_gpu(t, M, H, I, act, c["gate_mult"], c["down_mult"], mode=mode)
        assert not bad, f"guard band overwritten: {bad}"
        ref = {k: (np.array(c[k]) if c[k] is not None else None)
               for k in ("out", "dx", "dWg", "dWu", "dWd")}
        compare_full(got, ref, fuse=False)


SMALL = [  # (M, H, I): one tile; several tiles with ragged tails in every dimension
    (64, 128, 352),
    (300, 200, 392),
    (257, 264, 520),
    (1, 8, 8),
]


@pytest.mark.parametrize("tile_policy", [1, 2], indirect=True)
@pytest.mark.parametrize("act,gm,dm", [("swiglu", 1.0, 1.0), ("swiglu", 1.125, 2.0),
                                       ("relu_sq", 1.0, 1.0), ("gelu_tanh_approx", 0.75, 1.5)])
@pytest.mark.parametrize("shape", SMALL)
@pytest.mark.parametrize("mode,fuse", [("saved", False), ("recompute", False), ("saved", True),
                                       ("recompute", True)])
def test_small_parity(act, gm, dm, shape, mode, fuse, tile_policy):
    M, H, I = shape
    t = make_inputs(M, H, I, act, seed=1, dW_prev=fuse)
    tc = {k: v for k, v in t.items() if not k.endswith("_prev")}
    prev = {k: v for k, v in t.items() if k.endswith("_prev")} if fuse else None
    got, bad, _ = run_gpu(dev_tensors(tc), M, H, I, act, gm, dm, mode=mode, fuse=fuse, dW_prev=prev)
    assert not bad, f"guard band overwritten: {bad}"
    ref = oracle_full(tc, act, gm, dm, dW_prev=prev)
    compare_full(got, ref, fuse, floor=dw_floor(tc, act, gm, dm, mode, ref, prev) if fuse else None)


@pytest.mark.parametrize("act", list(m.ACTS))
def test_infer_equals_train_forward_bitwise(act):
    M, H, I = 300, 264, 392
    t = dev_tensors(make_inputs(M, H, I, act, seed=2))
    prob = m.problem(M, H, I, act, 1.125, 2.0)
    o1 = torch.empty(M, H, dtype=torch.bfloat16, device="cuda")
    o2 = torch.empty_like(o1)
    G = torch.empty(M, I, dtype=torch.bfloat16, device="cuda")
    U = torch.empty_like(G) if act in m.GATED_ACTS else None
    m.mlp_fwd(prob, t["x"], t["Wg"], t["Wu"], t["Wd"], o1, G, U)
    m.mlp_fwd_infer(prob, t["x"], t["Wg"], t["Wu"], t["Wd"], o2)
    torch.cuda.synchronize()
    assert torch.equal(o1, o2)


@pytest.mark.parametrize("act", ["swiglu", "relu_sq", "gelu_tanh_approx"])
def test_saved_equals_recompute(act):
    # Gated: both paths read bf16 preacts produced by the same GEMM tiles, so
    # out, dx, dWg and dWu agree exactly.  dWd differs by rounding only: the
    # recompute path takes the postact from the fp32 accumulators, the saved
    # path rebuilds it from the bf16 preacts.  Non-gated: the recompute path
    # takes the derivative from the fp32 preact too (rounded to bf16 where
    # the saved path rounds the preact), so only out is bitwise equal.
    M, H, I = 300, 264, 392
    tc = dev_tensors(make_inputs(M, H, I, act, seed=3))
    a, _, _ = run_gpu(tc, M, H, I, act, 1.0, 1.0, mode="saved")
    b, _, _ = run_gpu(tc, M, H, I, act, 1.0, 1.0, mode="recompute")
    exact = {"out", "dx", "dWg", "dWu"} if act in m.GATED_ACTS else {"out"}
    for k in a:
        if k in exact:
            assert torch.equal(a[k], b[k]), k
        else:
            assert rel_err(to_f64(a[k]), to_f64(b[k])) < TOL_BF16, k


@pytest.mark.parametrize("act", ["swiglu", "relu_sq"])
def test_single_cta_and_pair_tiles_agree(act):
    # Same fp32 accumulation order per output element: bitwise equal outputs.
    M, H, I = 300, 264, 392
    tc = dev_tensors(make_inputs(M, H, I, act, seed=6))
    try:
        m.mlp_set_tile_policy(1)
        a, _, _ = run_gpu(tc, M, H, I, act, 1.125, 2.0, mode="saved")
        m.mlp_set_tile_policy(2)
        b, _, _ = run_gpu(tc, M, H, I, act, 1.125, 2.0, mode="saved")
    finally:
        m.mlp_set_tile_policy(0)
    for k in a:
        assert torch.equal(a[k], b[k]), k


@pytest.mark.parametrize("act", ["swiglu", "relu_sq"])
@pytest.mark.parametrize("mode", ["saved", "recompute"])
@pytest.mark.parametrize("want", [("dWd",), ("dx",), ("dWg",), ("dx", "dWd")])
def test_partial_gradients(act, mode, want):
    # Unrequested gradients are skipped (NULL outputs); requested ones match.
    M, H, I = 200, 136, 264
    t = make_inputs(M, H, I, act, seed=4)
    got, bad, _ = run_gpu(dev_tensors(t), M, H, I, act, 1.125, 2.0, mode=mode, want=want)
    assert not bad
    ref = oracle_full(t, act, 1.125, 2.0)
    errs = compare_full(got, ref, fuse=False)
    assert set(errs) == {"out", *want}


@pytest.mark.parametrize("act", ["relu_sq", "gelu_tanh_approx", "relu"])
@pytest.mark.parametrize("M,H,I", [(64, 128, 352), (300, 200, 392), (1000, 768, 3072)])
def test_nongated_recompute_is_one_fused_kernel(act, M, H, I):
    # The non-gated recompute backward computes the preact and dout Wd in one
    # kernel (no separate recompute GEMM) and matches the oracle.
    t = make_inputs(M, H, I, act, seed=21, dW_prev=True)
    tc = {k: v for k, v in t.items() if not k.endswith("_prev")}
    prev = {k: v for k, v in t.items() if k.endswith("_prev")}
    m.mlp_trace_read()
    m.mlp_trace_enable(True)
    try:
        got, bad, _ = run_gpu(dev_tensors(tc), M, H, I, act, 0.75, 1.5, mode="recompute",
                              fuse=True, dW_prev=prev)
    finally:
        m.mlp_trace_enable(False)
    names = [n for n, _ in m.mlp_trace_read()]
    # the forward's gate/up GEMM is the only one: the backward recomputes
    # the preact inside the fused kernel
    assert names.count("gate_up_act") == 1 and names.count("dact_recompute") == 1, names
    assert "dgated" not in names, names
    assert not bad
    ref = oracle_full(tc, act, 0.75, 1.5, dW_prev=prev)
    compare_full(got, ref, fuse=True, floor=dw_floor(tc, act, 0.75, 1.5, "recompute", ref, prev))


def test_split_m_accumulation_matches_one_call():
    # The data-parallel invariant: two half-M backward calls accumulating into
    # the same fp32 gradients equal one full-M call.
    M, H, I, act = 512, 256, 384, "swiglu"
    t = dev_tensors(make_inputs(M, H, I, act, seed=5))
    prob_full = m.problem(M, H, I, act)
    z = lambda *s: torch.zeros(*s, dtype=torch.float32, device="cuda")  # noqa: E731
    full = {"dWg": z(I, H), "dWu": z(I, H), "dWd": z(H, I)}
    m.mlp_bwd_recompute(prob_full, t["dout"], t["x"], t["Wg"], t["Wu"], t["Wd"], None,
                        full["dWg"], full["dWu"], full["dWd"], fuse_grad_accum=True)
    half = {"dWg": z(I, H), "dWu": z(I, H), "dWd": z(H, I)}
    for sl in (slice(0, 200), slice(200, M)):
        n = sl.stop - sl.start
        prob = m.problem(n, H, I, act)
        m.mlp_bwd_recompute(prob, t["dout"][sl].contiguous(), t["x"][sl].contiguous(), t["Wg"],
                            t["Wu"], t["Wd"], None, half["dWg"], half["dWu"], half["dWd"],
                            fuse_grad_accum=True)
    torch.cuda.synchronize()
    for k in full:
        assert rel_err(to_f64(half[k]), to_f64(full[k])) < 1e-5, k


@pytest.mark.parametrize("tile_policy", [0, 1], indirect=True)
@pytest.mark.parametrize("act,mode", [("swiglu", "saved"), ("swiglu", "recompute"),
                                      ("relu_sq", "recompute")])
def test_wgrad_split_k_accumulate(act, mode, tile_policy):
    """Many tokens and small weights: the weight-gradient tiles cannot fill
    the GPU, so the token reduction is split into work units whose fp32
    partial sums meet by atomic adds in the pre-existing gradients.  The
    launch plan confirms the split; the result is held to the fp32 bound."""
    M, H, I = 8192, 256, 384
    prob = m.problem(M, H, I, act, 1.125, 2.0)
    pmode = m.MODE_BWD_RECOMPUTE if mode == "recompute" else m.MODE_BWD
    plan = m.mlp_plan(prob, pmode, fuse_grad_accum=True)
    assert plan["wgrad_split"] > 1, plan
    assert m.mlp_plan(prob, pmode, fuse_grad_accum=False)["wgrad_split"] == 1
    t = make_inputs(M, H, I, act, seed=15, dW_prev=True)
    tc = {k: v for k, v in t.items() if not k.endswith("_prev")}
    prev = {k: v for k, v in t.items() if k.endswith("_prev")}
    got, bad, _ = run_gpu(dev_tensors(tc), M, H, I, act, 1.125, 2.0, mode=mode, fuse=True,
                          dW_prev=prev)
    assert not bad
    errs = compare_full(got, oracle_full(tc, act, 1.125, 2.0, dW_prev=prev), fuse=True)


def test_device_status_ok_and_errors():
    M, H, I = 64, 128, 352
    t = dev_tensors(make_inputs(M, H, I, "swiglu"))
    prob = m.problem(M, H, I)
    out = torch.empty(M, H, dtype=torch.bfloat16, device="cuda")
    ws = m.alloc_workspace(prob, m.MODE_INFER)
    m.mlp_fwd_infer(prob, t["x"], t["Wg"], t["Wu"], t["Wd"], out, ws=ws)
    assert m.mlp_device_status(ws) == 0
    # workspace too small
    with pytest.raises(m.MlpError) as e:
        m.mlp_fwd_infer(prob, t["x"], t["Wg"], t["Wu"], t["Wd"], out, ws=ws[:1024])
    assert e.value.code == -4
    # misaligned input pointer (offset by one element = 2 bytes)
    xb = torch.empty(M * H + 8, dtype=torch.bfloat16, device="cuda")
    xmis = xb[1:1 + M * H].view(M, H)
    with pytest.raises(m.MlpError) as e:
        m.mlp_fwd_infer(prob, xmis, t["Wg"], t["Wu"], t["Wd"], out, ws=ws)
    assert e.value.code == -2
    # non-gated activation with an up weight
    with pytest.raises(m.MlpError) as e:
        m.mlp_fwd_infer(m.problem(M, H, I, "relu_sq"), t["x"], t["Wg"], t["Wu"], t["Wd"], out)
    assert e.value.code == -1


# ------------------------------------------------------------- full sizes (sampled)

@pytest.mark.parametrize("name", ["llama7b_swiglu", "falcon_h1_swiglu", "nanogpt_relu_sq",
                                  "llama3_8b_swiglu"])
def test_full_size_sampled(name):
    """The pages' shapes at full size, in the launch configuration the
    benchmark times; parity on sampled token rows (out, dx) and sampled
    intermediate units (rows of dWg/dWu, columns of dWd, each reduced over
    all M tokens), computed exactly by the oracle."""
    w = WORKLOADS[name]
    t = workload_inputs(w)
    tc = {k: v for k, v in t.items() if not k.endswith("_prev")}
    prev = {k: v for k, v in t.items() if k.endswith("_prev")} if w.fuse_grad_accum else None
    mode = "recompute" if w.recompute else "saved"
    got, bad, _ = run_gpu(dev_tensors(tc), w.M, w.H, w.I, w.act, w.gate_mult, w.down_mult,
                          mode=mode, fuse=w.fuse_grad_accum, dW_prev=prev)
    assert not bad
    rows = spread_sample(w.M, SAMPLE_ROWS)
    cols = spread_sample(w.I, SAMPLE_UNITS)
    r, c = oracle_sampled(tc, w.act, w.gate_mult, w.down_mult, rows, cols, dW_prev=prev)
    tol_w = TOL_F32 if w.fuse_grad_accum else TOL_BF16
    errs = {
        "out": rel_err(to_f64(got["out"][torch.as_tensor(rows)]), r["out"]),
        "dx": rel_err(to_f64(got["dx"][torch.as_tensor(rows)]), r["dx"]),
        "dWg": rel_err(to_f64(got["dWg"][torch.as_tensor(cols)]), c["dWg"]),
        "dWd": rel_err(to_f64(got["dWd"][:, torch.as_tensor(cols)]), c["dWd"]),
    }
    if w.gated:
        errs["dWu"] = rel_err(to_f64(got["dWu"][torch.as_tensor(cols)]), c["dWu"])
    for k, e in errs.items():
        tol = tol_w if k.startswith("dW") else TOL_BF16
        assert e <= tol, (name, k, errs)
    for k in ("out", "dx", "dWg", "dWd"):
        assert torch.isfinite(got[k].float()).all(), k
    if w.infer:
        out2 = torch.empty_like(got["out"])
        dt = dev_tensors(tc)
        m.mlp_fwd_infer(m.problem(w.M, w.H, w.I, w.act, w.gate_mult, w.down_mult),
                        dt["x"], dt["Wg"], dt["Wu"], dt["Wd"], out2)
        torch.cuda.synchronize()
        assert torch.equal(out2, got["out"])


@pytest.mark.parametrize("tile_policy", [1, 2], indirect=True)
@pytest.mark.parametrize("act", ["relu", "reglu", "geglu", "glu"])
@pytest.mark.parametrize("shape", [(64, 128, 352), (300, 200, 392)])
@pytest.mark.parametrize("mode,fuse", [("saved", False), ("recompute", True)])
def test_more_activations_parity(act, shape, mode, fuse, tile_policy):
    """The further activations of quack's Activation literal (relu, and the
    gated reglu, geglu, glu) through the same kernels."""
    M, H, I = shape
    t = make_inputs(M, H, I, act, seed=8, dW_prev=fuse)
    tc = {k: v for k, v in t.items() if not k.endswith("_prev")}
    prev = {k: v for k, v in t.items() if k.endswith("_prev")} if fuse else None
    got, bad, _ = run_gpu(dev_tensors(tc), M, H, I, act, 1.125, 2.0, mode=mode, fuse=fuse,
                          dW_prev=prev)
    assert not bad
    ref = oracle_full(tc, act, 1.125, 2.0, dW_prev=prev)
    compare_full(got, ref, fuse,
                 floor=dw_floor(tc, act, 1.125, 2.0, mode, ref, prev) if fuse else None)


@pytest.mark.parametrize("act", ["reglu", "glu", "relu"])
def test_dwd_only_postact_kernel(act):
    # only dWd requested in saved mode: the elementwise postact kernel path
    M, H, I = 200, 136, 264
    t = make_inputs(M, H, I, act, seed=9)
    got, bad, _ = run_gpu(dev_tensors(t), M, H, I, act, 1.125, 2.0, mode="saved", want=("dWd",))
    assert not bad
    compare_full(got, oracle_full(t, act, 1.125, 2.0), fuse=False)


# ------------------------------------------------ decode-sized token counts

@pytest.mark.parametrize("act", ["swiglu", "relu_sq"])
@pytest.mark.parametrize("M", [1, 16, 64, 200])
def test_small_m_split_k(act, M):
    """Few tokens: the down projection (and dx) split K so that their few
    output tiles still use the whole GPU; the partial sums meet in fp32.
    (1 token takes the weight-streaming forward, then the split dx.)"""
    H, I = 512, 2048  # 2 output tiles per 128 rows, K = 2048 (forward), 4096 (gated dx)
    t = make_inputs(M, H, I, act, seed=12)
    got, bad, _ = run_gpu(dev_tensors(t), M, H, I, act, 1.125, 2.0, mode="recompute")
    assert not bad
    compare_full(got, oracle_full(t, act, 1.125, 2.0), fuse=False)
    # the inference path agrees bitwise with the training forward
    d = dev_tensors(t)
    o2 = torch.empty(M, H, dtype=torch.bfloat16, device="cuda")
    m.mlp_fwd_infer(m.problem(M, H, I, act, 1.125, 2.0), d["x"], d["Wg"], d["Wu"], d["Wd"], o2)
    torch.cuda.synchronize()
    assert rel_err(to_f64(o2), to_f64(got["out"])) < 1e-2


@pytest.mark.parametrize("act", ["swiglu", "relu_sq"])
def test_forward_split_k_fills_a_partial_wave(act):
    """640 tokens with H = 2048: the down projection's 24 output tiles of
    256 x 256 would occupy a third of the 76 CTA pairs, so the forward splits
    K three ways (72 units, 95 % of one wave) and runs as two launches; the
    backward's dx stays whole.  Against the oracle, the training forward with
    its saved preacts and the backward from them."""
    M, H, I = 640, 2048, 4096
    prob = m.problem(M, H, I, act, 1.125, 2.0)
    assert m.mlp_plan(prob, m.MODE_INFER)["out_split"] == 3
    assert m.mlp_plan(prob, m.MODE_FWD)["out_split"] == 3
    assert m.mlp_plan(prob, m.MODE_BWD)["out_split"] == 1
    assert m.mlp_plan(prob, m.MODE_FWD)["fused_forward"] == 0
    t = make_inputs(M, H, I, act, seed=14)
    got, bad, _ = run_gpu(dev_tensors(t), M, H, I, act, 1.125, 2.0, mode="saved")
    assert not bad
    compare_full(got, oracle_full(t, act, 1.125, 2.0), fuse=False)


def test_inference_forward_in_a_cuda_graph():
    """mlp_fwd_infer captured into a CUDA graph (after one direct call has
    set up the library's caches) replays to the direct call's result.  At
    this token count the down projection splits K, and the fp32 partial sums
    meet through atomic adds in no fixed order, so the replays agree with the
    direct call to rounding, not bitwise."""
    M, H, I = 16, 1024, 4096
    t = dev_tensors(make_inputs(M, H, I, "swiglu", seed=13))
    prob = m.problem(M, H, I)
    ws = m.alloc_workspace(prob, m.MODE_INFER)
    ref = torch.empty(M, H, dtype=torch.bfloat16, device="cuda")
    out = torch.zeros_like(ref)
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        m.mlp_fwd_infer(prob, t["x"], t["Wg"], t["Wu"], t["Wd"], ref, ws=ws)
    torch.cuda.current_stream().wait_stream(s)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        m.mlp_fwd_infer(prob, t["x"], t["Wg"], t["Wu"], t["Wd"], out, ws=ws)
    for _ in range(3):
        out.zero_()
        g.replay()
        torch.cuda.synchronize()
        assert torch.isfinite(out.float()).all()
        assert rel_err(to_f64(out), to_f64(ref)) < 1e-2
    assert m.mlp_device_status(ws) == 0


def test_training_backward_in_a_cuda_graph():
    """mlp_bwd forks the weight gradients onto the library's second stream
    and joins them back; captured into a CUDA graph (after a direct call has
    created that stream and the caches) the fork and join become graph
    edges, and replays give the direct call's weight gradients bitwise and
    its dx to rounding (dx splits K at this size)."""
    M, H, I, act = 512, 512, 1024, "swiglu"
    t = dev_tensors(make_inputs(M, H, I, act, seed=14))
    prob = m.problem(M, H, I, act)
    bf = torch.bfloat16
    G = torch.empty(M, I, dtype=bf, device="cuda")
    U = torch.empty(M, I, dtype=bf, device="cuda")
    out = torch.empty(M, H, dtype=bf, device="cuda")
    wsf = m.alloc_workspace(prob, m.MODE_FWD)
    wsb = m.alloc_workspace(prob, m.MODE_BWD)

    def step(res):
        m.mlp_fwd(prob, t["x"], t["Wg"], t["Wu"], t["Wd"], out, G, U, ws=wsf)
        m.mlp_bwd(prob, t["dout"], t["x"], t["Wg"], t["Wu"], t["Wd"], G, U, res["dx"],
                  res["dWg"], res["dWu"], res["dWd"], ws=wsb)

    def bufs():
        return {"dx": torch.empty(M, H, dtype=bf, device="cuda"),
                "dWg": torch.empty(I, H, dtype=bf, device="cuda"),
                "dWu": torch.empty(I, H, dtype=bf, device="cuda"),
                "dWd": torch.empty(H, I, dtype=bf, device="cuda")}
    ref, got = bufs(), bufs()
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        step(ref)
    torch.cuda.current_stream().wait_stream(s)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        step(got)
    for _ in range(2):
        for v in got.values():
            v.fill_(float("nan"))
        g.replay()
        torch.cuda.synchronize()
        for k in ref:
            assert torch.isfinite(got[k].float()).all(), k
            if k == "dx":  # split K at this size: fp32 partial sums meet in no fixed order
                assert rel_err(to_f64(got[k]), to_f64(ref[k])) < 1e-2, k
            else:
                assert torch.equal(got[k], ref[k]), k
    assert m.mlp_device_status(wsb) == 0
