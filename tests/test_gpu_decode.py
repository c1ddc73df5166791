"""GPU parity of the decode-sized forward (one to sixteen tokens), which
streams the weights instead of running GEMM tiles, against the fp64 oracle,
through the C ABI.

Two weight streams: the warp-MMA one (three to eight tokens by default, up
to sixteen when forced) and the CUDA-core one (one or two tokens by default,
up to four whose rows fit shared memory when forced); the debug flags force
either.  From nine tokens on the library takes the tensor-core GEMMs.  The same guard bands and NaN-filled outputs as the
other parity tests; the training forward's saved preacts (G, U) come from
the same kernels."""
import contextlib

import pytest
import torch

import activated_mlp_gemms_gb300 as m
from activated_mlp_gemms_gb300.workloads import make_inputs, to_f64
from mlp_gpu_helpers import compare_full, dev_tensors, oracle_full, run_gpu
from oracle import mlp_forward, rel_err

pytestmark = pytest.mark.gpu

PLAN_MMA, PLAN_FMA, PLAN_TC = 2, 1, 0


@contextlib.contextmanager
def decode_kernel(kind):
    """kind "mma" or "fma": force that weight stream; others: the default choice."""
    m.mlp_debug_set_flags({"fma": m.DEBUG_DECODE_FMA, "mma": m.DEBUG_DECODE_MMA}.get(kind, 0))
    try:
        yield
    finally:
        m.mlp_debug_set_flags(0)


ACTS = ["swiglu", "relu_sq", "gelu_tanh_approx", "relu", "reglu", "geglu", "glu"]


@pytest.mark.parametrize("act", ACTS)
@pytest.mark.parametrize("M,kind", [(1, "mma"), (2, "mma"), (3, "mma"), (4, "mma"), (5, "mma"),
                                    (8, "mma"), (9, "mma"), (16, "mma"), (9, "tc"), (17, "tc"),
                                    (1, "fma"), (2, "fma"), (3, "fma"), (4, "fma")])
def test_decode_forward_parity(act, M, kind):
    """K = 1000 (a ragged last load group), I = 1544 rows (a ragged last
    16-row block; the down pass: K = 1544, 1000 rows); the forward saves
    G/U, the backward then runs on the tensor cores from them.  Without a
    flag M = 9 and M = 17 take the tensor-core GEMMs."""
    H, I = 1000, 1544
    t = make_inputs(M, H, I, act, seed=31)
    with decode_kernel(kind):
        want = {"mma": PLAN_MMA, "fma": PLAN_FMA, "tc": PLAN_TC}[kind]
        assert m.mlp_plan(m.problem(M, H, I, act), m.MODE_FWD)["decode"] == want
        got, bad, _ = run_gpu(dev_tensors(t), M, H, I, act, 1.125, 2.0, mode="saved")
    assert not bad
    compare_full(got, oracle_full(t, act, 1.125, 2.0), fuse=False)


@pytest.mark.parametrize("act", ["swiglu", "relu_sq"])
@pytest.mark.parametrize("M,kind", [(1, "mma"), (4, "mma"), (7, "mma"), (12, "mma"), (16, "mma"),
                                    (1, "fma"), (2, "fma"), (3, "fma"), (4, "fma")])
def test_decode_inference_long_k(act, M, kind):
    """Long rows (H = 4096 for gate/up, I = 5504 for the down projection),
    against the oracle and the tensor-core path."""
    H, I = 4096, 5504
    t = make_inputs(M, H, I, act, seed=32)
    d = dev_tensors(t)
    prob = m.problem(M, H, I, act, 0.5, 1.5)
    out = torch.full((M, H), float("nan"), dtype=torch.bfloat16, device="cuda")
    with decode_kernel(kind):
        ws = m.mlp_fwd_infer(prob, d["x"], d["Wg"], d["Wu"], d["Wd"], out)
    torch.cuda.synchronize()
    assert m.mlp_device_status(ws) == 0
    a = {k: to_f64(v) for k, v in t.items()}
    ref = mlp_forward(a["x"], a["Wg"], a["Wu"], a["Wd"], act, 0.5, 1.5)["out"]
    assert rel_err(to_f64(out), ref) <= 2e-2
    # the tensor-core path (forced by a tile policy) on the same inputs
    tc = torch.full_like(out, float("nan"))
    m.mlp_set_tile_policy(1)
    try:
        m.mlp_fwd_infer(prob, d["x"], d["Wg"], d["Wu"], d["Wd"], tc)
        torch.cuda.synchronize()
    finally:
        m.mlp_set_tile_policy(0)
    assert rel_err(to_f64(out), to_f64(tc)) <= 1e-2


@pytest.mark.parametrize("M,kind", [(2, "mma"), (13, "mma"), (2, "fma")])
def test_decode_path_is_two_kernels_and_graph_capturable(M, kind):
    """The decode forward launches the two weight-streaming kernels (traced
    as gate_up_act and down_proj), and replays of a CUDA graph of it are
    bitwise equal to the direct call (no atomics, fixed reduction order)."""
    H, I = 2048, 5632
    t = dev_tensors(make_inputs(M, H, I, "swiglu", seed=33))
    prob = m.problem(M, H, I)
    ws = m.alloc_workspace(prob, m.MODE_INFER)
    ref = torch.empty(M, H, dtype=torch.bfloat16, device="cuda")
    with decode_kernel(kind):
        m.mlp_trace_read()
        m.mlp_trace_enable(True)
        try:
            m.mlp_fwd_infer(prob, t["x"], t["Wg"], t["Wu"], t["Wd"], ref, ws=ws)
            torch.cuda.synchronize()
        finally:
            m.mlp_trace_enable(False)
        assert [n for n, _ in m.mlp_trace_read()] == ["gate_up_act", "down_proj"]
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
            assert torch.equal(out, ref)


@pytest.mark.parametrize("M,I,plan", [(1, 14336, PLAN_FMA), (2, 14336, PLAN_FMA),
                                      (2, 32768, PLAN_MMA), (3, 14336, PLAN_MMA),
                                      (8, 14336, PLAN_MMA), (9, 14336, PLAN_TC),
                                      (16, 14336, PLAN_TC), (17, 14336, PLAN_TC)])
def test_default_decode_stream(M, I, plan):
    """Without a flag: the CUDA-core stream for one or two tokens whose rows
    fit shared memory, the warp-MMA one for the others up to eight, then the
    tensor-core GEMMs; a tile policy keeps every size on the GEMMs."""
    prob = m.problem(M, 4096, I)
    assert m.mlp_plan(prob, m.MODE_INFER)["decode"] == plan
    assert m.mlp_plan(prob, m.MODE_FWD)["decode"] == plan
    m.mlp_set_tile_policy(1)
    try:
        assert m.mlp_plan(prob, m.MODE_INFER)["decode"] == PLAN_TC
    finally:
        m.mlp_set_tile_policy(0)


@pytest.mark.parametrize("M,I,plan", [(3, 14336, PLAN_FMA), (4, 14336, PLAN_FMA),
                                      (4, 16384, PLAN_MMA), (5, 14336, PLAN_MMA)])
def test_cuda_core_stream_needs_its_token_rows_in_shared_memory(M, I, plan):
    """Asked for, the CUDA-core stream takes up to four token rows of
    Llama-3-8B's intermediate size (14336: 112 KiB of staged rows); four
    rows of 16384, or five tokens, do not fit and take the warp-MMA stream,
    which reads the token rows through the caches."""
    H = 4096
    t = make_inputs(M, H, I, "swiglu", seed=34)
    d = dev_tensors(t)
    prob = m.problem(M, H, I)
    out = torch.full((M, H), float("nan"), dtype=torch.bfloat16, device="cuda")
    with decode_kernel("fma"):
        assert m.mlp_plan(prob, m.MODE_INFER)["decode"] == plan
        m.mlp_trace_read()
        m.mlp_trace_enable(True)
        try:
            ws = m.mlp_fwd_infer(prob, d["x"], d["Wg"], d["Wu"], d["Wd"], out)
            torch.cuda.synchronize()
        finally:
            m.mlp_trace_enable(False)
    assert [n for n, _ in m.mlp_trace_read()] == ["gate_up_act", "down_proj"]
    assert m.mlp_device_status(ws) == 0
    a = {k: to_f64(v) for k, v in t.items() if v is not None}
    ref = mlp_forward(a["x"], a["Wg"], a["Wu"], a["Wd"], "swiglu")["out"]
    assert rel_err(to_f64(out), ref) <= 2e-2


@pytest.mark.parametrize("M,kind", [(4, "fma"), (16, "mma")])
def test_decode_at_llama3_8b_width(M, kind):
    """Llama-3-8B's gate/up and down shapes (H = 4096, I = 14336): four
    tokens on the CUDA-core stream (112 KiB of staged token rows), sixteen on
    the warp-MMA stream (forced: two 8-token blocks), against the oracle and
    bitwise against a second call; every output row checked."""
    H, I = 4096, 14336
    t = make_inputs(M, H, I, "swiglu", seed=35)
    d = dev_tensors(t)
    prob = m.problem(M, H, I)
    out = torch.empty(M, H, dtype=torch.bfloat16, device="cuda")
    out2 = torch.empty_like(out)
    with decode_kernel(kind):
        assert m.mlp_plan(prob, m.MODE_INFER)["decode"] == (PLAN_FMA if kind == "fma" else PLAN_MMA)
        m.mlp_fwd_infer(prob, d["x"], d["Wg"], d["Wu"], d["Wd"], out)
        m.mlp_fwd_infer(prob, d["x"], d["Wg"], d["Wu"], d["Wd"], out2)
        torch.cuda.synchronize()
    a = {k: to_f64(v) for k, v in t.items() if v is not None}
    ref = mlp_forward(a["x"], a["Wg"], a["Wu"], a["Wd"], "swiglu")["out"]
    got = to_f64(out)
    for r in range(M):
        assert rel_err(got[r], ref[r]) <= 2e-2, r
    assert torch.equal(out, out2)


def test_warp_mma_stream_matches_the_cuda_core_stream():
    """Both weight streams on the same inputs (two tokens, a gated and a
    non-gated pass): the same sums up to fp32 rounding order."""
    for act in ("swiglu", "relu_sq"):
        M, H, I = 2, 1536, 4096
        t = dev_tensors(make_inputs(M, H, I, act, seed=36))
        prob = m.problem(M, H, I, act)
        outs = {}
        for kind in ("mma", "fma"):
            o = torch.empty(M, H, dtype=torch.bfloat16, device="cuda")
            with decode_kernel(kind):
                m.mlp_fwd_infer(prob, t["x"], t["Wg"], t["Wu"], t["Wd"], o)
            outs[kind] = o
        torch.cuda.synchronize()
        assert rel_err(to_f64(outs["mma"]), to_f64(outs["fma"])) <= 1e-2, act
