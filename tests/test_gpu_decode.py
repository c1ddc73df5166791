"""GPU parity of the decode-sized forward (one to four tokens), which streams
the weights on the CUDA cores, against the fp64 oracle, through the C ABI.

The same guard bands and NaN-filled outputs as the other parity tests; the
training forward's saved preacts (G, U) come from the same kernel."""
import pytest
import torch

import activated_mlp_gemms_gb300 as m
from activated_mlp_gemms_gb300.workloads import make_inputs, to_f64
from mlp_gpu_helpers import compare_full, dev_tensors, oracle_full, run_gpu
from oracle import mlp_forward, rel_err

pytestmark = pytest.mark.gpu

ACTS = ["swiglu", "relu_sq", "gelu_tanh_approx", "relu", "reglu", "geglu", "glu"]


@pytest.mark.parametrize("act", ACTS)
@pytest.mark.parametrize("M", [1, 2, 3, 4, 5])
def test_decode_forward_parity(act, M):
    """K = 1000 (a ragged last load group), I = 1544 rows (a ragged last
    round of rows); the forward saves G/U, the backward then runs on the
    tensor cores from them.  M = 5 takes the tensor-core forward."""
    H, I = 1000, 1544
    t = make_inputs(M, H, I, act, seed=31)
    got, bad, _ = run_gpu(dev_tensors(t), M, H, I, act, 1.125, 2.0, mode="saved")
    assert not bad
    compare_full(got, oracle_full(t, act, 1.125, 2.0), fuse=False)


@pytest.mark.parametrize("act", ["swiglu", "relu_sq"])
@pytest.mark.parametrize("M", [1, 2, 3, 4])
def test_decode_inference_long_k(act, M):
    """Long rows (H = 4096 for gate/up, I = 5504 for the down projection),
    against the oracle and the tensor-core path."""
    H, I = 4096, 5504
    t = make_inputs(M, H, I, act, seed=32)
    d = dev_tensors(t)
    prob = m.problem(M, H, I, act, 0.5, 1.5)
    out = torch.full((M, H), float("nan"), dtype=torch.bfloat16, device="cuda")
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


def test_decode_path_is_two_kernels_and_graph_capturable():
    """The decode forward launches the two weight-streaming kernels (traced
    as gate_up_act and down_proj), and replays of a CUDA graph of it are
    bitwise equal to the direct call (no atomics, fixed reduction order)."""
    M, H, I = 2, 2048, 5632
    t = dev_tensors(make_inputs(M, H, I, "swiglu", seed=33))
    prob = m.problem(M, H, I)
    ws = m.alloc_workspace(prob, m.MODE_INFER)
    ref = torch.empty(M, H, dtype=torch.bfloat16, device="cuda")
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


@pytest.mark.parametrize("M,I,path", [(3, 14336, ["gate_up_act", "down_proj"]),
                                      (4, 14336, ["gate_up_act", "down_proj"]),
                                      (4, 16384, None)])
def test_decode_token_rows_must_fit_shared_memory(M, I, path):
    """With Llama-3-8B's intermediate size (14336) up to four token rows of
    the postact (112 KiB) fit a CTA's shared memory and take the
    weight-streaming kernels; four rows of 16384 do not and take the tensor
    cores (a split-K down projection, then its fp32 -> bf16 pass)."""
    H = 4096
    t = make_inputs(M, H, I, "swiglu", seed=34)
    d = dev_tensors(t)
    prob = m.problem(M, H, I)
    out = torch.full((M, H), float("nan"), dtype=torch.bfloat16, device="cuda")
    m.mlp_trace_read()
    m.mlp_trace_enable(True)
    try:
        ws = m.mlp_fwd_infer(prob, d["x"], d["Wg"], d["Wu"], d["Wd"], out)
        torch.cuda.synchronize()
    finally:
        m.mlp_trace_enable(False)
    names = [n for n, _ in m.mlp_trace_read()]
    if path is not None:
        assert names == path, names
    else:
        assert names == ["gate_up_act", "down_proj", "convert"], names
    assert m.mlp_device_status(ws) == 0
    a = {k: to_f64(v) for k, v in t.items() if v is not None}
    ref = mlp_forward(a["x"], a["Wg"], a["Wu"], a["Wd"], "swiglu")["out"]
    assert rel_err(to_f64(out), ref) <= 2e-2


def test_decode_four_tokens_of_a_wide_intermediate():
    """Four tokens with I = 14336 (the Llama-3-8B width): 112 KiB of staged
    token rows for the down projection, still on the CUDA cores, against the
    oracle and bitwise against a second call."""
    M, H, I = 4, 1024, 14336
    t = make_inputs(M, H, I, "swiglu", seed=33)
    d = dev_tensors(t)
    prob = m.problem(M, H, I)
    assert m.mlp_plan(prob, m.MODE_INFER)["decode"] == 1
    out = torch.empty(M, H, dtype=torch.bfloat16, device="cuda")
    out2 = torch.empty_like(out)
    m.mlp_fwd_infer(prob, d["x"], d["Wg"], d["Wu"], d["Wd"], out)
    m.mlp_fwd_infer(prob, d["x"], d["Wg"], d["Wu"], d["Wd"], out2)
    torch.cuda.synchronize()
    a = {k: to_f64(v) for k, v in t.items() if v is not None}
    ref = mlp_forward(a["x"], a["Wg"], a["Wu"], a["Wd"], "swiglu")["out"]
    assert rel_err(to_f64(out), ref) <= 2e-2
    assert torch.equal(out, out2)
