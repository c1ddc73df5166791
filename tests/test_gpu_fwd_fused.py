"""The gated forward in one launch (gate/up tiles, then each 256-row block's
down tiles once its postact is stored) against the same forward as two
launches (tile policy 3) and against the fp64 oracle, through the C ABI.

Both schedules run the same tile computations in the same accumulation
order, so their outputs are bitwise equal; the oracle comparison is the
parity bar of the other tests."""
import time

import pytest
import torch

import activated_mlp_gemms_gb300 as m
from activated_mlp_gemms_gb300.workloads import make_inputs, to_f64
from mlp_gpu_helpers import TOL_BF16, dev_tensors, guard_intact, guarded
from oracle import block_forward, mlp_forward, rel_err

pytestmark = pytest.mark.gpu

GATED = ["swiglu", "reglu", "geglu", "glu"]


def _forward(prob, d, M, H, I, save, policy):
    bf = torch.bfloat16
    out, out_f = guarded((M, H), bf)
    G, G_f = guarded((M, I), bf)
    U, U_f = guarded((M, I), bf)
    m.mlp_set_tile_policy(policy)
    m.mlp_trace_read()
    m.mlp_trace_enable(True)
    try:
        ws = m.mlp_fwd(prob, d["x"], d["Wg"], d["Wu"], d["Wd"], out, G if save else None,
                       U if save else None)
        torch.cuda.synchronize()
    finally:
        m.mlp_trace_enable(False)
        m.mlp_set_tile_policy(0)
    names = [n for n, _ in m.mlp_trace_read()]
    assert m.mlp_device_status(ws) == 0
    assert guard_intact(out_f) and guard_intact(G_f) and guard_intact(U_f)
    return out, (G if save else None), (U if save else None), names


@pytest.mark.parametrize("act", GATED)
@pytest.mark.parametrize("M,H,I", [(300, 200, 392), (1000, 2568, 1544), (2048 + 77, 520, 1160)])
def test_fused_forward_equals_two_launches_and_the_oracle(act, M, H, I):
    """Ragged token blocks (M not a multiple of 256), a ragged last gate/up
    tile (I not a multiple of 128) and a ragged last down tile (H not a
    multiple of 256).  (Shapes whose down projection would split K keep the
    two launches: few output tiles and a long K, or at most 38 output tiles
    of 256 x 256, half the GPU's CTA pairs.)"""
    t = make_inputs(M, H, I, act, seed=41)
    d = dev_tensors(t)
    prob = m.problem(M, H, I, act, 1.125, 2.0)
    out, G, U, names = _forward(prob, d, M, H, I, True, 0)
    assert names == ["fwd_fused"], names
    out2, G2, U2, names2 = _forward(prob, d, M, H, I, True, 3)
    assert names2 == ["gate_up_act", "down_proj"], names2
    assert torch.equal(out, out2) and torch.equal(G, G2) and torch.equal(U, U2)
    a = {k: to_f64(v) for k, v in t.items() if v is not None}
    ref = mlp_forward(a["x"], a["Wg"], a["Wu"], a["Wd"], act, 1.125, 2.0)
    assert rel_err(to_f64(out), ref["out"]) <= TOL_BF16
    assert rel_err(to_f64(G), ref["g"]) <= TOL_BF16
    assert rel_err(to_f64(U), ref["u"]) <= TOL_BF16


@pytest.mark.parametrize("M,I", [(129, 960), (256, 960), (4096, 2816)])
def test_fused_inference_forward(M, I):
    """The no-grad forward (no G/U stores) takes the fused launch too; one
    256-row block (every down tile waits for all gate/up tiles) and many."""
    H = 1024
    t = make_inputs(M, H, I, "swiglu", seed=42)
    d = dev_tensors(t)
    prob = m.problem(M, H, I, "swiglu", 1.0, 1.0)
    outs = []
    for policy, want in ((0, ["fwd_fused"]), (3, ["gate_up_act", "down_proj"])):
        out = torch.full((M, H), float("nan"), dtype=torch.bfloat16, device="cuda")
        m.mlp_set_tile_policy(policy)
        m.mlp_trace_read()
        m.mlp_trace_enable(True)
        try:
            ws = m.mlp_fwd_infer(prob, d["x"], d["Wg"], d["Wu"], d["Wd"], out)
            torch.cuda.synchronize()
        finally:
            m.mlp_trace_enable(False)
            m.mlp_set_tile_policy(0)
        assert [n for n, _ in m.mlp_trace_read()] == want
        assert m.mlp_device_status(ws) == 0
        outs.append(out)
    assert torch.equal(outs[0], outs[1])
    a = {k: to_f64(v) for k, v in t.items() if v is not None}
    ref = mlp_forward(a["x"], a["Wg"], a["Wu"], a["Wd"], "swiglu", 1.0, 1.0)["out"]
    assert rel_err(to_f64(outs[0]), ref) <= TOL_BF16


def test_fused_block_forward():
    """The block's forward: the RMS norm's scale on the gate/up tiles and the
    residual add in the down tiles, fused the same way."""
    M, H, I = 1000, 2560, 1408
    kw = dict(resid_lambda=1.1 ** 0.5, post_lambda=0.8, eps=2.0 ** -7)
    t = make_inputs(M, H, I, "swiglu", seed=43)
    d = dev_tensors(t)
    prob = m.problem(M, H, I, "swiglu", 1.0, 1.0)
    blk = m.block(**kw)
    ys = []
    for policy, want in ((0, ["rstd", "fwd_fused"]), (3, ["rstd", "gate_up_act", "down_proj"])):
        y = torch.full((M, H), float("nan"), dtype=torch.bfloat16, device="cuda")
        m.mlp_set_tile_policy(policy)
        m.mlp_trace_read()
        m.mlp_trace_enable(True)
        try:
            _, ws = m.mlp_block_fwd(prob, blk, d["x"], d["Wg"], d["Wu"], d["Wd"], y)
            torch.cuda.synchronize()
        finally:
            m.mlp_trace_enable(False)
            m.mlp_set_tile_policy(0)
        assert [n for n, _ in m.mlp_trace_read()] == want
        assert m.mlp_device_status(ws) == 0
        ys.append(y)
    assert torch.equal(ys[0], ys[1])
    a = {k: to_f64(v) for k, v in t.items() if v is not None}
    ref = block_forward(a["x"], a["Wg"], a["Wu"], a["Wd"], "swiglu", gate_mult=1.0,
                        down_mult=1.0, **kw)["y"]
    assert rel_err(to_f64(ys[0]), ref) <= TOL_BF16


def test_fused_forward_graph_replays():
    """Captured in a CUDA graph, replays of the fused forward (its block
    counts reset by each call's control-block clear) give the direct call's
    result bitwise."""
    M, H, I = 2048, 1280, 2816
    d = dev_tensors(make_inputs(M, H, I, "swiglu", seed=44))
    prob = m.problem(M, H, I)
    ws = m.alloc_workspace(prob, m.MODE_FWD)
    ref = torch.empty(M, H, dtype=torch.bfloat16, device="cuda")
    m.mlp_fwd(prob, d["x"], d["Wg"], d["Wu"], d["Wd"], ref, ws=ws)
    torch.cuda.synchronize()
    out = torch.zeros_like(ref)
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        m.mlp_fwd(prob, d["x"], d["Wg"], d["Wu"], d["Wd"], out, ws=ws)
    torch.cuda.current_stream().wait_stream(s)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        m.mlp_fwd(prob, d["x"], d["Wg"], d["Wu"], d["Wd"], out, ws=ws)
    for _ in range(3):
        out.zero_()
        g.replay()
        torch.cuda.synchronize()
        assert torch.equal(out, ref)
    assert m.mlp_device_status(ws) == 0


def test_fused_forward_with_most_sms_held_by_another_stream():
    """The one-launch forward when only part of its grid is resident: a
    kernel on another stream keeps all but 40 SMs busy for 400 ms, far longer
    than the 100 ms bound put on the forward's waits.  Every work unit is
    claimed from the scheduler's counter, so the down units only wait for
    gate/up tiles that resident CTA pairs have claimed: the forward completes
    on the free SMs, with status 0 and the same output as without
    contention.  (With a unit per pair fixed in advance, the pairs that are
    not resident would own gate/up tiles the down units wait for, and the
    waits would expire.)"""
    M, H, I, act = 2048, 1280, 4096, "swiglu"
    t = make_inputs(M, H, I, act, seed=44)
    d = dev_tensors(t)
    prob = m.problem(M, H, I, act)
    assert m.mlp_plan(prob, m.MODE_FWD)["fused_forward"] == 1
    ref = torch.empty(M, H, dtype=torch.bfloat16, device="cuda")
    m.mlp_fwd_infer(prob, d["x"], d["Wg"], d["Wu"], d["Wd"], ref)
    torch.cuda.synchronize()
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    hold = torch.cuda.Stream()
    work = torch.cuda.Stream()
    out = torch.full((M, H), float("nan"), dtype=torch.bfloat16, device="cuda")
    ws = m.alloc_workspace(prob, m.MODE_INFER)
    torch.cuda.synchronize()
    try:
        m.mlp_set_wait_timeout_ms(100)
        m.mlp_debug_hold_sms(sms - 40, 400_000, stream=hold)
        time.sleep(0.02)  # the holding CTAs are resident before the forward starts
        with torch.cuda.stream(work):
            m.mlp_fwd_infer(prob, d["x"], d["Wg"], d["Wu"], d["Wd"], out, ws=ws, stream=work)
        work.synchronize()
        status = m.mlp_device_status(ws, stream=work)
        hold_busy = not hold.query()  # the holder was still running when the forward ended
        torch.cuda.synchronize()
    finally:
        m.mlp_set_wait_timeout_ms(0)
    assert hold_busy, "the forward did not overlap the holding kernel"
    assert status == 0, m.mlp_status_string(status)
    assert torch.equal(out, ref)
