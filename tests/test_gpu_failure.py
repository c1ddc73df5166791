"""Failure detection on the GPU without a fault: every device-side wait is
bounded, so when the tile scheduler publishes no work (MLP_DEBUG_NO_WORK,
no copy and no MMA is ever issued) the consumers' waits expire, the kernels
record MLP_ERR_TIMEOUT in the status word and return.  The host reads the
status; the context stays usable and the next normal call is correct."""
import pytest
import torch

import activated_mlp_gemms_gb300 as m
from activated_mlp_gemms_gb300.workloads import make_inputs, to_f64
from oracle import mlp_forward, rel_err

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("policy", [1, 2])
def test_bounded_wait_expiry_reports_timeout_and_recovers(policy):
    M, H, I = 300, 256, 512
    t = make_inputs(M, H, I, "swiglu", seed=7)
    g = {k: (v.cuda() if v is not None else None) for k, v in t.items()}
    prob = m.problem(M, H, I)
    out = torch.zeros(M, H, dtype=torch.bfloat16, device="cuda")
    ws = m.alloc_workspace(prob, m.MODE_INFER)
    m.mlp_set_tile_policy(policy)
    try:
        m.mlp_set_wait_timeout_ms(100)
        m.mlp_debug_set_flags(m.DEBUG_NO_WORK)
        m.mlp_fwd_infer(prob, g["x"], g["Wg"], g["Wu"], g["Wd"], out, ws=ws)
        assert m.mlp_device_status(ws) == -6  # MLP_ERR_TIMEOUT
    finally:
        m.mlp_debug_set_flags(0)
        m.mlp_set_wait_timeout_ms(0)
    # the context is still usable: a normal call succeeds and is correct
    m.mlp_fwd_infer(prob, g["x"], g["Wg"], g["Wu"], g["Wd"], out, ws=ws)
    assert m.mlp_device_status(ws) == 0
    m.mlp_set_tile_policy(0)
    a = {k: to_f64(v) for k, v in t.items() if v is not None}
    ref = mlp_forward(a["x"], a["Wg"], a["Wu"], a["Wd"], "swiglu")["out"]
    assert rel_err(to_f64(out), ref) <= 2e-2


@pytest.mark.parametrize("Md,flag", [(1, 0), (4, 0), (2, "mma")])
def test_decode_call_clears_a_stale_timeout(Md, flag):
    """A decode-sized forward enqueues no memset of the control block: its
    first kernel clears the status word.  After a call that timed out on the
    same workspace, the decode call (both weight streams) must report 0."""
    M, H, I = 300, 256, 512
    t = make_inputs(M, H, I, "swiglu", seed=8)
    g = {k: (v.cuda() if v is not None else None) for k, v in t.items()}
    prob = m.problem(M, H, I)
    out = torch.zeros(M, H, dtype=torch.bfloat16, device="cuda")
    ws = m.alloc_workspace(prob, m.MODE_INFER)
    try:
        m.mlp_set_wait_timeout_ms(100)
        m.mlp_debug_set_flags(m.DEBUG_NO_WORK)
        m.mlp_fwd_infer(prob, g["x"], g["Wg"], g["Wu"], g["Wd"], out, ws=ws)
        assert m.mlp_device_status(ws) == -6  # MLP_ERR_TIMEOUT
    finally:
        m.mlp_debug_set_flags(0)
        m.mlp_set_wait_timeout_ms(0)
    probd = m.problem(Md, H, I)
    assert m.mlp_workspace_size(probd, m.MODE_INFER) <= ws.numel()
    outd = torch.empty(Md, H, dtype=torch.bfloat16, device="cuda")
    m.mlp_debug_set_flags(m.DEBUG_DECODE_MMA if flag == "mma" else 0)
    try:
        assert m.mlp_plan(probd, m.MODE_INFER)["decode"] in (1, 2)
        m.mlp_fwd_infer(probd, g["x"][:Md], g["Wg"], g["Wu"], g["Wd"], outd, ws=ws)
        assert m.mlp_device_status(ws) == 0
    finally:
        m.mlp_debug_set_flags(0)
    a = {k: to_f64(v) for k, v in t.items() if v is not None}
    ref = mlp_forward(a["x"][:Md], a["Wg"], a["Wu"], a["Wd"], "swiglu")["out"]
    assert rel_err(to_f64(outd), ref) <= 2e-2
