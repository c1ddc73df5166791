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
