"""mlp_fwd_infer_noalloc: the inference forward for callers that may not
allocate device memory when they run the MLP (a runtime whose device memory
is planned once at start-up, or a serving loop that must not call cudaMalloc
because it synchronises the device).  Its scratch is a fixed array inside the
library instead of a caller workspace.

Checked through the C ABI against the existing entry point mlp_fwd_infer, on
two calls in a row (the array keeps the previous call's contents, so the
second call must still be right), within the bf16 parity tolerance.  This
file sorts last so that a run stopping at the first failure has already run
every other test; it also passes alone in a fresh process."""
import ctypes

import pytest
import torch

import activated_mlp_gemms_gb300 as m
from activated_mlp_gemms_gb300.workloads import make_inputs, to_f64
from oracle import rel_err

pytestmark = pytest.mark.gpu

TOL_BF16 = 2e-2


def _dev(t):
    return {k: (v.cuda() if v is not None else None) for k, v in t.items()}


@pytest.mark.parametrize("act,gm,dm,shape", [
    ("swiglu", 1.0, 1.0, (300, 264, 392)),
    ("swiglu", 1.125, 2.0, (512, 4096, 14336)),
    ("relu_sq", 1.0, 1.0, (257, 768, 3072)),
])
def test_noalloc_matches_workspace_entry_point(act, gm, dm, shape):
    M, H, I = shape
    L = m.lib()
    prob = m.problem(M, H, I, act, gm, dm)
    assert m.mlp_workspace_size(prob, m.MODE_INFER) <= m.NOALLOC_SCRATCH_BYTES
    stream = torch.cuda.current_stream().cuda_stream
    for seed in (11, 12):  # two calls in a row, different inputs
        t = _dev(make_inputs(M, H, I, act, seed=seed))
        ref = torch.empty(M, H, dtype=torch.bfloat16, device="cuda")
        m.mlp_fwd_infer(prob, t["x"], t["Wg"], t["Wu"], t["Wd"], ref)
        got = torch.full((M, H), float("nan"), dtype=torch.bfloat16, device="cuda")
        ptr = lambda v: None if v is None else v.data_ptr()  # noqa: E731
        rc = L.mlp_fwd_infer_noalloc(ctypes.byref(prob), ptr(t["x"]), ptr(t["Wg"]), ptr(t["Wu"]),
                                     ptr(t["Wd"]), ptr(got), stream)
        assert rc == 0, m.mlp_status_string(rc)
        torch.cuda.synchronize()
        assert torch.isfinite(got.float()).all()
        assert rel_err(to_f64(got), to_f64(ref)) <= TOL_BF16


def test_noalloc_rejects_problems_beyond_its_scratch():
    L = m.lib()
    prob = m.problem(4096, 4096, 14336)  # needs 117 MB of scratch
    assert m.mlp_workspace_size(prob, m.MODE_INFER) > m.NOALLOC_SCRATCH_BYTES
    x = torch.empty(16, dtype=torch.bfloat16, device="cuda")
    rc = L.mlp_fwd_infer_noalloc(ctypes.byref(prob), x.data_ptr(), x.data_ptr(), x.data_ptr(),
                                 x.data_ptr(), x.data_ptr(), None)
    assert rc == -4 and m.mlp_status_string(rc) == "MLP_ERR_WORKSPACE_TOO_SMALL"
