"""GPU parity of the e4m3 (FP8) forward of the ReLU^2 MLP (mlp_fp8_quantize,
mlp_fp8_fwd) against the fp64 oracle's e4m3 emulation, through the C ABI."""
import numpy as np
import pytest
import torch

import activated_mlp_gemms_gb300 as m
from activated_mlp_gemms_gb300.workloads import make_inputs, to_f64
from oracle import E4M3_MAX, fp8_relu_sq_forward, quantize, rel_err

pytestmark = pytest.mark.gpu


@pytest.fixture
def tile_policy(request):
    m.mlp_set_tile_policy(request.param)
    yield request.param
    m.mlp_set_tile_policy(0)


def _codes(t8):
    """e4m3 codes on the device -> float64 values on the host."""
    return t8.view(torch.float8_e4m3fn).cpu().to(torch.float64).numpy()


def _quantize_gpu(x, scale):
    s = torch.tensor([scale], dtype=torch.float32, device="cuda")
    amax = torch.zeros(1, dtype=torch.float32, device="cuda")
    q = torch.empty(x.shape, dtype=torch.uint8, device="cuda")
    m.mlp_fp8_quantize(x, s, q, amax)
    torch.cuda.synchronize()
    return q, float(amax.item())


@pytest.mark.parametrize("scale", ["pow2", "amax"])
def test_quantize_codes_are_bit_exact(scale):
    rng = np.random.default_rng(61)
    x = torch.tensor(rng.standard_normal((333, 96)) * 7, dtype=torch.float32).to(torch.bfloat16)
    xd = to_f64(x)
    s = 2.0 ** -4 if scale == "pow2" else float(np.float32(np.max(np.abs(xd)) / E4M3_MAX))
    q, amax = _quantize_gpu(x.cuda(), s)
    assert np.array_equal(_codes(q), quantize(xd, s))  # includes saturated codes for pow2
    assert amax == np.max(np.abs(xd))


@pytest.mark.parametrize("tile_policy", [1, 2], indirect=True)
@pytest.mark.parametrize("M,H,I", [(64, 128, 352), (300, 256, 400), (1000, 768, 3072)])
def test_fp8_forward_parity(M, H, I, tile_policy):
    t = make_inputs(M, H, I, "relu_sq", seed=62)
    x, W1, W2 = t["x"].cuda(), t["Wg"].cuda(), t["Wd"].cuda()
    xd, W1d, W2d = to_f64(t["x"]), to_f64(t["Wg"]), to_f64(t["Wd"])
    sx = 2.0 ** -4
    s1 = float(np.float32(np.max(np.abs(W1d)) / E4M3_MAX))
    s2 = float(np.float32(np.max(np.abs(W2d)) / E4M3_MAX))
    x8, _ = _quantize_gpu(x, sx)
    W1_8, _ = _quantize_gpu(W1, s1)
    W2_8, _ = _quantize_gpu(W2, s2)
    xc, W1c, W2c = quantize(xd, sx), quantize(W1d, s1), quantize(W2d, s2)
    assert np.array_equal(_codes(x8), xc) and np.array_equal(_codes(W1_8), W1c)
    # the delayed post scale: last step's amax x 1.03 / 448 (here: this step's, exactly)
    pre = (xc @ W1c.T) * (np.float32(sx) * np.float32(s1))
    s_post = float(np.float32(np.max(np.maximum(pre, 0) ** 2) * 1.03 / E4M3_MAX))
    scales = torch.tensor([sx, s1, s2, s_post], dtype=torch.float32, device="cuda")
    out = torch.full((M, H), float("nan"), dtype=torch.bfloat16, device="cuda")
    a8 = torch.empty(M, I, dtype=torch.uint8, device="cuda")
    amax = torch.zeros(1, dtype=torch.float32, device="cuda")
    ws = m.mlp_fp8_fwd(m.problem(M, H, I, "relu_sq"), x8, W1_8, W2_8, scales, out, a8, amax)
    torch.cuda.synchronize()
    assert m.mlp_device_status(ws) == 0
    ref = fp8_relu_sq_forward(xc, W1c, W2c, *[float(v) for v in scales.cpu().numpy()])
    got_a8 = _codes(a8)
    # the postact's codes: the kernel rounds its fp32 value, the oracle its
    # fp64 one; they may differ where the two straddle a rounding boundary,
    # and then by one code step
    diff = got_a8 != ref["a8"]
    assert diff.mean() < 2e-3, diff.mean()
    if diff.any():
        step = np.abs(got_a8[diff] - ref["a8"][diff]) / np.maximum(np.abs(ref["a8"][diff]), 2.0 ** -9)
        assert np.max(step) <= 0.25
    assert abs(float(amax.item()) - ref["amax_a"]) <= 1e-4 * ref["amax_a"]
    got = to_f64(out)
    assert np.all(np.isfinite(got))
    assert rel_err(got, ref["out"]) <= 2e-2, rel_err(got, ref["out"])
