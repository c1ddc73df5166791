"""GPU parity of the FP8 ReLU^2 MLP (mlp_fp8_quantize, mlp_fp8_fwd with its
e4m3 operands, mlp_fp8_bwd with e5m2 gradients) against the fp64 oracle's
8-bit emulation, through the C ABI."""
import numpy as np
import pytest
import torch

import activated_mlp_gemms_gb300 as m
from activated_mlp_gemms_gb300.workloads import make_inputs, to_f64
from mlp_gpu_helpers import SAMPLE_ROWS, SAMPLE_UNITS, spread_sample
from oracle import (E4M3_MAX, E5M2_MAX, fp8_relu_sq_backward, fp8_relu_sq_forward, quantize,
                    rel_err)

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
@pytest.mark.parametrize("M,H,I", [(1, 128, 256), (7, 256, 400), (64, 128, 352), (300, 256, 400),
                                   (1000, 768, 3072)])
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
    assert diff.sum() <= max(1, 2e-3 * diff.size), diff.mean()
    if diff.any():
        step = np.abs(got_a8[diff] - ref["a8"][diff]) / np.maximum(np.abs(ref["a8"][diff]), 2.0 ** -9)
        assert np.max(step) <= 0.25
    assert abs(float(amax.item()) - ref["amax_a"]) <= 1e-4 * ref["amax_a"]
    got = to_f64(out)
    assert np.all(np.isfinite(got))
    assert rel_err(got, ref["out"]) <= 2e-2, rel_err(got, ref["out"])


# ---------------------------------------------------------------- backward
def _f8_bytes(values, dtype):
    """Oracle code values (exactly on the 8-bit grid) -> their bytes on the device."""
    return torch.tensor(values, dtype=torch.float32).to(dtype).view(torch.uint8).cuda()


def _e5m2_codes(t8):
    return t8.view(torch.float8_e5m2).cpu().to(torch.float64).numpy()


def _bwd_case(M, H, I, seed, gate_mult=1.0, down_mult=1.0):
    """Oracle-made inputs of the backward (e4m3 codes, the bf16 preact, the
    e4m3 postact) and fp32 scales {sx, s1, s2, s_post, sg, s_dpre}; the
    delayed scales are taken from this step's amaxes."""
    t = make_inputs(M, H, I, "relu_sq", seed=seed)
    xd, W1d, W2d = to_f64(t["x"]), to_f64(t["Wg"]), to_f64(t["Wd"])
    f32 = lambda v: float(np.float32(v))
    sx = 2.0 ** -4
    s1, s2 = f32(np.max(np.abs(W1d)) / E4M3_MAX), f32(np.max(np.abs(W2d)) / E4M3_MAX)
    xc, W1c, W2c = quantize(xd, sx), quantize(W1d, s1), quantize(W2d, s2)
    pre = (xc @ W1c.T) * (sx * s1)
    s_post = f32(max(np.max(np.maximum(pre, 0) ** 2) * gate_mult, 1e-6) * 1.03 / E4M3_MAX)
    fwd = fp8_relu_sq_forward(xc, W1c, W2c, sx, s1, s2, s_post, gate_mult, down_mult)
    # the saved preact, in bf16 on both sides
    pre_bf = torch.tensor(pre, dtype=torch.float32).to(torch.bfloat16)
    pre_d = to_f64(pre_bf)
    sg = 2.0 ** -6
    probe = fp8_relu_sq_backward(to_f64(t["dout"]), xc, W1c, W2c, fwd["a8"], sx, s1, s2, s_post,
                                 sg, 1.0, gate_mult, down_mult, pre=pre_d)
    s_dpre = f32(max(probe["amax_dpre"], 1e-30) * 1.25 / E5M2_MAX)
    scales = [sx, s1, s2, s_post, sg, s_dpre]
    ref = fp8_relu_sq_backward(to_f64(t["dout"]), xc, W1c, W2c, fwd["a8"], *scales, gate_mult,
                               down_mult, pre=pre_d)
    dev = {"dout": t["dout"].cuda(), "x8": _f8_bytes(xc, torch.float8_e4m3fn),
           "W1_8": _f8_bytes(W1c, torch.float8_e4m3fn), "W2_8": _f8_bytes(W2c, torch.float8_e4m3fn),
           "pre": pre_bf.cuda(), "a8": _f8_bytes(fwd["a8"], torch.float8_e4m3fn),
           "scales": torch.tensor(scales, dtype=torch.float32, device="cuda")}
    return dev, ref


def _codes_close(got, ref, max_frac):
    """8-bit codes decided in fp32 (kernel) and fp64 (oracle): equal except
    where the two straddle a rounding boundary, and then one step apart."""
    diff = got != ref
    assert diff.sum() <= max(1, max_frac * diff.size), diff.mean()
    if diff.any():
        step = np.abs(got[diff] - ref[diff]) / np.maximum(np.abs(ref[diff]), 2.0 ** -16)
        assert np.max(step) <= 0.5, np.max(step)


@pytest.mark.parametrize("tile_policy", [1, 2], indirect=True)
@pytest.mark.parametrize("M,H,I", [(1, 128, 256), (7, 256, 400), (64, 128, 352), (300, 256, 400),
                                   (1000, 768, 3072)])
def test_fp8_backward_parity(M, H, I, tile_policy):
    dev, ref = _bwd_case(M, H, I, seed=63)
    dx = torch.full((M, H), float("nan"), dtype=torch.bfloat16, device="cuda")
    dW1 = torch.full((I, H), float("nan"), dtype=torch.bfloat16, device="cuda")
    dW2 = torch.full((H, I), float("nan"), dtype=torch.bfloat16, device="cuda")
    amax = torch.zeros(1, dtype=torch.float32, device="cuda")
    ws = m.mlp_fp8_bwd(m.problem(M, H, I, "relu_sq"), dev["dout"], dev["x8"], dev["W1_8"],
                       dev["W2_8"], dev["pre"], dev["a8"], dev["scales"], dx, dW1, dW2, amax)
    torch.cuda.synchronize()
    assert m.mlp_device_status(ws) == 0
    # the workspace holds the e5m2 codes of dout, then those of dpre
    off = 1024
    dout8 = ws[off:off + M * H].view(M, H)
    off += (M * H + 255) // 256 * 256
    dP8 = ws[off:off + M * I].view(M, I)
    assert np.array_equal(_e5m2_codes(dout8), ref["dout8"])
    _codes_close(_e5m2_codes(dP8), ref["dP8"], 2e-3)
    assert abs(float(amax.item()) - ref["amax_dpre"]) <= 1e-3 * ref["amax_dpre"]
    for name, got in (("dx", dx), ("dW1", dW1), ("dW2", dW2)):
        g = to_f64(got)
        assert np.all(np.isfinite(g)), name
        assert rel_err(g, ref[name]) <= 2e-2, (name, rel_err(g, ref[name]))


def test_fp8_backward_multipliers_and_partial_outputs():
    M, H, I = 200, 256, 512
    dev, ref = _bwd_case(M, H, I, seed=64, gate_mult=0.5, down_mult=2.0)
    prob = m.problem(M, H, I, "relu_sq", gate_mult=0.5, down_mult=2.0)
    args = (dev["dout"], dev["x8"], dev["W1_8"], dev["W2_8"], dev["pre"], dev["a8"], dev["scales"])
    # only dW2: no derivative GEMM, its operands may be absent
    dW2 = torch.empty(H, I, dtype=torch.bfloat16, device="cuda")
    m.mlp_fp8_bwd(prob, dev["dout"], None, None, None, None, dev["a8"], dev["scales"], dW2=dW2)
    torch.cuda.synchronize()
    assert rel_err(to_f64(dW2), ref["dW2"]) <= 2e-2
    # only dx
    dx = torch.empty(M, H, dtype=torch.bfloat16, device="cuda")
    m.mlp_fp8_bwd(prob, *args, dx=dx)
    torch.cuda.synchronize()
    assert rel_err(to_f64(dx), ref["dx"]) <= 2e-2
    # only dW1
    dW1 = torch.empty(I, H, dtype=torch.bfloat16, device="cuda")
    m.mlp_fp8_bwd(prob, *args, dW1=dW1)
    torch.cuda.synchronize()
    assert rel_err(to_f64(dW1), ref["dW1"]) <= 2e-2


def test_fp8_forward_saves_the_bf16_preact():
    M, H, I = 300, 256, 400
    t = make_inputs(M, H, I, "relu_sq", seed=65)
    xd, W1d, W2d = to_f64(t["x"]), to_f64(t["Wg"]), to_f64(t["Wd"])
    sx = 2.0 ** -4
    s1 = float(np.float32(np.max(np.abs(W1d)) / E4M3_MAX))
    s2 = float(np.float32(np.max(np.abs(W2d)) / E4M3_MAX))
    xc, W1c, W2c = quantize(xd, sx), quantize(W1d, s1), quantize(W2d, s2)
    scales = torch.tensor([sx, s1, s2, 1.0], dtype=torch.float32, device="cuda")
    out = torch.empty(M, H, dtype=torch.bfloat16, device="cuda")
    pre = torch.full((M, I), float("nan"), dtype=torch.bfloat16, device="cuda")
    m.mlp_fp8_fwd(m.problem(M, H, I, "relu_sq"), _f8_bytes(xc, torch.float8_e4m3fn),
                  _f8_bytes(W1c, torch.float8_e4m3fn), _f8_bytes(W2c, torch.float8_e4m3fn), scales,
                  out, pre_save=pre)
    torch.cuda.synchronize()
    ref = (xc @ W1c.T) * (np.float32(sx) * np.float32(s1))
    got = to_f64(pre)
    # bf16 rounding of the fp32 value: half an ulp (2^-9 relative), plus the
    # accumulation order
    assert np.all(np.abs(got - ref) <= 2.0 ** -8 * np.abs(ref) + 1e-6 * np.max(np.abs(ref)))


def test_fp8_negative_gate_mult_and_amax_of_magnitudes():
    """gate_mult < 0 flips the postact's sign: its e4m3 codes are negative and
    the recorded amax is the largest |a|."""
    M, H, I = 300, 256, 400
    t = make_inputs(M, H, I, "relu_sq", seed=66)
    xd, W1d, W2d = to_f64(t["x"]), to_f64(t["Wg"]), to_f64(t["Wd"])
    f32 = lambda v: float(np.float32(v))  # noqa: E731
    sx = 2.0 ** -4
    s1, s2 = f32(np.max(np.abs(W1d)) / E4M3_MAX), f32(np.max(np.abs(W2d)) / E4M3_MAX)
    xc, W1c, W2c = quantize(xd, sx), quantize(W1d, s1), quantize(W2d, s2)
    pre = (xc @ W1c.T) * (sx * s1)
    gm = -0.75
    s_post = f32(np.max(np.maximum(pre, 0) ** 2) * abs(gm) * 1.03 / E4M3_MAX)
    scales = torch.tensor([sx, s1, s2, s_post], dtype=torch.float32, device="cuda")
    out = torch.empty(M, H, dtype=torch.bfloat16, device="cuda")
    a8 = torch.empty(M, I, dtype=torch.uint8, device="cuda")
    amax = torch.zeros(1, dtype=torch.float32, device="cuda")
    m.mlp_fp8_fwd(m.problem(M, H, I, "relu_sq", gate_mult=gm), _f8_bytes(xc, torch.float8_e4m3fn),
                  _f8_bytes(W1c, torch.float8_e4m3fn), _f8_bytes(W2c, torch.float8_e4m3fn), scales,
                  out, a8, amax)
    torch.cuda.synchronize()
    ref = fp8_relu_sq_forward(xc, W1c, W2c, sx, s1, s2, s_post, gate_mult=gm)
    got = _codes(a8)
    assert np.all(got <= 0) and np.any(got < 0)
    diff = got != ref["a8"]
    assert diff.mean() < 2e-3, diff.mean()
    assert abs(float(amax.item()) - ref["amax_a"]) <= 1e-4 * ref["amax_a"]
    assert rel_err(to_f64(out), ref["out"]) <= 2e-2


def test_fp8_training_step_in_a_cuda_graph():
    """The FP8 forward (saving the preact) and backward captured into a CUDA
    graph, after a direct call has created the backward's second stream:
    replays give the direct call's outputs bitwise (no split-K, no
    order-dependent accumulation; the amaxes are maxima)."""
    M, H, I = 1000, 768, 3072
    dev, ref_o = _bwd_case(M, H, I, seed=67)
    prob = m.problem(M, H, I, "relu_sq")
    bf = torch.bfloat16
    pre = torch.empty(M, I, dtype=bf, device="cuda")
    a8 = torch.empty(M, I, dtype=torch.uint8, device="cuda")
    ws8 = m.alloc_workspace(prob, m.MODE_FP8_FWD)
    wsb = m.alloc_workspace(prob, m.MODE_FP8_BWD)

    def bufs():
        return {"out": torch.empty(M, H, dtype=bf, device="cuda"),
                "dx": torch.empty(M, H, dtype=bf, device="cuda"),
                "dW1": torch.empty(I, H, dtype=bf, device="cuda"),
                "dW2": torch.empty(H, I, dtype=bf, device="cuda"),
                "amax_a": torch.zeros(1, dtype=torch.float32, device="cuda"),
                "amax_d": torch.zeros(1, dtype=torch.float32, device="cuda")}

    def step(r):
        m.mlp_fp8_fwd(prob, dev["x8"], dev["W1_8"], dev["W2_8"], dev["scales"], r["out"], a8,
                      r["amax_a"], ws=ws8, pre_save=pre)
        m.mlp_fp8_bwd(prob, dev["dout"], dev["x8"], dev["W1_8"], dev["W2_8"], pre, a8,
                      dev["scales"], r["dx"], r["dW1"], r["dW2"], r["amax_d"], ws=wsb)
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
        for k, v in got.items():
            v.fill_(0.0 if k.startswith("amax") else float("nan"))
        g.replay()
        torch.cuda.synchronize()
        for k in ref:
            assert torch.equal(got[k], ref[k]), k
    # and the direct call is the oracle's backward (its own inputs, same scales)
    for name in ("dx", "dW1", "dW2"):
        assert rel_err(to_f64(ref[name]), ref_o[name]) <= 2e-2, name


def test_fp8_delayed_scaling_loop():
    """Three training steps with the page's delayed-scale refresh between
    them (post: amax x 1.03 / 448; dpre: amax x 1.25 / 57344): every step's
    recorded amaxes match the oracle's; from a deliberately wrong first
    scale (1.0) the second and third steps run on the refreshed scales,
    nothing saturates, and the outputs match the oracle run with the same
    scales."""
    M, H, I = 512, 256, 512
    t = make_inputs(M, H, I, "relu_sq", seed=68)
    xd, W1d, W2d, dout = to_f64(t["x"]), to_f64(t["Wg"]), to_f64(t["Wd"]), t["dout"].cuda()
    f32 = lambda v: float(np.float32(v))  # noqa: E731
    sx = 2.0 ** -4
    s1, s2 = f32(np.max(np.abs(W1d)) / E4M3_MAX), f32(np.max(np.abs(W2d)) / E4M3_MAX)
    xc, W1c, W2c = quantize(xd, sx), quantize(W1d, s1), quantize(W2d, s2)
    x8, W1_8, W2_8 = (_f8_bytes(v, torch.float8_e4m3fn) for v in (xc, W1c, W2c))
    # the oracle's own saved preact, in bf16 (the kernels save theirs)
    pre_o = to_f64(torch.tensor((xc @ W1c.T) * (sx * s1), dtype=torch.float64).to(torch.bfloat16))
    prob = m.problem(M, H, I, "relu_sq")
    bf = torch.bfloat16
    scales = torch.tensor([sx, s1, s2, 1.0, 2.0 ** -6, 1.0], dtype=torch.float32, device="cuda")
    out = torch.empty(M, H, dtype=bf, device="cuda")
    pre = torch.empty(M, I, dtype=bf, device="cuda")
    a8 = torch.empty(M, I, dtype=torch.uint8, device="cuda")
    dx = torch.empty(M, H, dtype=bf, device="cuda")
    amax_a = torch.zeros(1, dtype=torch.float32, device="cuda")
    amax_d = torch.zeros(1, dtype=torch.float32, device="cuda")
    for step in range(3):
        amax_a.zero_()
        amax_d.zero_()
        m.mlp_fp8_fwd(prob, x8, W1_8, W2_8, scales, out, a8, amax_a, pre_save=pre)
        m.mlp_fp8_bwd(prob, dout, x8, W1_8, W2_8, pre, a8, scales, dx=dx, amax_dpre=amax_d)
        torch.cuda.synchronize()
        sc = [float(v) for v in scales.cpu().numpy()]
        fw = fp8_relu_sq_forward(xc, W1c, W2c, *sc[:4])
        bw = fp8_relu_sq_backward(to_f64(dout), xc, W1c, W2c, fw["a8"], *sc, pre=pre_o)
        assert abs(float(amax_a.item()) - fw["amax_a"]) <= 1e-3 * fw["amax_a"]
        assert abs(float(amax_d.item()) - bw["amax_dpre"]) <= 1e-3 * bw["amax_dpre"]
        if step > 0:  # scales from the recorded maxima: nothing saturates
            assert np.max(np.abs(_codes(a8))) <= E4M3_MAX
            assert np.max(np.abs(fw["a"])) / sc[3] < E4M3_MAX
            assert rel_err(to_f64(out), fw["out"]) <= 2e-2
            assert rel_err(to_f64(dx), bw["dx"]) <= 2e-2
        # the page's refresh: last step's amax times the headroom over the
        # format's max (taken from the oracle's amaxes, which the kernels'
        # recorded ones match above, so that both sides get the same scales)
        scales[3] = f32(fw["amax_a"] * 1.03 / E4M3_MAX)
        scales[5] = f32(bw["amax_dpre"] * 1.25 / E5M2_MAX)


def test_fp8_golden_closed_form():
    """The stored closed-form fixture (integer codes, power-of-two scales,
    written by the oracle alone): every product and sum of fc1 and of the
    derivative is exact in fp32, so the e4m3 postact's and the e5m2 codes
    and both amaxes match bit for bit; out, dx, dW1, dW2 within the bf16
    tolerance."""
    import json
    import os
    from activated_mlp_gemms_gb300.workloads import fp8_closed_form_codes
    path = os.path.join(os.path.dirname(__file__), "golden", "fp8_closed_form.json")
    with open(path) as f:
        g = json.load(f)
    sc = g["scales"]
    for tile_policy in (1, 2):
        m.mlp_set_tile_policy(tile_policy)
        try:
            for c in g["cases"]:
                M, H, I = c["M"], c["H"], c["I"]
                t = fp8_closed_form_codes(M, H, I)
                x8, W1_8, W2_8 = (_f8_bytes(t[k].numpy(), torch.float8_e4m3fn)
                                  for k in ("x8", "W1_8", "W2_8"))
                scales = torch.tensor([sc["sx"], sc["s1"], sc["s2"], sc["s_post"], sc["sg"],
                                       c["s_dpre"]], dtype=torch.float32, device="cuda")
                prob = m.problem(M, H, I, "relu_sq", c["gate_mult"], c["down_mult"])
                bf = torch.bfloat16
                out = torch.full((M, H), float("nan"), dtype=bf, device="cuda")
                a8 = torch.empty(M, I, dtype=torch.uint8, device="cuda")
                amax_a = torch.zeros(1, dtype=torch.float32, device="cuda")
                m.mlp_fp8_fwd(prob, x8, W1_8, W2_8, scales, out, a8, amax_a)
                pre = torch.tensor(c["pre_bf16"], dtype=torch.float64).to(bf).cuda()
                dx = torch.full((M, H), float("nan"), dtype=bf, device="cuda")
                dW1 = torch.full((I, H), float("nan"), dtype=bf, device="cuda")
                dW2 = torch.full((H, I), float("nan"), dtype=bf, device="cuda")
                amax_d = torch.zeros(1, dtype=torch.float32, device="cuda")
                ws = m.mlp_fp8_bwd(prob, t["dout"].cuda(), x8, W1_8, W2_8, pre, a8, scales, dx,
                                   dW1, dW2, amax_d)
                torch.cuda.synchronize()
                assert m.mlp_device_status(ws) == 0
                assert np.array_equal(_codes(a8), np.array(c["a8"]))
                off = 1024
                dout8 = ws[off:off + M * H].view(M, H)
                off += (M * H + 255) // 256 * 256
                dP8 = ws[off:off + M * I].view(M, I)
                assert np.array_equal(_e5m2_codes(dout8), np.array(c["dout8"]))
                assert np.array_equal(_e5m2_codes(dP8), np.array(c["dP8"]))
                assert float(amax_a.item()) == c["amax_a"]
                assert float(amax_d.item()) == c["amax_dpre"]
                for name, got in (("out", out), ("dx", dx), ("dW1", dW1), ("dW2", dW2)):
                    assert rel_err(to_f64(got), np.array(c[name])) <= 2e-2, name
        finally:
            m.mlp_set_tile_policy(0)


def test_fp8_full_size_sampled():
    """The ReLU^2 workload at full size (49152 x 768 x 3072) through the FP8
    forward (saving the preact) and backward, in the launch configuration
    the benchmark times; parity on sampled token rows (out, dx) and sampled
    intermediate units (rows of dW1, columns of dW2, each reduced over all
    tokens), computed by the oracle on its own codes and preacts."""
    from activated_mlp_gemms_gb300.workloads import WORKLOADS, workload_inputs
    from oracle import fp8_relu_sq_sampled, quantize_e5m2
    w = WORKLOADS["nanogpt_relu_sq"]
    M, H, I = w.M, w.H, w.I
    t = workload_inputs(w)
    xd, W1d, W2d, doutd = (to_f64(t[k]) for k in ("x", "Wg", "Wd", "dout"))
    f32 = lambda v: float(np.float32(v))  # noqa: E731
    sx = 2.0 ** -4
    s1, s2 = f32(np.max(np.abs(W1d)) / E4M3_MAX), f32(np.max(np.abs(W2d)) / E4M3_MAX)
    xc, W1c, W2c = quantize(xd, sx), quantize(W1d, s1), quantize(W2d, s2)
    rows = spread_sample(M, SAMPLE_ROWS)
    units = spread_sample(I, SAMPLE_UNITS)

    def round_pre(v):  # the saved preact's bf16 rounding
        return to_f64(torch.tensor(v, dtype=torch.float64).to(torch.bfloat16))
    # delayed scales as they settle, from the oracle's own sampled rows
    pre_r = (xc[rows] @ W1c.T) * (sx * s1)
    s_post = f32(np.max(np.maximum(pre_r, 0) ** 2) * 1.03 / E4M3_MAX)
    sg = 2.0 ** -6
    da = (quantize_e5m2(doutd[rows], sg) @ W2c) * (sg * s2)
    s_dpre = f32(np.max(np.abs(da * 2 * np.maximum(round_pre(pre_r), 0))) * 1.25 / E5M2_MAX)
    scales = [sx, s1, s2, s_post, sg, s_dpre]
    ref = fp8_relu_sq_sampled(doutd, xc, W1c, W2c, *scales, rows, units, round_pre=round_pre)

    prob = m.problem(M, H, I, "relu_sq")
    bf = torch.bfloat16
    x8, W1_8, W2_8 = (_f8_bytes(v, torch.float8_e4m3fn) for v in (xc, W1c, W2c))
    sc = torch.tensor(scales, dtype=torch.float32, device="cuda")
    out = torch.full((M, H), float("nan"), dtype=bf, device="cuda")
    pre = torch.empty(M, I, dtype=bf, device="cuda")
    a8 = torch.empty(M, I, dtype=torch.uint8, device="cuda")
    dx = torch.full((M, H), float("nan"), dtype=bf, device="cuda")
    dW1 = torch.full((I, H), float("nan"), dtype=bf, device="cuda")
    dW2 = torch.full((H, I), float("nan"), dtype=bf, device="cuda")
    m.mlp_fp8_fwd(prob, x8, W1_8, W2_8, sc, out, a8, pre_save=pre)
    ws = m.mlp_fp8_bwd(prob, t["dout"].cuda(), x8, W1_8, W2_8, pre, a8, sc, dx, dW1, dW2)
    torch.cuda.synchronize()
    assert m.mlp_device_status(ws) == 0
    r_t, u_t = torch.as_tensor(rows), torch.as_tensor(units)
    errs = {"out": rel_err(to_f64(out[r_t]), ref["out"]),
            "dx": rel_err(to_f64(dx[r_t]), ref["dx"]),
            "dW1": rel_err(to_f64(dW1[u_t]), ref["dW1"]),
            "dW2": rel_err(to_f64(dW2[:, u_t]), ref["dW2"])}
    assert all(e <= 2e-2 for e in errs.values()), errs
    for v in (out, dx, dW1, dW2):
        assert torch.isfinite(v.float()).all()


def _refresh_host(amax, scale, gain, floor):
    """gpt.py's _refresh_delayed_scale restated on the host in fp32: the
    slot's amax (max over its row, NaN propagating), NaN / +-inf -> 0, at
    most 1e12; scale = max(a * gain, floor) where a > 0, else unchanged."""
    f = np.float32
    a = np.max(amax.astype(f), axis=1)
    a = np.nan_to_num(a, nan=0.0, posinf=0.0, neginf=0.0).astype(f)
    a = np.minimum(a, f(1e12))
    new = np.maximum(a * f(gain), f(floor))
    return np.where(a > 0, new, scale.astype(f)).astype(f)


@pytest.mark.parametrize("width", [1, 3])
def test_refresh_scales_matches_host_restatement(width):
    inf, nan = float("inf"), float("nan")
    rows = [[2.5], [0.0], [nan], [inf], [-inf], [-1.0], [3e13], [1e-9], [448.0], [6e-7]]
    rng = np.random.default_rng(70)
    amax = np.array([r * width for r in rows], dtype=np.float32)
    if width > 1:
        amax[:, 1:] = rng.uniform(0, 4, size=(len(rows), width - 1)).astype(np.float32)
        amax[2, 2] = nan  # a NaN anywhere in the row
    scale = rng.uniform(0.5, 2.0, size=len(rows)).astype(np.float32)
    for gain, floor in ((1.03 / 448.0, 1e-6), (1.25 / 57344.0, 1e-12)):
        a_d = torch.tensor(amax, device="cuda")
        s_d = torch.tensor(scale, device="cuda")
        m.mlp_fp8_refresh_scales(a_d, s_d, gain, floor)
        torch.cuda.synchronize()
        want = _refresh_host(amax, scale, gain, floor)
        got = s_d.cpu().numpy()
        assert np.array_equal(got.view(np.int32), want.view(np.int32)), (got, want)
        assert (a_d == 0).all()


def test_fp8_training_loop_in_a_graph_needs_no_host_sync():
    """Three FP8 training steps (forward saving the preact, backward, then the
    delayed-scale refresh of s_post and s_dpre from the amaxes the kernels
    recorded) as one captured CUDA graph replayed three times back to back,
    against the same steps run eagerly with the refresh restated on the
    host between them: the scales, amaxes and every output agree bit for
    bit.  The first scales are deliberately off (1.0)."""
    M, H, I = 512, 256, 512
    t = make_inputs(M, H, I, "relu_sq", seed=71)
    xd, W1d, W2d = to_f64(t["x"]), to_f64(t["Wg"]), to_f64(t["Wd"])
    f32 = lambda v: float(np.float32(v))  # noqa: E731
    sx = 2.0 ** -4
    s1, s2 = f32(np.max(np.abs(W1d)) / E4M3_MAX), f32(np.max(np.abs(W2d)) / E4M3_MAX)
    x8, W1_8, W2_8 = (_f8_bytes(quantize(v, s), torch.float8_e4m3fn)
                      for v, s in ((xd, sx), (W1d, s1), (W2d, s2)))
    dout = t["dout"].cuda()
    prob = m.problem(M, H, I, "relu_sq")
    bf = torch.bfloat16
    G_POST, F_POST = 1.03 / E4M3_MAX, 1e-6
    G_DPRE, F_DPRE = 1.25 / E5M2_MAX, 1e-12

    def state():
        return {"scales": torch.tensor([sx, s1, s2, 1.0, 2.0 ** -6, 1.0], dtype=torch.float32,
                                       device="cuda"),
                "amax_a": torch.zeros(1, dtype=torch.float32, device="cuda"),
                "amax_d": torch.zeros(1, dtype=torch.float32, device="cuda"),
                "out": torch.empty(M, H, dtype=bf, device="cuda"),
                "pre": torch.empty(M, I, dtype=bf, device="cuda"),
                "a8": torch.empty(M, I, dtype=torch.uint8, device="cuda"),
                "dx": torch.empty(M, H, dtype=bf, device="cuda"),
                "dW1": torch.empty(I, H, dtype=bf, device="cuda"),
                "dW2": torch.empty(H, I, dtype=bf, device="cuda"),
                "wsf": m.alloc_workspace(prob, m.MODE_FP8_FWD),
                "wsb": m.alloc_workspace(prob, m.MODE_FP8_BWD)}

    def step(s):
        m.mlp_fp8_fwd(prob, x8, W1_8, W2_8, s["scales"], s["out"], s["a8"], s["amax_a"],
                      ws=s["wsf"], pre_save=s["pre"])
        m.mlp_fp8_bwd(prob, dout, x8, W1_8, W2_8, s["pre"], s["a8"], s["scales"], s["dx"],
                      s["dW1"], s["dW2"], s["amax_d"], ws=s["wsb"])

    # eager: the refresh on the host after each step
    e = state()
    for _ in range(3):
        step(e)
        torch.cuda.synchronize()
        sc = e["scales"].cpu().numpy()
        sc[3] = _refresh_host(e["amax_a"].cpu().numpy()[None, :], sc[3:4], G_POST, F_POST)[0]
        sc[5] = _refresh_host(e["amax_d"].cpu().numpy()[None, :], sc[5:6], G_DPRE, F_DPRE)[0]
        e["scales"].copy_(torch.from_numpy(sc))
        e["amax_a"].zero_()
        e["amax_d"].zero_()
    torch.cuda.synchronize()

    # graph: the whole step including the refresh on the device
    g = state()
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):  # a direct call first sets up the library's caches
        step(state())
    torch.cuda.current_stream().wait_stream(s)
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        step(g)
        m.mlp_fp8_refresh_scales(g["amax_a"], g["scales"][3:4], G_POST, F_POST)
        m.mlp_fp8_refresh_scales(g["amax_d"], g["scales"][5:6], G_DPRE, F_DPRE)
    for _ in range(3):
        graph.replay()
    torch.cuda.synchronize()
    assert float(e["scales"][3]) != 1.0 and float(e["scales"][5]) != 1.0
    for k in ("scales", "amax_a", "amax_d", "out", "pre", "a8", "dx", "dW1", "dW2"):
        assert torch.equal(g[k], e[k]), k
    assert m.mlp_device_status(g["wsb"]) == 0


@pytest.mark.parametrize("tile_policy", [1, 2], indirect=True)
@pytest.mark.parametrize("M,H,I", [(7, 256, 400), (300, 256, 400), (1000, 768, 3072)])
def test_fp8_backward_recomputing_the_preact_equals_the_saved_path(M, H, I, tile_policy):
    """mlp_fp8_bwd without a saved preact recomputes it in the derivative
    GEMM's tile from x8 and W1_8 (the forward's own fp32 sums) and rounds
    2 relu(pre) to bf16 as the saved path does: the e5m2 derivative codes,
    their amax, dx, dW1 and dW2 are bitwise those of the saved path."""
    t = make_inputs(M, H, I, "relu_sq", seed=72)
    xd, W1d, W2d = to_f64(t["x"]), to_f64(t["Wg"]), to_f64(t["Wd"])
    f32 = lambda v: float(np.float32(v))  # noqa: E731
    sx = 2.0 ** -4
    s1, s2 = f32(np.max(np.abs(W1d)) / E4M3_MAX), f32(np.max(np.abs(W2d)) / E4M3_MAX)
    x8, W1_8, W2_8 = (_f8_bytes(quantize(v, sc), torch.float8_e4m3fn)
                      for v, sc in ((xd, sx), (W1d, s1), (W2d, s2)))
    prob = m.problem(M, H, I, "relu_sq", 1.125, 2.0)
    bf = torch.bfloat16
    pre = (xd[:64] @ W1d.T).clip(min=0) ** 2
    s_post = f32(np.max(pre) * 1.125 * 1.03 / E4M3_MAX)
    scales = torch.tensor([sx, s1, s2, s_post, 2.0 ** -6, 2.0 ** -10], dtype=torch.float32,
                          device="cuda")
    out = torch.empty(M, H, dtype=bf, device="cuda")
    a8 = torch.empty(M, I, dtype=torch.uint8, device="cuda")
    pre_s = torch.empty(M, I, dtype=bf, device="cuda")
    m.mlp_fp8_fwd(prob, x8, W1_8, W2_8, scales, out, a8, pre_save=pre_s)
    dout = t["dout"].cuda()
    res = {}
    for name, p_in in (("saved", pre_s), ("recompute", None)):
        dx = torch.full((M, H), float("nan"), dtype=bf, device="cuda")
        dW1 = torch.full((I, H), float("nan"), dtype=bf, device="cuda")
        dW2 = torch.full((H, I), float("nan"), dtype=bf, device="cuda")
        amax = torch.zeros(1, dtype=torch.float32, device="cuda")
        ws = m.mlp_fp8_bwd(prob, dout, x8, W1_8, W2_8, p_in, a8, scales, dx, dW1, dW2, amax)
        torch.cuda.synchronize()
        assert m.mlp_device_status(ws) == 0
        off = 1024 + (M * H + 255) // 256 * 256
        res[name] = {"dx": dx, "dW1": dW1, "dW2": dW2, "amax": amax,
                     "dP8": ws[off:off + M * I].clone()}
    for k in res["saved"]:
        assert torch.isfinite(res["recompute"][k].float()).all() if k != "dP8" else True
        assert torch.equal(res["saved"][k], res["recompute"][k]), k
