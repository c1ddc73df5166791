"""Pins of the FP8 oracle: the e4m3 rounding against torch's independent
float8_e4m3fn cast and against grid facts, the saturation reading, and the
forward on inputs whose codes and products are exact."""
import numpy as np
import pytest

import oracle.fp8_oracle as F8


def test_e4m3_matches_torch_cast_in_range():
    torch = pytest.importorskip("torch")
    rng = np.random.default_rng(51)
    v = np.concatenate([rng.standard_normal(20000) * s for s in (1e-3, 0.05, 1, 30, 200)])
    v = v[np.abs(v) <= 448]
    # include exact ties between neighbouring codes (round half to even)
    grid = np.array([1.0, 1.125, 1.25, 8, 9, 0.015625, 0.017578125, 0.001953125, 0.00390625])
    v = np.concatenate([v, (grid[:-1] + grid[1:]) / 2, -(grid[:-1] + grid[1:]) / 2, grid])
    ref = torch.tensor(v, dtype=torch.float64).to(torch.float8_e4m3fn).to(torch.float64).numpy()
    assert np.array_equal(F8.e4m3(v), ref)


def test_e4m3_grid_facts():
    assert F8.e4m3(448.0) == 448.0 and F8.e4m3(1000.0) == 448.0 and F8.e4m3(-1e9) == -448.0
    assert F8.e4m3(2.0 ** -9) == 2.0 ** -9          # smallest subnormal
    assert F8.e4m3(2.0 ** -10) == 0.0                # half of it: ties to even (0)
    assert F8.e4m3(1.0625) == 1.0 and F8.e4m3(1.1875) == 1.25  # half-way: even mantissa
    # 0, 7 subnormals and 15 x 8 - 1 normals (the all-ones pattern is NaN): 127 values
    v = np.concatenate([np.linspace(0, 0.05, 200001), np.linspace(0, 448, 200001)])
    assert len(np.unique(F8.e4m3(v))) == 127
    codes = [m * 2.0 ** -9 for m in range(1, 8)] + [
        (1 + m / 8) * 2.0 ** e for e in range(-6, 9) for m in range(8) if (e, m) != (8, 7)]
    assert len(codes) == 126 and np.array_equal(F8.e4m3(codes), codes)
    assert F8.e4m3(0.0) == 0.0


def test_quantize_with_power_of_two_scale_is_plain_rounding():
    rng = np.random.default_rng(52)
    x = rng.standard_normal(1000)
    assert np.array_equal(F8.quantize(x, 2.0 ** -4), F8.e4m3(np.float32(x).astype(np.float64) * 16))


def test_fp8_forward_exact_on_representable_inputs():
    # codes are small integers, scales powers of two: every product and sum
    # is exact in fp64, so the forward equals its closed form
    rng = np.random.default_rng(53)
    M, H, I = 4, 8, 6
    x8 = rng.integers(-3, 4, (M, H)).astype(float)
    W1 = rng.integers(-2, 3, (I, H)).astype(float)
    W2 = rng.integers(-2, 3, (H, I)).astype(float)
    sx, s1, s2 = 2.0 ** -2, 2.0 ** -1, 2.0 ** -3
    pre = (x8 @ W1.T) * sx * s1
    a = np.maximum(pre, 0) ** 2
    s_post = 2.0 ** -3
    assert np.max(a) / s_post <= 448
    fw = F8.fp8_relu_sq_forward(x8, W1, W2, sx, s1, s2, s_post)
    assert np.array_equal(fw["a"], a)
    assert np.array_equal(fw["a8"], F8.e4m3(a / s_post))
    assert np.array_equal(fw["out"], (fw["a8"] @ W2.T) * s_post * s2)
    assert fw["amax_a"] == np.max(a)
    # a negative gate_mult flips the postact's sign; the amax is of |a|
    fn = F8.fp8_relu_sq_forward(x8, W1, W2, sx, s1, s2, s_post, gate_mult=-0.5)
    assert np.array_equal(fn["a8"], -F8.e4m3(0.5 * a / s_post))
    assert fn["amax_a"] == 0.5 * np.max(a)


def test_fp8_forward_close_to_the_bf16_definition():
    # with page-like scales the FP8 forward stays near the exact MLP (the
    # quantisation error of e4m3, 3 mantissa bits, bounds it)
    rng = np.random.default_rng(54)
    M, H, I = 64, 128, 256
    x = rng.standard_normal((M, H))
    W1 = rng.standard_normal((I, H)) / np.sqrt(H)
    W2 = rng.standard_normal((H, I)) / np.sqrt(I)
    sx, s1, s2 = 2.0 ** -4, F8.weight_scale(W1), F8.weight_scale(W2)
    exact_a = np.maximum(x @ W1.T, 0) ** 2
    s_post = np.max(exact_a) * 1.03 / 448
    fw = F8.fp8_relu_sq_forward(F8.quantize(x, sx), F8.quantize(W1, s1), F8.quantize(W2, s2),
                                sx, s1, s2, s_post)
    exact = exact_a @ W2.T
    err = np.max(np.abs(fw["out"] - exact)) / np.max(np.abs(exact))
    assert err < 0.1


def test_planted_missing_dequant_is_caught():
    rng = np.random.default_rng(55)
    x8 = rng.integers(-3, 4, (3, 8)).astype(float)
    W1 = rng.integers(-2, 3, (5, 8)).astype(float)
    W2 = rng.integers(-2, 3, (8, 5)).astype(float)
    good = F8.fp8_relu_sq_forward(x8, W1, W2, 0.25, 0.5, 0.125, 0.125)["out"]
    bad = (F8.e4m3(np.maximum(x8 @ W1.T * 0.25, 0) ** 2 / 0.125) @ W2.T) * 0.125 * 0.125
    assert not np.array_equal(good, bad)


def test_e5m2_matches_torch_cast_in_range():
    torch = pytest.importorskip("torch")
    rng = np.random.default_rng(56)
    v = np.concatenate([rng.standard_normal(20000) * s for s in (1e-5, 1e-2, 1, 300, 20000)])
    v = v[np.abs(v) <= 57344]
    grid = np.array([1.0, 1.25, 1.5, 2.0 ** -14, 2.0 ** -16, 2.0 ** -15])
    v = np.concatenate([v, (grid[:-1] + grid[1:]) / 2, grid, -grid])
    ref = torch.tensor(v, dtype=torch.float64).to(torch.float8_e5m2).to(torch.float64).numpy()
    assert np.array_equal(F8.e5m2(v), ref)


def test_e5m2_grid_facts():
    assert F8.e5m2(57344.0) == 57344.0 and F8.e5m2(1e9) == 57344.0
    assert F8.e5m2(2.0 ** -16) == 2.0 ** -16 and F8.e5m2(2.0 ** -17) == 0.0
    assert F8.e5m2(1.125) == 1.0 and F8.e5m2(1.375) == 1.5  # ties to even mantissa


@pytest.mark.parametrize("M,H,I", [(3, 6, 5), (5, 8, 4)])
def test_fp8_backward_matches_finite_differences_of_the_dequantised_forward(M, H, I):
    # Inputs chosen so that no quantisation rounds: one-hot token rows for x
    # and dout, W1 in {-1..2}, W2 in {-1, 0, 1}, so that pre is in {-1..2},
    # dout W2 in {-1, 0, 1} and dpre = 2 (dout W2) relu(pre) in {0, 2, 4}
    # (exact e5m2 codes).  The backward must then be the derivative of the
    # dequantised forward out = relu(x W1^T)^2 W2^T (postact quantisation
    # as the identity): central differences.
    rng = np.random.default_rng(57)
    x8 = np.eye(H)[rng.integers(0, H, M)]
    W1 = rng.integers(-1, 3, (I, H)).astype(float)
    W2 = rng.integers(-1, 2, (H, I)).astype(float)
    dout = np.eye(H)[rng.integers(0, H, M)] * rng.choice([-1.0, 1.0], (M, 1))
    one = dict(sx=1.0, s1=1.0, s2=1.0, s_post=1.0, sg=1.0, s_dpre=1.0)
    a8 = F8.fp8_relu_sq_forward(x8, W1, W2, 1.0, 1.0, 1.0, 1.0)["a8"]
    bw = F8.fp8_relu_sq_backward(dout, x8, W1, W2, a8, **one)
    assert np.array_equal(bw["dP8"], bw["dpre"])  # exact codes

    def loss(x, W1_, W2_):
        return float(np.sum(dout * ((np.maximum(x @ W1_.T, 0) ** 2) @ W2_.T)))
    h = 1e-6
    for name, arr, key in (("x", x8, "dx"), ("W1", W1, "dW1"), ("W2", W2, "dW2")):
        num = np.zeros_like(arr)
        for idx in np.ndindex(arr.shape):
            old = arr[idx]
            arr[idx] = old + h
            lp = loss(x8, W1, W2)
            arr[idx] = old - h
            lm = loss(x8, W1, W2)
            arr[idx] = old
            num[idx] = (lp - lm) / (2 * h)
        assert np.max(np.abs(bw[key] - num)) <= 1e-5 * max(1.0, np.max(np.abs(num))), name


def test_planted_missing_relu_grad_factor_is_caught():
    rng = np.random.default_rng(58)
    x8 = rng.integers(-2, 3, (4, 6)).astype(float)
    W1 = rng.integers(-2, 3, (5, 6)).astype(float)
    W2 = rng.integers(-2, 3, (6, 5)).astype(float)
    dout = rng.integers(-2, 3, (4, 6)).astype(float)
    a8 = F8.fp8_relu_sq_forward(x8, W1, W2, 1.0, 1.0, 1.0, 1.0)["a8"]
    good = F8.fp8_relu_sq_backward(dout, x8, W1, W2, a8, 1.0, 1.0, 1.0, 1.0, 1.0, 1.0)["dx"]
    bad = ((dout @ W2) * np.maximum(x8 @ W1.T, 0)) @ W1  # the factor 2 dropped
    assert not np.array_equal(good, bad)


def test_fp8_sampled_equals_the_full_definition():
    """The sampled oracle (token rows, intermediate units) is the full
    forward and backward restricted to those rows and units, bit for bit."""
    rng = np.random.default_rng(57)
    M, H, I = 24, 32, 40
    x = rng.standard_normal((M, H))
    W1 = rng.standard_normal((I, H)) / np.sqrt(H)
    W2 = rng.standard_normal((H, I)) / np.sqrt(I)
    dout = rng.standard_normal((M, H))
    sx, s1, s2 = 2.0 ** -4, F8.weight_scale(W1), F8.weight_scale(W2)
    x8, W1_8, W2_8 = F8.quantize(x, sx), F8.quantize(W1, s1), F8.quantize(W2, s2)
    s_post, sg, s_dpre = 2.0 ** -9, 2.0 ** -6, 2.0 ** -12
    gm, dm = 0.75, 1.5
    round_pre = lambda v: np.round(v * 64) / 64  # noqa: E731  (any fixed rounding)
    fw = F8.fp8_relu_sq_forward(x8, W1_8, W2_8, sx, s1, s2, s_post, gm, dm)
    pre = (x8 @ W1_8.T) * (sx * s1)
    bw = F8.fp8_relu_sq_backward(dout, x8, W1_8, W2_8, fw["a8"], sx, s1, s2, s_post, sg, s_dpre,
                                 gm, dm, pre=round_pre(pre))
    rows, units = np.array([0, 5, 23]), np.array([1, 17, 39])
    sm = F8.fp8_relu_sq_sampled(dout, x8, W1_8, W2_8, sx, s1, s2, s_post, sg, s_dpre, rows, units,
                                gm, dm, round_pre=round_pre)
    assert np.array_equal(sm["out"], fw["out"][rows])
    assert np.array_equal(sm["dx"], bw["dx"][rows])
    assert np.array_equal(sm["dW1"], bw["dW1"][units])
    assert np.array_equal(sm["dW2"], bw["dW2"][:, units])
