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
