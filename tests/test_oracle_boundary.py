"""Pins for the oracle's sandwich-norm boundary."""
import json
import os

import numpy as np
import torch

from oracle import bf16
from oracle.boundary import boundary, residual, residual_coefficients, rmsnorm

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def test_worked_example_rounding_points():
    g = json.load(open(os.path.join(GOLDEN, "boundary_rounding_points.json")))
    h_new, z, y = boundary(np.array([g["h"]]), np.array([g["x"]]), np.array(g["w_post"]),
                           np.array(g["w_pre"]), g["n"], g["eps"])
    assert y[0].tolist() == g["y"]
    assert h_new[0].tolist() == g["h_new"]
    assert z[0].tolist() == g["z"]
    assert h_new[0].tolist() != g["h_new_if_y_not_rounded"]


def test_rmsnorm_matches_library():
    # torch.nn.functional.rms_norm computes v / sqrt(mean(v^2) + eps) * w.
    rng = np.random.default_rng(2)
    v = rng.standard_normal((7, 96)) * 3.0
    w = 1.0 + 0.02 * rng.standard_normal(96)
    for eps in (0.0, 1e-6, 0.5):
        ref = torch.nn.functional.rms_norm(torch.from_numpy(v), (96,), torch.from_numpy(w), eps).numpy()
        np.testing.assert_allclose(rmsnorm(v, w, eps), ref, rtol=1e-14, atol=0)


def test_eps_sits_inside_the_square_root():
    x = np.full((1, 64), 1e-4)
    _, _, y = boundary(np.zeros((1, 64)), x, np.ones(64), np.ones(64), 3, 1e-6)
    assert y[0, 0] == bf16.round_bf16(1e-4 / np.sqrt(1e-8 + 1e-6))


def test_coefficients_preserve_unit_variance():
    for n in range(1, 300):
        a, b = residual_coefficients(n)
        assert abs(a * a + b * b - 1.0) <= 4e-16
    assert residual_coefficients(1) == (0.0, 1.0)
    a, b = residual_coefficients(4)
    assert abs(a - np.sqrt(3) / 2) < 1e-16 and b == 0.5


def test_first_boundary_returns_the_normed_output():
    rng = np.random.default_rng(3)
    h = bf16.round_bf16(rng.standard_normal((5, 128)))
    x = bf16.round_bf16(rng.standard_normal((5, 128)))
    w = bf16.round_bf16(1 + 0.02 * rng.standard_normal(128))
    h_new, _, y = boundary(h, x, w, w, 1, 1e-6)
    assert np.array_equal(h_new, y)


def test_constant_row_normalises_to_one():
    for c in (0.1, 1.0, 3.0, -2.0, 1000.0):
        x = np.full((1, 256), c)
        _, _, y = boundary(np.zeros((1, 256)), x, np.ones(256), np.ones(256), 5, 1e-6)
        assert np.all(y == np.sign(c))


def test_residual_of_unit_variance_inputs_stays_unit_variance():
    rng = np.random.default_rng(4)
    T, H = 256, 1024
    h = bf16.round_bf16(rng.standard_normal((T, H)))
    x = bf16.round_bf16(rng.standard_normal((T, H)))
    ones = np.ones(H)
    sigma = np.sqrt(2.0 / (T * H))
    for n in (2, 10, 60):
        h_new, _, _ = boundary(h, x, ones, ones, n, 1e-6)
        assert abs(np.mean(h_new ** 2) - 1.0) < 5 * sigma
    # and plain addition would not
    assert np.mean((h + rmsnorm(x, ones, 1e-6)) ** 2) > 1.9


def test_outputs_are_bf16_values():
    rng = np.random.default_rng(5)
    h = bf16.round_bf16(rng.standard_normal((4, 256)))
    x = bf16.round_bf16(rng.standard_normal((4, 256)))
    w = bf16.round_bf16(1 + 0.02 * rng.standard_normal(256))
    for arr in boundary(h, x, w, w, 7, 1e-6):
        assert np.array_equal(bf16.round_bf16(arr), arr)


def test_residual_form_equals_the_pages_formula():
    rng = np.random.default_rng(6)
    h = bf16.round_bf16(rng.standard_normal(10000))
    y = bf16.round_bf16(rng.standard_normal(10000))
    for n in (1, 2, 3, 10, 20, 60, 100):
        a, b = residual_coefficients(n)
        np.testing.assert_allclose(residual(h, y, n), a * h + b * y, rtol=1e-12, atol=1e-15)


def test_exact_cancellation_gives_zero():
    # n - 1 a perfect square: sqrt((n-1)/n) h + y / sqrt(n) = 0 exactly when y = -sqrt(n-1) h
    h = np.array([1.0, -0.75, 3.0, 2.0 ** -20])
    for n, m in ((2, 1.0), (5, 2.0), (10, 3.0), (17, 4.0)):
        y = -m * h
        assert np.all(residual(h, y, n) == 0.0)
    # through the whole boundary: x = (-3, -3) normalises to y = -1, h = 1/3 would
    # not be bf16, so take h = 1 with n = 2 (y = -h)
    h_new, _, _ = boundary(np.ones((1, 2)), -np.ones((1, 2)), np.ones(2), np.ones(2), 2, 0.0)
    assert np.all(h_new == 0.0)
