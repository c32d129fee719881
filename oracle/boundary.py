"""Sandwich-norm boundary: post-norm -> depth-scaled residual -> next pre-norm.

Sources:
* vLLM Beam summary, section "MoE and residual stream": every sublayer has an
  RMSNorm before and after it, and the n-th residual add computes
  h <- sqrt((n-1)/n) * h + x / sqrt(n) instead of h + x, so unit-variance
  sublayer outputs keep the residual stream at unit variance;
* same page, kernel change 1: post-norm, scaled residual add and the next
  pre-norm run as one fused step with FP32 math and the reference's BF16
  rounding points;
* TokenSpeed blog, section "MNNVL all-reduce and SandwichNorm fusion": the
  order is post-norm, depth-scaled residual addition, next pre-norm;
* Gaudi cookbook port, "What was built -> Model code": the reference rounds to
  bf16 after the sandwich norms and the depth-scaled residuals.

Reading taken where the pages are silent: RMSNorm is x / sqrt(mean(x^2) + eps)
times the weight, the weight applied before the single rounding; exactly three
rounding points (post-norm output y, new residual h', pre-norm output z).

The residual add is evaluated as (sqrt(n-1) * h + y) / sqrt(n), the same real
number as sqrt((n-1)/n) * h + y / sqrt(n). In this form float64 is exact
whenever n-1 is a perfect square (n = 2, 5, 10, 17, ...), where h and y can
cancel exactly and the result must be exactly 0; for other n the cancellation
between bf16 inputs is bounded and float64 keeps far more than bf16 precision.
"""
from __future__ import annotations

import numpy as np

from .bf16 import round_bf16


def residual_coefficients(n: int):
    """(a, b) = (sqrt((n-1)/n), 1/sqrt(n)) for the n-th residual add, n >= 1."""
    if n < 1:
        raise ValueError("boundary index n must be >= 1")
    return np.sqrt((n - 1) / n), 1.0 / np.sqrt(n)


def residual(h, y, n: int) -> np.ndarray:
    """sqrt((n-1)/n) * h + y / sqrt(n), unrounded, as (sqrt(n-1) h + y) / sqrt(n)."""
    if n < 1:
        raise ValueError("boundary index n must be >= 1")
    return (np.sqrt(float(n - 1)) * np.asarray(h, dtype=np.float64) + np.asarray(y, dtype=np.float64)) / np.sqrt(
        float(n))


def rmsnorm(v: np.ndarray, w: np.ndarray, eps: float) -> np.ndarray:
    """Row-wise RMSNorm in float64: v / sqrt(mean(v^2) + eps) * w (no rounding)."""
    v = np.asarray(v, dtype=np.float64)
    ms = np.mean(v * v, axis=-1, keepdims=True)
    return v / np.sqrt(ms + eps) * np.asarray(w, dtype=np.float64)


def boundary(h, x, w_post, w_pre, n: int, eps: float):
    """One sandwich-norm boundary on float64 arrays holding bf16 values.

    Returns (h_new, z, y): the new residual, the next sublayer's normalised
    input and the post-normed sublayer output, each rounded to bf16 once.
    """
    y = round_bf16(rmsnorm(x, w_post, eps))
    h_new = round_bf16(residual(h, y, n))
    z = round_bf16(rmsnorm(h_new, w_pre, eps))
    return h_new, z, y
