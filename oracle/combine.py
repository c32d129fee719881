"""Weighted top-k combine.

TokenSpeed blog, "TensorRT-LLM NVFP4 MoE": the MoE kernel computes the weighted
sum of expert outputs for each token, using the FP32 routing weights. The vLLM
Beam summary (kernel change 3) combines the top-8 expert outputs per token.
y[t] = sum_k w[t, k] * Y_perm[inv_perm[t*K + k]], in float64.
"""
from __future__ import annotations

import numpy as np


def combine(Y_perm: np.ndarray, w: np.ndarray, inv_perm: np.ndarray) -> np.ndarray:
    w = np.asarray(w, dtype=np.float64)
    T, K = w.shape
    Y_perm = np.asarray(Y_perm, dtype=np.float64)
    y = np.zeros((T, Y_perm.shape[1]), dtype=np.float64)
    for t in range(T):
        for k in range(K):
            y[t] += w[t, k] * Y_perm[int(inv_perm[t * K + k])]
    return y
