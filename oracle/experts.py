"""Routed SwiGLU experts.

Sources: the vLLM Beam summary ("MoE and residual stream") gives 256 routed
experts with d_ff 2560 and no shared expert; the TokenSpeed blog ("TensorRT-LLM
NVFP4 MoE") runs both expert GEMMs with SwiGLU fused into the first and
computes the weighted sum of expert outputs per token. The Gaudi cookbook port
mentions the 2560-wide intermediate that feeds the down projection.

Per expert e with gate W_g [F][H], up W_u [F][H] and down W_d [H][F]:
    g = X W_g^T,  u = X W_u^T,  a = silu(g) * u,  Y = a W_d^T,
with silu(v) = v * sigmoid(v). Everything is float64 and unrounded.
"""
from __future__ import annotations

from concurrent.futures import ThreadPoolExecutor
from typing import Callable, Optional, Tuple

import numpy as np

from .bf16 import decode


def silu(v: np.ndarray) -> np.ndarray:
    v = np.asarray(v, dtype=np.float64)
    return v / (1.0 + np.exp(-v))


def swiglu_ffn(X: np.ndarray, Wg: np.ndarray, Wu: np.ndarray, Wd: np.ndarray) -> np.ndarray:
    """One expert's SwiGLU FFN on rows X [n][H] -> [n][H] (float64)."""
    X = np.asarray(X, dtype=np.float64)
    g = X @ np.asarray(Wg, dtype=np.float64).T
    u = X @ np.asarray(Wu, dtype=np.float64).T
    a = silu(g) * u
    return a @ np.asarray(Wd, dtype=np.float64).T


def intermediate(X: np.ndarray, Wg: np.ndarray, Wu: np.ndarray) -> np.ndarray:
    """a = silu(X W_g^T) * (X W_u^T), the input of the down projection."""
    X = np.asarray(X, dtype=np.float64)
    return silu(X @ np.asarray(Wg, dtype=np.float64).T) * (X @ np.asarray(Wu, dtype=np.float64).T)


def decoded_expert(W_gu_bits: np.ndarray, W_d_bits: np.ndarray, e: int, F: int):
    """Expert e's (W_g, W_u, W_d) in float64 from the packed bf16 arrays
    W_gu [E][2F][H] (gate rows then up rows) and W_d [E][H][F]."""
    gu = decode(W_gu_bits[e])
    return gu[:F], gu[F:], decode(W_d_bits[e])


ExpertFn = Callable[[int], Tuple[np.ndarray, np.ndarray, np.ndarray]]


def expert_outputs(z: np.ndarray, perm_token: np.ndarray, offsets: np.ndarray,
                   expert_fn: ExpertFn, workers: Optional[int] = None) -> np.ndarray:
    """Y_perm [T*K][H]: row p is FFN_e(z[perm_token[p]]) for the expert e whose
    range [offsets[e], offsets[e+1]) holds p."""
    z = np.asarray(z, dtype=np.float64)
    E = offsets.shape[0] - 1
    Y = np.zeros((perm_token.shape[0], z.shape[1]), dtype=np.float64)

    def one(e: int) -> None:
        lo, hi = int(offsets[e]), int(offsets[e + 1])
        if hi > lo:
            Wg, Wu, Wd = expert_fn(e)
            Y[lo:hi] = swiglu_ffn(z[perm_token[lo:hi]], Wg, Wu, Wd)

    _run(one, range(E), workers)
    return Y


def _run(fn, items, workers: Optional[int]) -> None:
    items = list(items)
    if not workers or workers <= 1:
        for it in items:
            fn(it)
    else:
        with ThreadPoolExecutor(workers) as ex:
            list(ex.map(fn, items))
