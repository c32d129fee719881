"""The whole MoE sublayer at a sandwich-norm boundary, in float64.

Order of the steps (vLLM Beam summary, "MoE and residual stream" and kernel
changes 1 and 4; TokenSpeed blog, "Fused FP32 routing" and "TensorRT-LLM
NVFP4 MoE"):

1. boundary: y = norm_post(x), h' = sqrt((n-1)/n) h + y / sqrt(n),
   z = norm_pre(h'), each rounded to bf16;
2. router: FP32 logits z W_r^T, sigmoid, correction bias, top 4 of 8 groups,
   top 8 experts, renormalised weights times 2.5;
3. experts: SwiGLU FFN of each chosen expert on z;
4. combine: y_out[t] = sum_k w[t, k] FFN_{ids[t, k]}(z[t]).

Layer inputs are the residual h and the previous sublayer's output x; its
outputs are the new residual h' and the MoE output y_out, which the next
boundary takes as its x. Tokens are independent, so the oracle can run on any
subset of tokens (``tokens``) and still give exact per-token results.
"""
from __future__ import annotations

from typing import Callable, Optional

import numpy as np

from . import boundary as _boundary
from . import routing as _routing
from .experts import ExpertFn, _run, swiglu_ffn


def layer(h, x, w_post, w_pre, W_r, bias, *, n: int, eps: float, G: int, TG: int,
          K: int, routed_scale: float, expert_fn: Optional[ExpertFn] = None,
          tokens: Optional[np.ndarray] = None, ids_override: Optional[np.ndarray] = None,
          workers: Optional[int] = None, rule: str = "top2sum",
          ffn: Optional[Callable[[int, np.ndarray], np.ndarray]] = None) -> dict:
    """Run the sublayer on float64 inputs (bf16 values) for ``tokens`` (default: all).

    ``ids_override`` [len(tokens)][K] replaces the routing decision (weights
    are then recomputed from the unbiased scores of those ids); it is used to
    evaluate the layer output under another implementation's near-tie
    choices ("routing-conditioned" comparison).

    The experts are the bf16 SwiGLU FFN of ``expert_fn(e)``'s matrices, or,
    when ``ffn`` is given, ``ffn(e, rows)`` (the NVFP4 experts of
    ``oracle.nvfp4``).
    """
    if (expert_fn is None) == (ffn is None):
        raise ValueError("give exactly one of expert_fn and ffn")
    h = np.asarray(h, dtype=np.float64)
    x = np.asarray(x, dtype=np.float64)
    if tokens is not None:
        h, x = h[tokens], x[tokens]
    h_new, z, y_post = _boundary.boundary(h, x, w_post, w_pre, n, eps)
    logits = _routing.router_logits(z, W_r)
    r = _routing.route(logits, bias, G, TG, K, routed_scale, rule)
    ids, w = r["ids"], r["w"]
    if ids_override is not None:
        ids = np.asarray(ids_override, dtype=np.int32)
        chosen = np.take_along_axis(r["s"], ids.astype(np.int64), axis=1)
        w = routed_scale * chosen / chosen.sum(axis=1, keepdims=True)
    T = z.shape[0]
    y = np.zeros_like(z)
    E = np.asarray(bias).shape[0]
    parts = {}

    def one(e: int) -> None:
        rows, slots = np.nonzero(ids == e)
        if rows.size:
            if ffn is not None:
                parts[e] = (rows, slots, ffn(e, z[rows]))
            else:
                Wg, Wu, Wd = expert_fn(e)
                parts[e] = (rows, slots, swiglu_ffn(z[rows], Wg, Wu, Wd))

    _run(one, range(E), workers)
    # the weighted sum in slot order for every token
    contrib = np.zeros((T, K, z.shape[1]), dtype=np.float64)
    for e, (rows, slots, Y) in parts.items():
        contrib[rows, slots] = Y
    for k in range(K):
        y += w[:, k:k + 1] * contrib[:, k]
    return {"h_new": h_new, "z": z, "y_post": y_post, "logits": logits, "route": r,
            "ids": ids, "w": w, "y": y}
