"""FP32 router, sigmoid scores, correction bias, group-limited top-k, weights.

Sources:
* vLLM Beam summary, section "MoE and residual stream": 256 routed experts,
  routing as in DeepSeek-V3 -- sigmoid scores and a correction bias pick the
  top 4 of 8 expert groups, then the top 8 experts; renormalised weights are
  scaled by 2.5; no shared expert; the 5120 x 256 router runs fully in FP32;
* TokenSpeed blog, "Model architecture and precision -> Architecture": the
  bias affects expert selection only; "Fused FP32 routing": BF16 activations
  times FP32 weights give FP32 scores, then sigmoid, bias addition, group
  top-k and final weights including the routed scale 2.5;
* Gaudi cookbook port, "What was built -> Model code": the bias is close to a
  constant of about 28, so bf16 loses the differences that pick experts;
  EP 8 holds "one group per card" with 32 experts per card, i.e. groups are
  contiguous blocks of E/G experts.

Readings taken where the pages are silent:
* group score = sum of the two largest biased scores in the group (the
  DeepSeek-V3 rule the pages name); ``rule="max"`` is offered for comparison;
* ties go to the lower group index and to the lower expert index; chosen
  experts are listed in descending biased score;
* w_k = scale * s_k / sum_j s_j over the chosen experts, using the unbiased
  sigmoid scores (s > 0, so no epsilon is needed).

The oracle decides in float64. ``margins`` reports how close each token's
decision was, so a comparison with an FP32 implementation can separate
near-ties (where both answers are valid) from real disagreements.
"""
from __future__ import annotations

import numpy as np


def router_logits(z: np.ndarray, W_r: np.ndarray) -> np.ndarray:
    """logits[t, e] = sum_h z[t, h] * W_r[e, h] in float64 (bf16 x fp32 products are exact)."""
    return np.asarray(z, dtype=np.float64) @ np.asarray(W_r, dtype=np.float64).T


def sigmoid(v: np.ndarray) -> np.ndarray:
    return 1.0 / (1.0 + np.exp(-np.asarray(v, dtype=np.float64)))


def group_scores(sb: np.ndarray, G: int, rule: str = "top2sum") -> np.ndarray:
    """Score of each of G contiguous groups from one token's biased scores."""
    E = sb.shape[0]
    per = E // G
    out = np.empty(G, dtype=np.float64)
    for g in range(G):
        vals = sorted(sb[g * per:(g + 1) * per].tolist(), reverse=True)
        if rule == "top2sum":
            out[g] = sum(vals[:min(2, per)])
        elif rule == "max":
            out[g] = vals[0]
        else:
            raise ValueError(rule)
    return out


def select_token(sb: np.ndarray, G: int, TG: int, K: int, rule: str = "top2sum"):
    """Group-limited top-k for one token.

    Returns (ids, groups, group_margin, expert_margin): ids in slot order
    (descending biased score, ties to the lower index), the chosen groups in
    order, the gap between the TG-th and (TG+1)-th group scores, and the
    smallest gap between consecutive biased scores among the first K+1
    candidates (it covers both the set boundary and the slot order).
    """
    E = sb.shape[0]
    per = E // G
    gs = group_scores(sb, G, rule)
    gorder = sorted(range(G), key=lambda g: (-gs[g], g))
    groups = gorder[:TG]
    gmargin = gs[gorder[TG - 1]] - gs[gorder[TG]] if TG < G else np.inf
    cand = [e for g in sorted(groups) for e in range(g * per, (g + 1) * per)]
    corder = sorted(cand, key=lambda e: (-sb[e], e))
    ids = corder[:K]
    top = [sb[e] for e in corder[:K + 1]]
    emargin = min((top[j] - top[j + 1] for j in range(len(top) - 1)), default=np.inf)
    return ids, groups, gmargin, emargin


def route(logits: np.ndarray, bias: np.ndarray, G: int, TG: int, K: int,
          routed_scale: float = 2.5, rule: str = "top2sum"):
    """Routing for a batch of tokens from float64 logits [T][E].

    Returns a dict with ids [T][K] int32, weights [T][K] float64, scores s,
    biased scores sb, chosen groups [T][TG] and the two margins [T].
    """
    logits = np.atleast_2d(np.asarray(logits, dtype=np.float64))
    T, E = logits.shape
    s = sigmoid(logits)
    sb = s + np.asarray(bias, dtype=np.float64)[None, :]
    ids = np.empty((T, K), dtype=np.int32)
    w = np.empty((T, K), dtype=np.float64)
    groups = np.empty((T, TG), dtype=np.int32)
    gm = np.empty(T)
    em = np.empty(T)
    for t in range(T):
        sel, grp, gm[t], em[t] = select_token(sb[t], G, TG, K, rule)
        ids[t] = sel
        groups[t] = grp
        chosen = s[t, sel]
        w[t] = routed_scale * chosen / chosen.sum()
    return {"ids": ids, "w": w, "s": s, "sb": sb, "groups": groups,
            "group_margin": gm, "expert_margin": em}


def near_tie(route_out: dict, threshold: float = 1e-5) -> np.ndarray:
    """Tokens whose group or expert decision is within ``threshold``."""
    return (route_out["group_margin"] <= threshold) | (route_out["expert_margin"] <= threshold)
