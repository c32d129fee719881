"""Token permutation by expert.

The vLLM Beam summary ("The fused decoding graph runs one MoE layer in 13
kernels") lists two routing kernels and two grouped GEMMs for the MoE path; a
grouped GEMM needs the (token, slot) pairs of each expert stored contiguously.
Reading taken: the pairs i = t*K + k are ordered by the key (expert, t) -- a
stable counting sort by expert -- and offsets[e] is the exclusive prefix sum
of the per-expert counts.
"""
from __future__ import annotations

import numpy as np


def permute(ids: np.ndarray, E: int):
    """ids [T][K] -> (counts [E], offsets [E+1], perm_token [T*K], inv_perm [T*K]).

    perm_token[p] is the token whose row sits at permuted position p;
    inv_perm[t*K + k] is the position of token t's k-th slot.
    """
    ids = np.asarray(ids)
    T, K = ids.shape
    flat = [int(v) for v in ids.reshape(-1)]
    if any(e < 0 or e >= E for e in flat):
        raise ValueError("expert id out of range")
    order = sorted(range(T * K), key=lambda i: (flat[i], i))
    counts = np.zeros(E, dtype=np.int32)
    for e in flat:
        counts[e] += 1
    offsets = np.zeros(E + 1, dtype=np.int32)
    for e in range(E):
        offsets[e + 1] = offsets[e] + counts[e]
    perm_token = np.empty(T * K, dtype=np.int32)
    inv_perm = np.empty(T * K, dtype=np.int32)
    for p, i in enumerate(order):
        perm_token[p] = i // K
        inv_perm[i] = p
    return counts, offsets, perm_token, inv_perm
