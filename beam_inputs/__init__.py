"""Seeded synthetic inputs for the Beam MoE sublayer.

This module only draws random numbers and packs them into the layouts that the
library's C ABI documents. It contains none of the sublayer's arithmetic (no
normalisation, routing, permutation, GEMM or combine), so both the fp64 oracle
and the GPU path can take their inputs from here without sharing any of the
method.

Shapes follow the Beam 501B-A23B MoE sublayer as the TokenSpeed blog on
Reflection Beam describes it (section "Model architecture and precision ->
Architecture": 256 routed experts, 8 active, top 4 of 8 groups, routed scale
2.5) and the vLLM Beam summary (section "MoE and residual stream": hidden 5120,
d_ff 2560, FP32 5120x256 router). The pages measured real layers and real
traffic; those are not available, so the recipes below stand in for them:

* residual ``h`` and sublayer output ``x``: bf16(N(0, 1)) rows; the
  ``shared_direction`` recipe adds ``shared_norm * u`` to every row of both,
  with ``u`` one seeded unit vector, so tokens correlate and expert loads vary;
* RMSNorm weights: bf16(1 + N(0, 0.02));
* router weight ``W_r`` [E][H]: fp32 N(0, std 1/sqrt(H));
* correction bias [E]: fp32 28 + N(0, 1e-3); the ``zipf`` recipe uses
  28 + amp * r**(-s) with r the 1-based rank of the expert under a seeded
  permutation;
* expert weights: bf16 N(0, std 1/sqrt(fan_in)) (fan_in H for gate/up, F for
  down).

Every tensor has its own ``numpy.random.SeedSequence`` stream keyed by
``(seed, stream id[, expert, matrix])`` so that any one expert can be
regenerated on its own. bf16 values are produced with PyTorch's CPU
float32 -> bfloat16 conversion (round to nearest even) and handed out as
uint16 bit patterns.
"""
from __future__ import annotations

import dataclasses
import os
from concurrent.futures import ThreadPoolExecutor
from typing import Dict, Optional, Tuple

import numpy as np

__all__ = [
    "BeamConfig", "CONFIGS", "make_activations", "shared_direction", "make_norm_weights",
    "make_router", "expert_weights", "make_all_expert_weights",
    "sample_tokens", "random_topk_ids", "to_bf16_bits", "bits_to_float32",
]

# stream ids inside SeedSequence(seed, spawn_key=(stream, ...))
_S_H, _S_X, _S_WPOST, _S_WPRE, _S_WR, _S_BIAS, _S_DIR, _S_ZIPF, _S_SAMPLE, _S_EXPERT, _S_IDS = range(11)


@dataclasses.dataclass(frozen=True)
class BeamConfig:
    """One synthetic workload of the MoE sublayer.

    T tokens, hidden H, E routed experts in G contiguous groups, top TG groups
    then top K experts, SwiGLU width F, boundary index n (1-based residual
    add), RMSNorm eps and the routed scale.
    """
    name: str
    T: int
    H: int = 5120
    E: int = 256
    G: int = 8
    TG: int = 4
    K: int = 8
    F: int = 2560
    n: int = 20
    eps: float = 1e-6
    routed_scale: float = 2.5
    activations: str = "iid"          # "iid" | "shared_direction"
    shared_norm: float = 0.0
    bias: str = "normal"              # "normal" | "zipf"
    bias_center: float = 28.0
    bias_std: float = 1e-3
    zipf_s: float = 1.1
    zipf_amp: float = 0.05
    oracle_sample: Optional[int] = None   # tokens the oracle checks (None: all)
    seed: int = 0

    def with_(self, **kw) -> "BeamConfig":
        return dataclasses.replace(self, **kw)

    @property
    def experts_per_group(self) -> int:
        return self.E // self.G

    def expert_bytes(self) -> int:
        """bf16 bytes of one expert's gate, up and down matrices."""
        return 2 * 3 * self.F * self.H


CONFIGS: Dict[str, BeamConfig] = {
    # toy sublayer: hidden 256, 16 experts in 4 groups, top 2 groups then top 4, d_ff 128
    "toy": BeamConfig("toy", T=16, H=256, E=16, G=4, TG=2, K=4, F=128, n=10),
    # Beam shapes, decode batch 1
    "decode_t1": BeamConfig("decode_t1", T=1, n=20),
    # Beam shapes, decode batch 64, iid activations (near-uniform routing)
    "decode_t64": BeamConfig("decode_t64", T=64, n=40),
    # Beam shapes, prefill chunk 2048, shared direction of norm 2
    "prefill_t2048": BeamConfig("prefill_t2048", T=2048, n=60,
                                activations="shared_direction", shared_norm=2.0),
    # Beam shapes, prefill 16384, Zipf-skewed correction bias, 512-token oracle sample
    "prefill_t16384": BeamConfig("prefill_t16384", T=16384, n=100, bias="zipf",
                                 oracle_sample=512),
}


def _rng(seed: int, *key: int) -> np.random.Generator:
    return np.random.Generator(np.random.PCG64(np.random.SeedSequence(seed, spawn_key=tuple(key))))


def to_bf16_bits(a: np.ndarray) -> np.ndarray:
    """float32 array -> bf16 bit patterns (uint16), round to nearest even (PyTorch CPU cast)."""
    import torch
    t = torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32))
    return t.to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)


def bits_to_float32(bits: np.ndarray) -> np.ndarray:
    """bf16 bit patterns -> float32 values (exact widening)."""
    return (np.asarray(bits, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32)


def make_activations(cfg: BeamConfig, T: Optional[int] = None, batch: int = 0) -> Tuple[np.ndarray, np.ndarray]:
    """Residual h and previous sublayer output x, bf16 bits [T][H].

    ``batch`` selects an independent draw of the same recipe (used to rotate
    inputs between timed steps)."""
    T = cfg.T if T is None else T
    h = _rng(cfg.seed, _S_H, batch).standard_normal((T, cfg.H), dtype=np.float32)
    x = _rng(cfg.seed, _S_X, batch).standard_normal((T, cfg.H), dtype=np.float32)
    u = shared_direction(cfg)
    if u is not None:
        h += u
        x += u
    return to_bf16_bits(h), to_bf16_bits(x)


def shared_direction(cfg: BeamConfig) -> Optional[np.ndarray]:
    """The vector ``shared_norm * u`` (float32 [H], u a seeded unit vector)
    that the ``shared_direction`` recipe adds to every row of h and x; None
    for iid activations."""
    if cfg.activations == "iid":
        return None
    if cfg.activations != "shared_direction":
        raise ValueError(cfg.activations)
    u = _rng(cfg.seed, _S_DIR).standard_normal(cfg.H).astype(np.float64)
    return (cfg.shared_norm * u / np.sqrt(np.dot(u, u))).astype(np.float32)


def make_norm_weights(cfg: BeamConfig) -> Tuple[np.ndarray, np.ndarray]:
    """Post-norm and pre-norm weights, bf16 bits [H], drawn as 1 + N(0, 0.02)."""
    wp = 1.0 + 0.02 * _rng(cfg.seed, _S_WPOST).standard_normal(cfg.H, dtype=np.float32)
    wq = 1.0 + 0.02 * _rng(cfg.seed, _S_WPRE).standard_normal(cfg.H, dtype=np.float32)
    return to_bf16_bits(wp), to_bf16_bits(wq)


def make_router(cfg: BeamConfig) -> Tuple[np.ndarray, np.ndarray]:
    """Router weight fp32 [E][H] (std 1/sqrt(H)) and correction bias fp32 [E]."""
    W = (_rng(cfg.seed, _S_WR).standard_normal((cfg.E, cfg.H), dtype=np.float64)
         / np.sqrt(cfg.H)).astype(np.float32)
    if cfg.bias == "normal":
        b = cfg.bias_center + cfg.bias_std * _rng(cfg.seed, _S_BIAS).standard_normal(cfg.E)
    elif cfg.bias == "zipf":
        order = _rng(cfg.seed, _S_ZIPF).permutation(cfg.E)
        rank = np.empty(cfg.E, dtype=np.float64)
        rank[order] = np.arange(1, cfg.E + 1, dtype=np.float64)
        b = cfg.bias_center + cfg.zipf_amp * rank ** (-cfg.zipf_s)
    else:
        raise ValueError(cfg.bias)
    return W, b.astype(np.float32)


def expert_weights(cfg: BeamConfig, e: int) -> Tuple[np.ndarray, np.ndarray, np.ndarray]:
    """One expert's (gate [F][H], up [F][H], down [H][F]) as bf16 bits."""
    F, H = cfg.F, cfg.H
    g = _rng(cfg.seed, _S_EXPERT, e, 0).standard_normal((F, H), dtype=np.float32)
    g *= np.float32(1.0 / np.sqrt(H))
    u = _rng(cfg.seed, _S_EXPERT, e, 1).standard_normal((F, H), dtype=np.float32)
    u *= np.float32(1.0 / np.sqrt(H))
    d = _rng(cfg.seed, _S_EXPERT, e, 2).standard_normal((H, F), dtype=np.float32)
    d *= np.float32(1.0 / np.sqrt(F))
    return to_bf16_bits(g), to_bf16_bits(u), to_bf16_bits(d)


_WEIGHT_CACHE: Dict[tuple, Tuple[np.ndarray, np.ndarray]] = {}


def make_all_expert_weights(cfg: BeamConfig, workers: Optional[int] = None,
                            cache: bool = True) -> Tuple[np.ndarray, np.ndarray]:
    """All experts packed for the C ABI, bf16 bits.

    Returns ``W_gu`` [E][2F][H] (rows 0..F-1 gate, F..2F-1 up) and ``W_down``
    [E][H][F]. Experts are drawn in parallel threads (numpy releases the GIL
    while filling); the result is cached per (seed, E, F, H)."""
    key = (cfg.seed, cfg.E, cfg.F, cfg.H)
    if cache and key in _WEIGHT_CACHE:
        return _WEIGHT_CACHE[key]
    E, F, H = cfg.E, cfg.F, cfg.H
    W_gu = np.empty((E, 2 * F, H), dtype=np.uint16)
    W_d = np.empty((E, H, F), dtype=np.uint16)

    def fill(e: int) -> None:
        g, u, d = expert_weights(cfg, e)
        W_gu[e, :F] = g
        W_gu[e, F:] = u
        W_d[e] = d

    if workers is None:
        workers = max(1, min(32, len(os.sched_getaffinity(0))))
    if workers == 1 or E == 1:
        for e in range(E):
            fill(e)
    else:
        import torch
        prev = torch.get_num_threads()
        torch.set_num_threads(1)
        try:
            with ThreadPoolExecutor(workers) as ex:
                list(ex.map(fill, range(E)))
        finally:
            torch.set_num_threads(prev)
    if cache:
        _WEIGHT_CACHE[key] = (W_gu, W_d)
    return W_gu, W_d


def sample_tokens(cfg: BeamConfig) -> np.ndarray:
    """Sorted token indices the oracle checks (all tokens when no sample is set)."""
    if cfg.oracle_sample is None or cfg.oracle_sample >= cfg.T:
        return np.arange(cfg.T, dtype=np.int64)
    idx = _rng(cfg.seed, _S_SAMPLE).choice(cfg.T, size=cfg.oracle_sample, replace=False)
    return np.sort(idx).astype(np.int64)


def random_topk_ids(T: int, E: int, K: int, seed: int = 0, skew: float = 0.0) -> np.ndarray:
    """Random expert ids [T][K] int32, distinct within each token.

    ``skew`` > 0 draws experts with probability proportional to
    (rank)**(-skew) so that some experts receive many tokens. Used to exercise
    the permutation and the grouped GEMM independently of routing."""
    rng = _rng(seed, _S_IDS, T, E, K)
    if skew > 0:
        p = np.arange(1, E + 1, dtype=np.float64) ** (-skew)
        p = p[rng.permutation(E)]
        p /= p.sum()
    else:
        p = None
    out = np.empty((T, K), dtype=np.int32)
    for t in range(T):
        out[t] = rng.choice(E, size=K, replace=False, p=p)
    return out
