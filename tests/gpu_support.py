"""Helpers shared by the GPU parity tests: device copies of the seeded inputs,
comparisons against the oracle, and a per-process cache of the Beam expert
weights (20 GB on the device, generated and uploaded once)."""
from __future__ import annotations

import functools
import os
from typing import Optional

import numpy as np
import pytest
import torch

from beam_inputs import (BeamConfig, CONFIGS, make_activations, make_all_expert_weights, make_norm_weights,
                         make_router)
from oracle import bf16 as obf
from oracle.experts import decoded_expert

WORKERS = max(1, min(32, len(os.sched_getaffinity(0))))


def require_gpu():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")


@functools.lru_cache(maxsize=None)
def beam_module():
    require_gpu()
    from routed_expert_layer_post_gb300 import build as b
    b.build()
    import routed_expert_layer_post_gb300 as m
    m.library()
    return m


def dev_bf16(bits: np.ndarray) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).cuda().view(torch.bfloat16)


def bits_of(t: torch.Tensor) -> np.ndarray:
    return t.contiguous().view(torch.int16).cpu().numpy().view(np.uint16)


def f64_of(t: torch.Tensor) -> np.ndarray:
    if t.dtype == torch.bfloat16:
        return obf.decode(bits_of(t))
    return t.cpu().numpy().astype(np.float64)


def moe_config(cfg: BeamConfig):
    m = beam_module()
    return m.make_config(cfg.H, cfg.E, cfg.G, cfg.TG, cfg.K, cfg.F, cfg.routed_scale, cfg.eps)


class Model:
    """Seeded inputs and weights of one configuration, on host and device."""

    def __init__(self, cfg: BeamConfig):
        self.cfg = cfg
        self.h_bits, self.x_bits = make_activations(cfg)
        self.wp_bits, self.wq_bits = make_norm_weights(cfg)
        self.W_r, self.bias = make_router(cfg)
        self.W_gu_bits, self.W_d_bits = make_all_expert_weights(cfg, workers=WORKERS)
        self.dev = _device_weights(cfg.seed, cfg.E, cfg.F, cfg.H)
        self.w_post = dev_bf16(self.wp_bits)
        self.w_pre = dev_bf16(self.wq_bits)
        self.router_w = torch.from_numpy(self.W_r).cuda()
        self.bias_d = torch.from_numpy(self.bias).cuda()
        m = beam_module()
        self.mc = moe_config(cfg)
        self.weights = m.weights_struct(self.w_post, self.w_pre, self.router_w, self.bias_d, self.dev[0],
                                        self.dev[1])
        self._cache = {}

    def h(self):
        return dev_bf16(self.h_bits)

    def x(self):
        return dev_bf16(self.x_bits)

    def expert_fn(self, e: int):
        if e not in self._cache:
            self._cache[e] = decoded_expert(self.W_gu_bits, self.W_d_bits, e, self.cfg.F)
        return self._cache[e]

    def expert_fn_nocache(self, e: int):
        return decoded_expert(self.W_gu_bits, self.W_d_bits, e, self.cfg.F)

    def oracle_layer(self, tokens: Optional[np.ndarray] = None, ids_override=None):
        from oracle.layer import layer
        c = self.cfg
        return layer(obf.decode(self.h_bits), obf.decode(self.x_bits), obf.decode(self.wp_bits),
                     obf.decode(self.wq_bits), self.W_r, self.bias, n=c.n, eps=c.eps, G=c.G, TG=c.TG, K=c.K,
                     routed_scale=c.routed_scale, expert_fn=self.expert_fn_nocache, tokens=tokens,
                     ids_override=ids_override, workers=WORKERS)


_DEV_WEIGHTS = {}


def _device_weights(seed: int, E: int, F: int, H: int):
    key = (seed, E, F, H)
    if key not in _DEV_WEIGHTS:
        cfg = BeamConfig("w", T=1, H=H, E=E, F=F, seed=seed)
        W_gu, W_d = make_all_expert_weights(cfg, workers=WORKERS)
        _DEV_WEIGHTS[key] = (dev_bf16(W_gu), dev_bf16(W_d))
    return _DEV_WEIGHTS[key]


@functools.lru_cache(maxsize=None)
def model(name: str) -> Model:
    require_gpu()
    return Model(CONFIGS[name])


def assert_bf16_within_ulp(gpu_bits: np.ndarray, ref_f64: np.ndarray, ulps: int = 1, what: str = ""):
    d = obf.ulp_distance(gpu_bits, obf.encode(ref_f64))
    worst = int(d.max()) if d.size else 0
    assert worst <= ulps, f"{what}: {int((d > ulps).sum())} elements beyond {ulps} bf16 ulp (worst {worst})"


def layer_errors(y_gpu: np.ndarray, y_ref: np.ndarray):
    diff = np.abs(y_gpu - y_ref)
    rel = float(np.linalg.norm(y_gpu - y_ref) / max(np.linalg.norm(y_ref), 1e-300))
    return float(diff.max()) if diff.size else 0.0, rel
