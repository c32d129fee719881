"""Pins for the oracle's SwiGLU experts and the whole-layer composition."""
import math

import numpy as np
import torch

from beam_inputs import (CONFIGS, expert_weights, make_activations, make_all_expert_weights, make_norm_weights,
                         make_router)
from oracle import bf16
from oracle.boundary import boundary
from oracle.combine import combine
from oracle.experts import decoded_expert, expert_outputs, intermediate, silu, swiglu_ffn
from oracle.layer import layer
from oracle.permute import permute


def test_silu_matches_library():
    v = np.linspace(-40, 40, 2001)
    ref = torch.nn.functional.silu(torch.from_numpy(v)).numpy()
    np.testing.assert_allclose(silu(v), ref, rtol=1e-15, atol=1e-300)
    assert silu(np.array([0.0]))[0] == 0.0


def test_swiglu_structure_with_selection_matrices():
    # gate rows pick column c_f with gain s_f, up rows pick column d_f, down
    # rows pick intermediate p_j: then Y_j = silu(s_{p_j} x_{c_{p_j}}) x_{d_{p_j}}.
    rng = np.random.default_rng(12)
    H, F = 6, 4
    c, d, s = [5, 0, 2, 2], [1, 3, 4, 0], [0.5, -2.0, 1.5, 3.0]
    p = [2, 0, 3, 1, None, 0]
    Wg, Wu, Wd = np.zeros((F, H)), np.zeros((F, H)), np.zeros((H, F))
    for f in range(F):
        Wg[f, c[f]] = s[f]
        Wu[f, d[f]] = 1.0
    for j in range(H):
        if p[j] is not None:
            Wd[j, p[j]] = 1.0
    X = rng.standard_normal((3, H))
    Y = swiglu_ffn(X, Wg, Wu, Wd)
    for t in range(3):
        for j in range(H):
            if p[j] is None:
                assert Y[t, j] == 0.0
                continue
            f = p[j]
            g = s[f] * X[t, c[f]]
            expect = g / (1.0 + math.exp(-g)) * X[t, d[f]]
            assert abs(Y[t, j] - expect) <= 1e-15 * max(1.0, abs(expect))


def test_swiglu_homogeneity_and_linearity():
    rng = np.random.default_rng(13)
    X = rng.standard_normal((5, 16))
    Wg, Wu = rng.standard_normal((8, 16)), rng.standard_normal((8, 16))
    Wd1, Wd2 = rng.standard_normal((16, 8)), rng.standard_normal((16, 8))
    Y = swiglu_ffn(X, Wg, Wu, Wd1)
    np.testing.assert_allclose(swiglu_ffn(X, Wg, 3 * Wu, Wd1), 3 * Y, rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(swiglu_ffn(X, Wg, Wu, Wd1 + Wd2), Y + swiglu_ffn(X, Wg, Wu, Wd2),
                               rtol=1e-12, atol=1e-12)
    assert np.all(swiglu_ffn(X, np.zeros_like(Wg), Wu, Wd1) == 0.0)
    assert np.array_equal(intermediate(X, Wg, Wu) @ Wd1.T, Y)


def _toy():
    cfg = CONFIGS["toy"]
    h, x = make_activations(cfg)
    wp, wq = make_norm_weights(cfg)
    W, b = make_router(cfg)
    cache = {}

    def fn(e):
        if e not in cache:
            cache[e] = tuple(bf16.decode(m) for m in expert_weights(cfg, e))
        return cache[e]
    args = (bf16.decode(h), bf16.decode(x), bf16.decode(wp), bf16.decode(wq), W, b)
    kw = dict(n=cfg.n, eps=cfg.eps, G=cfg.G, TG=cfg.TG, K=cfg.K, routed_scale=cfg.routed_scale)
    return cfg, args, kw, fn


def test_identical_experts_give_scale_times_one_ffn():
    # sum_k w_k = 2.5, so if every expert is the same FFN the layer output is
    # 2.5 * FFN(z) whatever the routing decided.
    cfg, args, kw, fn = _toy()
    out = layer(*args, **kw, expert_fn=lambda e: fn(0))
    ref = 2.5 * swiglu_ffn(out["z"], *fn(0))
    np.testing.assert_allclose(out["y"], ref, rtol=1e-12, atol=1e-12)


def test_permuted_path_equals_per_token_definition():
    cfg, args, kw, fn = _toy()
    out = layer(*args, **kw, expert_fn=fn)
    _, offsets, perm, inv = permute(out["ids"], cfg.E)
    y2 = combine(expert_outputs(out["z"], perm, offsets, fn), out["w"], inv)
    np.testing.assert_allclose(out["y"], y2, rtol=1e-12, atol=1e-12)


def test_token_subset_matches_full_batch():
    cfg, args, kw, fn = _toy()
    full = layer(*args, **kw, expert_fn=fn)
    idx = np.array([1, 5, 11])
    sub = layer(*args, **kw, expert_fn=fn, tokens=idx)
    for key in ("h_new", "z", "ids"):
        assert np.array_equal(sub[key], full[key][idx])
    np.testing.assert_allclose(sub["y"], full["y"][idx], rtol=1e-12, atol=1e-12)


def test_layer_boundary_and_override():
    cfg, args, kw, fn = _toy()
    out = layer(*args, **kw, expert_fn=fn)
    h_new, z, _ = boundary(args[0], args[1], args[2], args[3], cfg.n, cfg.eps)
    assert np.array_equal(out["h_new"], h_new) and np.array_equal(out["z"], z)
    same = layer(*args, **kw, expert_fn=fn, ids_override=out["ids"])
    np.testing.assert_allclose(same["y"], out["y"], rtol=1e-13, atol=1e-13)
    # the output magnitude is O(1) for unit-variance inputs and 1/sqrt(fan_in) weights
    assert 0.05 < np.sqrt(np.mean(out["y"] ** 2)) < 5


def test_decoded_expert_reads_gate_up_and_down_planes():
    # The packed arrays the C ABI takes (W_gu [E][2F][H]: gate rows, then up
    # rows; W_down [E][H][F]) are unpacked by the oracle into the same three
    # matrices the generator draws for each expert, gate and up separately.
    cfg = CONFIGS["toy"].with_(E=6, G=3, F=64, H=128)
    W_gu, W_d = make_all_expert_weights(cfg, workers=1, cache=False)
    for e in (0, 2, 5):
        g_bits, u_bits, d_bits = expert_weights(cfg, e)
        Wg, Wu, Wd = decoded_expert(W_gu, W_d, e, cfg.F)
        assert Wg.shape == (cfg.F, cfg.H) and Wu.shape == (cfg.F, cfg.H) and Wd.shape == (cfg.H, cfg.F)
        assert np.array_equal(Wg, bf16.decode(g_bits))
        assert np.array_equal(Wu, bf16.decode(u_bits))
        assert np.array_equal(Wd, bf16.decode(d_bits))
        # the three draws differ, so a swapped or shifted plane cannot pass
        assert not np.array_equal(Wg, Wu)
    other = decoded_expert(W_gu, W_d, 1, cfg.F)
    assert not np.array_equal(other[0], bf16.decode(expert_weights(cfg, 0)[0]))
