"""Pins for the oracle's router, group-limited top-k and routing weights."""
import itertools
import json
import os

import numpy as np
import pytest

from beam_inputs import CONFIGS, make_activations, make_norm_weights, make_router
from oracle import bf16
from oracle.boundary import boundary
from oracle.routing import group_scores, near_tie, route, router_logits, sigmoid

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


@pytest.mark.parametrize("rule", ["top2sum", "max"])
def test_worked_example(rule):
    g = json.load(open(os.path.join(GOLDEN, "routing_group_topk.json")))
    for t in range(2):
        r = route(np.array([g["logits"][t]]), np.array(g["bias"][t]), g["G"], g["TG"], g["K"],
                  g["routed_scale"], rule)
        assert r["ids"][0].tolist() == g[rule]["ids"][t]
        assert r["groups"][0].tolist() == g[rule]["groups"][t]
        if rule == "top2sum":
            np.testing.assert_allclose(r["w"][0], g[rule]["w"][t], rtol=1e-13)


def _brute_force(sb, G, TG, K):
    """Enumerate every group subset and every expert subset; return the best sets."""
    E = sb.size
    per = E // G
    gs = [max(sb[g * per + i] + sb[g * per + j] for i in range(per) for j in range(per) if i != j)
          if per >= 2 else sb[g] for g in range(G)]
    best_groups = max(itertools.combinations(range(G), TG), key=lambda c: sum(gs[g] for g in c))
    cand = [e for g in best_groups for e in range(g * per, (g + 1) * per)]
    best = max(itertools.combinations(cand, K), key=lambda c: sum(sb[e] for e in c))
    return set(best_groups), set(best)


@pytest.mark.parametrize("E,G,TG,K", [(8, 4, 2, 3), (12, 3, 2, 4), (16, 4, 2, 4), (16, 8, 3, 5),
                                      (12, 6, 1, 2), (10, 5, 5, 6), (8, 2, 1, 4)])
def test_selection_equals_brute_force(E, G, TG, K):
    rng = np.random.default_rng(E * 100 + G * 10 + K)
    for _ in range(40):
        logits = rng.standard_normal((1, E)) * 2
        bias = 28 + 1e-3 * rng.standard_normal(E)
        r = route(logits, bias, G, TG, K)
        groups, experts = _brute_force(r["sb"][0], G, TG, K)
        assert set(r["groups"][0].tolist()) == groups
        assert set(r["ids"][0].tolist()) == experts


def _toy_routing():
    cfg = CONFIGS["toy"]
    h, x = make_activations(cfg)
    wp, wq = make_norm_weights(cfg)
    W, b = make_router(cfg)
    _, z, _ = boundary(bf16.decode(h), bf16.decode(x), bf16.decode(wp), bf16.decode(wq), cfg.n, cfg.eps)
    return cfg, route(router_logits(z, W), b, cfg.G, cfg.TG, cfg.K, cfg.routed_scale)


def test_invariants():
    cfg, r = _toy_routing()
    rng = np.random.default_rng(7)
    per = cfg.E // cfg.G
    r2 = route(rng.standard_normal((50, 256)), 28 + 1e-3 * rng.standard_normal(256), 8, 4, 8)
    for rr, G, K, per_ in ((r, cfg.G, cfg.K, per), (r2, 8, 8, 32)):
        np.testing.assert_allclose(rr["w"].sum(axis=1), 2.5, rtol=0, atol=1e-12)
        for t in range(rr["ids"].shape[0]):
            ids = rr["ids"][t].tolist()
            assert len(set(ids)) == K
            assert {e // per_ for e in ids} <= set(rr["groups"][t].tolist())
            sb = rr["sb"][t, ids]
            assert np.all(np.diff(sb) <= 0)
        assert np.all(rr["w"] > 0)


def test_zero_router_weight_closed_form():
    # W_r = 0 -> every score is sigmoid(0) = 1/2: the bias alone selects and
    # every weight is scale / K.
    rng = np.random.default_rng(8)
    bias = 28 + 1e-3 * rng.standard_normal(256)
    z = rng.standard_normal((3, 64))
    r = route(router_logits(z, np.zeros((256, 64))), bias, 8, 4, 8)
    assert np.all(r["w"] == 2.5 / 8)
    for t in range(3):
        gs = group_scores(bias + 0.5, 8)
        top_groups = sorted(range(8), key=lambda g: -gs[g])[:4]
        cand = [e for g in top_groups for e in range(32 * g, 32 * g + 32)]
        expect = sorted(cand, key=lambda e: -bias[e])[:8]
        assert r["ids"][t].tolist() == expect


def test_logits_select_the_right_operand_axes():
    # Router rows that are unit basis vectors pick single activation columns.
    rng = np.random.default_rng(9)
    z = rng.standard_normal((4, 10))
    W = np.zeros((6, 10))
    cols = [3, 0, 9, 9, 5, 1]
    for e, c in enumerate(cols):
        W[e, c] = 1.0
    assert np.array_equal(router_logits(z, W), z[:, cols])


def test_sigmoid_values():
    assert sigmoid(np.array([0.0]))[0] == 0.5
    np.testing.assert_allclose(sigmoid(np.log(np.array([3.0, 1 / 3.0]))), [0.75, 0.25], rtol=1e-15)
    v = np.linspace(-30, 30, 101)
    np.testing.assert_allclose(sigmoid(v) + sigmoid(-v), 1.0, rtol=0, atol=1e-15)


def test_bias_only_affects_selection():
    rng = np.random.default_rng(10)
    logits = rng.standard_normal((1, 16))
    r1 = route(logits, np.zeros(16), 4, 2, 4)
    ids = r1["ids"][0]
    s = 1 / (1 + np.exp(-logits[0, ids]))
    np.testing.assert_allclose(r1["w"][0], 2.5 * s / s.sum(), rtol=1e-15)
    # a large bias on one group forces its experts in, with unbiased weights
    bias = np.zeros(16)
    bias[12:16] = 5.0
    r2 = route(logits, bias, 4, 2, 4)
    assert 3 in r2["groups"][0].tolist()
    # every chosen expert lies in a chosen group, and both sets are the
    # exhaustive search's optimum for these biased scores
    assert {e // 4 for e in r2["ids"][0].tolist()} <= set(r2["groups"][0].tolist())
    groups, experts = _brute_force(r2["sb"][0], 4, 2, 4)
    assert set(r2["groups"][0].tolist()) == groups
    assert set(r2["ids"][0].tolist()) == experts
    # the forced group holds the four largest biased scores: all four are taken
    assert set(r2["ids"][0].tolist()) == {12, 13, 14, 15}
    chosen = r2["ids"][0]
    s2 = 1 / (1 + np.exp(-logits[0, chosen]))
    np.testing.assert_allclose(r2["w"][0], 2.5 * s2 / s2.sum(), rtol=1e-15)


def test_near_tie_flags():
    r = route(np.zeros((1, 8)), np.array([1.0, 1.0, 0, 0, 0, 0, 0, 0]), 4, 2, 2)
    assert near_tie(r)[0]            # groups 1..3 tie at the TG boundary
    r = route(np.zeros((1, 8)), np.array([3.0, 2.0, 1.0, 0.5, 0, 0, 0, 0]), 4, 2, 2)
    assert not near_tie(r)[0]
