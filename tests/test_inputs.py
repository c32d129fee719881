"""The seeded input generator: deterministic, per-tensor streams, stated distributions."""
import numpy as np

from beam_inputs import (CONFIGS, bits_to_float32, expert_weights, make_activations,
                         make_all_expert_weights, make_norm_weights, make_router, random_topk_ids,
                         sample_tokens)


def test_deterministic_and_independent_streams():
    cfg = CONFIGS["toy"]
    h1, x1 = make_activations(cfg)
    h2, x2 = make_activations(cfg)
    assert np.array_equal(h1, h2) and np.array_equal(x1, x2)
    assert not np.array_equal(h1, x1)
    h3, _ = make_activations(cfg, batch=1)
    assert not np.array_equal(h1, h3)


def test_distributions():
    cfg = CONFIGS["decode_t64"]
    h, x = make_activations(cfg)
    hv = bits_to_float32(h)
    assert h.shape == (64, 5120) and abs(hv.mean()) < 0.01 and abs(hv.std() - 1) < 0.01
    wp, wq = make_norm_weights(cfg)
    assert abs(bits_to_float32(wp).std() - 0.02) < 0.002
    W, b = make_router(cfg)
    assert W.dtype == np.float32 and W.shape == (256, 5120)
    assert abs(W.std() * np.sqrt(5120) - 1) < 0.01
    assert abs(b.mean() - 28) < 1e-3 and 0.5e-3 < b.std() < 1.5e-3


def test_zipf_bias_and_shared_direction():
    cfg = CONFIGS["prefill_t16384"]
    _, b = make_router(cfg)
    off = np.sort(b.astype(np.float64) - 28)[::-1]
    # fp32 spacing at 28 is 1.9e-6
    np.testing.assert_allclose(off[:3], 0.05 * np.arange(1, 4) ** -1.1, rtol=0, atol=2e-6)
    s = sample_tokens(cfg)
    assert s.size == 512 and np.all(np.diff(s) > 0) and s[-1] < cfg.T
    c4 = CONFIGS["prefill_t2048"].with_(T=8)
    h, x = make_activations(c4)
    hx = bits_to_float32(h).astype(np.float64)
    # a shared direction makes rows correlate
    cos = hx[0] @ hx[1] / np.linalg.norm(hx[0]) / np.linalg.norm(hx[1])
    assert cos > 0.0


def test_packed_experts_match_single_expert_draws():
    cfg = CONFIGS["toy"]
    W_gu, W_d = make_all_expert_weights(cfg, workers=4, cache=False)
    for e in (0, 7, 15):
        g, u, d = expert_weights(cfg, e)
        assert np.array_equal(W_gu[e, :cfg.F], g) and np.array_equal(W_gu[e, cfg.F:], u)
        assert np.array_equal(W_d[e], d)
    std = bits_to_float32(W_gu).std() * np.sqrt(cfg.H)
    assert abs(std - 1) < 0.02


def test_random_ids_are_distinct_per_token():
    ids = random_topk_ids(100, 32, 8, seed=3, skew=1.0)
    assert all(len(set(r)) == 8 for r in ids.tolist())
    assert ids.min() >= 0 and ids.max() < 32
