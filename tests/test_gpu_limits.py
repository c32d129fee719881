"""The largest supported shapes against the fp64 oracle: hidden size 8192
(1024 threads per boundary block) and 16 experts per token out of 64 in 8
groups, which takes the general routing, top-k and combine kernels rather
than Beam's specialised ones."""
import functools

import numpy as np
import pytest

from beam_inputs import BeamConfig, make_activations, make_norm_weights
from oracle import bf16 as obf
from oracle.boundary import boundary
from oracle.routing import near_tie
from tests.gpu_support import (Model, assert_bf16_within_ulp, beam_module, bits_of, dev_bf16, f64_of, layer_errors,
                               require_gpu)

pytestmark = pytest.mark.gpu


@functools.lru_cache(maxsize=None)
def limit_model() -> Model:
    require_gpu()
    return Model(BeamConfig("limits", T=40, H=8192, E=64, G=8, TG=4, K=16, F=256, n=7))


@pytest.mark.parametrize("T", [1, 37, 1030])  # 1030: two chunks per thread from 1024 tokens
def test_boundary_at_the_largest_hidden_size(T):
    beam = beam_module()
    cfg = limit_model().cfg.with_(T=T)
    h_bits, x_bits = make_activations(cfg, batch=900 + T)
    wp, wq = make_norm_weights(cfg)
    h_out, z = beam.beam_boundary_norm(dev_bf16(h_bits), dev_bf16(x_bits), dev_bf16(wp), dev_bf16(wq), cfg.eps,
                                       cfg.n)
    ref_h, ref_z, _ = boundary(obf.decode(h_bits), obf.decode(x_bits), obf.decode(wp), obf.decode(wq), cfg.n,
                               cfg.eps)
    assert_bf16_within_ulp(bits_of(h_out), ref_h, 1, "h'")
    assert_bf16_within_ulp(bits_of(z), ref_z, 1, "z")


def test_layer_at_the_largest_hidden_size_and_top_k():
    beam = beam_module()
    m = limit_model()
    cfg = m.cfg
    h_out, y, dbg = beam.beam_moe_layer(m.h(), m.x(), cfg.n, m.weights, m.mc, debug=True)
    assert beam.beam_get_device_error() == 0
    ref = m.oracle_layer()
    assert_bf16_within_ulp(bits_of(h_out), ref["h_new"], 1, "h'")
    ids = dbg["topk_ids"].cpu().numpy()
    tie = near_tie(ref["route"])
    same = np.all(ids == ref["ids"], axis=1)
    assert np.all(same | tie), f"{int((~same & ~tie).sum())} non-near-tie tokens routed differently"
    w = dbg["topk_w"].cpu().numpy()
    assert np.allclose(w.sum(axis=1), cfg.routed_scale, rtol=1e-5)
    yg = f64_of(y)
    mx, rel = layer_errors(yg[same], ref["y"][same])
    assert mx <= 2e-2 and rel <= 5e-3, (mx, rel)
    if (~same).any():
        tokens = np.nonzero(~same)[0]
        cond = m.oracle_layer(tokens=tokens, ids_override=ids[~same])
        mx2, rel2 = layer_errors(yg[~same], cond["y"])
        assert mx2 <= 2e-2 and rel2 <= 5e-3, (mx2, rel2)
