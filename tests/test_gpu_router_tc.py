"""The layer's tensor-core FP32 router (more than 128 tokens): each fp32 router
weight split exactly into three bf16 terms, all three accumulated in fp32.
Logits must match the fp64 product of the layer's own z with the fp32 weights
within 1e-5 of the row's largest magnitude (the same bar as the SIMT router),
and the routing must follow from them (ids equal away from near-ties)."""
import numpy as np
import pytest
import torch

from beam_inputs import make_activations
from oracle.routing import near_tie, route
from tests.gpu_support import beam_module, dev_bf16, f64_of, model

pytestmark = pytest.mark.gpu


# token tiles of 32 (up to 4863 tokens), 64 (5000) and 128 (10000)
@pytest.mark.parametrize("T", [129, 1000, 2048, 5000, 10000])
def test_layer_tc_router_matches_fp64(T):
    beam = beam_module()
    m = model("decode_t64")
    cfg = m.cfg.with_(T=T)
    hb, xb = make_activations(cfg, batch=400 + T)
    _, _, dbg = beam.beam_moe_layer(dev_bf16(hb), dev_bf16(xb), cfg.n, m.weights, m.mc, debug=True)
    torch.cuda.synchronize()
    assert beam.beam_get_device_error() == 0
    z = f64_of(dbg["z"])
    L = z @ m.W_r.astype(np.float64).T
    gl = dbg["logits"].double().cpu().numpy()
    rowmax = np.abs(L).max(axis=1, keepdims=True)
    err = np.abs(gl - L) / rowmax
    print(f"T={T}: max row-relative logit error {err.max():.2e}")
    assert np.all(err <= 1e-5), float(err.max())
    r = route(L, m.bias, cfg.G, cfg.TG, cfg.K, cfg.routed_scale)
    ids = dbg["topk_ids"].cpu().numpy()
    same = np.all(ids == r["ids"], axis=1)
    assert np.all(same | near_tie(r))


def test_tc_router_logits_close_to_simt_router():
    # the standalone router entry point keeps the SIMT kernel; on the same z
    # both stay within the router's 1e-5 bar of each other
    beam = beam_module()
    m = model("decode_t64")
    cfg = m.cfg.with_(T=512)
    hb, xb = make_activations(cfg, batch=77)
    _, _, dbg = beam.beam_moe_layer(dev_bf16(hb), dev_bf16(xb), cfg.n, m.weights, m.mc, debug=True)
    logits, _, _ = beam.beam_router_topk(dbg["z"], m.router_w, m.bias_d, m.mc)
    torch.cuda.synchronize()
    a = dbg["logits"].double().cpu().numpy()
    b = logits.double().cpu().numpy()
    rowmax = np.abs(b).max(axis=1, keepdims=True)
    d = np.abs(a - b) / rowmax
    print(f"tensor-core vs SIMT router: max row-relative difference {d.max():.2e}")
    assert np.all(d <= 1e-5), float(d.max())
