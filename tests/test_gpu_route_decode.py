"""The layer's decode-size routing (one launch for boundary, router, top-k,
permutation and row gather, up to 8 tokens with 256 experts in 8 groups)
against the separate entry points and the fp64 oracle: h' and z bit-identical
to the boundary kernel, logits within 1e-5 of the row's largest magnitude,
routing equal away from near-ties, the layer output within the layer
tolerances, in-place residual updates, and repeated calls (the launch leaves
its ticket at zero)."""
import numpy as np
import pytest
import torch

from beam_inputs import make_activations
from oracle import bf16 as obf
from oracle.layer import layer
from oracle.routing import near_tie
from tests.gpu_support import beam_module, bits_of, dev_bf16, f64_of, layer_errors, model

pytestmark = pytest.mark.gpu


def staged(m, h, x, n):
    beam = beam_module()
    h_out, z = beam.beam_boundary_norm(h, x, m.w_post, m.w_pre, m.cfg.eps, n)
    logits, ids, w = beam.beam_router_topk(z, m.router_w, m.bias_d, m.mc)
    offsets, _, _, _ = beam.beam_moe_permute(ids, z, m.mc, gather=False)
    torch.cuda.synchronize()
    return h_out, z, logits, ids, offsets


@pytest.mark.parametrize("T", [1, 2, 3, 4, 5, 8, 9])
def test_fused_routing_matches_staged_path_and_oracle(T):
    beam = beam_module()
    m = model("decode_t64")
    cfg = m.cfg.with_(T=T)
    hb, xb = make_activations(cfg, batch=100 + T)
    h, x = dev_bf16(hb), dev_bf16(xb)
    h_out, y, dbg = beam.beam_moe_layer(h, x, cfg.n, m.weights, m.mc, debug=True)
    torch.cuda.synchronize()
    assert beam.beam_get_device_error() == 0
    sh, sz, slog, sids, soff = staged(m, h, x, cfg.n)
    assert torch.equal(h_out.view(torch.int16), sh.view(torch.int16))
    assert torch.equal(dbg["z"].view(torch.int16), sz.view(torch.int16))
    lg, sl = dbg["logits"].double().cpu().numpy(), slog.double().cpu().numpy()
    scale = np.abs(sl).max(axis=1, keepdims=True)
    assert np.all(np.abs(lg - sl) <= 1e-5 * scale)

    tokens = np.arange(T)
    ref = layer(obf.decode(hb), obf.decode(xb), obf.decode(m.wp_bits), obf.decode(m.wq_bits), m.W_r, m.bias,
                n=cfg.n, eps=cfg.eps, G=cfg.G, TG=cfg.TG, K=cfg.K, routed_scale=cfg.routed_scale,
                expert_fn=m.expert_fn_nocache, tokens=tokens, workers=16)
    ids = dbg["topk_ids"].cpu().numpy()
    tie = near_tie(ref["route"])
    same = np.all(ids == ref["ids"], axis=1)
    assert np.all(same | tie)
    assert np.all(np.all(ids == sids.cpu().numpy(), axis=1) | tie)
    if np.array_equal(ids, sids.cpu().numpy()):
        assert torch.equal(dbg["expert_offsets"], soff)
    counts = np.bincount(ids.ravel(), minlength=cfg.E)
    assert np.array_equal(np.diff(dbg["expert_offsets"].cpu().numpy()), counts)
    mx, rel = layer_errors(f64_of(y)[same], ref["y"][same])
    assert mx <= 2e-2 and rel <= 5e-3, (mx, rel)
    # the experts and combine stages give the same bits as the separate
    # experts entry point on the layer's own routing
    offs2, _, inv2, xp2 = beam.beam_moe_permute(dbg["topk_ids"], dbg["z"], m.mc)
    y2 = beam.beam_moe_experts(xp2, offs2, m.dev[0], m.dev[1], dbg["topk_w"], inv2, m.mc, T)
    torch.cuda.synchronize()
    assert torch.equal(y.view(torch.int16), y2.view(torch.int16))


@pytest.mark.parametrize("T", [1, 8])
def test_fused_routing_in_place_residual(T):
    # h_out aliases h: every expert block reads h, so only the block that
    # finishes last may write h'
    beam = beam_module()
    m = model("decode_t64")
    cfg = m.cfg.with_(T=T)
    hb, xb = make_activations(cfg, batch=200 + T)
    h_ref, y_ref, _ = beam.beam_moe_layer(dev_bf16(hb), dev_bf16(xb), cfg.n, m.weights, m.mc)
    h = dev_bf16(hb)
    h_out, y, _ = beam.beam_moe_layer(h, dev_bf16(xb), cfg.n, m.weights, m.mc, h_out=h)
    torch.cuda.synchronize()
    assert h_out.data_ptr() == h.data_ptr()
    assert torch.equal(h.view(torch.int16), h_ref.view(torch.int16))
    assert torch.equal(y.view(torch.int16), y_ref.view(torch.int16))


def test_fused_routing_repeated_calls_share_a_workspace():
    beam = beam_module()
    m = model("decode_t1")
    ws = beam.Workspace()
    outs = [beam.beam_moe_layer(m.h(), m.x(), m.cfg.n, m.weights, m.mc, ws=ws)[1] for _ in range(3)]
    torch.cuda.synchronize()
    assert beam.beam_get_device_error() == 0
    assert all(torch.equal(o.view(torch.int16), outs[0].view(torch.int16)) for o in outs[1:])
    # the same bits from a workspace full of garbage (the ticket is cleared by the layer)
    junk = beam.Workspace()
    junk.get(beam.beam_moe_workspace_size(m.mc, m.cfg.T)).fill_(0xFF)
    _, y, _ = beam.beam_moe_layer(m.h(), m.x(), m.cfg.n, m.weights, m.mc, ws=junk)
    torch.cuda.synchronize()
    assert beam.beam_get_device_error() == 0
    assert torch.equal(y.view(torch.int16), outs[0].view(torch.int16))
