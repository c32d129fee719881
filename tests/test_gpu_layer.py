"""GPU parity of the whole MoE sublayer (beam_moe_layer through the C ABI)
against the fp64 oracle on the five workloads: h' within 1 bf16 ulp, routing
bit-exact away from near-ties, layer output within max-abs 2e-2 and rel-L2
5e-3 (near-tie tokens checked against the oracle re-run with the GPU's
routing)."""
import numpy as np
import pytest
import torch

from beam_inputs import CONFIGS, sample_tokens
from oracle import bf16 as obf
from oracle.routing import near_tie
from tests.gpu_support import (assert_bf16_within_ulp, beam_module, bits_of, dev_bf16, f64_of, layer_errors,
                               model)

pytestmark = pytest.mark.gpu


def run_layer(m, h=None, x=None, n=None):
    beam = beam_module()
    h = m.h() if h is None else h
    x = m.x() if x is None else x
    h_out, y, dbg = beam.beam_moe_layer(h, x, m.cfg.n if n is None else n, m.weights, m.mc, debug=True)
    torch.cuda.synchronize()
    assert beam.beam_get_device_error() == 0
    return h_out, y, dbg


@pytest.mark.parametrize("name", ["toy", "decode_t1", "decode_t64", "prefill_t2048", "prefill_t16384"])
def test_layer_matches_oracle(name):
    m = model(name)
    cfg = m.cfg
    h_out, y, dbg = run_layer(m)
    tokens = sample_tokens(cfg)
    ref = m.oracle_layer(tokens=tokens)
    assert_bf16_within_ulp(bits_of(h_out)[tokens], ref["h_new"], 1, "h'")
    ids = dbg["topk_ids"].cpu().numpy()[tokens]
    tie = near_tie(ref["route"])
    same = np.all(ids == ref["ids"], axis=1)
    assert np.all(same | tie), f"{int((~same & ~tie).sum())} non-near-tie tokens routed differently"
    yg = f64_of(y)[tokens]
    mx, rel = layer_errors(yg[same], ref["y"][same])
    print(f"{name}: tokens {tokens.size}, near-ties {int(tie.sum())}, differing {int((~same).sum())}, "
          f"max|dy| {mx:.3e}, rel-L2 {rel:.3e}")
    assert mx <= 2e-2 and rel <= 5e-3, (mx, rel)
    if (~same).any():
        # routing-conditioned check: the oracle evaluated with the GPU's choices
        cond = m.oracle_layer(tokens=tokens[~same], ids_override=ids[~same])
        mx2, rel2 = layer_errors(yg[~same], cond["y"])
        assert mx2 <= 2e-2 and rel2 <= 5e-3, (mx2, rel2)
    # load statistics for the record
    off = dbg["expert_offsets"].cpu().numpy()
    counts = np.diff(off)
    print(f"{name}: touched experts {int((counts > 0).sum())}, max share {counts.max() / counts.sum():.3f}")


def test_layer_is_deterministic():
    m = model("decode_t64")
    _, y1, d1 = run_layer(m)
    _, y2, d2 = run_layer(m)
    assert torch.equal(y1, y2) and torch.equal(d1["topk_ids"], d2["topk_ids"])


# besides ragged sizes, both sides of every point where the layer changes
# kernels: one-launch routing (T <= 8), router with fused top-k (T <= 32),
# tensor-core router (T > 128), one-kernel permutation (T * K <= 2048)
@pytest.mark.parametrize("T", [2, 8, 9, 32, 33, 37, 128, 129, 256, 257, 1000])
def test_ragged_batches(T):
    from beam_inputs import make_activations
    m = model("decode_t64")
    cfg = m.cfg.with_(T=T)
    hb, xb = make_activations(cfg, batch=T)
    h_out, y, dbg = run_layer(m, dev_bf16(hb), dev_bf16(xb))
    from oracle.layer import layer
    tokens = np.arange(T) if T <= 64 else np.arange(0, T, 32)
    ref = layer(obf.decode(hb), obf.decode(xb), obf.decode(m.wp_bits), obf.decode(m.wq_bits), m.W_r, m.bias,
                n=cfg.n, eps=cfg.eps, G=cfg.G, TG=cfg.TG, K=cfg.K, routed_scale=cfg.routed_scale,
                expert_fn=m.expert_fn_nocache, tokens=tokens, workers=16)
    ids = dbg["topk_ids"].cpu().numpy()[tokens]
    same = np.all(ids == ref["ids"], axis=1)
    assert np.all(same | near_tie(ref["route"]))
    mx, rel = layer_errors(f64_of(y)[tokens][same], ref["y"][same])
    assert mx <= 2e-2 and rel <= 5e-3, (mx, rel)


def test_all_tokens_on_one_group():
    # a dominant correction bias on group 0 sends every token to the same
    # experts: one expert receives all T rows (several token tiles), the rest none
    beam = beam_module()
    m = model("toy")
    cfg = m.cfg
    bias = m.bias.copy()
    bias[:4] += 5.0
    bias[4:8] += 4.0
    bias_d = torch.from_numpy(bias).cuda()   # keep the tensor alive while the library uses its pointer
    w = beam.weights_struct(m.w_post, m.w_pre, m.router_w, bias_d, m.dev[0], m.dev[1])
    h_out, y, dbg = beam.beam_moe_layer(m.h(), m.x(), cfg.n, w, m.mc, debug=True)
    torch.cuda.synchronize()
    off = dbg["expert_offsets"].cpu().numpy()
    assert set(np.nonzero(np.diff(off))[0].tolist()) <= set(range(8))
    from oracle.layer import layer
    ref = layer(obf.decode(m.h_bits), obf.decode(m.x_bits), obf.decode(m.wp_bits), obf.decode(m.wq_bits), m.W_r,
                bias, n=cfg.n, eps=cfg.eps, G=cfg.G, TG=cfg.TG, K=cfg.K, routed_scale=cfg.routed_scale,
                expert_fn=m.expert_fn)
    assert np.array_equal(dbg["topk_ids"].cpu().numpy(), ref["ids"])
    mx, rel = layer_errors(f64_of(y), ref["y"])
    assert mx <= 2e-2 and rel <= 5e-3, (mx, rel)


@pytest.mark.parametrize("T,pinned_out", [(1, True), (1, False), (8, True), (16, True), (64, True), (300, False),
                                         (2048, True), (8192, True), (16384, True)])
def test_host_buffer_entry_point_matches_device_entry_point(T, pinned_out):
    # up to 8 tokens with page-locked buffers the layer reads and writes the
    # mapped host memory directly; otherwise it copies in and out (from 64
    # tokens the copy of h' back overlaps the rest of the layer; from 8192 the
    # layer is pipelined with the copies in four token chunks, eight from
    # 16384, whose router launches take narrower token tiles than the whole
    # batch's)
    from beam_inputs import make_activations
    beam = beam_module()
    m = model("decode_t64")
    cfg = m.cfg.with_(T=T)
    hb, xb = make_activations(cfg, batch=600 + T)
    h_dev, y_dev, _ = run_layer(m, dev_bf16(hb), dev_bf16(xb), n=cfg.n)
    h_host = torch.from_numpy(hb.view(np.int16)).view(torch.bfloat16).pin_memory()
    x_host = torch.from_numpy(xb.view(np.int16)).view(torch.bfloat16).pin_memory()
    h_out = torch.empty_like(h_host)
    y_out = torch.empty_like(h_host)
    if pinned_out:
        h_out, y_out = h_out.pin_memory(), y_out.pin_memory()
    h_out, y = beam.beam_moe_layer_host(h_host, x_host, cfg.n, m.weights, m.mc, h_out_host=h_out, y_out_host=y_out)
    assert torch.equal(y.view(torch.int16), y_dev.cpu().view(torch.int16))
    assert torch.equal(h_out.view(torch.int16), h_dev.cpu().view(torch.int16))


def test_empty_batch():
    beam = beam_module()
    m = model("toy")
    e = torch.empty(0, m.cfg.H, dtype=torch.bfloat16, device="cuda")
    h_out, y, _ = beam.beam_moe_layer(e, e.clone(), 3, m.weights, m.mc)
    assert y.shape == (0, m.cfg.H)


def test_skewed_routing_several_token_tiles_per_expert():
    # 32 of 64 tokens are copies of one token, so its 8 experts each receive
    # 32+ rows: several 16-row token tiles per expert inside the fused launch
    # (the down units of a token tile wait for all of that tile's gate/up rows)
    from beam_inputs import make_activations
    m = model("decode_t64")
    cfg = m.cfg.with_(T=64)
    hb, xb = make_activations(cfg, batch=500)
    hb[:32] = hb[0]
    xb[:32] = xb[0]
    h_out, y, dbg = run_layer(m, dev_bf16(hb), dev_bf16(xb))
    ids = dbg["topk_ids"].cpu().numpy()
    counts = np.diff(dbg["expert_offsets"].cpu().numpy())
    assert counts[ids[0]].min() >= 32
    yb = bits_of(y)
    assert all(np.array_equal(yb[t], yb[0]) for t in range(1, 32))  # identical rows, identical bits
    from oracle.layer import layer
    tokens = np.array([0, 31, 32, 45, 63])
    ref = layer(obf.decode(hb), obf.decode(xb), obf.decode(m.wp_bits), obf.decode(m.wq_bits), m.W_r, m.bias,
                n=cfg.n, eps=cfg.eps, G=cfg.G, TG=cfg.TG, K=cfg.K, routed_scale=cfg.routed_scale,
                expert_fn=m.expert_fn_nocache, tokens=tokens, workers=16)
    same = np.all(ids[tokens] == ref["ids"], axis=1)
    assert np.all(same | near_tie(ref["route"]))
    mx, rel = layer_errors(f64_of(y)[tokens][same], ref["y"][same])
    assert mx <= 2e-2 and rel <= 5e-3, (mx, rel)


def test_concurrent_layers_on_two_streams():
    # two layer calls in flight at once on separate streams and workspaces
    # share no device state: each gives the bits it gives alone
    from beam_inputs import make_activations
    beam = beam_module()
    m = model("decode_t64")
    runs = []
    for T, batch in ((1, 950), (8, 951)):
        cfg = m.cfg.with_(T=T)
        hb, xb = make_activations(cfg, batch=batch)
        runs.append((dev_bf16(hb), dev_bf16(xb)))
    alone = []
    for h, x in runs:
        h_out, y, _ = beam.beam_moe_layer(h, x, m.cfg.n, m.weights, m.mc, ws=beam.Workspace())
        torch.cuda.synchronize()
        alone.append((h_out.clone(), y.clone()))
    streams = [torch.cuda.Stream(), torch.cuda.Stream()]
    wss = [beam.Workspace(), beam.Workspace()]
    outs = [None, None]
    torch.cuda.synchronize()
    for rep in range(3):
        for i, (h, x) in enumerate(runs):
            with torch.cuda.stream(streams[i]):
                outs[i] = beam.beam_moe_layer(h, x, m.cfg.n, m.weights, m.mc, ws=wss[i])
        torch.cuda.synchronize()
        for i in range(2):
            assert torch.equal(outs[i][0].view(torch.int16), alone[i][0].view(torch.int16)), (rep, i)
            assert torch.equal(outs[i][1].view(torch.int16), alone[i][1].view(torch.int16)), (rep, i)
    assert beam.beam_get_device_error() == 0


@pytest.mark.parametrize("first", [0, 1])
def test_concurrent_prefill_and_decode_layers(first):
    # A 256-token layer (the fused expert launch with one CTA per SM, whose
    # down units wait on gate/up units of other CTAs) and a one-token layer
    # in flight at once on two streams, launched in both orders, 20 times:
    # each call gives the bits it gives alone, and no bounded wait gives up
    # (the expert launch hands out its units from a counter, so its progress
    # does not depend on all of its CTAs being resident).
    from beam_inputs import make_activations
    beam = beam_module()
    m = model("decode_t64")
    runs = []
    for T, batch in ((256, 960), (1, 961)):
        cfg = m.cfg.with_(T=T)
        hb, xb = make_activations(cfg, batch=batch)
        runs.append((dev_bf16(hb), dev_bf16(xb)))
    alone = []
    for h, x in runs:
        h_out, y, _ = beam.beam_moe_layer(h, x, m.cfg.n, m.weights, m.mc, ws=beam.Workspace())
        torch.cuda.synchronize()
        alone.append((h_out.clone(), y.clone()))
    assert beam.beam_get_device_error() == 0
    streams = [torch.cuda.Stream(), torch.cuda.Stream()]
    wss = [beam.Workspace(), beam.Workspace()]
    order = [first, 1 - first]
    torch.cuda.synchronize()
    for rep in range(20):
        outs = [None, None]
        for i in order:
            h, x = runs[i]
            with torch.cuda.stream(streams[i]):
                outs[i] = beam.beam_moe_layer(h, x, m.cfg.n, m.weights, m.mc, ws=wss[i])
        torch.cuda.synchronize()
        for i in range(2):
            assert torch.equal(outs[i][0].view(torch.int16), alone[i][0].view(torch.int16)), (rep, i)
            assert torch.equal(outs[i][1].view(torch.int16), alone[i][1].view(torch.int16)), (rep, i)
    assert beam.beam_get_device_error() == 0
