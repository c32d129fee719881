"""The layer captured in a CUDA graph: every step of beam_moe_layer is a
stream-ordered launch or memset, so a captured graph replays the same work.
Replays must give the same bits as direct calls, also after new inputs are
copied into the captured buffers, at a decode size (one routing launch and
the fused experts launch) and at a size that takes the separate kernels."""
import pytest
import torch

from beam_inputs import make_activations
from tests.gpu_support import beam_module, dev_bf16, model

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("name,T", [("decode_t1", 1), ("decode_t64", 64), ("decode_t64", 5)])
def test_graph_replay_matches_direct_calls(name, T):
    beam = beam_module()
    m = model(name)
    cfg = m.cfg.with_(T=T)
    batches = [make_activations(cfg, batch=300 + b) for b in range(3)]
    # direct calls, one workspace
    ws = beam.Workspace()
    ref = []
    for hb, xb in batches:
        h_out, y, _ = beam.beam_moe_layer(dev_bf16(hb), dev_bf16(xb), cfg.n, m.weights, m.mc, ws=ws)
        ref.append((h_out.clone(), y.clone()))
    torch.cuda.synchronize()

    # capture once on fixed buffers (the workspace is sized before capture)
    h = dev_bf16(batches[0][0])
    x = dev_bf16(batches[0][1])
    h_out = torch.empty_like(h)
    y = torch.empty_like(h)
    gws = beam.Workspace()
    gws.get(beam.beam_moe_workspace_size(m.mc, T))
    beam.beam_moe_layer(h, x, cfg.n, m.weights, m.mc, h_out=h_out, y_out=y, ws=gws)  # warm-up outside capture
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        beam.beam_moe_layer(h, x, cfg.n, m.weights, m.mc, h_out=h_out, y_out=y, ws=gws)
    for rep in range(2):
        for b, (hb, xb) in enumerate(batches):
            h.copy_(dev_bf16(hb))
            x.copy_(dev_bf16(xb))
            g.replay()
            torch.cuda.synchronize()
            assert beam.beam_get_device_error() == 0
            assert torch.equal(h_out.view(torch.int16), ref[b][0].view(torch.int16)), (rep, b)
            assert torch.equal(y.view(torch.int16), ref[b][1].view(torch.int16)), (rep, b)
