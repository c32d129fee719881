"""Repeated host-buffer layer calls (beam_moe_layer_host on page-locked
buffers, up to 8 tokens): the first call with a given argument set runs as
direct launches, the second captures a CUDA graph, later ones replay it. The
buffers' contents change between calls; every call must give the bits of the
device entry point on that call's inputs (which the layer parity tests tie to
the oracle)."""
import numpy as np
import pytest
import torch

from beam_inputs import make_activations
from tests.gpu_support import beam_module, dev_bf16, model

pytestmark = pytest.mark.gpu


def _bf16(a: np.ndarray) -> torch.Tensor:
    return torch.from_numpy(a.view(np.int16)).view(torch.bfloat16)


def _device_call(beam, m, hb, xb, n):
    h, y, _ = beam.beam_moe_layer(dev_bf16(hb), dev_bf16(xb), n, m.weights, m.mc)
    torch.cuda.synchronize()
    return h.cpu(), y.cpu()


@pytest.mark.parametrize("T", [1, 8])
def test_repeated_host_calls_replay_with_fresh_inputs(T):
    beam = beam_module()
    m = model("decode_t64")
    cfg = m.cfg.with_(T=T)
    H = cfg.H
    beam.beam_release_host_graphs()
    ws = beam.Workspace()
    # two buffer sets: two argument sets, so two graphs
    sets = [[torch.empty(T, H, dtype=torch.bfloat16).pin_memory() for _ in range(4)] for _ in range(2)]
    counts = []
    # (buffer set, n): each set is seen three times with n (direct, capture,
    # replay), then set 0 twice with another n (a new argument set)
    plan = [(0, cfg.n), (1, cfg.n), (0, cfg.n), (1, cfg.n), (0, cfg.n), (1, cfg.n), (0, cfg.n + 1), (0, cfg.n + 1)]
    for i, (j, n) in enumerate(plan):
        h_in, x_in, h_out, y_out = sets[j]
        hb, xb = make_activations(cfg, batch=720 + i)
        h_in.copy_(_bf16(hb))
        x_in.copy_(_bf16(xb))
        h_out.fill_(0)
        y_out.fill_(0)
        beam.beam_moe_layer_host(h_in, x_in, n, m.weights, m.mc, h_out_host=h_out, y_out_host=y_out, ws=ws)
        counts.append(beam.beam_last_launch_count())
        assert beam.beam_get_device_error() == 0
        h_dev, y_dev = _device_call(beam, m, hb, xb, n)
        assert torch.equal(y_out.view(torch.int16), y_dev.view(torch.int16)), i
        assert torch.equal(h_out.view(torch.int16), h_dev.view(torch.int16)), i
    # a replay reports the same kernels as the direct launches it captured
    assert len(set(counts)) == 1 and counts[0] > 1, counts
    beam.beam_release_host_graphs()
    # after the release the same call runs (directly) again with the same bits
    h_in, x_in, h_out, y_out = sets[0]
    hb, xb = make_activations(cfg, batch=730)
    h_in.copy_(_bf16(hb))
    x_in.copy_(_bf16(xb))
    beam.beam_moe_layer_host(h_in, x_in, cfg.n, m.weights, m.mc, h_out_host=h_out, y_out_host=y_out, ws=ws)
    h_dev, y_dev = _device_call(beam, m, hb, xb, cfg.n)
    assert torch.equal(y_out.view(torch.int16), y_dev.view(torch.int16))
    assert torch.equal(h_out.view(torch.int16), h_dev.view(torch.int16))


def test_host_call_with_in_place_residual_replays():
    # h_out may alias h: a decode loop that updates its residual buffer in
    # place makes the same call every step
    beam = beam_module()
    m = model("decode_t64")
    cfg = m.cfg.with_(T=1)
    ws = beam.Workspace()
    h_buf = torch.empty(1, cfg.H, dtype=torch.bfloat16).pin_memory()
    x_buf = torch.empty(1, cfg.H, dtype=torch.bfloat16).pin_memory()
    y_buf = torch.empty(1, cfg.H, dtype=torch.bfloat16).pin_memory()
    hb, _ = make_activations(cfg, batch=740)
    h_buf.copy_(_bf16(hb))
    h_ref = dev_bf16(hb)
    for i in range(4):
        _, xb = make_activations(cfg, batch=741 + i)
        x_buf.copy_(_bf16(xb))
        beam.beam_moe_layer_host(h_buf, x_buf, cfg.n, m.weights, m.mc, h_out_host=h_buf, y_out_host=y_buf, ws=ws)
        h_ref, y_ref, _ = beam.beam_moe_layer(h_ref, dev_bf16(xb), cfg.n, m.weights, m.mc, h_out=h_ref)
        torch.cuda.synchronize()
        assert torch.equal(y_buf.view(torch.int16), y_ref.cpu().view(torch.int16)), i
        assert torch.equal(h_buf.view(torch.int16), h_ref.cpu().view(torch.int16)), i


def test_more_argument_sets_than_graph_slots():
    # n is part of an argument set: 100 sets called twice are captured, 300
    # more then overflow the 256-entry table (evicting the captured graphs),
    # and the first sets come back; every checked call must give the device
    # entry point's bits
    beam = beam_module()
    m = model("decode_t64")
    cfg = m.cfg.with_(T=1)
    beam.beam_release_host_graphs()
    ws = beam.Workspace()
    h_in, x_in, h_out, y_out = (torch.empty(1, cfg.H, dtype=torch.bfloat16).pin_memory() for _ in range(4))
    hb, xb = make_activations(cfg, batch=760)
    h_in.copy_(_bf16(hb))
    x_in.copy_(_bf16(xb))

    def call(n, check):
        beam.beam_moe_layer_host(h_in, x_in, n, m.weights, m.mc, h_out_host=h_out, y_out_host=y_out, ws=ws)
        if check:
            h_dev, y_dev = _device_call(beam, m, hb, xb, n)
            assert torch.equal(y_out.view(torch.int16), y_dev.view(torch.int16)), n
            assert torch.equal(h_out.view(torch.int16), h_dev.view(torch.int16)), n

    for rep in range(2):
        for n in range(2, 102):
            call(n, check=(rep == 1 and n % 25 == 0))
    for n in range(102, 402):
        call(n, check=(n % 100 == 0))
    for n in range(2, 12):
        call(n, check=True)
    assert beam.beam_get_device_error() == 0
    beam.beam_release_host_graphs()
