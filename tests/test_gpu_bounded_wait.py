"""Failure detection on the device without a fault: a bounded wait on a flag
that nothing sets gives up after its limit, reports its site code through the
library's error word, and leaves the context usable (the next layer call
matches a call made before it)."""
import time

import pytest
import torch

from tests.gpu_support import beam_module, model

pytestmark = pytest.mark.gpu


def test_bounded_wait_times_out_and_reports():
    beam = beam_module()
    m = model("toy")
    _, y_before, _ = beam.beam_moe_layer(m.h(), m.x(), m.cfg.n, m.weights, m.mc)
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    site = beam.beam_check_bounded_wait(50)
    elapsed = time.perf_counter() - t0
    assert site == 99
    assert 0.04 <= elapsed < 5.0, elapsed
    assert beam.beam_get_device_error() == 0  # cleared by the check
    _, y_after, _ = beam.beam_moe_layer(m.h(), m.x(), m.cfg.n, m.weights, m.mc)
    torch.cuda.synchronize()
    assert torch.equal(y_before.view(torch.int16), y_after.view(torch.int16))


@pytest.mark.parametrize("T", [1, 16])
def test_host_entry_reports_a_pending_timeout(T):
    # A timed-out bounded wait left in the device error word is reported by
    # the next host-buffer layer call (status BEAM_ERR_DEVICE_TIMEOUT), which
    # clears it: the call after gives the bits of a call made before, with
    # status OK. T = 1 takes the mapped-memory path, T = 16 the copy path.
    beam = beam_module()
    m = model("toy")
    H = m.cfg.H
    h_in = m.h().cpu()[:T].contiguous().pin_memory()
    x_in = m.x().cpu()[:T].contiguous().pin_memory()
    outs = [[torch.empty(T, H, dtype=torch.bfloat16).pin_memory() for _ in range(2)] for _ in range(3)]
    ws = beam.Workspace()
    beam.beam_release_host_graphs()
    assert beam.beam_get_device_error() == 0
    beam.beam_moe_layer_host(h_in, x_in, m.cfg.n, m.weights, m.mc, h_out_host=outs[0][0], y_out_host=outs[0][1],
                             ws=ws)
    beam.beam_check_bounded_wait_pending(20)
    with pytest.raises(beam.BeamError, match="status 6"):
        beam.beam_moe_layer_host(h_in, x_in, m.cfg.n, m.weights, m.mc, h_out_host=outs[1][0],
                                 y_out_host=outs[1][1], ws=ws)
    assert beam.beam_get_device_error() == 0  # cleared by the call that reported it
    beam.beam_moe_layer_host(h_in, x_in, m.cfg.n, m.weights, m.mc, h_out_host=outs[2][0], y_out_host=outs[2][1],
                             ws=ws)
    assert torch.equal(outs[0][0].view(torch.int16), outs[2][0].view(torch.int16))
    assert torch.equal(outs[0][1].view(torch.int16), outs[2][1].view(torch.int16))
    beam.beam_release_host_graphs()
