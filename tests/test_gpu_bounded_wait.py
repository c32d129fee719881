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
