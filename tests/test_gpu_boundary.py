"""GPU parity: the fused sandwich-norm boundary against the fp64 oracle (<= 1 bf16 ulp)."""
import numpy as np
import pytest
import torch

from beam_inputs import CONFIGS, make_activations, make_norm_weights
from oracle import bf16 as obf
from oracle.boundary import boundary
from tests.gpu_support import assert_bf16_within_ulp, beam_module, bits_of, dev_bf16

pytestmark = pytest.mark.gpu


def _run(cfg, T=None, n=None, inplace=False, batch=0):
    beam = beam_module()
    h_bits, x_bits = make_activations(cfg, T=T, batch=batch)
    wp, wq = make_norm_weights(cfg)
    n = cfg.n if n is None else n
    h = dev_bf16(h_bits)
    h_out, z = beam.beam_boundary_norm(h, dev_bf16(x_bits), dev_bf16(wp), dev_bf16(wq), cfg.eps, n,
                                       h_out=h if inplace else None)
    torch.cuda.synchronize()
    ref_h, ref_z, _ = boundary(obf.decode(h_bits), obf.decode(x_bits), obf.decode(wp), obf.decode(wq), n, cfg.eps)
    return bits_of(h_out), bits_of(z), ref_h, ref_z, h_out, h


@pytest.mark.parametrize("name", ["toy", "decode_t1", "decode_t64", "prefill_t2048", "prefill_t16384"])
def test_boundary_matches_oracle(name):
    cfg = CONFIGS[name]
    hb, zb, ref_h, ref_z, _, _ = _run(cfg)
    assert_bf16_within_ulp(hb, ref_h, 1, f"{name} h'")
    assert_bf16_within_ulp(zb, ref_z, 1, f"{name} z")
    # the vast majority is bit-exact; a 1-ulp difference needs a value within
    # fp32 rounding of a bf16 midpoint
    exact = np.mean(obf.ulp_distance(zb, obf.encode(ref_z)) == 0)
    assert exact > 0.999, exact


@pytest.mark.parametrize("T", [3, 37, 129])
def test_ragged_token_counts_and_in_place(T):
    cfg = CONFIGS["decode_t64"]
    hb, zb, ref_h, ref_z, h_out, h = _run(cfg, T=T, inplace=True, batch=T)
    assert h_out.data_ptr() == h.data_ptr()
    assert_bf16_within_ulp(hb, ref_h, 1, "h' in place")
    assert_bf16_within_ulp(zb, ref_z, 1, "z")


def test_first_residual_add_and_toy_hidden():
    cfg = CONFIGS["toy"]
    hb, zb, ref_h, ref_z, _, _ = _run(cfg, n=1)
    assert_bf16_within_ulp(hb, ref_h, 1, "n=1 h'")
    assert_bf16_within_ulp(zb, ref_z, 1, "n=1 z")


def test_empty_batch_is_a_no_op():
    beam = beam_module()
    e = torch.empty(0, 256, dtype=torch.bfloat16, device="cuda")
    w = torch.ones(256, dtype=torch.bfloat16, device="cuda")
    h_out, z = beam.beam_boundary_norm(e, e.clone(), w, w, 1e-6, 3)
    assert h_out.shape == (0, 256)


@pytest.mark.parametrize("n,w", [(2, 1.0), (10, 3.0), (17, 4.0)])
def test_exact_cancellation_gives_zero(n, w):
    # h = 1 and x = -1 with post-norm weight w make y = -w; with w = sqrt(n-1)
    # the residual (sqrt(n-1) h + y) / sqrt(n) is exactly 0
    beam = beam_module()
    H = 256
    h = torch.ones(4, H, dtype=torch.bfloat16, device="cuda")
    x = -torch.ones(4, H, dtype=torch.bfloat16, device="cuda")
    wp = torch.full((H,), w, dtype=torch.bfloat16, device="cuda")
    wq = torch.ones(H, dtype=torch.bfloat16, device="cuda")
    h_out, _ = beam.beam_boundary_norm(h, x, wp, wq, 0.0, n)
    assert torch.all(h_out.float() == 0.0)
