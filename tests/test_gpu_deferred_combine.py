"""The combine deferred into the next boundary (vLLM Beam summary, kernel
change list: the norm kernel after the MoE also combines the top-8 outputs).

beam_boundary_norm_combine must give the bits of beam_moe_combine followed by
beam_boundary_norm; against the fp64 oracle, its outputs are within 1 bf16
ulp of the oracle boundary applied to the GPU's combined x, and that x is
within one bf16 rounding of the oracle combine. beam_moe_layer_uncombined
followed by it must give the bits of beam_moe_layer followed by the plain
boundary."""
import numpy as np
import pytest
import torch

from beam_inputs import CONFIGS, make_activations, make_norm_weights, random_topk_ids
from oracle import bf16 as obf
from oracle.boundary import boundary
from oracle.combine import combine
from oracle.permute import permute
from tests.gpu_support import assert_bf16_within_ulp, beam_module, bits_of, dev_bf16, f64_of, model

pytestmark = pytest.mark.gpu


def _combine_inputs(T, K, H, E, seed, drop=0.0):
    rng = np.random.default_rng(seed)
    ids = random_topk_ids(T, E, K, seed=seed)
    _, _, _, inv = permute(ids, E)
    inv = np.asarray(inv, dtype=np.int32).copy()
    if drop:
        inv[rng.random(T * K) < drop] = -1  # dropped pairs (no valid expert)
    yp_bits = obf.encode(0.05 * rng.standard_normal((T * K, H)))
    w = (0.6 * rng.random((T, K))).astype(np.float32)
    return yp_bits, w, inv


def _both_paths(cfg, T, K, yp_bits, w, inv, batch, inplace=False):
    beam = beam_module()
    E = 16
    mc = beam.make_config(cfg.H, E, 4, 4, K, 128, cfg.routed_scale, cfg.eps)
    h_bits, _ = make_activations(cfg, T=T, batch=batch)
    wp, wq = make_norm_weights(cfg)
    y_perm, tw, ti = dev_bf16(yp_bits), torch.from_numpy(w).cuda(), torch.from_numpy(inv).cuda()
    w_post, w_pre = dev_bf16(wp), dev_bf16(wq)
    # separate: combine, then the boundary on its output
    x = beam.beam_moe_combine(y_perm, tw, ti, mc, T)
    h_sep, z_sep = beam.beam_boundary_norm(dev_bf16(h_bits), x, w_post, w_pre, cfg.eps, cfg.n)
    # fused
    h = dev_bf16(h_bits)
    h_fus, z_fus = beam.beam_boundary_norm_combine(h, y_perm, tw, ti, w_post, w_pre, cfg.eps, cfg.n,
                                                   h_out=h if inplace else None)
    torch.cuda.synchronize()
    return h_bits, wp, wq, bits_of(x), (bits_of(h_sep), bits_of(z_sep)), (bits_of(h_fus), bits_of(z_fus))


@pytest.mark.parametrize("T,K,H", [(1, 8, 5120), (5, 8, 5120), (64, 8, 5120), (300, 8, 2048), (37, 16, 1024),
                                   (16, 4, 256)])
def test_fused_boundary_equals_combine_then_boundary(T, K, H):
    cfg = CONFIGS["decode_t64"].with_(H=H, T=T)
    yp_bits, w, inv = _combine_inputs(T, K, H, 16, seed=800 + T)
    h_bits, wp, wq, x_bits, sep, fus = _both_paths(cfg, T, K, yp_bits, w, inv, batch=800 + T)
    assert np.array_equal(fus[0], sep[0]) and np.array_equal(fus[1], sep[1])
    # against the oracle: x is one bf16 rounding of the fp32 sum, the boundary on that x within 1 ulp
    x_ref = combine(obf.decode(yp_bits), w.astype(np.float64), inv)
    x_gpu = obf.decode(x_bits)
    assert np.all(np.abs(x_gpu - x_ref) <= 2.0 ** -8 * np.abs(x_ref) + 1e-6)
    ref_h, ref_z, _ = boundary(obf.decode(h_bits), x_gpu, obf.decode(wp), obf.decode(wq), cfg.n, cfg.eps)
    assert_bf16_within_ulp(fus[0], ref_h, 1, "h'")
    assert_bf16_within_ulp(fus[1], ref_z, 1, "z")


def test_fused_boundary_with_dropped_pairs_and_in_place():
    T, K, H = 33, 8, 5120
    cfg = CONFIGS["decode_t64"].with_(T=T)
    yp_bits, w, inv = _combine_inputs(T, K, H, 16, seed=850, drop=0.2)
    assert (inv < 0).any()
    _, _, _, _, sep, fus = _both_paths(cfg, T, K, yp_bits, w, inv, batch=850, inplace=True)
    assert np.array_equal(fus[0], sep[0]) and np.array_equal(fus[1], sep[1])


def test_fused_boundary_empty_batch():
    beam = beam_module()
    cfg = CONFIGS["decode_t64"]
    wp, wq = make_norm_weights(cfg)
    e = torch.empty(0, cfg.H, dtype=torch.bfloat16, device="cuda")
    h_out, z = beam.beam_boundary_norm_combine(e, e, torch.empty(0, 8, device="cuda"),
                                               torch.empty(0, dtype=torch.int32, device="cuda"), dev_bf16(wp),
                                               dev_bf16(wq), cfg.eps, cfg.n)
    assert h_out.shape == (0, cfg.H) and beam.beam_last_launch_count() == 0


@pytest.mark.parametrize("name,T", [("toy", None), ("decode_t1", None), ("decode_t64", 8), ("decode_t64", None)])
def test_layer_uncombined_then_fused_boundary(name, T):
    # the next sublayer's boundary: the residual h' of this layer, norm weights of the next
    beam = beam_module()
    m = model(name)
    cfg = m.cfg if T is None else m.cfg.with_(T=T)
    h_bits, x_bits = make_activations(cfg, batch=870)
    wp2, wq2 = make_norm_weights(cfg.with_(seed=cfg.seed + 1))
    w_post2, w_pre2 = dev_bf16(wp2), dev_bf16(wq2)
    n2 = cfg.n + 1
    h1, y, _ = beam.beam_moe_layer(dev_bf16(h_bits), dev_bf16(x_bits), cfg.n, m.weights, m.mc)
    h2_sep, z2_sep = beam.beam_boundary_norm(h1, y, w_post2, w_pre2, cfg.eps, n2)
    torch.cuda.synchronize()
    ws = beam.Workspace()
    h1u, pend = beam.beam_moe_layer_uncombined(dev_bf16(h_bits), dev_bf16(x_bits), cfg.n, m.weights, m.mc, ws=ws)
    h2_fus, z2_fus = beam.beam_boundary_norm_combine(h1u, *pend, w_post2, w_pre2, cfg.eps, n2, h_out=h1u)
    torch.cuda.synchronize()
    assert beam.beam_get_device_error() == 0
    assert torch.equal(h2_fus.view(torch.int16), h2_sep.view(torch.int16))
    assert torch.equal(z2_fus.view(torch.int16), z2_sep.view(torch.int16))
