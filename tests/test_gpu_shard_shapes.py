"""The expert stage at the per-GPU shapes of a Beam layer sharded over eight
GPUs (TokenSpeed blog, "TensorRT-LLM NVFP4 MoE": the MoE kernels are compared
on the TP8 and EP8 per-GPU shapes), against the fp64 oracle:
- TP8: all 256 experts, each a 320-wide slice of d_ff (2560 / 8), so the
  gate/up row blocks end in a half-empty 128-row block;
- EP8: 32 whole experts; tokens are routed over all 256, the pairs routed to
  the other GPUs' experts are dropped by the permutation (ids outside [0, 32)),
  and the combine sums this GPU's share of each token."""
import functools

import numpy as np
import pytest
import torch

from beam_inputs import CONFIGS, random_topk_ids
from oracle import bf16 as obf
from oracle.experts import intermediate
from oracle.permute import permute
from tests.gpu_support import Model, beam_module, dev_bf16, f64_of, layer_errors, moe_config, require_gpu

pytestmark = pytest.mark.gpu


@functools.lru_cache(maxsize=None)
def shard_model(shape: str) -> Model:
    require_gpu()
    base = CONFIGS["decode_t1"]
    if shape == "tp8":
        return Model(base.with_(name="tp8", F=base.F // 8))
    return Model(base.with_(name="ep8", E=base.E // 8, G=8, TG=4))


def _check_rows(got, ref, what):
    tol = 2.0 ** -8 * np.abs(ref) + 1e-4
    bad = np.abs(got - ref) > tol
    assert not bad.any(), f"{what}: {int(bad.sum())} of {bad.size} beyond tolerance"


@pytest.mark.parametrize("T,limit", [(1, None), (8, None), (64, 24), (2048, 12)])
def test_tp8_gate_up_and_down(T, limit):
    # d_ff = 320: gate/up rows in blocks of 128, 128 and 64 (zero-filled to 128)
    beam = beam_module()
    m = shard_model("tp8")
    cfg = m.cfg
    assert cfg.F == 320
    mc = moe_config(cfg)
    ids = random_topk_ids(T, cfg.E, cfg.K, seed=900 + T)
    rng = np.random.default_rng(900 + T)
    z_bits = obf.encode(rng.standard_normal((T, cfg.H)))
    counts, offsets, perm, inv = permute(ids, cfg.E)
    xp_bits = z_bits[perm]
    off_d = torch.from_numpy(offsets).cuda()
    act = beam.beam_moe_gate_up(dev_bf16(xp_bits), off_d, m.dev[0], mc, T)
    touched = np.nonzero(counts)[0]
    if limit is not None and touched.size > limit:
        touched = np.sort(np.random.default_rng(T).choice(touched, size=limit, replace=False))
    X = obf.decode(xp_bits)
    a_ref = np.zeros((T * cfg.K, cfg.F))
    rows = []
    for e in touched:
        lo, hi = offsets[e], offsets[e + 1]
        Wg, Wu, _ = m.expert_fn_nocache(int(e))
        a_ref[lo:hi] = intermediate(X[lo:hi], Wg, Wu)
        rows.append(np.arange(lo, hi))
    rows = np.concatenate(rows)
    _check_rows(f64_of(act)[rows], a_ref[rows], "gate/up")
    A_bits = obf.encode(a_ref)
    y_perm = beam.beam_moe_down(dev_bf16(A_bits), off_d, m.dev[1], mc, T)
    A = obf.decode(A_bits)
    y_ref = np.zeros((T * cfg.K, cfg.H))
    for e in touched:
        lo, hi = offsets[e], offsets[e + 1]
        y_ref[lo:hi] = A[lo:hi] @ m.expert_fn_nocache(int(e))[2].T
    _check_rows(f64_of(y_perm)[rows], y_ref[rows], "down")
    assert beam.beam_get_device_error() == 0


def _expert_out(m, e, z_row):
    Wg, Wu, Wd = m.expert_fn(int(e))
    a = obf.decode(obf.encode(intermediate(z_row[None, :], Wg, Wu)))  # the bf16 intermediate
    return (a @ Wd.T)[0]


@pytest.mark.parametrize("shape,T", [("tp8", 1), ("tp8", 8), ("tp8", 64), ("ep8", 1), ("ep8", 8), ("ep8", 64),
                                     ("ep8", 512)])
def test_shard_shape_experts_and_combine(shape, T):
    beam = beam_module()
    m = shard_model(shape)
    cfg = m.cfg
    mc = moe_config(cfg)
    E_route = 256  # routing spans all experts of the layer
    ids = random_topk_ids(T, E_route, cfg.K, seed=950 + T).astype(np.int32)
    rng = np.random.default_rng(950 + T)
    z_bits = obf.encode(rng.standard_normal((T, cfg.H)))
    w = rng.random((T, cfg.K)) + 0.1
    w = (cfg.routed_scale * w / w.sum(axis=1, keepdims=True)).astype(np.float32)
    # the GPU's own permutation: for EP8 the ids >= 32 (other GPUs' experts) are dropped
    offsets, perm, inv, x_perm = beam.beam_moe_permute(torch.from_numpy(ids).cuda(), dev_bf16(z_bits), mc)
    inv_h = inv.cpu().numpy()
    local = ids.reshape(-1) < cfg.E
    assert np.array_equal(inv_h < 0, ~local)
    y = beam.beam_moe_experts(x_perm, offsets, m.dev[0], m.dev[1], torch.from_numpy(w).cuda(), inv, mc, T)
    torch.cuda.synchronize()
    Z = obf.decode(z_bits)
    y_ref = np.zeros((T, cfg.H))
    sample = range(T) if T <= 64 else np.random.default_rng(T).choice(T, size=32, replace=False)
    for t in sample:
        for k in range(cfg.K):
            e = int(ids[t, k])
            if e < cfg.E:
                y_ref[t] += float(w[t, k]) * _expert_out(m, e, Z[t])
    sample = np.array(sorted(sample))
    mx, rel = layer_errors(f64_of(y)[sample], y_ref[sample])
    assert mx <= 2e-2 and rel <= 5e-3, (mx, rel)
    assert beam.beam_get_device_error() == 0
