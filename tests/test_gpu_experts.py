"""GPU parity: the tcgen05 grouped GEMMs (gate/up + SwiGLU, down) and the
combine, against the fp64 oracle, at toy and Beam shapes, with split-K,
ragged expert tails and every token-tile width."""
import numpy as np
import pytest
import torch

from beam_inputs import CONFIGS, random_topk_ids
from oracle import bf16 as obf
from oracle.combine import combine
from oracle.experts import intermediate
from oracle.permute import permute
from tests.gpu_support import WORKERS, beam_module, bits_of, dev_bf16, f64_of, layer_errors, model

pytestmark = pytest.mark.gpu


def _inputs(m, T, skew, seed):
    cfg = m.cfg
    ids = random_topk_ids(T, cfg.E, cfg.K, seed=seed, skew=skew)
    rng = np.random.default_rng(seed)
    z_bits = obf.encode(rng.standard_normal((T, cfg.H)))
    counts, offsets, perm, inv = permute(ids, cfg.E)
    x_perm_bits = z_bits[perm]
    return ids, z_bits, counts, offsets, perm, inv, x_perm_bits


def _sample_experts(counts, limit):
    touched = np.nonzero(counts)[0]
    if limit is None or touched.size <= limit:
        return touched
    order = np.argsort(-counts[touched], kind="stable")
    rng = np.random.default_rng(int(counts.sum()))
    pick = set(touched[order[:2]].tolist())            # the most loaded experts
    pick |= set(rng.choice(touched, size=limit - 2, replace=False).tolist())
    return np.array(sorted(pick))


@pytest.mark.parametrize("name,T,skew,limit", [
    ("toy", 16, 0.0, None),
    ("toy", 200, 1.5, None),          # multi-tile experts with ragged tails
    ("decode_t1", 1, 0.0, None),      # split-K, token tile 16
    ("decode_t1", 3, 0.0, None),
    ("decode_t1", 64, 0.0, 24),       # ~213 experts with 1-3 rows
    ("decode_t1", 512, 0.0, 12),      # token tile 32
    ("decode_t1", 1024, 0.0, 12),     # token tile 64
    ("decode_t1", 2048, 1.1, 12),     # token tile 128, skewed loads
    ("decode_t1", 4096, 0.0, 8),      # down GEMM with 256-token tiles
    ("toy", 1024, 1.5, None),         # paired-SM GEMMs: 256-token tiles, skewed, ragged tails
    ("decode_t1", 8192, 1.1, 8),      # paired-SM GEMMs at Beam shapes
])
def test_gate_up_and_down(name, T, skew, limit):
    m = model(name)
    ids, z_bits, counts, offsets, perm, inv, xp_bits = _inputs(m, T, skew, seed=T * 7 + 1)
    _check_gate_up_and_down(m, T, counts, offsets, xp_bits, limit)


def _ids_with_counts(counts, T, K):
    """Routing ids [T][K] in which expert e is chosen by counts[e] tokens,
    each token's K experts distinct: the experts' slots laid out expert by
    expert and dealt column by column (a block of at most T consecutive
    slots never meets the same token twice)."""
    assert sum(counts) == T * K and max(counts) <= T
    slots = np.repeat(np.arange(len(counts), dtype=np.int32), counts)
    return slots.reshape(K, T).T.copy()


def test_paired_gemm_tail_widths():
    """Paired-SM GEMMs (256-token tiles) with every kind of last tile: the
    experts' row counts leave 1, 15, 16, 17, 31, 32, 33, 63, 64, 65, 127, 128,
    129 and 200 rows in the last tile, one expert fills its last tile exactly
    and the last one takes the remaining rows (1127: a fifth tile of 103)."""
    m = model("toy")
    cfg = m.cfg
    tails = [1, 15, 16, 17, 31, 32, 33, 63, 64, 65, 127, 128, 129, 200, 256]
    counts = [256 + t for t in tails]
    T = 1536
    counts.append(T * cfg.K - sum(counts))
    assert counts[-1] == 1127
    ids = _ids_with_counts(counts, T, cfg.K)
    rng = np.random.default_rng(17)
    z_bits = obf.encode(rng.standard_normal((T, cfg.H)))
    cnt, offsets, perm, inv = permute(ids, cfg.E)
    assert list(cnt) == counts
    _check_gate_up_and_down(m, T, cnt, offsets, z_bits[perm], None)


def _check_gate_up_and_down(m, T, counts, offsets, xp_bits, limit):
    beam = beam_module()
    cfg = m.cfg
    mc = beam.make_config(cfg.H, cfg.E, cfg.G, cfg.TG, cfg.K, cfg.F, cfg.routed_scale, cfg.eps)
    off_d = torch.from_numpy(offsets).cuda()
    act = beam.beam_moe_gate_up(dev_bf16(xp_bits), off_d, m.dev[0], mc, T)
    # the down GEMM takes the oracle's rounded intermediate, so the two GEMMs are checked independently
    experts = _sample_experts(counts, limit)
    X = obf.decode(xp_bits)
    a_ref = np.zeros((T * cfg.K, cfg.F))
    rows_all = []
    for e in experts:
        lo, hi = offsets[e], offsets[e + 1]
        Wg, Wu, _ = m.expert_fn_nocache(int(e))
        a_ref[lo:hi] = intermediate(X[lo:hi], Wg, Wu)
        rows_all.append(np.arange(lo, hi))
    rows = np.concatenate(rows_all)
    act_gpu = f64_of(act)[rows]
    tol = 2.0 ** -8 * np.abs(a_ref[rows]) + 1e-4
    bad = np.abs(act_gpu - a_ref[rows]) > tol
    assert not bad.any(), f"gate/up: {int(bad.sum())} of {bad.size} beyond tolerance"

    act_in_bits = obf.encode(a_ref)
    y_perm = beam.beam_moe_down(dev_bf16(act_in_bits), off_d, m.dev[1], mc, T)
    A = obf.decode(act_in_bits)
    y_ref = np.zeros((T * cfg.K, cfg.H))
    for e in experts:
        lo, hi = offsets[e], offsets[e + 1]
        y_ref[lo:hi] = A[lo:hi] @ m.expert_fn_nocache(int(e))[2].T
    yg = f64_of(y_perm)[rows]
    tol = 2.0 ** -8 * np.abs(y_ref[rows]) + 1e-4
    bad = np.abs(yg - y_ref[rows]) > tol
    assert not bad.any(), f"down: {int(bad.sum())} of {bad.size} beyond tolerance"
    assert beam.beam_get_device_error() == 0


@pytest.mark.parametrize("name,T", [("toy", 16), ("decode_t1", 1), ("decode_t1", 8)])
def test_experts_and_combine(name, T):
    beam = beam_module()
    m = model(name)
    cfg = m.cfg
    mc = beam.make_config(cfg.H, cfg.E, cfg.G, cfg.TG, cfg.K, cfg.F, cfg.routed_scale, cfg.eps)
    ids, z_bits, counts, offsets, perm, inv, xp_bits = _inputs(m, T, 0.0, seed=T + 11)
    rng = np.random.default_rng(T)
    w = rng.random((T, cfg.K)) + 0.1
    w = (cfg.routed_scale * w / w.sum(axis=1, keepdims=True)).astype(np.float32)
    y = beam.beam_moe_experts(dev_bf16(xp_bits), torch.from_numpy(offsets).cuda(), m.dev[0], m.dev[1],
                              torch.from_numpy(w).cuda(), torch.from_numpy(inv).cuda(), mc, T)
    Z = obf.decode(z_bits)
    y_ref = np.zeros((T, cfg.H))
    for t in range(T):
        for k in range(cfg.K):
            Wg, Wu, Wd = m.expert_fn_nocache(int(ids[t, k]))
            y_ref[t] += float(w[t, k]) * (intermediate(Z[t:t + 1], Wg, Wu) @ Wd.T)[0]
    mx, rel = layer_errors(f64_of(y), y_ref)
    assert mx <= 2e-2 and rel <= 5e-3, (mx, rel)


def test_combine_unpermutes_with_one_slot():
    beam = beam_module()
    T, E, H = 300, 16, 256
    mc = beam.make_config(H, E, 4, 4, 1, 128)
    ids = random_topk_ids(T, E, 1, seed=2)
    _, _, perm, inv = permute(ids, E)
    x = torch.randn(T, H, device="cuda").to(torch.bfloat16)
    y_perm = x[torch.from_numpy(perm).long().cuda()]
    y = beam.beam_moe_combine(y_perm, torch.ones(T, 1, device="cuda"), torch.from_numpy(inv).cuda(), mc, T)
    assert torch.equal(y, x)


def test_combine_weighted_sum():
    beam = beam_module()
    T, E, K, H = 64, 16, 4, 512
    mc = beam.make_config(H, E, 4, 2, K, 128)
    ids = random_topk_ids(T, E, K, seed=4)
    _, _, perm, inv = permute(ids, E)
    rng = np.random.default_rng(5)
    yp_bits = obf.encode(rng.standard_normal((T * K, H)))
    w = rng.random((T, K)).astype(np.float32)
    y = beam.beam_moe_combine(dev_bf16(yp_bits), torch.from_numpy(w).cuda(), torch.from_numpy(inv).cuda(), mc, T)
    ref = combine(obf.decode(yp_bits), w.astype(np.float64), inv)
    # one bf16 rounding of an fp32 sum of K terms
    assert np.all(np.abs(f64_of(y) - ref) <= 2.0 ** -8 * np.abs(ref) + 1e-6)
