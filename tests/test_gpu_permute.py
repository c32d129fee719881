"""GPU parity: permutation by expert is bit-exact against the oracle's stable sort."""
import numpy as np
import pytest
import torch

from beam_inputs import random_topk_ids
from oracle.permute import permute
from tests.gpu_support import beam_module

pytestmark = pytest.mark.gpu


def _cfg(beam, E, K, H=256):
    G = 8 if E % 8 == 0 else 1
    return beam.make_config(H, E, G, G, K, 128)


@pytest.mark.parametrize("T,E,K,skew", [(1, 256, 8, 0.0), (16, 16, 4, 0.0), (37, 256, 8, 0.0),
                                        (64, 256, 8, 0.0), (300, 64, 8, 1.5), (2048, 256, 8, 0.0),
                                        (2049, 256, 8, 1.1), (16384, 256, 8, 1.1)])
def test_permutation_bit_exact(T, E, K, skew):
    beam = beam_module()
    ids = random_topk_ids(T, E, K, seed=T + E, skew=skew)
    H = 256
    z = torch.randn(T, H, device="cuda").to(torch.bfloat16)
    offsets, perm, inv, x_perm = beam.beam_moe_permute(torch.from_numpy(ids).cuda(), z, _cfg(beam, E, K, H))
    torch.cuda.synchronize()
    counts, o_off, o_perm, o_inv = permute(ids, E)
    assert np.array_equal(offsets.cpu().numpy(), o_off)
    assert np.array_equal(perm.cpu().numpy(), o_perm)
    assert np.array_equal(inv.cpu().numpy(), o_inv)
    assert torch.equal(x_perm, z[perm.long()])


def test_permutation_is_deterministic():
    beam = beam_module()
    ids = torch.from_numpy(random_topk_ids(5000, 256, 8, seed=9, skew=1.3)).cuda()
    cfg = _cfg(beam, 256, 8)
    a = beam.beam_moe_permute(ids, None, cfg, gather=False)
    b = beam.beam_moe_permute(ids, None, cfg, gather=False)
    for u, v in zip(a[:3], b[:3]):
        assert torch.equal(u, v)


def test_out_of_range_ids_are_dropped():
    beam = beam_module()
    ids = random_topk_ids(40, 16, 4, seed=3)
    ids[5, 1] = -1
    ids[7, 3] = 16
    offsets, perm, inv, _ = beam.beam_moe_permute(torch.from_numpy(ids).cuda(), None, _cfg(beam, 16, 4),
                                                  gather=False)
    inv = inv.cpu().numpy()
    assert inv[5 * 4 + 1] == -1 and inv[7 * 4 + 3] == -1
    assert offsets.cpu().numpy()[-1] == 40 * 4 - 2
    valid = ids.copy()
    keep = (valid >= 0) & (valid < 16)
    counts = np.bincount(valid[keep], minlength=16)
    assert np.array_equal(np.diff(offsets.cpu().numpy()), counts)
