"""beam_moe_permute_no_alloc: the permutation for callers that cannot pass a
workspace (for example an operator plugin that only receives the tensors it
declares, or a loop where a device allocation is not allowed). It must give
exactly what beam_moe_permute gives, call after call, even though every call
reuses the same fixed scratch array inside the library.

This file is named to be collected last, so that a run stopping at the first
failure has already run every other test."""
import ctypes

import numpy as np
import pytest
import torch

from beam_inputs import random_topk_ids
from tests.gpu_support import beam_module

pytestmark = pytest.mark.gpu


def _call_no_alloc(beam, ids, z, cfg):
    T = ids.shape[0]
    rows = T * cfg.topk
    dev = ids.device
    offsets = torch.full((cfg.num_experts + 1,), -7, dtype=torch.int32, device=dev)
    perm = torch.full((rows,), -7, dtype=torch.int32, device=dev)
    inv = torch.full((rows,), -7, dtype=torch.int32, device=dev)
    x_perm = torch.zeros(rows, cfg.hidden, dtype=torch.bfloat16, device=dev)
    st = beam.library().beam_moe_permute_no_alloc(
        ids.data_ptr(), z.data_ptr(), T, ctypes.byref(cfg), offsets.data_ptr(), perm.data_ptr(), inv.data_ptr(),
        x_perm.data_ptr(), torch.cuda.current_stream().cuda_stream)
    assert st == 0, beam.beam_status_string(st)
    return offsets, perm, inv, x_perm


@pytest.mark.parametrize("cases", [[(37, 256, 8, 0.0, 1), (16384, 256, 8, 1.1, 2)],
                                   [(5000, 64, 6, 1.3, 3), (1, 256, 8, 0.0, 4)]])
def test_no_alloc_matches_regular_entry_point_on_consecutive_calls(cases):
    beam = beam_module()
    for T, E, K, skew, seed in cases:       # two calls in a row share the library's scratch array
        H = 256
        cfg = beam.make_config(H, E, 8, 8, K, 128)
        ids = torch.from_numpy(random_topk_ids(T, E, K, seed=seed, skew=skew)).cuda()
        z = torch.randn(T, H, device="cuda").to(torch.bfloat16)
        got = _call_no_alloc(beam, ids, z, cfg)
        ref = beam.beam_moe_permute(ids, z, cfg)
        torch.cuda.synchronize()
        for g, r in zip(got, ref):
            assert torch.equal(g, r)                 # integer and copy outputs: bit-exact


def test_no_alloc_rejects_sizes_beyond_its_array():
    beam = beam_module()
    lib = beam.library()
    cfg = beam.make_config(256, 256, 8, 4, 8, 128)
    too_many_tokens = 131072 // 8 + 1
    p = 0x10000
    st = lib.beam_moe_permute_no_alloc(p, p, too_many_tokens, ctypes.byref(cfg), p, p, p, None, None)
    assert st == 4 and "workspace" in beam.beam_status_string(st)
    # an empty batch is still a no-op
    assert lib.beam_moe_permute_no_alloc(None, None, 0, ctypes.byref(cfg), None, None, None, None, None) == 0
