"""Pins for the oracle's permutation and weighted combine."""
import json
import os

import numpy as np

from beam_inputs import random_topk_ids
from oracle.combine import combine
from oracle.permute import permute

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def test_permutation_worked_example():
    g = json.load(open(os.path.join(GOLDEN, "permute_small.json")))
    counts, offsets, perm, inv = permute(np.array(g["ids"]), g["E"])
    assert counts.tolist() == g["counts"]
    assert offsets.tolist() == g["offsets"]
    assert perm.tolist() == g["perm_token"]
    assert inv.tolist() == g["inv_perm"]


def test_permutation_is_a_stable_sort_by_expert():
    for T, E, K, skew in ((1, 256, 8, 0), (37, 16, 4, 0), (300, 64, 8, 1.2)):
        ids = random_topk_ids(T, E, K, seed=T, skew=skew)
        counts, offsets, perm, inv = permute(ids, E)
        flat = ids.reshape(-1)
        order = np.lexsort((np.arange(T * K), flat))          # library stable sort by (expert, pair)
        assert np.array_equal(perm, order // K)
        assert np.array_equal(np.sort(inv), np.arange(T * K))  # bijection
        assert np.array_equal(order[inv], np.arange(T * K))
        assert counts.sum() == T * K and np.array_equal(counts, np.bincount(flat, minlength=E))
        assert offsets[0] == 0 and np.array_equal(np.diff(offsets), counts)
        for e in range(E):
            seg = perm[offsets[e]:offsets[e + 1]]
            assert np.all(np.diff(seg) > 0)                    # tokens ascending within an expert


def test_combine_worked_example():
    Y = np.array([[1, 0, 0], [0, 1, 0], [0, 0, 1], [1, 1, 1]], dtype=np.float64)
    inv = np.array([2, 0, 3, 1])
    w = np.array([[0.5, 2.0], [1.0, -1.0]])
    # y0 = 0.5*Y[2] + 2*Y[0] = (2, 0, 0.5);  y1 = Y[3] - Y[1] = (1, 0, 1)
    assert combine(Y, w, inv).tolist() == [[2.0, 0.0, 0.5], [1.0, 0.0, 1.0]]


def test_combine_with_one_slot_and_unit_weight_unpermutes():
    rng = np.random.default_rng(11)
    T, E = 50, 7
    ids = rng.integers(0, E, (T, 1)).astype(np.int32)
    _, _, perm, inv = permute(ids, E)
    X = rng.standard_normal((T, 5))
    Y_perm = X[perm]
    assert np.array_equal(combine(Y_perm, np.ones((T, 1)), inv), X)
