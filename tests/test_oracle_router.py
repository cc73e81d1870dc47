"""Pins for oracle.router: selection against a sort with an explicit
(-logit, id) key and brute force over tiny rows with many ties; the top-k
softmax against scipy's softmax (k = E) and torch's; logits against torch
float64 matmul."""

import itertools

import numpy as np
import pytest
import scipy.special
import torch

from oracle import router as R


def test_selection_matches_keyed_sort_with_ties():
    rng = np.random.default_rng(0)
    z = rng.integers(-3, 4, size=(200, 17)).astype(np.float32)   # many ties
    ids = R.select_topk(z, 5)
    for t in range(z.shape[0]):
        order = sorted(range(17), key=lambda e: (-float(z[t, e]), e))[:5]
        assert ids[t].tolist() == order


def test_selection_brute_force_tiny():
    for row in itertools.product([0.0, 1.0, -1.0], repeat=4):
        z = np.array([row])
        for k in range(1, 5):
            ids = R.select_topk(z, k)[0].tolist()
            # every chosen logit >= every unchosen; ties resolved to lower ids
            rest = [e for e in range(4) if e not in ids]
            assert all(z[0, a] >= z[0, b] for a in ids for b in rest)
            for a, b in zip(ids, ids[1:]):
                assert z[0, a] > z[0, b] or (z[0, a] == z[0, b] and a < b)
            for a in ids:
                for b in rest:
                    assert z[0, a] > z[0, b] or a < b


def test_topk_softmax_against_libraries():
    rng = np.random.default_rng(1)
    z = rng.standard_normal((50, 12))
    full = R.topk_softmax(z, np.tile(np.arange(12), (50, 1)))
    assert np.allclose(full, scipy.special.softmax(z, axis=1), rtol=1e-14, atol=0)
    ids = R.select_topk(z, 4)
    w = R.topk_softmax(z, ids)
    ref = torch.softmax(torch.from_numpy(np.take_along_axis(z, ids, axis=1)), dim=1).numpy()
    assert np.allclose(w, ref, rtol=1e-14, atol=1e-16)
    assert np.allclose(w.sum(axis=1), 1.0, rtol=0, atol=1e-15)


def test_logits_against_torch():
    rng = np.random.default_rng(2)
    x = torch.randn(20, 300).to(torch.bfloat16).double().numpy()
    w = rng.standard_normal((9, 300)).astype(np.float32)
    assert np.allclose(R.logits(x, w), (torch.from_numpy(x) @ torch.from_numpy(w.astype(np.float64)).T).numpy(),
                       rtol=1e-13, atol=1e-13)
