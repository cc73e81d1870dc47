"""Pins for oracle.layout: brute force over all routings of tiny problems, the
hand-evaluated worked examples under tests/golden/, and the layout invariants
stated in "Support DeepGEMM for standard MoE dispatch" (sglang PR #33128
report): every padding row is -1 and every token row is written exactly once.
"""

import itertools
import os

import numpy as np
import pytest

from oracle import layout as L

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _parse_rows(s):
    return np.array([[int(v) for v in r.split()] for r in s.split("|")])


def load_worked_example():
    d = {}
    for line in open(os.path.join(GOLDEN, "layout_worked_example.txt")):
        line = line.split("#")[0].strip()
        if line:
            k, v = line.split(":")
            d[k.strip()] = v.strip()
    return d


def test_worked_example_compact_and_masked():
    g = load_worked_example()
    ids = _parse_rows(g["topk_ids"])
    p = L.plan_layout(ids, E_global=4, E_local=3, expert_start=1, layout="compact", block_e=4)
    assert p["counts"].tolist() == [int(v) for v in g["counts"].split()]
    assert p["padded"].tolist() == [int(v) for v in g["padded"].split()]
    assert p["start"].tolist() == [int(v) for v in g["start"].split()]
    assert p["all_tokens"] == int(g["all_tokens"])
    assert p["m_indices"].tolist() == [int(v) for v in g["m_indices"].split()]
    assert np.array_equal(p["src2dst"], _parse_rows(g["src2dst"]))
    m = L.plan_layout(ids, E_global=4, E_local=3, expert_start=1, layout="masked", max_m=6)
    assert m["masked_m"].tolist() == [int(v) for v in g["masked_m"].split()]
    assert np.array_equal(m["src2dst"], _parse_rows(g["masked_src2dst"]))
    assert not p["errors"] and not m["errors"]


def test_compact_bound_golden_values():
    for line in open(os.path.join(GOLDEN, "compact_bound.txt")):
        line = line.split("#")[0].split()
        if line:
            A, E, bound = map(int, line)
            assert L.compact_all_tokens(A, E, 128) == bound


def _padded_rows(counts, block_e):
    return sum(-(-c // block_e) * block_e for c in counts)


@pytest.mark.parametrize("T,k,E,block_e", [(t, k, e, b) for t in (1, 2, 3, 4) for k in (1, 2)
                                           for e in (1, 2, 3, 4) for b in (1, 2, 4) if k <= e])
def test_bound_holds_and_is_tight_brute_force(T, k, E, block_e):
    """Enumerate every routing (distinct experts per token): the padded row
    count never exceeds the static bound, and some routing reaches it."""
    rows_choices = list(itertools.permutations(range(E), k))
    bound = L.compact_all_tokens(T * k, E, block_e)
    best = 0
    for routing in itertools.product(rows_choices, repeat=T):
        counts = np.bincount(np.array(routing).reshape(-1), minlength=E)
        best = max(best, _padded_rows(counts, block_e))
    assert best <= bound
    # Tightness over unconstrained assignment multisets (the bound's own
    # premise: assignments may land on any expert).
    A = T * k
    worst = 0
    for counts in itertools.product(range(A + 1), repeat=E):
        if sum(counts) == A:
            worst = max(worst, _padded_rows(counts, block_e))
    assert worst == bound


def test_bound_random_large_routings():
    rng = np.random.default_rng(3)
    for _ in range(200):
        E = int(rng.integers(1, 300))
        A = int(rng.integers(0, 70000))
        counts = np.bincount(rng.integers(0, E, size=A), minlength=E)
        assert _padded_rows(counts, 128) <= L.compact_all_tokens(A, E, 128)


def test_masked_choice():
    assert L.use_masked_layout(256, 32) and L.use_masked_layout(64, 8)
    assert not L.use_masked_layout(256, 33) and not L.use_masked_layout(32, 32)
    assert not L.use_masked_layout(128, 128)


def check_plan_invariants(ids, E_global, E_local, expert_start, block_e, max_m):
    T, k = ids.shape
    flat = ids.reshape(-1)
    loc = flat - expert_start
    is_local = (flat >= 0) & (flat < E_global) & (loc >= 0) & (loc < E_local)
    p = L.plan_layout(ids, E_global, E_local, expert_start, "compact", block_e)
    src = p["src2dst"].reshape(-1)
    mi = p["m_indices"]
    assert np.all(src[~is_local] == -1)
    d = src[is_local]
    assert len(np.unique(d)) == d.size                          # injective
    assert np.array_equal(mi[d], loc[is_local])                  # row -> its expert
    assert np.count_nonzero(mi >= 0) == d.size                   # onto the token rows
    assert np.all(p["padded"] % block_e == 0) and np.all(p["padded"] >= p["counts"])
    assert np.all(p["padded"] - p["counts"] < block_e)
    assert p["padded"].sum() <= p["all_tokens"] == mi.size
    for e in range(E_local):                                     # stable order inside experts
        de = src[is_local & (loc == e)]
        assert np.array_equal(de, p["start"][e] + np.arange(de.size))
        seg = mi[p["start"][e]:p["start"][e] + p["padded"][e]]
        assert np.all(seg[:de.size] == e) and np.all(seg[de.size:] == -1)
    assert np.all(mi[p["padded"].sum():] == -1)
    m = L.plan_layout(ids, E_global, E_local, expert_start, "masked", block_e, max_m)
    msrc = m["src2dst"].reshape(-1)
    assert np.array_equal(m["masked_m"], np.minimum(p["counts"], max_m))
    for e in range(E_local):
        de = msrc[is_local & (loc == e)]
        n = min(de.size, max_m)
        assert np.array_equal(de[:n], e * max_m + np.arange(n))
        assert np.all(de[n:] == -1)


def test_plan_invariants_random():
    rng = np.random.default_rng(11)
    for _ in range(60):
        T = int(rng.integers(1, 200))
        E_global = int(rng.integers(1, 40))
        k = int(rng.integers(1, min(E_global, 8) + 1))
        E_local = int(rng.integers(1, E_global + 1))
        expert_start = int(rng.integers(0, E_global - E_local + 1))
        ids = np.stack([rng.permutation(E_global)[:k] for _ in range(T)])
        drop = rng.random(ids.shape) < 0.1
        ids[drop] = -1
        block_e = int(rng.choice([1, 4, 128]))
        max_m = int(rng.integers(1, T + 1))
        check_plan_invariants(ids, E_global, E_local, expert_start, block_e, max_m)


def test_bad_ids_are_reported_and_dropped():
    ids = np.array([[0, 5], [1, -3]])
    p = L.plan_layout(ids, E_global=4, E_local=4, expert_start=0, layout="compact")
    assert p["errors"] == {"expert_id"}
    assert p["src2dst"].tolist() == [[0, -1], [128, -1]]
    m = L.plan_layout(np.array([[0], [0], [0]]), 4, 4, 0, "masked", max_m=2)
    assert m["errors"] == {"masked_overflow"} and m["masked_m"].tolist() == [2, 0, 0, 0]
    assert m["src2dst"].reshape(-1).tolist() == [0, 1, -1]
