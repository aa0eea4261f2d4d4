"""Pins for the oracle's tree-shape policies (static tree, batched chains,
confidence ratio): worked examples whose trees are written out by hand from
the ratios, reductions of one policy to another, brute-force children from a
stable argsort, closed-form sizes, and the ancestor mask against the
transitive closure of the parent relation."""

import math

import numpy as np
import pytest

from oracle.tree_build import mask_to_bool
from oracle.tree_policies import (candidate_chains, confidence_tree, static_tree,
                                  static_tree_size)


def _rows(n_rows, V, seed):
    return np.random.default_rng(seed).standard_normal((n_rows, V)).astype(np.float32)


def _closure(parents):
    """Ancestor-or-self matrix by repeated squaring of the parent relation."""
    m = len(parents)
    a = np.eye(m, dtype=bool)
    for i in range(1, m):
        a[i, parents[i]] = True
    while True:
        b = (a.astype(np.int64) @ a.astype(np.int64)) > 0
        if (b == a).all():
            return a
        a = b


def _stable_top(row, n):
    return list(np.argsort(-np.asarray(row, dtype=np.float64), kind="stable")[:n])


def _check_common(t):
    m = t["m"]
    par, dep = t["parents"], t["depth"]
    assert par[0] == -1 and dep[0] == 0
    for i in range(1, m):
        assert 0 <= par[i] < i and dep[i] == dep[par[i]] + 1
    assert (np.diff(dep) >= 0).all() and (np.diff(par[1:]) >= 0).all()   # breadth-first
    np.testing.assert_array_equal(mask_to_bool(t["mask"], m), _closure(par))
    np.testing.assert_array_equal(t["pos"], dep)


# ------------------------------------------------------------ confidence ratio

def _hand_rows():
    """Three rows over 8 tokens whose probabilities are set through logs."""
    x = np.zeros((8, 8), dtype=np.float32)
    # root: p(5) / p(2) = 6 / 2 = 3 > tau = 2 -> one child, token 5
    x[0, 5], x[0, 2] = math.log(6.0), math.log(2.0)
    # node 1: p(3) : p(6) : p(0) : p(7) = 4 : 3 : 2.5 : 1.9 -> C = 4/3 <= 2;
    # within a factor 2 of the best: 6 (1.33) and 0 (1.6), not 7 (2.1) -> 3 children
    x[1, 3], x[1, 6], x[1, 0], x[1, 7] = (math.log(4.0), math.log(3.0), math.log(2.5),
                                          math.log(1.9))
    # node 2: a flat row -> C = 1, every token within the factor -> 4 children
    # (lowest ids), cut by the budget of 8 nodes after three of them
    return x


def test_confidence_hand_example():
    t = confidence_tree(_hand_rows(), 2.0, 8, 99)
    assert t["m"] == 8
    assert list(t["parents"]) == [-1, 0, 1, 1, 1, 2, 2, 2]
    assert list(t["tokens"]) == [99, 5, 3, 6, 0, 0, 1, 2]
    assert list(t["depth"]) == [0, 1, 2, 2, 2, 3, 3, 3]
    assert list(t["node_row"]) == [0, 1, 2, -1, -1, -1, -1, -1]
    assert t["rows_used"] == 3
    _check_common(t)


def test_confidence_hand_example_larger_budget():
    # with room for all four children of node 2, then nodes 3 and 4 expand
    # (their rows are flat as well: four children each; the budget of 14 leaves
    # node 4 one child)
    t = confidence_tree(_hand_rows(), 2.0, 14, 99)
    assert list(t["parents"]) == [-1, 0, 1, 1, 1, 2, 2, 2, 2, 3, 3, 3, 3, 4]
    assert list(t["tokens"]) == [99, 5, 3, 6, 0, 0, 1, 2, 3, 0, 1, 2, 3, 0]
    _check_common(t)


def test_confidence_chain_to_max_depth():
    # one dominant token per row (ratio e^3 > 2): a chain, stopped by max_depth
    x = _rows(12, 50, 3)
    best = [7, 11, 0, 49, 23]
    for i, b in enumerate(best):
        x[i, b] = 10.0
    t = confidence_tree(x, 2.0, 40, 1, max_depth=4)
    assert t["m"] == 5
    assert list(t["tokens"]) == [1] + best[:4]
    assert list(t["parents"]) == [-1, 0, 1, 2, 3]
    _check_common(t)


@pytest.mark.parametrize("seed", [0, 1, 2])
def test_confidence_below_one_is_the_argmax_chain(seed):
    # tau < 1: C >= 1 > tau at every node, so every node has one child
    x = _rows(20, 300, seed)
    t = confidence_tree(x, 0.5, 50, 4, max_depth=9)
    s = static_tree(x, 1, 9, 4)
    for key in ("parents", "tokens", "depth"):
        np.testing.assert_array_equal(t[key], s[key])


@pytest.mark.parametrize("seed,m", [(0, 30), (1, 57), (2, 200)])
def test_confidence_huge_tau_is_the_static_tree_cut(seed, m):
    # tau beyond every ratio: every node branches to max_branch = 4 children,
    # i.e. the full 4-ary tree in node order, cut after m nodes
    x = _rows(100, 120, seed)        # the static tree reads rows 0..84
    t = confidence_tree(x, 1e30, m, 9, max_depth=10, max_branch=4)
    s = static_tree(x, 4, 4, 9)      # 341 nodes, enough for every m here
    assert t["m"] == m
    for key in ("parents", "tokens", "depth"):
        np.testing.assert_array_equal(t[key], s[key][:m])


@pytest.mark.parametrize("seed", [0, 5])
def test_confidence_children_follow_the_ratio(seed):
    # brute force over a random tree: each expanded node has 1 child iff its
    # top-two logit gap exceeds ln tau, else every token within a factor tau
    # of the best, between 2 and 4, in stable-argsort order (the last expanded
    # node may be cut by the budget)
    x = _rows(200, 40, seed) * 0.7
    tau = 2.0
    t = confidence_tree(x, tau, 150, 0, max_depth=6)
    par, tok = t["parents"], t["tokens"]
    expanded = [i for i in range(t["m"]) if t["node_row"][i] >= 0]
    for i in expanded:
        kids = [j for j in range(t["m"]) if par[j] == i]
        order = _stable_top(x[i], 40)
        gap = float(x[i][order[0]]) - float(x[i][order[1]])
        if gap > math.log(tau):
            want = order[:1]
        else:
            within = [v for v in order if float(x[i][order[0]]) - float(x[i][v]) <= math.log(tau)]
            want = order[:min(4, max(2, len(within)))]
        got = [int(tok[j]) for j in kids]
        if i == expanded[-1]:
            assert got == want[:len(got)]
        else:
            assert got == want
    assert all(t["depth"] <= 6) and t["m"] <= 150
    _check_common(t)


# ------------------------------------------------------------ static tree

@pytest.mark.parametrize("n,D", [(1, 5), (2, 4), (3, 3), (5, 2), (4, 0)])
def test_static_tree_sizes_and_children(n, D):
    x = _rows(200, 64, 11)
    t = static_tree(x, n, D, 2)
    assert t["m"] == static_tree_size(n, D) == (D + 1 if n == 1 else (n ** (D + 1) - 1) // (n - 1))
    internal = static_tree_size(n, D - 1) if D >= 1 else 0
    assert t["rows_used"] == internal
    for i in range(internal):
        kids = [j for j in range(t["m"]) if t["parents"][j] == i]
        assert [int(t["tokens"][j]) for j in kids] == _stable_top(x[i], n)
    _check_common(t)


def test_static_chain_is_the_argmax_path():
    x = _rows(8, 500, 4)
    t = static_tree(x, 1, 6, 3)
    assert list(t["tokens"]) == [3] + [int(np.argmax(x[i])) for i in range(6)]


def test_static_ties_take_lower_ids():
    x = np.zeros((4, 10), dtype=np.float32)
    t = static_tree(x, 3, 1, 0)
    assert list(t["tokens"]) == [0, 0, 1, 2]


# ------------------------------------------------------------ batched chains

@pytest.mark.parametrize("n,D", [(3, 4), (10, 6), (2, 1)])
def test_chains_by_brute_force(n, D):
    x = _rows(1 + n * D, 200, 6)
    t = candidate_chains(x, n, D, 8)
    assert t["m"] == 1 + n * D
    first = _stable_top(x[0], n)
    for j in range(n):
        node, chain = 1 + j, [first[j]]
        for d in range(2, D + 1):
            chain.append(int(np.argmax(x[node])))
            node += n
        got = [int(t["tokens"][1 + (d - 1) * n + j]) for d in range(1, D + 1)]
        assert got == chain
    _check_common(t)


def test_one_chain_is_the_static_chain():
    x = _rows(10, 80, 7)
    a = candidate_chains(x, 1, 7, 5)
    b = static_tree(x, 1, 7, 5)
    for key in ("parents", "tokens", "depth", "mask"):
        np.testing.assert_array_equal(a[key], b[key])
