"""Pins for the oracle's acceptance walk.

Greedy: hand-worked walk, forced-argmax full chain, and a brute force over
every node (the accepted path ends at the deepest node whose whole root path
matches the parents' argmaxes).  Sampling: closed forms of the warped
distribution on rows of log-probabilities, the inverse CDF on a hand case,
and the losslessness the pages claim -- over many seeds the first emitted
token follows the warped target distribution of the root (chi-square), each
child is accepted with probability p(token), and a single-child chain reduces
to standard speculative sampling with a one-hot draft.
"""

import numpy as np
import pytest
from scipy import stats

from oracle import philox
from oracle.verify import inverse_cdf, verify_tree, warped_distribution

# tree used by the hand cases (same shape as the hand-worked build example)
PARENTS = [-1, 0, 0, 1, 1, 2, 3]
TOKENS = [2, 3, 1, 2, 0, 5, 1]


def _rows(V, m, seed):
    rng = np.random.default_rng(seed)
    return (rng.standard_normal((m, V)) * 2.0).astype(np.float32)


# ------------------------------------------------------------------ greedy
def test_greedy_hand_walk():
    x = _rows(6, 7, 0)
    x[0, 1] = 50.0      # root predicts tok1 -> node 2
    x[2, 5] = 50.0      # node 2 predicts tok5 -> node 5 (a leaf)
    x[5, 4] = 50.0      # bonus at node 5 = tok4
    r = verify_tree(x, PARENTS, TOKENS)
    assert r["path"] == [0, 2, 5] and r["n_accepted"] == 2 and r["bonus"] == 4


def test_greedy_first_discrepancy_stops():
    x = _rows(6, 7, 1)
    x[0, 4] = 50.0      # tok4 is no child of the root
    r = verify_tree(x, PARENTS, TOKENS)
    assert r["path"] == [0] and r["bonus"] == 4


def test_greedy_forced_first_child_chain():
    x = _rows(6, 7, 2)
    x[0, 3] = 50.0      # -> node 1
    x[1, 2] = 50.0      # -> node 3 (first child of node 1)
    x[3, 1] = 50.0      # -> node 6 (leaf)
    x[6, 0] = 50.0
    r = verify_tree(x, PARENTS, TOKENS)
    assert r["path"] == [0, 1, 3, 6] and r["bonus"] == 0


def test_greedy_ties_go_to_lower_token_id():
    x = np.zeros((7, 6), dtype=np.float32)
    x[0, 1] = x[0, 3] = 9.0           # tie: tok1 < tok3 -> node 2
    r = verify_tree(x, PARENTS, TOKENS)
    assert r["path"][:2] == [0, 2]


@pytest.mark.parametrize("seed", range(20))
def test_greedy_bruteforce_all_nodes(seed):
    rng = np.random.default_rng(seed)
    V = 6
    x = _rows(V, 7, 100 + seed)
    for i in range(7):                 # make matches likely
        if rng.random() < 0.7:
            kids = [c for c in range(1, 7) if PARENTS[c] == i]
            if kids:
                x[i, TOKENS[kids[int(rng.integers(len(kids)))]]] = 30.0
    am = [int(np.argmax(x[i])) for i in range(7)]      # no ties with N(0,4) draws
    ok = [True] + [False] * 6
    for i in range(1, 7):
        ok[i] = ok[PARENTS[i]] and TOKENS[i] == am[PARENTS[i]]
    depth = [0, 1, 1, 2, 2, 2, 3]
    deepest = max((i for i in range(7) if ok[i]), key=lambda i: depth[i])
    r = verify_tree(x, PARENTS, TOKENS)
    assert r["path"][-1] == deepest and r["bonus"] == am[deepest]


# ------------------------------------------------------- warped distribution
def test_warped_distribution_closed_forms():
    p = np.array([0.0625, 0.5, 0.125, 0.25, 0.0625])       # ids 0..4
    row = np.log(p).astype(np.float32)
    ids, q = warped_distribution(row, 1.0, 0, 1.0)
    np.testing.assert_allclose(q, p, rtol=1e-6)
    ids, q = warped_distribution(row, 1.0, 2, 1.0)          # top-2: ids 1, 3
    assert ids.tolist() == [1, 3]
    np.testing.assert_allclose(q, [2 / 3, 1 / 3], rtol=1e-6)
    ids, q = warped_distribution(row, 1.0, 0, 0.6)          # .5 + .25 >= .6
    assert ids.tolist() == [1, 3]
    np.testing.assert_allclose(q, [2 / 3, 1 / 3], rtol=1e-6)
    ids, q = warped_distribution(row, 1.0, 0, 0.5)          # .5 alone reaches .5
    assert ids.tolist() == [1]
    ids, q = warped_distribution(row, 1.0, 4, 0.85)         # top-4 renorm: .533 .8 .933
    assert ids.tolist() == [1, 2, 3]
    ids, q = warped_distribution(row, 0.5, 0, 1.0)          # T = 0.5 squares p
    np.testing.assert_allclose(q, p ** 2 / np.sum(p ** 2), rtol=1e-6)


def test_inverse_cdf_hand_case():
    ids = np.array([2, 5, 7, 9])
    p = np.array([0.1, 0.4, 0.3, 0.2])
    assert inverse_cdf(ids, p, [], 0.05) == 2
    assert inverse_cdf(ids, p, [], 0.10) == 5            # strict: cum must exceed
    assert inverse_cdf(ids, p, [5], 0.35) == 7           # cum .1, .1, .4, .6
    assert inverse_cdf(ids, p, [5, 7], 0.25) == 9
    assert inverse_cdf(ids, p, [], 0.9999) == 9


# ------------------------------------------------------------ losslessness
def _first_token(res, tokens):
    return tokens[res["path"][1]] if res["n_accepted"] else res["bonus"]


@pytest.mark.parametrize("T,top_k,top_p", [(1.0, 0, 1.0), (0.7, 5, 0.9)])
def test_sampling_is_lossless_on_the_first_token(T, top_k, top_p):
    V = 8
    parents = [-1, 0, 0, 0, 1, 1, 2]
    tokens = [0, 3, 1, 6, 2, 7, 4]
    rng = np.random.default_rng(7)
    x = (rng.standard_normal((7, V)) * 1.2).astype(np.float32)
    x[0, 3] += 1.0
    ids, p = warped_distribution(x[0], T, top_k, top_p)
    target = np.zeros(V)
    target[ids] = p
    N = 30000
    counts = np.zeros(V)
    acc_child = np.zeros(V)
    for seed in range(N):
        r = verify_tree(x, parents, tokens, greedy=False, temperature=T, top_k=top_k,
                        top_p=top_p, seed=seed, step=3)
        counts[_first_token(r, tokens)] += 1
        if r["n_accepted"]:
            acc_child[tokens[r["path"][1]]] += 1
    assert counts[target == 0].sum() == 0
    keep = target > 0
    assert stats.chisquare(counts[keep], target[keep] * N).pvalue > 1e-3
    # a child token is emitted only by accepting that child: P = p(token)
    for c in (1, 2, 3):
        tok = tokens[c]
        assert acc_child[tok] == counts[tok]
    # nothing accepted with probability 1 - sum of children's p
    p_none = 1.0 - sum(target[tokens[c]] for c in (1, 2, 3))
    n_none = N - acc_child.sum()
    assert abs(n_none / N - p_none) < 5 * np.sqrt(p_none * (1 - p_none) / N) + 1e-9


def test_single_child_reduces_to_one_hot_speculative_sampling():
    V = 5
    parents = [-1, 0]
    tokens = [0, 2]
    x = np.log(np.array([[0.1, 0.2, 0.3, 0.15, 0.25], [0.2] * 5])).astype(np.float32)
    N = 20000
    acc = 0
    for seed in range(N):
        r = verify_tree(x, parents, tokens, greedy=False, seed=seed, step=0)
        acc += r["n_accepted"]
        if r["n_accepted"] == 0:
            assert r["bonus"] != 2            # rejected token never re-drawn
    # one-hot draft on token 2: accepted with probability p(2) = 0.3
    assert abs(acc / N - 0.3) < 5 * np.sqrt(0.3 * 0.7 / N)


def test_sampling_uses_the_keyed_uniforms():
    # with u known, the acceptance of the first child is decided by u < p
    V = 4
    x = np.log(np.array([[0.4, 0.3, 0.2, 0.1], [0.25] * 4])).astype(np.float32)
    for seed in range(50):
        u = philox.uniform(seed, 9, 0, 0)
        r = verify_tree(x, [-1, 0], [0, 0], greedy=False, seed=seed, step=9)
        assert (r["n_accepted"] == 1) == (u < 0.4 * (1 + 1e-7))
