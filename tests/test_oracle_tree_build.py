"""Pins for the oracle's draft-tree construction.

Checked against: library routines (scipy logsumexp), closed forms (uniform
rows, rows of log-probabilities), a tree worked out by hand, special cases
whose shape is known in advance (chain, star, full expansion, identical
rows), brute-force pairwise checks of every selection, and an independent
transitive closure (Warshall) of the parent relation for the mask.
"""

import numpy as np
import pytest
from scipy.special import logsumexp

from oracle.tree_build import (build_draft_tree, mask_to_bool, row_logsumexp,
                               row_top_k, tree_sizes)
from eagle_speculative_decoding_verify_gb300 import workloads as wl


def _beats(v_a, i_a, v_b, i_b):
    return v_a > v_b or (v_a == v_b and i_a < i_b)


# --------------------------------------------------------------- row stats
def test_logsumexp_matches_library_and_closed_forms():
    rng = np.random.default_rng(0)
    for sigma in (1.0, 3.0, 6.0, 40.0):
        row = (rng.standard_normal(5000) * sigma).astype(np.float32)
        assert abs(row_logsumexp(row) - logsumexp(row.astype(np.float64))) < 1e-12
    # uniform row: log(V) + c exactly
    for V in (1, 7, 1000, 128256):
        c = -3.25
        assert abs(row_logsumexp(np.full(V, c)) - (c + np.log(V))) < 1e-12
    # row of log-probabilities that sum to one: logsumexp is 0
    p = np.array([0.5, 0.25, 0.125, 0.0625, 0.0625])
    assert abs(row_logsumexp(np.log(p))) < 1e-15


def test_top_k_bruteforce_with_ties():
    rng = np.random.default_rng(1)
    for trial in range(50):
        V = int(rng.integers(1, 40))
        row = rng.integers(-3, 4, size=V).astype(np.float32)   # many ties
        k = int(rng.integers(1, V + 1))
        sel = list(row_top_k(row, k))
        assert len(set(sel)) == k
        rest = [i for i in range(V) if i not in sel]
        for a in sel:                       # every selected beats every other
            for b in rest:
                assert _beats(row[a], a, row[b], b)
        for x, y in zip(sel, sel[1:]):      # selected come best first
            assert _beats(row[x], x, row[y], y)


# --------------------------------------------------------- hand-worked tree
# V = 6, top_k = 2, depth = 3 (R = 5 rows, C = 10 candidates).  Each row holds
# log-probabilities, so a node's value is the log of the product of the
# probabilities along its path.  Worked by hand:
#   row 0 (root):            tok3 .60, tok1 .30          -> c0 (tok3, .60), c1 (tok1, .30)
#   frontier depth 1:        slot0 = c0, slot1 = c1
#   row 1 (slot0, under c0): tok2 .70, tok0 .20          -> c2 (.42), c3 (.12)
#   row 2 (slot1, under c1): tok5 .55, tok4 .35          -> c4 (.165), c5 (.105)
#   frontier depth 2:        best two of {.42,.12,.165,.105} -> slot0 = c2, slot1 = c4
#   row 3 (slot0, under c2): tok1 .80, tok5 .10          -> c6 (.336), c7 (.042)
#   row 4 (slot1, under c4): tok0 .45, tok3 .44          -> c8 (.07425), c9 (.0726)
#   ranking: c0 .6 > c2 .42 > c6 .336 > c1 .3 > c4 .165 > c3 .12 > c5 .105 > ...
#   m = 7 keeps c0 c2 c6 c1 c4 c3 -> nodes in candidate order c0 c1 c2 c3 c4 c6
_HAND_P = [
    {3: .60, 1: .30, 0: .04, 2: .03, 4: .02, 5: .01},
    {2: .70, 0: .20, 1: .05, 3: .03, 4: .01, 5: .01},
    {5: .55, 4: .35, 0: .05, 1: .03, 2: .01, 3: .01},
    {1: .80, 5: .10, 0: .04, 2: .03, 3: .02, 4: .01},
    {0: .45, 3: .44, 1: .05, 2: .03, 4: .02, 5: .01},
]


def _hand_logits():
    out = np.zeros((5, 6), dtype=np.float32)
    for r, probs in enumerate(_HAND_P):
        for t, p in probs.items():
            out[r, t] = np.log(p)
    return out


def test_hand_worked_tree():
    t = build_draft_tree(_hand_logits(), top_k=2, depth=3, total_tokens=7, root_token=2)
    assert t["parents"].tolist() == [-1, 0, 0, 1, 1, 2, 3]
    assert t["tokens"].tolist() == [2, 3, 1, 2, 0, 5, 1]
    assert t["depth"].tolist() == [0, 1, 1, 2, 2, 2, 3]
    assert t["pos"].tolist() == t["depth"].tolist()
    assert t["selected"].tolist() == [0, 1, 2, 3, 4, 6]
    np.testing.assert_allclose(np.exp(t["values"][1:]), [.60, .30, .42, .12, .165, .336], rtol=1e-6)
    rows = [{0}, {0, 1}, {0, 2}, {0, 1, 3}, {0, 1, 4}, {0, 2, 5}, {0, 1, 3, 6}]
    mb = mask_to_bool(t["mask"], 7)
    for i, expect in enumerate(rows):
        assert set(np.nonzero(mb[i])[0].tolist()) == expect
    assert [f.tolist() for f in t["frontiers"]] == [[0, 1], [2, 4]]
    np.testing.assert_allclose(np.exp(t["cand_value"]),
                               [.6, .3, .42, .12, .165, .105, .336, .042, .07425, .0726], rtol=1e-6)
    assert not t["log"]


def test_hand_worked_tree_other_sizes():
    full = build_draft_tree(_hand_logits(), 2, 3, 11, 2)          # m = 1 + C
    assert full["selected"].tolist() == list(range(10))
    only_root = build_draft_tree(_hand_logits(), 2, 3, 1, 2)
    assert only_root["parents"].tolist() == [-1] and only_root["tokens"].tolist() == [2]
    three = build_draft_tree(_hand_logits(), 2, 3, 4, 2)          # c0, c2, c6: a chain
    assert three["parents"].tolist() == [-1, 0, 1, 2]
    assert three["tokens"].tolist() == [2, 3, 2, 1]


# ------------------------------------------------------------ special cases
def _random_rows(R, V, seed):
    rng = np.random.default_rng(seed)
    sig = rng.choice([1.0, 3.0, 6.0], size=R)
    return (rng.standard_normal((R, V)) * sig[:, None]).astype(np.float32)


def test_top_k_one_is_a_chain_of_row_argmaxes():
    D, V = 5, 300
    logits = _random_rows(D, V, 3)
    t = build_draft_tree(logits, 1, D, D + 1, 7)
    assert t["parents"].tolist() == [-1] + list(range(D))
    assert t["tokens"].tolist() == [7] + [int(np.argmax(logits[r])) for r in range(D)]


def test_depth_one_is_a_star_of_root_top_tokens():
    V, k = 500, 9
    logits = _random_rows(1, V, 4)
    t = build_draft_tree(logits, k, 1, 6, 0)
    assert t["parents"].tolist() == [-1, 0, 0, 0, 0, 0]
    order = np.argsort(-logits[0].astype(np.float64), kind="stable")
    assert t["tokens"][1:].tolist() == order[:5].tolist()


def test_identical_rows_give_slot_symmetric_tree():
    k, D, V = 3, 3, 50
    R, C = tree_sizes(k, D)
    row = _random_rows(1, V, 5)[0]
    logits = np.tile(row, (R, 1))
    t = build_draft_tree(logits, k, D, 1 + C, 0)
    # every depth-2 frontier slot sees the same row: children tokens repeat per parent
    kids = {}
    for i in range(1, t["m"]):
        kids.setdefault(int(t["parents"][i]), []).append(int(t["tokens"][i]))
    lists = [v for p, v in kids.items() if t["depth"][p] >= 1]
    assert all(lst == lists[0] for lst in lists)


def test_confident_rows_grow_deeper_trees():
    k, D, m, V = 4, 6, 24, 1000
    R, _ = tree_sizes(k, D)
    rng = np.random.default_rng(6)
    sharp = (rng.standard_normal((R, V)) * 6.0).astype(np.float32)
    flat = (rng.standard_normal((R, V)) * 1.0).astype(np.float32)
    deep = build_draft_tree(sharp, k, D, m, 0)["depth"].mean()
    wide = build_draft_tree(flat, k, D, m, 0)["depth"].mean()
    assert deep > wide


# ------------------------------------------------ brute-force invariants
def _check_invariants(t, k, D):
    m = t["m"]
    par, dep = t["parents"], t["depth"]
    val = t["cand_value"]
    C = val.size
    # parent before child, depth = parent depth + 1, pos = depth
    for i in range(1, m):
        assert 0 <= par[i] < i and dep[i] == dep[par[i]] + 1
    assert (t["pos"] == dep).all()
    # mask == reflexive transitive closure of the parent relation (Warshall)
    reach = np.eye(m, dtype=bool)
    for i in range(1, m):
        reach[i, par[i]] = True
    for via in range(m):
        reach = reach | (reach[:, [via]] & reach[[via], :])
    assert (mask_to_bool(t["mask"], m) == reach).all()
    # selection = best m-1 candidates overall (pairwise)
    sel = set(t["selected"].tolist())
    for a in sel:
        for b in range(C):
            if b not in sel:
                assert _beats(val[a], a, val[b], b)
    # ancestor closure of the selected candidate set
    for a in sel:
        pa = int(t["cand_parent"][a])
        assert pa < 0 or pa in sel
    # each frontier = best k of its depth, best first (pairwise)
    for lvl, fr in enumerate(t["frontiers"], start=1):
        level = np.nonzero(t["cand_depth"] == lvl)[0]
        fr = fr.tolist()
        for a in fr:
            for b in level:
                if b not in fr:
                    assert _beats(val[a], a, val[b], b)
        for x, y in zip(fr, fr[1:]):
            assert _beats(val[x], x, val[y], y)
    # values are sums of per-row log-probabilities along the path
    for c in range(C):
        r = int(t["cand_row"][c])
        pa = int(t["cand_parent"][c])
        base = 0.0 if pa < 0 else val[pa]
        assert val[c] <= base


@pytest.mark.parametrize("seed", range(6))
def test_tiny_workload_invariants(seed):
    w = wl.WORKLOADS["c0"]
    logits = _random_rows(w.n_rows, w.vocab, 100 + seed)
    t = build_draft_tree(logits, w.top_k, w.depth, w.total_tokens, 1)
    _check_invariants(t, w.top_k, w.depth)


def test_generated_tiny_workload_invariants():
    w = wl.WORKLOADS["c0"]
    logits = wl.draft_logits(w).numpy()
    t = build_draft_tree(logits, w.top_k, w.depth, w.total_tokens, wl.root_token(w))
    _check_invariants(t, w.top_k, w.depth)
    assert not t["log"], t["log"].summary()


def test_rows_follow_frontier_slots():
    # changing a row that no frontier slot reads must not change the tree;
    # changing the row of slot 0 at depth 1 must change its children
    k, D, V = 3, 3, 200
    R, C = tree_sizes(k, D)
    logits = _random_rows(R, V, 9)
    base = build_draft_tree(logits, k, D, 1 + C, 0)
    alt = logits.copy()
    alt[1] = _random_rows(1, V, 10)[0]
    changed = build_draft_tree(alt, k, D, 1 + C, 0)
    slot0 = int(base["frontiers"][0][0])
    kids_base = [int(base["cand_token"][c]) for c in range(C) if base["cand_parent"][c] == slot0]
    kids_alt = [int(changed["cand_token"][c]) for c in range(C) if changed["cand_parent"][c] == slot0]
    assert kids_base != kids_alt
    assert kids_alt == row_top_k(alt[1], k).tolist()
