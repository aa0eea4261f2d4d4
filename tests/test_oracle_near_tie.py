"""Pins for the oracle's near-tie bookkeeping (``oracle/near_tie.py``) and for
the places where the oracle logs its decisive comparisons.

Every GPU parity test leans on this module: a decision whose two operands
lie within 1e-6 relative may legitimately come out differently in the
library's fp32 arithmetic, so the tests compare validity instead of identity
there.  An over-flagging bug (an absolute instead of a relative margin, a
wrong scale, a decision on derived values logged as exact) would quietly turn
parity comparisons into validity checks, and an under-flagging one would make
legitimate near ties fail; the hand cases below catch both.

Source of the 1e-6 rule: the method statement of the verify step (tree,
mask, positions and accepted path bit-exact, ties to the lowest index, any
comparison within 1e-6 relative flagged and reported rather than passed).
"""

import numpy as np
import pytest

from oracle import philox
from oracle.near_tie import REL_TOL, NearTieLog, rel_margin
from oracle.tree_build import build_draft_tree
from oracle.verify import inverse_cdf, verify_tree, warped_distribution


# ------------------------------------------------------------ rel_margin
@pytest.mark.parametrize("a,b,want", [
    (1.0, 1.0 + 5e-7, 5e-7 / (1.0 + 5e-7)),
    (1.0, 1.0 + 2e-6, 2e-6 / (1.0 + 2e-6)),
    (-3.0, -3.0, 0.0),
    (0.0, 0.0, 0.0),                 # both zero: an exact tie, margin 0
    (0.0, 1e-30, 1.0),               # one zero: scale is the other operand
    (-2.0, 2.0, 2.0),                # opposite signs: |a-b| / max(|a|, |b|)
    (1000.0, 1000.0005, 0.0005 / 1000.0005),
])
def test_rel_margin_hand_values(a, b, want):
    assert rel_margin(a, b) == pytest.approx(want, rel=1e-9, abs=0)
    assert rel_margin(b, a) == rel_margin(a, b)       # symmetric


def test_rel_margin_is_relative_not_absolute():
    # an absolute rule would flag the small pair and pass the large one
    assert rel_margin(1e-3, 1e-3 + 2e-9) > REL_TOL
    assert rel_margin(1e3, 1e3 + 5e-4) < REL_TOL


# ------------------------------------------------------------ NearTieLog
def test_check_flags_inside_and_not_outside_the_tolerance():
    log = NearTieLog()
    log.check("a", "x", 1.0, 1.0 + 5e-7)           # inside: flagged
    log.check("b", "y", 1.0, 1.0 + 2e-6)           # outside: not flagged
    log.check("c", "z", 0.0, 0.0)                  # zero operands: margin 0, flagged
    log.check("d", "w", 7.5, 7.5, exact=True)      # exact decision: kept apart
    assert log.n_checked == 4
    assert [f["kind"] for f in log.flags] == ["a", "c", "d"]
    assert [f["kind"] for f in log.inexact_flags] == ["a", "c"]
    assert bool(log)
    assert "a@x" in log.summary() and "d@w" not in log.summary()


def test_exact_flags_alone_do_not_make_the_log_true():
    log = NearTieLog()
    log.check("draft_topk_cut", "row0", 2.0, 2.0, exact=True)
    assert log.flags and not log.inexact_flags and not bool(log)
    assert log.summary() == ""


def test_check_returns_the_margin():
    log = NearTieLog()
    assert log.check("k", "w", 4.0, 5.0) == pytest.approx(0.2)
    assert not log.flags


# ---------------------------------------------- decisive comparisons logged
def _kinds(log, exact=False):
    return {f["kind"] for f in (log.flags if exact else log.inexact_flags)}


def test_frontier_cut_near_tie_is_logged():
    # k 2, depth 3: the root's two children tie exactly (values equal), so the
    # depth-2 candidates are (child value) + (log-prob in rows 1 and 2).  Rows
    # 1 and 2 differ in their second logit by ~1e-7: the two best depth-2
    # candidates are within 1e-6 relative -- a frontier decision.
    V = 4
    x = np.full((5, V), -50.0)
    x[0, :2] = 0.0
    x[1, :2] = [0.0, -1.0]
    x[2, :2] = [0.0, -1.0000001]
    r = build_draft_tree(x, 2, 3, 7, 0)
    assert "frontier" in _kinds(r["log"])
    # control: a clear gap between the two rows leaves the frontier unflagged
    x[2, 1] = -1.5
    r = build_draft_tree(x, 2, 3, 7, 0)
    assert "frontier" not in _kinds(r["log"])


def test_rerank_cut_near_tie_is_logged():
    # a star (depth 1): the rerank keeps the best m-1 = 1 of k = 3 children;
    # the best two logits differ by 2.4e-7 (relative margin of the values
    # ~3e-7), the third and fourth tie exactly (an exact, raw-logit cut)
    x = np.array([[2.0, np.float32(2.0000002), -5.0, -5.0]])
    r = build_draft_tree(x, 3, 1, 2, 0)
    assert "rerank_cut" in _kinds(r["log"])
    assert "draft_topk_cut" in _kinds(r["log"], exact=True)
    assert "draft_topk_cut" not in _kinds(r["log"])
    # control: a clear winner
    x[0, 1] = 3.0
    r = build_draft_tree(x, 3, 1, 2, 0)
    assert "rerank_cut" not in _kinds(r["log"])


def _logit(p):
    return np.log(p) - np.log1p(-p)


def test_accept_test_near_tie_is_logged():
    # root with one child (token 0), V = 2: p(token 0) = sigmoid(l0 - l1) is
    # set to u * (1 + 3e-7) with u the child's uniform
    seed, step = 11, 4
    u = philox.uniform(seed, step, 0, 0)
    parents, tokens = [-1, 0], [9, 0]
    x = np.zeros((2, 2))
    x[0, 0] = _logit(u * (1 + 3e-7))
    r = verify_tree(x, parents, tokens, greedy=False, seed=seed, step=step)
    assert "accept" in _kinds(r["log"])
    x[0, 0] = _logit(min(0.999, u * 1.01))
    r = verify_tree(x, parents, tokens, greedy=False, seed=seed, step=step)
    assert "accept" not in _kinds(r["log"])


def test_top_p_cut_near_tie_is_logged():
    # p(token 0) = 0.9 (1 + 1e-9): the nucleus cut at top_p 0.9 is a near tie
    p0 = 0.9 * (1 + 1e-9)
    row = np.log(np.array([p0, (1 - p0) / 2, (1 - p0) / 2]))
    log = NearTieLog()
    warped_distribution(row, 1.0, 0, 0.9, log, "n0")
    assert "top_p_cut" in _kinds(log)
    log = NearTieLog()
    warped_distribution(np.log(np.array([0.95, 0.03, 0.02])), 1.0, 0, 0.9, log, "n0")
    assert "top_p_cut" not in _kinds(log)


def test_inverse_cdf_threshold_near_tie_is_logged():
    log = NearTieLog()
    ids, p = np.array([0, 1, 2]), np.array([0.25, 0.5, 0.25])
    inverse_cdf(ids, p, [], 0.25 * (1 + 4e-7), log, "n0")
    assert "inverse_cdf" in _kinds(log)
    log = NearTieLog()
    assert inverse_cdf(ids, p, [], 0.3, log, "n0") == 1
    assert "inverse_cdf" not in _kinds(log)


def test_residual_draw_near_tie_is_logged_through_the_walk():
    # a leaf root: the bonus is the residual draw with u = U(seed, step, 0,
    # 0xffffffff); make the first token's mass u (1 + 2e-7)
    seed, step = 5, 2
    u = philox.uniform(seed, step, 0, philox.RESIDUAL_CHILD)
    p0 = u * (1 + 2e-7)
    x = np.log(np.array([[p0, 1 - p0]]))
    r = verify_tree(x, [-1], [3], greedy=False, seed=seed, step=step)
    assert "inverse_cdf" in _kinds(r["log"])


def test_greedy_walk_logs_no_inexact_decision():
    # greedy decisions compare raw logits: exact on both sides
    rng = np.random.default_rng(0)
    x = rng.standard_normal((7, 50)).astype(np.float32)
    r = verify_tree(x, [-1, 0, 0, 1, 1, 2, 3], [2, 3, 1, 2, 0, 5, 1])
    assert not r["log"]
