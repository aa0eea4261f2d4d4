"""GPU parity of the per-depth tree build (eagle_tree_expand, one call per
depth, then eagle_tree_finalize) against the oracle's tree build and the
one-shot eagle_tree_build on the same rows, through the C ABI: identical
tree arrays, and after every level the frontier the drafting loop needs."""

import numpy as np
import pytest
import torch

from eagle_speculative_decoding_verify_gb300 import binding as eb
from eagle_speculative_decoding_verify_gb300 import workloads as wl
from oracle.tree_build import build_draft_tree
from tests.parity import to_device_rows, tree_matches

pytestmark = pytest.mark.gpu


def _level_rows(logits, k, level):
    return logits[0:1] if level == 0 else logits[1 + (level - 1) * k: 1 + level * k]


def _grow(logits, k, D, m, root, growth=None):
    V = logits.shape[1]
    g = growth or eb.TreeGrowth(k, D, V)
    fronts = []
    for level in range(D):
        f = g.expand(to_device_rows(_level_rows(logits, k, level)), level)
        fronts.append(f.cpu().numpy().copy())
    tree = g.finalize(m, root)
    torch.cuda.synchronize()
    assert eb.workspace_error(g.ws) == (0, 0)
    return tree, fronts, g


def _check(tree, fronts, ref, k, D):
    # the same bar as the one-shot build: bit-exact structure, values within
    # 1e-5, near ties reported instead of compared
    if not tree_matches(tree, ref, "expand"):
        return
    # frontier after level L = the oracle's best k candidates of depth L + 1
    for L in range(D - 1):
        cand = ref["frontiers"][L]
        assert np.array_equal(fronts[L][0], ref["cand_token"][cand]), f"frontier tokens, level {L}"
        if L == 0:
            assert np.all(fronts[L][1] == 0)
        else:
            base = k + (L - 1) * k * k
            assert np.array_equal(fronts[L][1], (cand - base) // k), f"parent slots, level {L}"


@pytest.mark.parametrize("key", ["c0", "c1", "c2"])
def test_workloads_match_oracle_and_one_shot_build(key):
    w = wl.WORKLOADS[key]
    logits = wl.draft_logits(w)
    root = wl.root_token(w)
    ref = build_draft_tree(logits.numpy(), w.top_k, w.depth, w.total_tokens, root)
    tree, fronts, _ = _grow(logits, w.top_k, w.depth, w.total_tokens, root)
    _check(tree, fronts, ref, w.top_k, w.depth)
    one = eb.eagle_tree_build(to_device_rows(logits), w.top_k, w.depth, w.total_tokens, root)
    torch.cuda.synchronize()
    assert torch.equal(one.parents, tree.parents) and torch.equal(one.mask, tree.mask)


@pytest.mark.parametrize("V,k,D,m,seed", [
    (1000, 1, 6, 7, 1),      # top_k 1: a chain
    (777, 6, 1, 7, 2),       # depth 1: a star
    (513, 3, 4, 1 + 3 + 3 * 9, 3),     # every candidate kept
    (4099, 12, 3, 80, 4),    # ragged vocabulary
    (300, 5, 5, 2, 5),       # root and one node
])
def test_shapes(V, k, D, m, seed):
    rng = np.random.default_rng(seed)
    R = 1 + (D - 1) * k
    logits = torch.from_numpy((rng.standard_normal((R, V)) *
                               rng.choice([1.0, 3.0, 6.0], size=(R, 1))).astype(np.float32))
    ref = build_draft_tree(logits.numpy(), k, D, m, 17)
    tree, fronts, _ = _grow(logits, k, D, m, 17)
    _check(tree, fronts, ref, k, D)


def test_state_is_reused_across_rounds():
    w = wl.WORKLOADS["c1"]
    g = None
    for item in range(3):
        logits = wl.draft_logits(w, item)
        root = wl.root_token(w, item)
        ref = build_draft_tree(logits.numpy(), w.top_k, w.depth, w.total_tokens, root)
        tree, fronts, g = _grow(logits, w.top_k, w.depth, w.total_tokens, root, g)
        _check(tree, fronts, ref, w.top_k, w.depth)


def test_calls_out_of_order_are_reported():
    k, D, V = 4, 3, 500
    rows = to_device_rows(torch.randn(k, V))
    g = eb.TreeGrowth(k, D, V)
    g.expand(rows, 2)                       # level 2 before levels 0 and 1
    assert eb.workspace_error(g.ws)[0] == eb.EAGLE_ERR_DEVICE_ASSERT
    g2 = eb.TreeGrowth(k, D, V)
    g2.expand(rows[:1], 0)
    out = eb.Tree(5)
    g2.finalize(5, 0, out=out)              # finalize after one of three levels
    assert eb.workspace_error(g2.ws)[0] == eb.EAGLE_ERR_DEVICE_ASSERT
