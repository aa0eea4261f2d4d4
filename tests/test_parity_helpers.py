"""CPU checks of the parity helpers the GPU tests rely on (tests/parity.py):
the validity checks accept every oracle tree and walk, and reject planted
mistakes (a wrong parent, depth, position or mask bit, a duplicated sibling
token, a path that jumps branches, a bonus outside the kept set); the
near-tie branches still compare what is unique."""

import numpy as np
import pytest
import torch

from oracle.near_tie import NearTieLog
from oracle.tree_build import build_draft_tree
from oracle.verify import verify_tree
from tests import parity


class _FakeTree:
    """The attributes of binding.Tree that the helpers read, on the CPU."""

    def __init__(self, ref, **override):
        a = {k: np.array(ref[k]).copy() for k in ("parents", "tokens", "depth", "pos", "mask",
                                                   "values")}
        a.update(override)
        self.m = ref["m"]
        self.parents = torch.from_numpy(a["parents"].astype(np.int32))
        self.tokens = torch.from_numpy(a["tokens"].astype(np.int32))
        self.depth = torch.from_numpy(a["depth"].astype(np.int32))
        self.pos = torch.from_numpy(a["pos"].astype(np.int32))
        self.values = torch.from_numpy(a["values"].astype(np.float64))
        self._mask = a["mask"].astype(np.uint64)

    def mask_u64(self):
        return self._mask


def _ref(seed=0, k=3, D=4, m=20, V=200):
    rng = np.random.default_rng(seed)
    R = 1 + (D - 1) * k
    x = (rng.standard_normal((R, V)) * rng.choice([1.0, 3.0, 6.0], size=(R, 1))).astype(
        np.float32)
    return build_draft_tree(x, k, D, m, 5)


def test_oracle_trees_pass():
    for seed in range(6):
        ref = _ref(seed)
        assert parity.tree_matches(_FakeTree(ref), ref)


def test_ancestor_closure_by_hand():
    par = [-1, 0, 0, 1, 3]
    want = np.array([[1, 0, 0, 0, 0],
                     [1, 1, 0, 0, 0],
                     [1, 0, 1, 0, 0],
                     [1, 1, 0, 1, 0],
                     [1, 1, 0, 1, 1]], dtype=bool)
    np.testing.assert_array_equal(parity.ancestor_closure(par), want)


@pytest.mark.parametrize("plant", ["parent", "depth", "pos", "mask", "sibling", "value"])
def test_planted_tree_mistakes_fail_validity(plant):
    ref = _ref(1)
    par, tok = ref["parents"].copy(), ref["tokens"].copy()
    dep, pos, mask, val = ref["depth"].copy(), ref["pos"].copy(), ref["mask"].copy(), \
        ref["values"].copy()
    i = ref["m"] - 1
    if plant == "parent":
        par[i] = i          # not before the node
    elif plant == "depth":
        dep[i] += 1
        pos[i] += 1
    elif plant == "pos":
        pos[i] += 1
    elif plant == "mask":
        mask[i, 0] ^= np.uint64(1) << np.uint64(i - 1 if par[i] != i - 1 else i - 2)
    elif plant == "sibling":
        pairs = [(a, b) for a in range(1, ref["m"]) for b in range(a + 1, ref["m"])
                 if par[a] == par[b]]
        a, b = pairs[-1]
        tok[b] = tok[a]
    elif plant == "value":
        val[i] = val[par[i]] + 1.0
    fake = _FakeTree(ref, parents=par, tokens=tok, depth=dep, pos=pos, mask=mask, values=val)
    with pytest.raises(AssertionError):
        parity.check_tree_valid(fake.parents.numpy(), fake.tokens.numpy(), fake.depth.numpy(),
                                fake.pos.numpy(), fake.mask_u64(), int(ref["tokens"][0]), "t",
                                fake.values.numpy())


def test_rerank_near_tie_compares_selected_values():
    # a star: the best two children are a near tie at the cut (m - 1 = 1)
    x = np.array([[2.0, np.float32(2.0000002), -5.0, -5.0]])
    ref = build_draft_tree(x, 3, 1, 2, 0)
    assert ref["log"]
    # the other side of the tie is a valid answer
    other = int(np.argsort(-x[0], kind="stable")[1])
    alt = _FakeTree(ref, tokens=np.array([0, other]),
                    values=np.array([0.0, ref["cand_value"][1 - ref["selected"][0]]]))
    with pytest.warns(UserWarning):
        assert not parity.tree_matches(alt, ref)
    # a clearly worse child is not
    bad = _FakeTree(ref, tokens=np.array([0, 2]), values=np.array([0.0, ref["cand_value"][2]]))
    with pytest.warns(UserWarning), pytest.raises(AssertionError):
        parity.tree_matches(bad, ref)


# ------------------------------------------------------------------- paths
PARENTS = [-1, 0, 0, 1, 1, 2, 3]
TOKENS = [2, 3, 1, 2, 0, 5, 1]


def _walk_case(seed):
    rng = np.random.default_rng(seed)
    x = (rng.standard_normal((7, 6)) * 0.5).astype(np.float32)
    params = (0, 1.0, 0, 1.0)
    v = verify_tree(x, PARENTS, TOKENS, greedy=False, seed=seed, step=1)
    return x, v, params


def test_oracle_walks_pass():
    for seed in range(20):
        x, v, params = _walk_case(seed)
        acc = np.array(v["path"] + [-1] * (7 - len(v["path"])))
        assert parity.path_matches(acc, v["n_accepted"], v["bonus"], v, "w", PARENTS, TOKENS, x,
                                   params)


def test_path_that_jumps_branches_fails():
    x, v, params = _walk_case(0)
    with pytest.raises(AssertionError):
        parity.check_path_valid([0, 1, 5], 0, PARENTS, TOKENS, "w", x, params)


def test_bonus_equal_to_a_rejected_child_token_fails():
    x, v, params = _walk_case(0)
    with pytest.raises(AssertionError):   # node 2's only child carries token 5
        parity.check_path_valid([0, 2], 5, PARENTS, TOKENS, "w", x, params)


def test_greedy_bonus_must_be_the_argmax():
    x = np.zeros((7, 6), dtype=np.float32)
    x[0, 4] = 9.0                          # argmax 4: no child of the root
    parity.check_path_valid([0], 4, PARENTS, TOKENS, "w", x, (1, 1.0, 0, 1.0))
    with pytest.raises(AssertionError):
        parity.check_path_valid([0], 0, PARENTS, TOKENS, "w", x, (1, 1.0, 0, 1.0))


def test_bonus_outside_the_top_k_fails():
    x = np.zeros((7, 6), dtype=np.float32)
    x[0] = [0.0, 5.0, 0.0, 6.0, 0.0, 0.0]
    # top_k 2 keeps tokens 3 and 1, both children of the root: any bonus at
    # the root is outside what it may be
    with pytest.raises(AssertionError):
        parity.check_path_valid([0], 4, PARENTS, TOKENS, "w", x, (0, 1.0, 2, 1.0))


def test_near_tie_walk_must_agree_up_to_the_flagged_node():
    ref = dict(path=[0, 1, 3], bonus=4, log=NearTieLog())
    ref["log"].check("accept", "node1/child0", 0.5, 0.5 + 1e-8)
    acc_ok = np.array([0, 1, 4, -1, -1, -1, -1])        # departs after node 1: allowed
    with pytest.warns(UserWarning):
        assert not parity.path_matches(acc_ok, 2, 1, ref, "w", PARENTS, TOKENS)
    acc_bad = np.array([0, 2, 5, -1, -1, -1, -1])       # departs at the root: not allowed
    with pytest.warns(UserWarning), pytest.raises(AssertionError):
        parity.path_matches(acc_bad, 2, 0, ref, "w", PARENTS, TOKENS)
