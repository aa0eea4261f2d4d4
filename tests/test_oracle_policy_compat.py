"""The oracle's verify walk and tree attention take the trees of every shape
policy: a target that agrees with the tree along one root-to-leaf path is
accepted along exactly that path, and each node's tree attention equals
ordinary attention over the prefix plus its own ancestor chain."""

import numpy as np
import pytest

from oracle.tree_attn import tree_attention
from oracle.tree_policies import candidate_chains, confidence_tree, static_tree
from oracle.verify import verify_tree


def _policy_tree(kind, seed):
    x = np.random.default_rng(seed).standard_normal((200, 64)).astype(np.float32)
    if kind == "static":
        return static_tree(x, 3, 3, 7)
    if kind == "chains":
        return candidate_chains(x, 4, 5, 7)
    return confidence_tree(x * 0.6, 2.0, 60, 7, max_depth=7)


def _path_to(parents, node):
    path = [node]
    while parents[path[-1]] >= 0:
        path.append(int(parents[path[-1]]))
    return path[::-1]


@pytest.mark.parametrize("kind", ["static", "chains", "confidence"])
@pytest.mark.parametrize("seed", [0, 1])
def test_greedy_walk_follows_the_agreeing_path(kind, seed):
    t = _policy_tree(kind, seed)
    m, par, tok = t["m"], t["parents"], t["tokens"]
    rng = np.random.default_rng(100 + seed)
    deepest = [i for i in range(m) if t["depth"][i] == t["depth"].max()]
    leaf = int(rng.choice(deepest))
    path = _path_to(par, leaf)
    V = 64
    target = rng.standard_normal((m, V)).astype(np.float32)
    for a, b in zip(path[:-1], path[1:]):
        target[a, tok[b]] = 50.0                 # the target's argmax is the next path token
    # at the leaf, a token the leaf has no child for (it has none)
    target[leaf, 5] = 50.0
    # off the path, argmaxes that match no child: each node's row peaks at a
    # token none of its children carry
    for i in range(m):
        if i in path:
            continue
        kids = {int(tok[c]) for c in range(m) if par[c] == i}
        free = next(v for v in range(V) if v not in kids)
        target[i, free] = 50.0
    res = verify_tree(target, par, tok, greedy=True)
    assert res["path"] == path and res["n_accepted"] == len(path) - 1 and res["bonus"] == 5


@pytest.mark.parametrize("kind", ["static", "chains", "confidence"])
def test_tree_attention_is_attention_over_each_ancestor_chain(kind):
    t = _policy_tree(kind, 3)
    m = t["m"]
    rng = np.random.default_rng(7)
    hq, hkv, d, S = 4, 2, 16, 9
    q = rng.standard_normal((m, hq, d))
    kc = rng.standard_normal((hkv, S, d))
    vc = rng.standard_normal((hkv, S, d))
    tk = rng.standard_normal((m, hkv, d))
    tv = rng.standard_normal((m, hkv, d))
    out = tree_attention(q, kc, vc, tk, tv, t["mask"], S)
    for i in range(m):
        chain = _path_to(t["parents"], i)
        for h in range(hq):
            g = h // (hq // hkv)
            keys = np.concatenate([kc[g], tk[chain, g]])
            vals = np.concatenate([vc[g], tv[chain, g]])
            s = keys @ q[i, h] / np.sqrt(d)
            w = np.exp(s - s.max())
            np.testing.assert_allclose(out[i, h], (w / w.sum()) @ vals, rtol=1e-12, atol=1e-12)
