"""Pins for the oracle's KV commit.

Checked against: a hand-worked example (which rows move where, and that no
other row changes); and the property the commit exists for -- after it, plain
causal attention of the last accepted node over the new prefix (PyTorch's
scaled_dot_product_attention in fp64, a library routine) equals attention of
that node over the old prefix plus its ancestor chain, the chain found by
walking parent pointers from the node (not from the accepted list).
"""

import numpy as np
import torch

from oracle.kv_commit import kv_commit
from oracle.tree_build import build_draft_tree


def test_hand_worked_example():
    Hkv, cap, d, m, S = 2, 10, 3, 6, 4
    k_cache = np.full((Hkv, cap, d), -1.0)
    v_cache = np.full((Hkv, cap, d), -2.0)
    # tree row t of head h holds 100 t + 10 h (keys) / its negation (values)
    tree_k = np.array([[[100.0 * t + 10 * h] * d for h in range(Hkv)] for t in range(m)])
    tree_v = -tree_k
    k, v, new_len = kv_commit(k_cache, v_cache, S, tree_k, tree_v, [0, 2, 5, 4], 2)
    assert new_len == 7
    for h in range(Hkv):
        assert k[h, :S].tolist() == [[-1.0] * d] * S             # prefix untouched
        assert [r[0] for r in k[h, S:S + 3]] == [10 * h, 200 + 10 * h, 500 + 10 * h]
        assert [r[0] for r in v[h, S:S + 3]] == [-10 * h, -200 - 10 * h, -500 - 10 * h]
        assert k[h, S + 3:].tolist() == [[-1.0] * d] * (cap - S - 3)   # accepted[3] not used
        assert v[h, S + 3:].tolist() == [[-2.0] * d] * (cap - S - 3)


def test_root_only():
    k, v, new_len = kv_commit(np.zeros((1, 3, 2)), np.zeros((1, 3, 2)), 0,
                              np.arange(8.0).reshape(4, 1, 2), -np.arange(8.0).reshape(4, 1, 2),
                              [0], 0)
    assert new_len == 1 and k[0, 0].tolist() == [0.0, 1.0] and k[0, 1:].sum() == 0.0


def test_committed_cache_is_the_accepted_nodes_context():
    rng = np.random.default_rng(5)
    k, D, m, V = 3, 4, 14, 40
    R = 1 + (D - 1) * k
    t = build_draft_tree((rng.standard_normal((R, V)) * 3).astype(np.float32), k, D, m, 0)
    parents = t["parents"]
    Hkv, d, S = 2, 8, 9
    cap = S + m
    g = torch.Generator().manual_seed(11)
    r = lambda *s: torch.randn(*s, generator=g, dtype=torch.float64)
    k_cache, v_cache, tree_k, tree_v = r(Hkv, cap, d), r(Hkv, cap, d), r(m, Hkv, d), r(m, Hkv, d)
    q = r(d)
    for last in range(m):
        chain = []
        node = last
        while node >= 0:
            chain.append(node)
            node = int(parents[node])
        chain = chain[::-1]                       # root first
        kk, vv, new_len = kv_commit(k_cache.numpy(), v_cache.numpy(), S, tree_k.numpy(),
                                    tree_v.numpy(), chain, len(chain) - 1)
        assert new_len == S + len(chain)
        for h in range(Hkv):
            keys_new = torch.from_numpy(kk[h, :new_len])
            vals_new = torch.from_numpy(vv[h, :new_len])
            keys_ref = torch.cat([k_cache[h, :S], tree_k[chain, h]])
            vals_ref = torch.cat([v_cache[h, :S], tree_v[chain, h]])
            sdpa = lambda K_, V_: torch.nn.functional.scaled_dot_product_attention(
                q[None, None, None], K_[None, None], V_[None, None])[0, 0, 0]
            assert torch.allclose(sdpa(keys_new, vals_new), sdpa(keys_ref, vals_ref),
                                  rtol=0, atol=1e-12)
