"""Commit of the accepted path's keys and values to the target's KV cache
(oracle side).

TEST INFRASTRUCTURE ONLY -- see the package docstring.

Source: "Support Eagle-3 Speculative Decoding in llama.cpp", the reply on KV
caches: the target model keeps a KV cache of the accepted (correct) tokens
only, while the draft side also holds candidates that may be rejected.
"EAGLE-2: Feature-Level Speculative Decoding Guide", "Single-Pass Tree
Verification": the target computes keys and values for every tree token in
one pass, and the accepted tokens are a root-to-node path of the tree.

Definition written out: with the accepted path a_0 = root, a_1 .. a_n (node
ids, as the acceptance walk reports them) and the tree keys / values
tree_k, tree_v [m, Hkv, d],
    k_cache[h, prefix_len + i] = tree_k[a_i, h]   for i = 0 .. n, every h
and the same for v; every other cache row keeps its value.  Reading: the
root is a tree token (its keys and values come with the tree, not with the
prefix), so the commit appends n + 1 rows and the new prefix length is
prefix_len + n + 1; the bonus token has no keys or values yet (the next
step computes them as the root of its tree).
"""

import numpy as np


def kv_commit(k_cache, v_cache, prefix_len, tree_k, tree_v, accepted, n_accepted):
    """k/v_cache [Hkv, cap, d] (cap >= prefix_len + n_accepted + 1); tree_k/v
    [m, Hkv, d]; accepted: node ids, accepted[0] the root.  Returns updated
    copies of the two caches and the new prefix length."""
    k_out = np.array(k_cache, copy=True)
    v_out = np.array(v_cache, copy=True)
    m = np.asarray(tree_k).shape[0]
    assert 0 <= n_accepted < m and prefix_len + n_accepted + 1 <= k_out.shape[1]
    for i in range(n_accepted + 1):
        node = int(accepted[i])
        assert 0 <= node < m
        k_out[:, prefix_len + i, :] = np.asarray(tree_k)[node]
        v_out[:, prefix_len + i, :] = np.asarray(tree_v)[node]
    return k_out, v_out, prefix_len + n_accepted + 1
