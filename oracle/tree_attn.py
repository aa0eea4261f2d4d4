"""Tree-masked GQA attention of the tree queries (oracle side).

TEST INFRASTRUCTURE ONLY -- see the package docstring.

Source: "EAGLE-2: Feature-Level Speculative Decoding Guide", "Single-Pass
Tree Verification": the whole draft tree goes through the target model in one
pass; a token attends to its ancestors (and, as in any causal pass, to itself
and to the committed prefix) and never to other branches.  "Support Eagle-3
Speculative Decoding in llama.cpp" (reply on the KV cache): the target keeps a
KV cache of the accepted context, which is the prefix every tree token sees.

Definition written out (fp64, plain softmax with the row maximum subtracted):
    o[i, h] = sum_j softmax_j( scale * q[i, h] . k_j ) v_j
over j in the prefix keys of kv head h // g plus the tree keys j allowed by
mask row i.  Reading: scale = 1/sqrt(d) (the pages do not give one).
Inputs are whatever values the caller hands in (the tests pass the same
bf16-rounded values the GPU reads, widened to fp64).
"""

import numpy as np


def mask_bits(mask, m):
    """uint64 mask words [m, W] -> bool [m, m], bit j of row i = tree key j visible."""
    mask = np.asarray(mask, dtype=np.uint64)
    j = np.arange(m)
    words = mask[:, j // 64]
    return ((words >> (j % 64).astype(np.uint64)) & np.uint64(1)).astype(bool)


def tree_attention(q, k_cache, v_cache, tree_k, tree_v, mask, prefix_len,
                   scale=None, heads=None):
    """q [m, Hq, d]; k/v_cache [Hkv, >=prefix_len, d]; tree_k/v [m, Hkv, d];
    mask uint64 [m, W].  Returns fp64 [m, Hq, d] (rows of heads not listed in
    ``heads`` are left zero)."""
    q = np.asarray(q, dtype=np.float64)
    m, n_q_heads, d = q.shape
    n_kv_heads = k_cache.shape[0]
    assert n_q_heads % n_kv_heads == 0
    group = n_q_heads // n_kv_heads
    if scale is None or scale == 0.0:
        scale = 1.0 / np.sqrt(d)
    visible_tree = mask_bits(mask, m)
    visible = np.concatenate([np.ones((m, prefix_len), dtype=bool), visible_tree], axis=1)
    out = np.zeros((m, n_q_heads, d), dtype=np.float64)
    for h in (range(n_q_heads) if heads is None else heads):
        kvh = h // group
        keys = np.concatenate([np.asarray(k_cache[kvh, :prefix_len], dtype=np.float64),
                               np.asarray(tree_k[:, kvh], dtype=np.float64)], axis=0)
        vals = np.concatenate([np.asarray(v_cache[kvh, :prefix_len], dtype=np.float64),
                               np.asarray(tree_v[:, kvh], dtype=np.float64)], axis=0)
        scores = (q[:, h] @ keys.T) * scale
        scores = np.where(visible, scores, -np.inf)
        scores = scores - scores.max(axis=1, keepdims=True)
        weights = np.exp(scores)
        weights = weights / weights.sum(axis=1, keepdims=True)
        out[:, h] = weights @ vals
    return out


def tree_attention_rows(q, k_cache, v_cache, tree_k, tree_v, mask, prefix_len,
                        rows, scale=None):
    """Same definition for a list of (query i, head h) pairs only; returns
    fp64 [len(rows), d].  Used for sampled checks at full size."""
    q = np.asarray(q)
    m, n_q_heads, d = q.shape
    n_kv_heads = k_cache.shape[0]
    group = n_q_heads // n_kv_heads
    if scale is None or scale == 0.0:
        scale = 1.0 / np.sqrt(d)
    visible_tree = mask_bits(mask, m)
    out = np.zeros((len(rows), d), dtype=np.float64)
    for n, (i, h) in enumerate(rows):
        kvh = h // group
        tree_sel = np.nonzero(visible_tree[i])[0]
        keys = np.concatenate([np.asarray(k_cache[kvh, :prefix_len], dtype=np.float64),
                               np.asarray(tree_k[tree_sel, kvh], dtype=np.float64)], axis=0)
        vals = np.concatenate([np.asarray(v_cache[kvh, :prefix_len], dtype=np.float64),
                               np.asarray(tree_v[tree_sel, kvh], dtype=np.float64)], axis=0)
        s = (keys @ np.asarray(q[i, h], dtype=np.float64)) * scale
        s = s - s.max()
        w = np.exp(s)
        out[n] = (w / w.sum()) @ vals
    return out


def gather_pages(pool, block_table, prefix_len, page=128):
    """A paged KV cache back to the contiguous layout: pool [Hkv, rows, d],
    page j of the sequence (prefix tokens page*j .. page*j + page - 1) at pool
    rows block_table[j]*page .. +page.  Returns [Hkv, prefix_len, d].

    Source: "EAGLE-2: Feature-Level Speculative Decoding Guide", production
    section (serving engines keep the KV cache in a shared pool for high
    concurrency).  Reading: fixed pages of `page` tokens, one block table of
    page ids per sequence (the pages give no layout)."""
    pool = np.asarray(pool)
    n_pages = (prefix_len + page - 1) // page
    parts = [pool[:, int(block_table[j]) * page: int(block_table[j]) * page + page]
             for j in range(n_pages)]
    if not parts:
        return pool[:, :0]
    return np.concatenate(parts, axis=1)[:, :prefix_len]


def tree_attention_paged(q, k_pool, v_pool, block_table, tree_k, tree_v, mask, prefix_len,
                         scale=None, heads=None, page=128):
    """tree_attention over a paged prefix cache (gather, then the definition)."""
    return tree_attention(q, gather_pages(k_pool, block_table, prefix_len, page),
                          gather_pages(v_pool, block_table, prefix_len, page),
                          tree_k, tree_v, mask, prefix_len, scale=scale, heads=heads)
