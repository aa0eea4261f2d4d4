"""Draft-tree construction (oracle side): per-row log-softmax statistics,
top-k frontier expansion per depth, final top-(m-1) rerank, ancestor mask.

TEST INFRASTRUCTURE ONLY -- see the package docstring.

Sources:
* "EAGLE-2: Feature-Level Speculative Decoding Guide", "The Recurrent
  Feature Drafting Step": the draft distribution of the next token is the
  softmax of the LM-head logits, so a node's log-probability is
  logit - logsumexp(row) (draft temperature 1: the page gives a plain softmax).
  Its toy listing takes the top candidates of that softmax; the top-k of the
  softmax is the top-k of the raw logits.
* "Support Eagle-3 Speculative Decoding in llama.cpp", reply on the dynamic
  tree: node value approximates acceptance by draft confidence, the tree is
  grown per drafting step and pruned at the end of drafting.  Read as: value =
  cumulative log-probability along the path; expand the k best nodes of each
  depth; keep the best m-1 nodes overall at the end.
* "EAGLE-2: Feature-Level Speculative Decoding Guide", "Single-Pass Tree
  Verification": a token attends to its ancestors (and itself) only.

Readings where the pages are silent:
* depth D = deepest drafted level; root has depth 0; rows R = 1 + (D-1)k,
  candidates C = k + (D-1)k^2.
* row map: row 0 is the root; the j-th frontier slot at depth l (frontier
  ordered by value desc, ties -> lower candidate index) reads row
  1 + (l-1)k + j; its rank-c child is candidate base_{l+1} + j*k + c.
* m = total_tokens counts the root; nodes are the root plus the m-1 selected
  candidates sorted by candidate index; pos = depth.
* ties everywhere -> lower index.
"""

import numpy as np

from .near_tie import NearTieLog


def row_logsumexp(row):
    """log(sum(exp(row))) in fp64 with the maximum factored out."""
    x = np.asarray(row, dtype=np.float64)
    top = np.max(x)
    return float(top + np.log(np.sum(np.exp(x - top))))


def row_top_k(row, k):
    """Indices of the k largest entries, largest first, equal values by lower index."""
    x = np.asarray(row, dtype=np.float64)
    order = np.lexsort((np.arange(x.size), -x))   # primary: -x, secondary: index
    return order[:k]


def _ranked(values, indices):
    """Candidate indices sorted by (value desc, index asc)."""
    values = np.asarray(values, dtype=np.float64)
    indices = np.asarray(indices)
    return indices[np.lexsort((indices, -values))]


def tree_sizes(top_k, depth):
    """(draft rows R, candidates C) for a tree of the given top_k and depth."""
    n_rows = 1 + (depth - 1) * top_k
    n_cand = top_k + (depth - 1) * top_k * top_k
    return n_rows, n_cand


def build_draft_tree(draft_logits, top_k, depth, total_tokens, root_token, log=None):
    """Build the dynamic draft tree from draft logits of shape [R, V].

    Returns a dict with node arrays (parents, tokens, depth, pos, mask words,
    values) plus the candidate table, the frontier of each depth and the
    per-row statistics, for inspection by the tests.
    """
    if log is None:
        log = NearTieLog()
    logits = np.asarray(draft_logits)
    k, D, m = int(top_k), int(depth), int(total_tokens)
    R, C = tree_sizes(k, D)
    assert logits.ndim == 2 and logits.shape[0] >= R, "need R draft rows"
    V = logits.shape[1]
    assert 1 <= k <= V and D >= 1 and 1 <= m <= 1 + C

    # Per-row statistics: top-k token ids and their log-probabilities.
    top_ids = np.zeros((R, k), dtype=np.int64)
    top_logp = np.zeros((R, k), dtype=np.float64)
    lse = np.zeros(R, dtype=np.float64)
    for r in range(R):
        row = logits[r].astype(np.float64)
        lse[r] = row_logsumexp(row)
        ranked = row_top_k(row, min(k + 1, V))
        ids = ranked[:k]
        top_ids[r] = ids
        top_logp[r] = row[ids] - lse[r]
        if V > k:   # k-th vs (k+1)-th logit: raw fp32 values, exact on both sides
            log.check("draft_topk_cut", f"row{r}", row[ids[-1]], row[ranked[k]], exact=True)

    value = np.zeros(C, dtype=np.float64)
    token = np.zeros(C, dtype=np.int64)
    parent = np.full(C, -1, dtype=np.int64)       # -1 = the root
    cdepth = np.zeros(C, dtype=np.int64)
    crow = np.full(C, -1, dtype=np.int64)         # draft row that produced it

    # Depth 1: the root's top-k, in rank order.
    for c in range(k):
        value[c] = top_logp[0, c]
        token[c] = top_ids[0, c]
        cdepth[c] = 1
        crow[c] = 0
    frontiers = []
    level_base = 0            # first candidate index of the current depth
    frontier = _ranked(value[:k], np.arange(k))
    for lvl in range(1, D):
        # frontier: the k best candidates at depth lvl, best first
        frontiers.append(frontier.copy())
        child_base = level_base + (k if lvl == 1 else k * k)
        for j, pc in enumerate(frontier):
            r = 1 + (lvl - 1) * k + j
            for c in range(k):
                idx = child_base + j * k + c
                value[idx] = value[pc] + top_logp[r, c]
                token[idx] = top_ids[r, c]
                parent[idx] = pc
                cdepth[idx] = lvl + 1
                crow[idx] = r
        level_base = child_base
        if lvl + 1 < D:
            level = np.arange(level_base, level_base + k * k)
            ranked = _ranked(value[level], level)
            for a in range(min(k, ranked.size - 1)):      # slot order + cut
                log.check("frontier", f"depth{lvl + 1}/pos{a}",
                          value[ranked[a]], value[ranked[a + 1]])
            frontier = ranked[:k]

    # Final rerank: best m-1 candidates overall.
    ranked_all = _ranked(value, np.arange(C))
    n_sel = m - 1
    if 0 < n_sel < C:
        log.check("rerank_cut", f"pos{n_sel - 1}",
                  value[ranked_all[n_sel - 1]], value[ranked_all[n_sel]])
    selected = np.sort(ranked_all[:n_sel])
    node_of = {int(c): i + 1 for i, c in enumerate(selected)}

    parents = np.zeros(m, dtype=np.int64)
    tokens = np.zeros(m, dtype=np.int64)
    depth_arr = np.zeros(m, dtype=np.int64)
    values = np.zeros(m, dtype=np.float64)
    parents[0] = -1
    tokens[0] = int(root_token)
    for i, c in enumerate(selected, start=1):
        pc = int(parent[c])
        if pc < 0:
            parents[i] = 0
        else:
            assert pc in node_of, "selected set must be ancestor-closed"
            parents[i] = node_of[pc]
        tokens[i] = token[c]
        depth_arr[i] = cdepth[c]
        values[i] = value[c]

    mask_words = (m + 63) // 64
    mask = np.zeros((m, mask_words), dtype=np.uint64)
    for i in range(m):
        if i > 0:
            mask[i] = mask[parents[i]]
        mask[i, i // 64] |= np.uint64(1) << np.uint64(i % 64)

    return dict(
        parents=parents, tokens=tokens, depth=depth_arr, pos=depth_arr.copy(),
        mask=mask, values=values, m=m, mask_words=mask_words,
        selected=selected, cand_value=value, cand_token=token,
        cand_parent=parent, cand_depth=cdepth, cand_row=crow,
        frontiers=frontiers, top_ids=top_ids, top_logp=top_logp, lse=lse,
        log=log,
    )


def mask_to_bool(mask, m):
    """Expand uint64 mask words [m, W] to a boolean [m, m] matrix."""
    mask = np.asarray(mask, dtype=np.uint64)
    out = np.zeros((m, m), dtype=bool)
    for i in range(m):
        for j in range(m):
            out[i, j] = bool((int(mask[i, j // 64]) >> (j % 64)) & 1)
    return out
