"""Draft-tree shape policies other than the dynamic top-k tree (oracle side):
a static tree, batched candidate chains, and the confidence-ratio policy.

TEST INFRASTRUCTURE ONLY -- see the package docstring.

Sources:
* "Support Eagle-3 Speculative Decoding in llama.cpp", the reply on PR #3624:
  a static expansion of the token tree, n candidate tokens taken at every
  decoding step to form the next nodes; and the proposal to start with static
  tree sampling together with batched verification of candidate sequences.
* "EAGLE-2: Feature-Level Speculative Decoding Guide", "Context-Aware Dynamic
  Tree Construction in EAGLE-2": the confidence score C = P(y_(1)) / P(y_(2))
  of a node's draft distribution; above a threshold tau the token budget goes
  to depth (a linear chain, up to 7 deep), otherwise to breadth (2 to 4
  branches at that node); the page's listing compares the ratio with 2.0.
* "EAGLE-2: Feature-Level Speculative Decoding Guide", "The Recurrent Feature
  Drafting Step": the draft distribution is the softmax of the logits, so
  P(y_(1)) / P(y_(j)) = exp(l_(1) - l_(j)) and every ranking is by raw logit.

Readings where the pages are silent:
* Nodes are numbered breadth-first (by depth; within a depth by parent, then
  by the child's rank in its parent's row); node 0 is the root, pos = depth.
* Draft row i is node i's draft output: the rows a policy reads are those of
  the nodes it expands, in node order (the real drafting loop produces one
  row per expanded node, level by level).
* Static tree: every node above depth D gets the n best tokens of its row
  (a full n-ary tree, 1 + n + ... + n^D nodes).
* Batched chains: the root gets the n best tokens of row 0, then every chain
  is extended by the best token of its last node's row until depth D
  (1 + n D nodes).
* Confidence ratio: a node above max_depth whose row has
  l_(1) - l_(2) > ln tau gets one child (its best token); otherwise it gets
  the b best tokens, b = the number of tokens within a factor tau of the best
  (l_(1) - l_(j) <= ln tau), at least 2 by construction, at most max_branch
  (4: the page's "2 to 4").  Nodes are expanded in node order and children
  appended in rank order while the tree has fewer than m nodes; m is a cap
  and the tree can come out smaller.
* Ties everywhere -> lower token id.
"""

import math

import numpy as np

from .near_tie import NearTieLog
from .tree_build import row_top_k


def _finish(parents, tokens, depths, node_row, log):
    """Node arrays, ancestor mask words and bookkeeping of a finished tree."""
    m = len(parents)
    parents = np.asarray(parents, dtype=np.int64)
    depth = np.asarray(depths, dtype=np.int64)
    mask_words = (m + 63) // 64
    mask = np.zeros((m, mask_words), dtype=np.uint64)
    for i in range(m):
        if i > 0:
            assert 0 <= parents[i] < i, "parents precede children"
            mask[i] = mask[parents[i]]
        mask[i, i // 64] |= np.uint64(1) << np.uint64(i % 64)
    return dict(parents=parents, tokens=np.asarray(tokens, dtype=np.int64), depth=depth,
                pos=depth.copy(), mask=mask, m=m, mask_words=mask_words,
                node_row=np.asarray(node_row, dtype=np.int64),
                rows_used=int(max(node_row) + 1) if max(node_row) >= 0 else 0, log=log)


def static_tree(draft_logits, n, depth, root_token, log=None):
    """Full n-ary tree of the given depth; node i reads draft row i."""
    if log is None:
        log = NearTieLog()
    x = np.asarray(draft_logits)
    n, D = int(n), int(depth)
    V = x.shape[1]
    assert 1 <= n <= V and D >= 0
    parents, tokens, depths, node_row = [-1], [int(root_token)], [0], [-1]
    i = 0
    while i < len(parents):
        if depths[i] < D:
            node_row[i] = i
            row = x[i].astype(np.float64)
            ranked = row_top_k(row, min(n + 1, V))
            if V > n:
                log.check("static_cut", f"node{i}", row[ranked[n - 1]], row[ranked[n]],
                          exact=True)
            for t in ranked[:n]:
                parents.append(i)
                tokens.append(int(t))
                depths.append(depths[i] + 1)
                node_row.append(-1)
        i += 1
    return _finish(parents, tokens, depths, node_row, log)


def candidate_chains(draft_logits, n, depth, root_token, log=None):
    """n chains of length depth from the root's n best tokens; node i reads
    draft row i (chain j's node at depth d is node 1 + (d-1) n + j)."""
    if log is None:
        log = NearTieLog()
    x = np.asarray(draft_logits)
    n, D = int(n), int(depth)
    V = x.shape[1]
    assert 1 <= n <= V and D >= 0
    parents, tokens, depths, node_row = [-1], [int(root_token)], [0], [-1]
    if D >= 1:
        node_row[0] = 0
        row = x[0].astype(np.float64)
        ranked = row_top_k(row, min(n + 1, V))
        if V > n:
            log.check("chains_root_cut", "node0", row[ranked[n - 1]], row[ranked[n]], exact=True)
        for t in ranked[:n]:
            parents.append(0)
            tokens.append(int(t))
            depths.append(1)
            node_row.append(-1)
    for d in range(2, D + 1):
        for j in range(n):
            p = 1 + (d - 2) * n + j        # chain j's node at depth d-1
            node_row[p] = p
            row = x[p].astype(np.float64)
            ranked = row_top_k(row, min(2, V))
            if V > 1:
                log.check("chain_argmax", f"node{p}", row[ranked[0]], row[ranked[1]], exact=True)
            parents.append(p)
            tokens.append(int(ranked[0]))
            depths.append(d)
            node_row.append(-1)
    return _finish(parents, tokens, depths, node_row, log)


def confidence_tree(draft_logits, tau, total_tokens, root_token, max_depth=7, max_branch=4,
                    log=None):
    """Tree grown breadth-first by the confidence ratio of every node's row;
    at most total_tokens nodes (root included)."""
    if log is None:
        log = NearTieLog()
    x = np.asarray(draft_logits)
    m_cap, Dmax, bmax = int(total_tokens), int(max_depth), int(max_branch)
    V = x.shape[1]
    assert m_cap >= 1 and Dmax >= 0 and 2 <= bmax <= V and tau > 0
    ln_tau = math.log(tau)
    parents, tokens, depths, node_row = [-1], [int(root_token)], [0], [-1]
    i = 0
    while i < len(parents) and len(parents) < m_cap:
        if depths[i] < Dmax:
            node_row[i] = i
            row = x[i].astype(np.float64)
            ranked = row_top_k(row, min(bmax + 1, V))
            gap = row[ranked[0]] - row[ranked[1]]          # ln C, exact in fp64
            log.check("confidence", f"node{i}", gap, ln_tau)
            if gap > ln_tau:
                b = 1
            else:
                b = 2
                while b < bmax and row[ranked[0]] - row[ranked[b]] <= ln_tau:
                    b += 1
                if b < bmax:   # the count stopped at the ratio, not at the cap
                    log.check("branch_count", f"node{i}", row[ranked[0]] - row[ranked[b]], ln_tau)
            for t in ranked[:b]:
                if len(parents) >= m_cap:
                    break
                parents.append(i)
                tokens.append(int(t))
                depths.append(depths[i] + 1)
                node_row.append(-1)
        i += 1
    return _finish(parents, tokens, depths, node_row, log)


def static_tree_size(n, depth):
    """Nodes of the full n-ary tree of the given depth, root included."""
    return sum(n ** d for d in range(depth + 1))
