"""Acceptance walk over the target logits (oracle side): greedy argmax or
recursive speculative sampling over tree children.

TEST INFRASTRUCTURE ONLY -- see the package docstring.

Sources:
* "EAGLE-2: Feature-Level Speculative Decoding Guide", "Single-Pass Tree
  Verification": the target produces logits for every node at once; a greedy
  or sampling verifier walks the tree from the root, accepting matching
  tokens until the first discrepancy; the result equals vanilla decoding.
  "True Lossless Acceleration" (production section): every emitted token is
  verified by the target model.
* "Support Eagle-3 Speculative Decoding in llama.cpp", proposal: an
  acceptance / rejection (speculative sampling) strategy for draft tokens.
  "EAGLE-2: ...", problem section: classical speculative sampling
  (Leviathan et al., Chen et al.).
* "EAGLE-2 Speculative Decoding Support for llama.cpp - Phase 1",
  "Performance Notes": mixed sampling = temperature + top_k + top_p.

Readings where the pages are silent or ambiguous:
* row i of the target logits predicts the token after node i.
* warped target distribution: logits / T; keep the top_k largest (ties ->
  lower id; top_k = 0 keeps all); softmax over the kept set; if top_p < 1 keep
  the shortest prefix (probability desc, ties -> lower id) whose cumulative
  mass reaches top_p, the crossing token included; renormalise.
* tree children are deterministic top-k picks, so the draft distribution of
  each child is one-hot on its token.  Recursive speculative sampling then
  reads: try children in node order with u_j = U(seed, step, node, j); with
  rho the mass already rejected, accept child j iff u_j * (1 - rho) < p(x_j),
  otherwise rho += p(x_j).  If none is accepted (or the node is a leaf) the
  bonus token is drawn from p restricted to the non-rejected tokens by
  inverse CDF over token ids ascending with u = U(seed, step, node, 0xffffffff):
  the first token whose cumulative mass exceeds u * (1 - rho).
* greedy: a = argmax of the row (ties -> lower id); accept the child whose
  token is a (siblings carry distinct tokens); the bonus token is a at the
  last accepted node.
"""

import numpy as np

from . import philox
from .near_tie import NearTieLog
from .tree_build import row_top_k


def children_lists(parents):
    """children[i] = child node ids of node i in node order."""
    m = len(parents)
    out = [[] for _ in range(m)]
    for i in range(1, m):
        out[int(parents[i])].append(i)
    return out


def row_argmax(row):
    """Index of the largest entry, equal values -> lower index."""
    return int(row_top_k(row, 1)[0])


def warped_distribution(row, temperature, top_k, top_p, log=None, where=""):
    """Kept token ids (ascending) and their fp64 probabilities."""
    x = np.asarray(row, dtype=np.float64)
    V = x.size
    z = x / np.float64(temperature)
    if 0 < top_k < V:
        keep = row_top_k(x, top_k)              # same order as z since T > 0
    elif top_p < 1.0:
        keep = row_top_k(x, V)
    else:
        keep = np.arange(V)
    zk = z[keep]
    p = np.exp(zk - zk.max())
    p = p / p.sum()
    if top_p < 1.0:
        # keep is ordered by probability desc, ties by lower id
        csum = np.cumsum(p)
        reach = np.nonzero(csum >= np.float64(top_p))[0]
        last = int(reach[0]) if reach.size else p.size - 1
        if log is not None:
            log.check("top_p_cut", f"{where}/pos{last}", csum[last], np.float64(top_p))
            if last > 0:
                log.check("top_p_cut", f"{where}/pos{last - 1}", csum[last - 1], np.float64(top_p))
        keep = keep[: last + 1]
        p = p[: last + 1]
        p = p / p.sum()
    order = np.argsort(keep, kind="stable")
    return keep[order], p[order]


def inverse_cdf(ids, probs, excluded, threshold, log=None, where=""):
    """First id (ascending) whose cumulative mass, excluded ids removed,
    exceeds ``threshold``; the last eligible id with mass if none does."""
    ids = np.asarray(ids)
    p = np.asarray(probs, dtype=np.float64).copy()
    if len(excluded):
        p[np.isin(ids, np.asarray(list(excluded)))] = 0.0
    csum = np.cumsum(p)
    over = np.nonzero(csum > threshold)[0]
    if over.size:
        pick = int(over[0])
    else:
        nz = np.nonzero(p > 0)[0]
        pick = int(nz[-1]) if nz.size else int(ids.size - 1)
    if log is not None:
        log.check("inverse_cdf", f"{where}/hi", csum[pick], threshold)
        if pick > 0:
            log.check("inverse_cdf", f"{where}/lo", csum[pick - 1], threshold)
    return int(ids[pick])


def verify_tree(target_logits, parents, tokens, greedy=True, temperature=1.0,
                top_k=0, top_p=1.0, seed=0, step=0, log=None):
    """Walk the tree over target logits [m, V].

    Returns dict(path = accepted node ids starting with the root,
    n_accepted = len(path) - 1, bonus = bonus token, log).
    """
    if log is None:
        log = NearTieLog()
    logits = np.asarray(target_logits)
    kids = children_lists(parents)
    node = 0
    path = [0]
    bonus = None
    while True:
        row = logits[node].astype(np.float64)
        if greedy:
            a = row_argmax(row)
            nxt = [c for c in kids[node] if int(tokens[c]) == a]
            if nxt:
                node = nxt[0]
                path.append(node)
                continue
            bonus = a
            break
        ids, p = warped_distribution(row, temperature, top_k, top_p, log, f"node{node}")
        prob_of = dict(zip(ids.tolist(), p.tolist()))
        rejected_mass = 0.0
        rejected = []
        accepted = None
        for j, c in enumerate(kids[node]):
            u = philox.uniform(seed, step, node, j)
            tok = int(tokens[c])
            p_tok = prob_of.get(tok, 0.0)
            lhs = u * (1.0 - rejected_mass)
            log.check("accept", f"node{node}/child{j}", lhs, p_tok)
            if lhs < p_tok:
                accepted = c
                break
            rejected_mass += p_tok
            rejected.append(tok)
        if accepted is not None:
            node = accepted
            path.append(node)
            continue
        u = philox.uniform(seed, step, node, philox.RESIDUAL_CHILD)
        bonus = inverse_cdf(ids, p, rejected, u * (1.0 - rejected_mass), log, f"node{node}")
        break
    return dict(path=path, n_accepted=len(path) - 1, bonus=int(bonus), log=log)
