"""Helpers shared by the GPU parity tests: compare library outputs with the
oracle, with near ties (decisions within 1e-6 relative, recorded by the
oracle) reported instead of silently passed.

Every comparison first checks that the library's output is valid on its own
(a well-formed tree with the ancestor-closure mask, a root-to-node path with
an admissible bonus token).  Then, without a near tie, it must equal the
oracle's output exactly; with one, the parts that are still unique are
compared (the path up to the first flagged node; the selected node values
when only the final cut was a near tie)."""

import re
import warnings

import numpy as np

ATTN_TOL = 2e-3     # max abs error of attention outputs (fp32 out, bf16/fp32 inputs)


def peaked_tol(values):
    """Error bound of the tensor-core attention when a few keys dominate a
    row: the softmax weights enter the P V product as bf16, each within 2^-9
    (relative) of its fp32 value, and the row sum uses the same rounded
    weights, so the output moves by at most 2^-8 * max |v| (the weights'
    errors sum to at most 2 * 2^-9 after normalisation).  For the workloads'
    N(0, 1) inputs no key dominates and the 2e-3 bar applies."""
    import numpy as np
    return max(ATTN_TOL, 2.0 ** -8 * float(np.abs(np.asarray(values, dtype=np.float64)).max()))
VALUE_TOL = 1e-5    # node values: fp32-derived on the GPU, fp64 in the oracle


def report_near_ties(log, what):
    if log:
        warnings.warn(f"{what}: near ties within 1e-6 relative: {log.summary()}")
        return True
    return False


# ------------------------------------------------------------------ trees
def ancestor_closure(parents):
    """bool [m, m]: row i has node i and every ancestor of i (Warshall's
    transitive closure of the parent relation, plus the diagonal)."""
    m = len(parents)
    reach = np.zeros((m, m), dtype=bool)
    for i in range(1, m):
        reach[i, int(parents[i])] = True
    for k in range(m):
        reach |= reach[:, k:k + 1] & reach[k:k + 1, :]
    reach |= np.eye(m, dtype=bool)
    return reach


def mask_words_to_bool(mask, m):
    mask = np.asarray(mask, dtype=np.uint64).reshape(m, -1)
    j = np.arange(m)
    return ((mask[:, j // 64] >> (j % 64).astype(np.uint64)) & np.uint64(1)).astype(bool)


def check_tree_valid(par, tok, dep, pos, mask, root_token, what, values=None, n_nodes=None):
    """A well-formed draft tree: root first, parents before children, depth =
    parent depth + 1 = position id, distinct tokens among siblings, mask =
    the ancestor closure of its own parents, values never increasing along a
    path.  Only the first n_nodes slots are checked (default: all)."""
    dep_all = np.asarray(dep)
    m = len(par) if n_nodes is None else int(n_nodes)
    par, tok, dep, pos = (np.asarray(a)[:m] for a in (par, tok, dep, pos))
    assert par[0] == -1 and dep[0] == 0 and tok[0] == root_token, f"{what}: root"
    for i in range(1, m):
        assert 0 <= par[i] < i, f"{what}: parent of node {i} is {par[i]}"
        assert dep[i] == dep[par[i]] + 1, f"{what}: depth of node {i}"
    np.testing.assert_array_equal(pos, dep, err_msg=f"{what}: pos != depth")
    seen = set()
    for i in range(1, m):
        key = (int(par[i]), int(tok[i]))
        assert key not in seen, f"{what}: siblings share token {key[1]}"
        seen.add(key)
    words = np.asarray(mask, dtype=np.uint64).reshape(len(np.asarray(dep_all)), -1)[:m]
    got = mask_words_to_bool(words, m)
    np.testing.assert_array_equal(got, ancestor_closure(par), err_msg=f"{what}: mask")
    if values is not None:
        v = np.asarray(values)[:m]
        assert v[0] == 0.0, f"{what}: root value"
        for i in range(1, m):
            assert v[i] <= v[par[i]] + VALUE_TOL, f"{what}: value grows at node {i}"


def _candidate_of(par, tok, ref):
    """Oracle candidate index of every library node (root -1), matched by
    (parent's candidate, token); None when some node is no oracle candidate."""
    key = {(int(p), int(t)): c for c, (p, t) in
           enumerate(zip(ref["cand_parent"], ref["cand_token"]))}
    cand = [-1] * len(par)
    for i in range(1, len(par)):
        c = key.get((cand[int(par[i])], int(tok[i])))
        if c is None:
            return None
        cand[i] = c
    return cand


def tree_matches(gpu, ref, what="tree"):
    """Compare a library Tree with an oracle tree.  Returns True when it was
    compared bit-exactly, False when a near tie limited the comparison."""
    m = ref["m"]
    par = gpu.parents.cpu().numpy()
    tok = gpu.tokens.cpu().numpy()
    dep = gpu.depth.cpu().numpy()
    pos = gpu.pos.cpu().numpy()
    mask = gpu.mask_u64()
    vals = gpu.values.cpu().numpy() if gpu.values is not None else None
    check_tree_valid(par, tok, dep, pos, mask, int(ref["tokens"][0]), what, vals)
    if report_near_ties(ref["log"], what):
        kinds = {f["kind"] for f in ref["log"].inexact_flags}
        if kinds <= {"rerank_cut"}:
            # the candidate table is the oracle's: every node is one of its
            # candidates, and the selected values are the best m-1 (unique
            # as a sorted list even when the cut's identity is not)
            cand = _candidate_of(par, tok, ref)
            assert cand is not None, f"{what}: a node is no candidate of the oracle's table"
            got = np.sort(ref["cand_value"][cand[1:]])
            want = np.sort(ref["values"][1:])
            np.testing.assert_allclose(got, want, rtol=0, atol=VALUE_TOL,
                                       err_msg=f"{what}: selected values")
            if vals is not None:
                np.testing.assert_allclose(vals[1:], ref["cand_value"][cand[1:]], rtol=0,
                                           atol=VALUE_TOL, err_msg=f"{what}: values")
        return False
    np.testing.assert_array_equal(par, ref["parents"], err_msg=f"{what} parents")
    np.testing.assert_array_equal(tok, ref["tokens"], err_msg=f"{what} tokens")
    np.testing.assert_array_equal(dep, ref["depth"], err_msg=f"{what} depth")
    np.testing.assert_array_equal(pos, ref["pos"], err_msg=f"{what} pos")
    np.testing.assert_array_equal(mask, ref["mask"], err_msg=f"{what} mask")
    if vals is not None:
        np.testing.assert_allclose(vals, ref["values"], rtol=0, atol=VALUE_TOL,
                                   err_msg=f"{what} values")
    return True


# ------------------------------------------------------------------- paths
def kept_tokens(row, params):
    """Tokens the bonus may be drawn from at a node: the argmax (greedy) or
    the support of the warped target distribution (sampling)."""
    from oracle.verify import row_argmax, warped_distribution
    greedy, T, k, p = params
    row = np.asarray(row, dtype=np.float64)
    if greedy:
        return {row_argmax(row)}
    ids, probs = warped_distribution(row, T, k, p)
    return {int(i) for i, q in zip(ids, probs) if q > 0.0}


def check_path_valid(path, bonus, parents, tokens, what, target=None, params=None):
    """path[0] is the root and every next node is a child of the previous
    one; the walk stopped at its last node, so every child of that node was
    rejected (sampling: the bonus is none of their tokens; greedy: none of
    them carries the bonus token) and the bonus lies in the node's kept set."""
    assert len(path) >= 1 and path[0] == 0, f"{what}: path does not start at the root"
    for a, b in zip(path, path[1:]):
        assert 0 < b < len(parents) and int(parents[b]) == a, f"{what}: {b} is no child of {a}"
    last = path[-1]
    kids_tokens = {int(tokens[c]) for c in range(1, len(parents)) if int(parents[c]) == last}
    assert int(bonus) not in kids_tokens, f"{what}: bonus {bonus} is a child token of node {last}"
    if target is not None and params is not None:
        row = np.asarray(target[last])
        assert int(bonus) in kept_tokens(row, params), \
            f"{what}: bonus {bonus} outside the kept set of node {last}"


def _flagged_nodes(log):
    out = set()
    for f in log.inexact_flags:
        mm = re.match(r"node(\d+)", f["where"])
        if mm:
            out.add(int(mm.group(1)))
    return out


def path_matches(acc, n_acc, bonus, ref, what="verify", parents=None, tokens=None,
                 target=None, params=None):
    """Compare a library walk with the oracle's.  parents / tokens (the tree
    walked), target (its logits [m, V]) and params ((greedy, T, top_k,
    top_p)) enable the validity checks, which run before any comparison."""
    n = int(n_acc)
    got_path = [int(x) for x in acc[: n + 1]]
    if parents is not None:
        check_path_valid(got_path, bonus, parents, tokens, what, target, params)
    if report_near_ties(ref["log"], what):
        # identical up to and including the first node whose decision was a
        # near tie (the walk visits nodes in path order)
        flagged = _flagged_nodes(ref["log"])
        ref_path = ref["path"]
        first = next((i for i, node in enumerate(ref_path) if node in flagged), len(ref_path) - 1)
        assert got_path[: first + 1] == ref_path[: first + 1], \
            f"{what}: path {got_path} departs from {ref_path} before the near tie"
        return False
    assert got_path == ref["path"], f"{what}: path {got_path} != {ref['path']}"
    assert int(bonus) == ref["bonus"], f"{what}: bonus {int(bonus)} != {ref['bonus']}"
    return True


# ------------------------------------------------------------------ inputs
# Pad value past the vocabulary in padded rows: large and positive, so that
# any read of a pad element into a maximum, a top-k list or a sum changes the
# result and fails the comparison.
PAD = 3.0e38


def to_device_rows(x, stride=None):
    """Copy fp32 rows [R, V] to the GPU with a row stride that is a multiple of
    4 elements (the library's alignment rule); returns the [R, V] view.  The
    elements past V are PAD."""
    import torch
    R, V = x.shape
    stride = stride or (V + 3) // 4 * 4
    full = torch.full((R, stride), PAD, dtype=torch.float32, device="cuda")
    full[:, :V] = x.to("cuda")
    return full[:, :V]


# worst attention error seen per workload in this session (printed at the end)
ATTN_ERRORS = {}


def record_attn_error(what, err):
    ATTN_ERRORS[what] = max(float(err), ATTN_ERRORS.get(what, 0.0))


def max_abs(a, b):
    return float(np.abs(np.asarray(a, dtype=np.float64) - np.asarray(b, dtype=np.float64)).max())
