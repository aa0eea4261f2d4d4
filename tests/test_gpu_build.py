"""GPU parity of eagle_tree_build against the oracle (bit-exact tree, mask,
positions; node values within 1e-5), through the C ABI."""

import numpy as np
import pytest
import torch

from eagle_speculative_decoding_verify_gb300 import binding as eb
from eagle_speculative_decoding_verify_gb300 import workloads as wl
from oracle.tree_build import build_draft_tree, tree_sizes
from tests.parity import PAD, to_device_rows, tree_matches

pytestmark = pytest.mark.gpu


def _rows(R, V, seed, stride=None):
    g = torch.Generator().manual_seed(seed)
    sig = torch.tensor([1.0, 3.0, 6.0])[torch.randint(0, 3, (R,), generator=g)]
    x = torch.randn(R, V, generator=g) * sig[:, None]
    if stride is not None and stride > V:
        big = torch.full((R, stride), PAD)
        big[:, :V] = x
        return big[:, :V]
    return x


def _run(x, k, D, m, root=3):
    """Copy x to the GPU (row stride rounded up to 4 elements, or x's own
    stride when it is a slice of a wider buffer) and build the tree there."""
    xd = to_device_rows(x, x.stride(0) if not x.is_contiguous() else None)
    t = eb.eagle_tree_build(xd, k, D, m, root)
    torch.cuda.synchronize()
    return t


@pytest.mark.parametrize("key", ["c0", "c1", "c2", "c3"])
def test_workload_trees(key):
    w = wl.WORKLOADS[key]
    x = wl.draft_logits(w)
    root = wl.root_token(w)
    ref = build_draft_tree(x.numpy(), w.top_k, w.depth, w.total_tokens, root)
    t = _run(x, w.top_k, w.depth, w.total_tokens, root)
    tree_matches(t, ref, key)


@pytest.mark.parametrize("V,k,D,m,seed", [
    (5003, 4, 3, 16, 1),       # ragged vocab (not a multiple of 4 or 1024)
    (1024, 5, 4, 40, 2),       # one tile per row
    (777, 3, 5, 30, 3),        # vocab below one tile
    (20000, 1, 6, 7, 4),       # top_k 1: a chain
    (3000, 9, 1, 10, 5),       # depth 1: a star
    (2048, 3, 3, 22, 6),       # m = 1 + C: every candidate kept
    (4096, 7, 3, 1, 7),        # root only
    (70001, 64, 1, 65, 8),     # maximum top_k
    (9000, 2, 16, 31, 9),      # maximum depth
    (130000, 10, 6, 256, 10),  # maximum tree
])
def test_shapes(V, k, D, m, seed):
    R, C = tree_sizes(k, D)
    x = _rows(R, V, seed)
    ref = build_draft_tree(x.numpy(), k, D, m, 11)
    t = _run(x, k, D, m, 11)
    tree_matches(t, ref, f"V{V} k{k} D{D} m{m}")


def test_padded_row_stride():
    k, D, m, V = 4, 3, 12, 3001
    R, _ = tree_sizes(k, D)
    x = _rows(R, V, 21, stride=3004)
    ref = build_draft_tree(x.contiguous().numpy(), k, D, m, 0)
    t = _run(x, k, D, m, 0)
    tree_matches(t, ref, "padded stride")


def test_ties_go_to_lower_ids():
    # constant rows: every candidate ties; the lowest token ids / candidate
    # indices must win everywhere
    k, D, m, V = 3, 3, 10, 2500
    R, _ = tree_sizes(k, D)
    x = torch.zeros(R, V)
    ref = build_draft_tree(x.numpy(), k, D, m, 0)
    t = _run(x, k, D, m, 0)
    np.testing.assert_array_equal(t.parents.cpu().numpy(), ref["parents"])
    np.testing.assert_array_equal(t.tokens.cpu().numpy(), ref["tokens"])
    np.testing.assert_array_equal(t.mask_u64(), ref["mask"])


def test_batched_ragged16_drafts():
    w = wl.WORKLOADS["c4"]
    xs = [wl.draft_logits(w, item=b) for b in range(w.items)]
    roots = [wl.root_token(w, b) for b in range(w.items)]
    dev = torch.device("cuda")
    trees = eb.eagle_tree_build_batched([x.to(dev) for x in xs], w.top_k, w.depth,
                                        w.total_tokens, roots)
    torch.cuda.synchronize()
    for b in range(w.items):
        ref = build_draft_tree(xs[b].numpy(), w.top_k, w.depth, w.total_tokens, roots[b])
        tree_matches(trees[b], ref, f"item{b}")


def test_repeated_calls_reuse_workspace():
    w = wl.WORKLOADS["c1"]
    x = wl.draft_logits(w).cuda()
    root = wl.root_token(w)
    ws = eb.workspace(eb.eagle_tree_build_workspace_size(1, w.n_rows, w.vocab, w.top_k, w.depth,
                                                         w.total_tokens))
    t1 = eb.eagle_tree_build(x, w.top_k, w.depth, w.total_tokens, root, ws=ws)
    p1 = t1.parents.clone()
    m1 = t1.mask.clone()
    for _ in range(3):
        t2 = eb.eagle_tree_build(x, w.top_k, w.depth, w.total_tokens, root, ws=ws)
    torch.cuda.synchronize()
    assert torch.equal(p1, t2.parents) and torch.equal(m1, t2.mask)
    assert eb.workspace_error(ws) == (0, 0)


def _adversarial(kind, R, V, k, seed):
    """Rows that stress the two-pass top-K bound of the row stream."""
    g = torch.Generator().manual_seed(seed)
    x = torch.randn(R, V, generator=g)
    if kind == "one_lane":
        # every row's best k in the 16 elements one thread reads from its
        # first slot (positions q * 1024 + c): a single lane holds them all
        pos = [q * 1024 + c for q in range(4) for c in range(4)][:k]
        x[:, pos] = 100.0 + torch.rand(R, len(pos), generator=g)
    elif kind == "duplicates":
        # 100 copies of each row's maximum at random places: lowest ids win
        for r in range(R):
            idx = torch.randperm(V, generator=g)[:100]
            x[r, idx] = 50.0
    elif kind == "tail":
        # the best k in the last elements of a row whose length is no
        # multiple of 4 (read element-wise by the stream)
        x[:, V - k:] = 100.0 + torch.rand(R, k, generator=g)
    elif kind == "slots":
        # one element of every 4096-element slot (16 KB of a row) raised to
        # 5 + U(0, 1): the thread that reads that place of each slot has
        # every slot at or above the second pass's bound, more than the five
        # candidate slots a thread records, so its warp revisits every
        # qualifying slot of its CTA's share
        pos = torch.arange(0, V, 4096)
        x[:, pos] = 5.0 + torch.rand(R, len(pos), generator=g)
    elif kind == "negative":
        x = x - 1000.0
    return x


@pytest.mark.parametrize("kind,V,k,D,m", [
    ("one_lane", 40000, 10, 3, 40),
    ("one_lane", 152064, 16, 2, 60),
    ("duplicates", 30000, 10, 3, 40),
    ("duplicates", 152064, 50, 1, 51),
    ("tail", 5003, 10, 3, 40),
    ("tail", 152063, 64, 1, 65),
    ("negative", 20000, 8, 3, 30),
    ("slots", 152064, 10, 6, 60),    # row shares of 5+ slots: the fallback runs
    ("slots", 152064, 16, 4, 60),
    ("plain", 100, 64, 1, 65),       # fewer valid lanes than the bound needs: no bound
])
def test_adversarial_top_k_rows(kind, V, k, D, m):
    R, _ = tree_sizes(k, D)
    x = _adversarial(kind, R, V, k, 31)
    ref = build_draft_tree(x.numpy(), k, D, m, 5)
    t = _run(x, k, D, m, 5)
    if kind == "duplicates":
        # exact ties (the oracle reports them): the lowest token ids and
        # candidate indices decide, so the tree is still unique
        np.testing.assert_array_equal(t.parents.cpu().numpy(), ref["parents"])
        np.testing.assert_array_equal(t.tokens.cpu().numpy(), ref["tokens"])
        np.testing.assert_array_equal(t.mask_u64(), ref["mask"])
    else:
        tree_matches(t, ref, f"{kind} V{V} k{k}")
