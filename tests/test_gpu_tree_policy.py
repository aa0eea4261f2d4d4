"""GPU parity of eagle_tree_build_policy against the oracle's tree-shape
policies (static tree, batched candidate chains, confidence ratio), through
the C ABI: node arrays, ancestor masks and the tree size bit-exact (both
sides rank the same float logits and compare the same double gaps), unused
node slots padded."""

import math

import numpy as np
import pytest
import torch

from eagle_speculative_decoding_verify_gb300 import binding as eb
from eagle_speculative_decoding_verify_gb300 import workloads as wl
from oracle.tree_policies import candidate_chains, confidence_tree, static_tree, static_tree_size
from tests.parity import to_device_rows

pytestmark = pytest.mark.gpu


def _rows(R, V, seed, scale=1.0, dominant=0.0):
    """Normal rows; with dominant > 0 every third row gets one clear winner."""
    g = torch.Generator().manual_seed(seed)
    x = torch.randn(R, V, generator=g) * scale
    if dominant > 0:
        for r in range(0, R, 3):
            x[r, int(torch.randint(0, V, (1,), generator=g))] += dominant
    return x


def _build(x, pol, m, root):
    xd = to_device_rows(x)
    ws = eb.workspace(eb.eagle_tree_policy_workspace_size(x.shape[1], pol, m))
    t, nn = eb.eagle_tree_build_policy(xd, pol, m, root, ws=ws)
    torch.cuda.synchronize()
    assert eb.workspace_error(ws) == (0, 0)
    return t, nn


def _compare(t, nn, ref, what):
    m = ref["m"]
    assert int(nn.item()) == m, f"{what}: size {int(nn.item())} != {m}"
    par = t.parents.cpu().numpy()
    tok = t.tokens.cpu().numpy()
    dep = t.depth.cpu().numpy()
    pos = t.pos.cpu().numpy()
    mask = t.mask_u64()
    np.testing.assert_array_equal(par[:m], ref["parents"], err_msg=f"{what} parents")
    np.testing.assert_array_equal(tok[:m], ref["tokens"], err_msg=f"{what} tokens")
    np.testing.assert_array_equal(dep[:m], ref["depth"], err_msg=f"{what} depth")
    np.testing.assert_array_equal(pos[:m], ref["pos"], err_msg=f"{what} pos")
    w = ref["mask_words"]
    np.testing.assert_array_equal(mask[:m, :w], ref["mask"], err_msg=f"{what} mask")
    assert not mask[:m, w:].any() and not mask[m:].any(), f"{what}: stray mask bits"
    assert (par[m:] == -1).all() and (tok[m:] == -1).all() and (dep[m:] == 0).all(), what


@pytest.mark.parametrize("V,n,D", [(1000, 1, 6), (5003, 2, 4), (3000, 3, 3), (152064, 4, 3),
                                   (777, 10, 2), (4096, 7, 0)])
def test_static_tree(V, n, D):
    m = static_tree_size(n, D)
    x = _rows(max(1, static_tree_size(n, D - 1) if D else 1), V, 3 + n)
    ref = static_tree(x.numpy(), n, D, 17)
    t, nn = _build(x, eb.tree_policy(eb.EAGLE_POLICY_STATIC, n, D), m, 17)
    _compare(t, nn, ref, f"static V{V} n{n} D{D}")


@pytest.mark.parametrize("V,n,D", [(1000, 3, 4), (152064, 10, 6), (2000, 2, 1), (4096, 64, 3)])
def test_candidate_chains(V, n, D):
    m = 1 + n * D
    x = _rows(1 + n * (D - 1), V, 5 + D)
    ref = candidate_chains(x.numpy(), n, D, 2)
    t, nn = _build(x, eb.tree_policy(eb.EAGLE_POLICY_CHAINS, n, D), m, 2)
    _compare(t, nn, ref, f"chains V{V} n{n} D{D}")


@pytest.mark.parametrize("V,width,depth,tau,m,scale,dominant", [
    (152064, 4, 7, 2.0, 60, 1.0, 0.0),
    (1000, 4, 7, 2.0, 60, 0.7, 4.0),      # chains and branches mixed
    (5003, 8, 5, 3.0, 256, 0.5, 0.0),     # widest branching, largest tree
    (3000, 2, 7, 1.5, 40, 1.0, 3.0),
    (2000, 4, 3, 0.5, 30, 1.0, 0.0),      # tau < 1: the argmax chain, cut at depth 3
    (2000, 4, 10, 1e30, 100, 1.0, 0.0),   # tau past every ratio: the 4-ary tree cut at 100
    (4099, 3, 7, 2.0, 1, 1.0, 0.0),       # root only
])
def test_confidence_tree(V, width, depth, tau, m, scale, dominant):
    x = _rows(max(1, m - 1), V, 11 + width, scale, dominant)
    ref = confidence_tree(x.numpy(), tau, m, 9, max_depth=depth, max_branch=width)
    t, nn = _build(x, eb.tree_policy(eb.EAGLE_POLICY_CONFIDENCE, width, depth, tau), m, 9)
    _compare(t, nn, ref, f"confidence V{V} w{width} tau{tau} m{m}")


def test_confidence_hand_rows():
    # root: p(5)/p(2) = 3 > 2 -> one child; node 1: ratios 4:3:2.5:1.9 -> three
    # children; node 2 flat -> four children, cut by the budget of 8 after three
    x = torch.zeros(8, 8)
    x[0, 5], x[0, 2] = math.log(6.0), math.log(2.0)
    x[1, 3], x[1, 6], x[1, 0], x[1, 7] = (math.log(4.0), math.log(3.0), math.log(2.5),
                                          math.log(1.9))
    t, nn = _build(x, eb.tree_policy(eb.EAGLE_POLICY_CONFIDENCE, 4, 7, 2.0), 8, 99)
    assert int(nn.item()) == 8
    assert t.parents.cpu().tolist() == [-1, 0, 1, 1, 1, 2, 2, 2]
    assert t.tokens.cpu().tolist() == [99, 5, 3, 6, 0, 0, 1, 2]
    assert t.depth.cpu().tolist() == [0, 1, 2, 2, 2, 3, 3, 3]


def test_confidence_on_workload_draft_rows():
    # the c2 draft rows (sigma per row from {1, 3, 6}): 51 rows -> a cap of 52 nodes
    w = wl.WORKLOADS["c2"]
    x = wl.draft_logits(w)
    root = wl.root_token(w)
    ref = confidence_tree(x.numpy(), 2.0, 52, root, max_depth=7, max_branch=4)
    t, nn = _build(x, eb.tree_policy(eb.EAGLE_POLICY_CONFIDENCE, 4, 7, 2.0), 52, root)
    _compare(t, nn, ref, "confidence c2 rows")
