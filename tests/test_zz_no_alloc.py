"""GPU check of eagle_tree_build_noalloc (the allocation-free variant of
eagle_tree_build on the library's fixed static scratch), through the C ABI:
two calls in a row, on different shapes, each matching eagle_tree_build
(which runs on a caller-owned workspace) exactly, and the size limit.

Named so that pytest collects it last; it also passes alone in a fresh
process."""

import numpy as np
import pytest
import torch

from eagle_speculative_decoding_verify_gb300 import binding as eb
from eagle_speculative_decoding_verify_gb300 import workloads as wl

pytestmark = pytest.mark.gpu

FIELDS = ("parents", "tokens", "depth", "pos", "mask", "values")


def _same(a, b, what):
    for f in FIELDS:
        x, y = getattr(a, f).cpu().numpy(), getattr(b, f).cpu().numpy()
        assert np.array_equal(x, y), f"{what}: {f} differs"


def _rows(R, V, seed):
    g = torch.Generator().manual_seed(seed)
    return (torch.randn(R, V, generator=g) * 3.0).cuda()


def test_two_calls_match_the_workspace_entry_point():
    cases = []
    for key in ("c2", "c0"):          # different R / top_k: different scratch layouts
        w = wl.WORKLOADS[key]
        cases.append((wl.draft_logits(w).cuda(), w.top_k, w.depth, w.total_tokens,
                      wl.root_token(w)))
    got = []
    for x, k, D, m, root in cases:    # two allocation-free calls back to back
        got.append(eb.eagle_tree_build_noalloc(x, k, D, m, root))
    torch.cuda.synchronize()
    for (x, k, D, m, root), t in zip(cases, got):
        ref = eb.eagle_tree_build(x, k, D, m, root)
        torch.cuda.synchronize()
        _same(t, ref, f"k{k} D{D} m{m}")


def test_repeat_after_a_larger_shape_leaves_no_stale_state():
    # the largest fitting shape of top_k 10 (depth 16), then a small one twice
    big = (_rows(151, 4100, 1), 10, 16, 256, 7)
    small = (_rows(13, 3000, 2), 4, 4, 20, 3)
    for x, k, D, m, root in (big, small, small):
        t = eb.eagle_tree_build_noalloc(x, k, D, m, root)
        ref = eb.eagle_tree_build(x, k, D, m, root)
        torch.cuda.synchronize()
        _same(t, ref, f"k{k} D{D} m{m}")


def test_rejects_shapes_beyond_the_scratch():
    k, D, m = 12, 13, 64                       # workspace 16,896 bytes
    R = 1 + (D - 1) * k
    assert eb.eagle_tree_build_workspace_size(1, R, 1000, k, D, m) > \
        eb.EAGLE_NOALLOC_SCRATCH_BYTES
    x = _rows(R, 1000, 3)
    with pytest.raises(eb.EagleError) as e:
        eb.eagle_tree_build_noalloc(x, k, D, m, 0)
    assert e.value.status == eb.EAGLE_ERR_WORKSPACE_TOO_SMALL
    # the same shape still works through a caller-owned workspace
    t = eb.eagle_tree_build(x, k, D, m, 0)
    torch.cuda.synchronize()
    assert int(t.parents[0]) == -1


def test_reused_output_tree_and_error_word():
    # a caller that cannot allocate also reuses its output arrays: two calls
    # in stream order into the same tree with different roots, each result
    # read before the next call, each equal to the workspace entry point's
    w = wl.WORKLOADS["c1"]
    x = wl.draft_logits(w).cuda()
    out = eb.Tree(w.total_tokens)
    for root in (17, 90210):
        t = eb.eagle_tree_build_noalloc(x, w.top_k, w.depth, w.total_tokens, root, out=out)
        assert t is out
        ref = eb.eagle_tree_build(x, w.top_k, w.depth, w.total_tokens, root)
        torch.cuda.synchronize()
        _same(out, ref, f"root {root}")
        assert int(out.tokens[0]) == root
        # the static scratch's device error word is clear after a good call
        assert eb.eagle_tree_build_noalloc_error() == (0, 0)
