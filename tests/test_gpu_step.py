"""End-to-end verify step on the GPU (build -> attention -> verify, stream
ordered, all through the C ABI) against the oracle, plus the smoke entry."""

import numpy as np
import pytest
import torch

from eagle_speculative_decoding_verify_gb300 import binding as eb
from eagle_speculative_decoding_verify_gb300 import workloads as wl
from oracle.tree_attn import tree_attention
from oracle.tree_build import build_draft_tree
from oracle.verify import verify_tree
from tests.parity import ATTN_TOL, max_abs, path_matches, tree_matches

pytestmark = pytest.mark.gpu
NAMES = ("q", "k_cache", "v_cache", "tree_k", "tree_v")


@pytest.mark.parametrize("key", ["c0", "c2"])
def test_full_step(key):
    w = wl.WORKLOADS[key]
    draft = wl.draft_logits(w)
    root = wl.root_token(w)
    ref = build_draft_tree(draft.numpy(), w.top_k, w.depth, w.total_tokens, root)
    target = wl.target_logits(w, ref["parents"], ref["tokens"])
    a = wl.attention_inputs(w)
    gr, T, k, p = w.sampling_of(0)
    dev = {n: a[n].cuda() for n in NAMES}
    d_draft, d_target = draft.cuda(), target.cuda()
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        tree = eb.eagle_tree_build(d_draft, w.top_k, w.depth, w.total_tokens, root, stream=s)
        out = eb.eagle_tree_attn(*(dev[n] for n in NAMES), tree.mask, stream=s)
        acc, n, bonus = eb.eagle_tree_verify(d_target, tree, eb.sampling(gr, T, k, p), 42, 0,
                                             stream=s)
    s.synchronize()
    tree_matches(tree, ref, key)
    o_ref = tree_attention(*(a[n].double().numpy() for n in NAMES), ref["mask"], w.prefix)
    assert max_abs(out.cpu().numpy(), o_ref) <= ATTN_TOL
    v = verify_tree(target.numpy(), ref["parents"], ref["tokens"], greedy=bool(gr),
                    temperature=T, top_k=k, top_p=p, seed=42, step=0)
    path_matches(acc.cpu().numpy(), int(n.item()), int(bonus.item()), v, key, ref["parents"],
                 ref["tokens"], target.numpy(), (gr, T, k, p))


def test_smoke_entry():
    import __graft_entry__
    __graft_entry__.smoke()
