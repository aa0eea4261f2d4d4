"""A bounded device wait that runs out (failure detection without a GPU
fault): the tensor-core attention's producers are told, through the
workspace header's test hook, to issue no copy, so every wait on a copy or on
the MMAs behind it runs out after a short limit.  The call must come back,
record EAGLE_ERR_TIMEOUT in the workspace's error word, leave the context
usable, and -- after eagle_workspace_init -- the same workspace must give the
correct result."""

import numpy as np
import pytest
import torch

from eagle_speculative_decoding_verify_gb300 import binding as eb
from oracle.tree_attn import tree_attention
from oracle.tree_build import build_draft_tree, tree_sizes
from tests.parity import ATTN_TOL, max_abs

pytestmark = pytest.mark.gpu
NAMES = ("q", "k_cache", "v_cache", "tree_k", "tree_v")


def _case(m=60, hq=32, hkv=8, d=128, S=2048, seed=3):
    R, _ = tree_sizes(10, 6)
    g = torch.Generator().manual_seed(seed)
    ref = build_draft_tree((torch.randn(R, 300, generator=g) * 3).numpy(), 10, 6, m, 0)
    r = lambda *s: torch.randn(*s, generator=g).to(torch.bfloat16)
    a = dict(q=r(m, hq, d), k_cache=r(hkv, S, d), v_cache=r(hkv, S, d), tree_k=r(m, hkv, d),
             tree_v=r(m, hkv, d))
    mask = torch.from_numpy(ref["mask"].view(np.int64).reshape(-1).copy()).cuda()
    return a, ref, mask, S


def test_attention_wait_runs_out_then_the_workspace_recovers():
    a, ref, mask, S = _case()
    dev = {n: a[n].cuda() for n in NAMES}
    m, hq, d = a["q"].shape
    hkv = a["k_cache"].shape[0]
    ws = eb.workspace(eb.eagle_tree_attn_workspace_size(m, hq, hkv, d, S, eb.EAGLE_BF16))
    eb.workspace_test_hook(ws, no_copies=True, wait_us=2000)
    out = eb.eagle_tree_attn(*(dev[n] for n in NAMES), mask, prefix_len=S, ws=ws)
    st, detail = eb.workspace_error(ws)
    assert st == eb.EAGLE_ERR_TIMEOUT, (st, detail)
    assert detail in (29, 30, 31, 32, 33, 34, 40, 41, 42), detail   # a wait of the kernel
    # the context is usable; re-initialised, the same workspace works
    eb.eagle_workspace_init(ws)
    out = eb.eagle_tree_attn(*(dev[n] for n in NAMES), mask, prefix_len=S, ws=ws)
    torch.cuda.synchronize()
    assert eb.workspace_error(ws) == (0, 0)
    o_ref = tree_attention(*(a[n].double().numpy() for n in NAMES), ref["mask"], S)
    assert max_abs(out.cpu().numpy(), o_ref) <= ATTN_TOL


def test_default_limit_is_not_hit_in_normal_use():
    # the hook words left at zero: no timeout, correct output (batched form)
    a, ref, mask, S = _case(S=1000, seed=4)
    dev = {n: a[n].cuda() for n in NAMES}
    m, hq, d = a["q"].shape
    hkv = a["k_cache"].shape[0]
    out = torch.empty(m, hq, d, device="cuda")
    item = eb.attn_item(dev["q"], dev["k_cache"], dev["v_cache"], dev["tree_k"], dev["tree_v"],
                        mask, out, prefix_len=S)
    ws = eb.workspace(eb.eagle_tree_attn_batched_workspace_size([item], hq, hkv, d,
                                                                eb.EAGLE_BF16))
    eb.eagle_tree_attn_batched([item], hq, hkv, d, eb.EAGLE_BF16, ws=ws)
    torch.cuda.synchronize()
    assert eb.workspace_error(ws) == (0, 0)
    o_ref = tree_attention(*(a[n].double().numpy() for n in NAMES), ref["mask"], S)
    assert max_abs(out.cpu().numpy(), o_ref) <= ATTN_TOL
