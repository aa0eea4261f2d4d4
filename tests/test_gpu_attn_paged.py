"""GPU parity of eagle_tree_attn_paged_batched (prefix cache in 128-token
pages of a shared pool, one block table per item): bit-identical to the
contiguous call on the same keys and values, and within the attention
tolerance of the oracle's paged attention; a page id outside the pool is
reported, not faulted on."""

import numpy as np
import pytest
import torch

from eagle_speculative_decoding_verify_gb300 import binding as eb
from oracle.tree_attn import tree_attention_paged
from oracle.tree_build import build_draft_tree

pytestmark = pytest.mark.gpu
PAGE = eb.EAGLE_KV_PAGE_TOKENS


def _tree(seed, k=6, D=5, m=60, V=400):
    rng = np.random.default_rng(seed)
    R = 1 + (D - 1) * k
    return build_draft_tree((rng.standard_normal((R, V)) * 3).astype(np.float32), k, D, m, 0)


def _problem(seed, m, hq, hkv, d, S, pool_pages):
    """Contiguous inputs plus the same prefix scattered into shuffled pool pages."""
    g = torch.Generator().manual_seed(seed)
    r = lambda *s: torch.randn(*s, generator=g).to(torch.bfloat16)
    q, kc, vc, tk, tv = r(m, hq, d), r(hkv, S, d), r(hkv, S, d), r(m, hkv, d), r(m, hkv, d)
    n_pages = (S + PAGE - 1) // PAGE
    table = torch.from_numpy(np.random.default_rng(seed).permutation(pool_pages)[:n_pages]
                             .astype(np.int32))
    kp = r(hkv, pool_pages * PAGE, d)   # unused rows hold noise
    vp = r(hkv, pool_pages * PAGE, d)
    for j in range(n_pages):
        lo, hi = j * PAGE, min(S, (j + 1) * PAGE)
        kp[:, table[j] * PAGE: table[j] * PAGE + hi - lo] = kc[:, lo:hi]
        vp[:, table[j] * PAGE: table[j] * PAGE + hi - lo] = vc[:, lo:hi]
    return q, kc, vc, tk, tv, kp, vp, table


@pytest.mark.parametrize("hq,hkv,d,sizes", [
    (28, 4, 128, [8192]),                  # the c2 layer shape
    (32, 8, 128, [1000, 0, 4099, 128]),    # ragged, empty prefix, partial and whole pages
    (8, 2, 64, [300, 2500]),
])
def test_paged_equals_contiguous_and_oracle(hq, hkv, d, sizes):
    t = _tree(hq + d)
    m = t["m"]
    mask = torch.from_numpy(t["mask"].view(np.int64).reshape(-1)).cuda()
    items_p, items_c, keep, outs_p, outs_c, host = [], [], [], [], [], []
    for i, S in enumerate(sizes):
        q, kc, vc, tk, tv, kp, vp, table = _problem(7 * i + d, m, hq, hkv, d, S,
                                                    (S + PAGE - 1) // PAGE + 3)
        dv = [x.cuda() for x in (q, kc, vc, tk, tv, kp, vp, table)]
        op = torch.empty(m, hq, d, device="cuda")
        oc = torch.empty(m, hq, d, device="cuda")
        keep.append(dv)
        outs_p.append(op)
        outs_c.append(oc)
        host.append((q, kp, vp, table, tk, tv, S))
        items_p.append(eb.attn_paged_item(dv[0], dv[5], dv[6], dv[7], dv[3], dv[4], mask, op, S))
        items_c.append(eb.attn_item(dv[0], dv[1], dv[2], dv[3], dv[4], mask, oc, S))
    ws = eb.eagle_tree_attn_paged_batched(items_p, hq, hkv, d)
    eb.eagle_tree_attn_batched(items_c, hq, hkv, d, eb.EAGLE_BF16)
    torch.cuda.synchronize()
    assert eb.workspace_error(ws) == (0, 0)
    for op, oc, (q, kp, vp, table, tk, tv, S) in zip(outs_p, outs_c, host):
        assert torch.equal(op, oc)
        f = lambda x: x.double().numpy()
        ref = tree_attention_paged(f(q), f(kp), f(vp), table.numpy(), f(tk), f(tv), t["mask"], S)
        assert np.abs(op.cpu().numpy() - ref).max() <= 2e-3


def test_page_outside_the_pool_is_reported():
    t = _tree(1)
    m, hq, hkv, d, S = t["m"], 8, 2, 128, 700
    q, kc, vc, tk, tv, kp, vp, table = _problem(3, m, hq, hkv, d, S, 8)
    table[2] = 8                                  # the pool has pages 0..7
    mask = torch.from_numpy(t["mask"].view(np.int64).reshape(-1)).cuda()
    dv = [x.cuda() for x in (q, tk, tv, kp, vp, table)]
    out = torch.empty(m, hq, d, device="cuda")
    ws = eb.eagle_tree_attn_paged_batched(
        [eb.attn_paged_item(dv[0], dv[3], dv[4], dv[5], dv[1], dv[2], mask, out, S)], hq, hkv, d)
    torch.cuda.synchronize()
    assert eb.workspace_error(ws)[0] == eb.EAGLE_ERR_DEVICE_ASSERT


def test_rejects_bad_arguments():
    t = _tree(2)
    m, hq, hkv, S = t["m"], 4, 2, 200
    mask = torch.from_numpy(t["mask"].view(np.int64).reshape(-1)).cuda()
    for d in (96, 128):
        q, kc, vc, tk, tv, kp, vp, table = _problem(5, m, hq, hkv, d, S, 4)
        dv = [x.cuda() for x in (q, tk, tv, kp, vp, table)]
        out = torch.empty(m, hq, d, device="cuda")
        item = eb.attn_paged_item(dv[0], dv[3], dv[4], dv[5], dv[1], dv[2], mask, out, S)
        if d == 128:
            item.block_table = None                # a prefix without a block table
        with pytest.raises(eb.EagleError):
            eb.eagle_tree_attn_paged_batched([item], hq, hkv, d, ws=eb.workspace(1 << 20))
