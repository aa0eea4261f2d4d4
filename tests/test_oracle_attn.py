"""Pins for the oracle's tree attention.

Checked against: PyTorch's scaled_dot_product_attention in fp64 (a library
routine) on (a) every node's own causal sequence -- prefix plus its ancestor
chain found by walking parent pointers, not through the mask -- and (b) a
chain tree over an empty prefix, which is plain causal attention; plus the
closed form for identical keys (uniform weights = mean of visible values).
"""

import numpy as np
import pytest
import torch

from oracle.tree_attn import tree_attention, tree_attention_rows
from oracle.tree_build import build_draft_tree


def _tree(seed, k=3, D=3, m=10, V=64):
    rng = np.random.default_rng(seed)
    R = 1 + (D - 1) * k
    logits = (rng.standard_normal((R, V)) * rng.choice([1.0, 3.0, 6.0], size=(R, 1))).astype(np.float32)
    return build_draft_tree(logits, k, D, m, 0)


def _inputs(seed, m, Hq, Hkv, d, S):
    g = torch.Generator().manual_seed(seed)
    r = lambda *s: torch.randn(*s, generator=g, dtype=torch.float64)
    return r(m, Hq, d), r(Hkv, S + 5, d), r(Hkv, S + 5, d), r(m, Hkv, d), r(m, Hkv, d)


def _sdpa_one(q, keys, vals, scale):
    out = torch.nn.functional.scaled_dot_product_attention(
        q[None, None, None, :], keys[None, None], vals[None, None], scale=scale)
    return out[0, 0, 0]


@pytest.mark.parametrize("Hq,Hkv,S,scale", [(4, 2, 16, None), (6, 3, 0, None), (8, 1, 33, None),
                                            (4, 2, 16, 0.05), (2, 1, 9, 0.7)])
def test_each_node_equals_causal_attention_over_its_chain(Hq, Hkv, S, scale):
    # scale None: the default 1/sqrt(d); otherwise the caller's score scale
    t = _tree(Hq + S)
    m, d = t["m"], 16
    q, kc, vc, tk, tv = _inputs(S, m, Hq, Hkv, d, S)
    out = tree_attention(q.numpy(), kc.numpy(), vc.numpy(), tk.numpy(), tv.numpy(),
                         t["mask"], S, scale=scale)
    g = Hq // Hkv
    scale = 1.0 / np.sqrt(d) if scale is None else scale
    for i in range(m):
        chain = []
        n = i
        while n >= 0:
            chain.append(n)
            n = int(t["parents"][n]) if n > 0 else -1
        chain = chain[::-1]
        for h in range(Hq):
            kv = h // g
            keys = torch.cat([kc[kv, :S], tk[chain, kv]])
            vals = torch.cat([vc[kv, :S], tv[chain, kv]])
            ref = _sdpa_one(q[i, h], keys, vals, scale)
            np.testing.assert_allclose(out[i, h], ref.numpy(), rtol=1e-12, atol=1e-12)
    rows = [(0, 0), (m - 1, Hq - 1), (m // 2, 1)]
    sampled = tree_attention_rows(q.numpy(), kc.numpy(), vc.numpy(), tk.numpy(), tv.numpy(),
                                  t["mask"], S, rows, scale=scale)
    for n, (i, h) in enumerate(rows):
        np.testing.assert_allclose(sampled[n], out[i, h], rtol=1e-12, atol=1e-12)


def test_chain_tree_without_prefix_is_causal_attention():
    m, Hq, Hkv, d = 7, 4, 2, 8
    parents = np.array([-1] + list(range(m - 1)))
    mask = np.zeros((m, 1), dtype=np.uint64)
    for i in range(m):
        mask[i, 0] = np.uint64((1 << (i + 1)) - 1)
    q, kc, vc, tk, tv = _inputs(3, m, Hq, Hkv, d, 0)
    out = tree_attention(q.numpy(), kc.numpy(), vc.numpy(), tk.numpy(), tv.numpy(), mask, 0)
    kx = tk.repeat_interleave(Hq // Hkv, dim=1).permute(1, 0, 2)   # [Hq, m, d]
    vx = tv.repeat_interleave(Hq // Hkv, dim=1).permute(1, 0, 2)
    ref = torch.nn.functional.scaled_dot_product_attention(
        q.permute(1, 0, 2)[None], kx[None], vx[None], is_causal=True)[0].permute(1, 0, 2)
    np.testing.assert_allclose(out, ref.numpy(), rtol=1e-12, atol=1e-12)
    assert parents[0] == -1


def test_identical_keys_average_visible_values():
    t = _tree(11)
    m, Hq, Hkv, d, S = t["m"], 2, 1, 4, 5
    q, kc, vc, tk, tv = _inputs(4, m, Hq, Hkv, d, S)
    kc[:] = 0.5
    tk[:] = 0.5
    out = tree_attention(q.numpy(), kc.numpy(), vc.numpy(), tk.numpy(), tv.numpy(), t["mask"], S)
    for i in range(m):
        anc = [j for j in range(m) if (int(t["mask"][i, j // 64]) >> (j % 64)) & 1]
        vals = torch.cat([vc[0, :S], tv[anc, 0]])
        np.testing.assert_allclose(out[i, 0], vals.mean(0).numpy(), rtol=1e-12, atol=1e-13)


def test_paged_prefix_equals_the_contiguous_cache():
    """A contiguous cache scattered into shuffled pages of a larger pool (by
    hand, page by page) and gathered back gives the same attention; the pool's
    unused rows hold values that would change the result if read."""
    from oracle.tree_attn import gather_pages, tree_attention_paged
    t = _tree(9)
    m, Hq, Hkv, d, S, page = t["m"], 4, 2, 16, 300, 128
    q, kc, vc, tk, tv = _inputs(3, m, Hq, Hkv, d, S)
    n_pages = (S + page - 1) // page
    rng = np.random.default_rng(1)
    table = rng.permutation(7)[:n_pages]                 # pages anywhere in a 7-page pool
    kpool = np.full((Hkv, 7 * page, d), 1e3)
    vpool = np.full((Hkv, 7 * page, d), -1e3)
    for j in range(n_pages):
        lo, hi = j * page, min(S, (j + 1) * page)
        kpool[:, table[j] * page: table[j] * page + hi - lo] = kc[:, lo:hi].numpy()
        vpool[:, table[j] * page: table[j] * page + hi - lo] = vc[:, lo:hi].numpy()
    assert np.array_equal(gather_pages(kpool, table, S, page), kc[:, :S].numpy())
    ref = tree_attention(q.numpy(), kc.numpy(), vc.numpy(), tk.numpy(), tv.numpy(), t["mask"], S)
    got = tree_attention_paged(q.numpy(), kpool, vpool, table, tk.numpy(), tv.numpy(), t["mask"],
                               S, page=page)
    assert np.array_equal(got, ref)
