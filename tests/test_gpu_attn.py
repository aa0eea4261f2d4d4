"""GPU parity of eagle_tree_attn against the oracle (max abs error <= 2e-3 on
the same bf16-rounded / fp32 inputs), through the C ABI."""

import numpy as np
import pytest
import torch

from eagle_speculative_decoding_verify_gb300 import binding as eb
from eagle_speculative_decoding_verify_gb300 import workloads as wl
from oracle.tree_attn import tree_attention, tree_attention_rows
from oracle.tree_build import build_draft_tree, tree_sizes
from tests.parity import ATTN_TOL, max_abs, peaked_tol, record_attn_error

pytestmark = pytest.mark.gpu
NAMES = ("q", "k_cache", "v_cache", "tree_k", "tree_v")


def _tree(k, D, m, V=300, seed=0):
    R, _ = tree_sizes(k, D)
    g = torch.Generator().manual_seed(seed)
    x = torch.randn(R, V, generator=g) * 3.0
    return build_draft_tree(x.numpy(), k, D, m, 0)


def _mask_dev(ref):
    return torch.from_numpy(ref["mask"].view(np.int64).reshape(-1).copy()).cuda()


def _inputs(m, hq, hkv, d, S, dtype, seed, cap=None):
    g = torch.Generator().manual_seed(seed)
    cap = S if cap is None else cap
    r = lambda *s: torch.randn(*s, generator=g).to(dtype)
    return dict(q=r(m, hq, d), k_cache=r(hkv, cap, d), v_cache=r(hkv, cap, d),
                tree_k=r(m, hkv, d), tree_v=r(m, hkv, d))


def _check(a, ref, S, tol=ATTN_TOL, scale=0.0):
    dev = {n: a[n].cuda() for n in NAMES}
    out = eb.eagle_tree_attn(*(dev[n] for n in NAMES), _mask_dev(ref), prefix_len=S, scale=scale)
    torch.cuda.synchronize()
    o_ref = tree_attention(*(a[n].double().numpy() for n in NAMES), ref["mask"], S,
                           scale=scale or None)
    err = max_abs(out.cpu().numpy(), o_ref)
    assert err <= tol, f"max abs err {err}"
    return err


def _workload_name(key):
    w = wl.WORKLOADS[key]
    return f"{key} {w.name} (full)"


@pytest.mark.parametrize("key", ["c0", "c1", "c2"])
def test_workload_attention(key):
    w = wl.WORKLOADS[key]
    ref = build_draft_tree(wl.draft_logits(w).numpy(), w.top_k, w.depth, w.total_tokens,
                           wl.root_token(w))
    err = _check(wl.attention_inputs(w), ref, w.prefix)
    record_attn_error(_workload_name(key), err)


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
@pytest.mark.parametrize("m,hq,hkv,d,S", [
    (16, 4, 2, 64, 0),        # empty prefix: tree keys only
    (1, 8, 8, 128, 300),      # root only, no GQA sharing
    (60, 28, 4, 128, 1000),   # g = 7, ragged prefix
    (45, 8, 1, 64, 4099),     # MQA, prefix not a multiple of any tile
    (100, 16, 4, 128, 257),   # two tree chunks
    (256, 4, 4, 128, 130),    # maximum tree
])
def test_shapes(dtype, m, hq, hkv, d, S):
    ref = _tree(10, 6, m, seed=m + S)
    a = _inputs(m, hq, hkv, d, S, dtype, seed=S + d)
    _check(a, ref, S)


@pytest.mark.parametrize("S,kscale", [(2048, 40.0), (5000, 12.0), (300, 80.0)])
def test_peaked_scores(S, kscale):
    # keys scaled up: a few keys dominate every row, the case where the
    # weights' bf16 rounding must cancel in the normalisation
    m, hq, hkv, d = 60, 32, 8, 128
    ref = _tree(10, 6, m, seed=S)
    a = _inputs(m, hq, hkv, d, S, torch.bfloat16, seed=S + 1)
    a["k_cache"] = (a["k_cache"].float() * kscale).to(torch.bfloat16)
    a["tree_k"] = (a["tree_k"].float() * kscale).to(torch.bfloat16)
    tol = peaked_tol(torch.cat([a["v_cache"].float().flatten(), a["tree_v"].float().flatten()]))
    err = _check(a, ref, S, tol=tol)
    record_attn_error(f"peaked scores S{S} x{kscale} (bound {tol:.2e})", err)


def test_custom_scale_and_cache_capacity():
    m, hq, hkv, d, S = 20, 8, 2, 128, 700
    ref = _tree(4, 3, m, seed=5)
    a = _inputs(m, hq, hkv, d, S, torch.bfloat16, seed=9, cap=1024)   # cache longer than prefix
    _check(a, ref, S, scale=0.05)


def test_long32_all_layers():
    """32 layers x 32K prefix in one batched launch: layers 0 and 31 compared
    element by element, every other layer on sampled rows."""
    w = wl.WORKLOADS["c3"]
    ref = build_draft_tree(wl.draft_logits(w).numpy(), w.top_k, w.depth, w.total_tokens,
                           wl.root_token(w))
    mask = _mask_dev(ref)
    layers = [wl.attention_inputs(w, layer=l, device="cuda") for l in range(w.layers)]
    outs = [torch.empty(w.total_tokens, w.n_q_heads, w.head_dim, device="cuda")
            for _ in range(w.layers)]
    items = [eb.attn_item(a["q"], a["k_cache"], a["v_cache"], a["tree_k"], a["tree_v"], mask, o)
             for a, o in zip(layers, outs)]
    eb.eagle_tree_attn_batched(items, w.n_q_heads, w.n_kv_heads, w.head_dim, eb.EAGLE_BF16,
                               device=torch.device("cuda"))
    torch.cuda.synchronize()
    worst = 0.0
    for l in (0, w.layers - 1):
        a = {n: layers[l][n].cpu().double().numpy() for n in NAMES}
        o_ref = tree_attention(*(a[n] for n in NAMES), ref["mask"], w.prefix)
        err = max_abs(outs[l].cpu().numpy(), o_ref)
        assert err <= ATTN_TOL, (l, err)
        worst = max(worst, err)
    rng = np.random.default_rng(0)
    for l in range(1, w.layers - 1):
        a = {n: layers[l][n].cpu().double().numpy() for n in NAMES}
        rows = [(int(rng.integers(w.total_tokens)), int(rng.integers(w.n_q_heads)))
                for _ in range(3)]
        o_ref = tree_attention_rows(*(a[n] for n in NAMES), ref["mask"], w.prefix, rows)
        got = outs[l].cpu().numpy()
        for n, (i, h) in enumerate(rows):
            err = max_abs(got[i, h], o_ref[n])
            assert err <= ATTN_TOL, (l, i, h, err)
            worst = max(worst, err)
    record_attn_error("c3 long32 (layers 0, 31 in full; 30 layers sampled)", worst)


def test_ragged16_all_items():
    """16 sequences with prefixes U[512, 16384], 64/8 heads, one launch; every
    item compared element by element."""
    w = wl.WORKLOADS["c4"]
    lens = wl.prefix_lengths(w)
    items, keep = [], []
    for b in range(w.items):
        ref = build_draft_tree(wl.draft_logits(w, b).numpy(), w.top_k, w.depth, w.total_tokens,
                               wl.root_token(w, b))
        a = wl.attention_inputs(w, item=b, prefix=lens[b])
        dev = {n: a[n].cuda() for n in NAMES}
        mask = _mask_dev(ref)
        out = torch.empty(w.total_tokens, w.n_q_heads, w.head_dim, device="cuda")
        items.append(eb.attn_item(dev["q"], dev["k_cache"], dev["v_cache"], dev["tree_k"],
                                  dev["tree_v"], mask, out))
        keep.append((a, ref, dev, mask, out))
    eb.eagle_tree_attn_batched(items, w.n_q_heads, w.n_kv_heads, w.head_dim, eb.EAGLE_BF16,
                               device=torch.device("cuda"))
    torch.cuda.synchronize()
    worst = 0.0
    for b in range(w.items):
        a, ref, _, _, out = keep[b]
        o_ref = tree_attention(*(a[n].double().numpy() for n in NAMES), ref["mask"], lens[b])
        err = max_abs(out.cpu().numpy(), o_ref)
        assert err <= ATTN_TOL, (b, lens[b], err)
        worst = max(worst, err)
    record_attn_error("c4 ragged16 (all 16 items in full)", worst)


def test_rejects_bad_arguments():
    m, hq, hkv, d, S = 8, 4, 2, 64, 64
    ref = _tree(2, 3, m)
    a = {n: t.cuda() for n, t in _inputs(m, hq, hkv, d, S, torch.bfloat16, 0).items()}
    with pytest.raises(eb.EagleError) as e:   # heads not divisible
        eb.eagle_tree_attn(a["q"][:, :3], a["k_cache"], a["v_cache"], a["tree_k"], a["tree_v"],
                           _mask_dev(ref))
    assert e.value.status in (1, 2)
    need = eb.eagle_tree_attn_workspace_size(m, hq, hkv, d, S, eb.EAGLE_BF16)
    if need > 256:
        with pytest.raises(eb.EagleError) as e:
            eb.eagle_tree_attn(a["q"], a["k_cache"], a["v_cache"], a["tree_k"], a["tree_v"],
                               _mask_dev(ref), ws=eb.workspace(256))
        assert e.value.status == 3
