"""GPU parity of the tree attention over an E4M3 prefix cache (one scale per
(kv head, 128-token page)) with the oracle, which decodes the same codes with
its own E4M3 decoder and applies the attention definition in fp64; max abs
error <= 2e-3."""

import numpy as np
import pytest
import torch

from eagle_speculative_decoding_verify_gb300 import binding as eb
from eagle_speculative_decoding_verify_gb300 import workloads as wl
from oracle.kv_fp8 import tree_attention_fp8
from oracle.tree_build import build_draft_tree, tree_sizes
from tests.parity import ATTN_TOL, max_abs, peaked_tol, record_attn_error
from oracle.kv_fp8 import dequantize_cache

pytestmark = pytest.mark.gpu


def _problem(m, hq, hkv, S, seed, scale_k=1.0):
    R, _ = tree_sizes(10, 6)
    g = torch.Generator().manual_seed(seed)
    ref = build_draft_tree((torch.randn(R, 300, generator=g) * 3).numpy(), 10, 6, m, 0)
    d = 128
    r = lambda *s: torch.randn(*s, generator=g).to(torch.bfloat16)
    kx = torch.randn(hkv, S, d, generator=g) * scale_k
    vx = torch.randn(hkv, S, d, generator=g)
    kc, ks = wl.fp8_kv(kx)
    vc, vs = wl.fp8_kv(vx)
    a = dict(q=r(m, hq, d), tree_k=r(m, hkv, d), tree_v=r(m, hkv, d), kc=kc, vc=vc, ks=ks, vs=vs)
    return a, ref


def _oracle(a, ref, S):
    return tree_attention_fp8(a["q"].double().numpy(), a["kc"].numpy(), a["ks"].double().numpy(),
                              a["vc"].numpy(), a["vs"].double().numpy(),
                              a["tree_k"].double().numpy(), a["tree_v"].double().numpy(),
                              ref["mask"], S)


def _run(problems, hq, hkv, expect=(0, 0)):
    items, keep = [], []
    for a, ref, S in problems:
        dev = {k: v.cuda() for k, v in a.items()}
        mask = torch.from_numpy(ref["mask"].view(np.int64).reshape(-1).copy()).cuda()
        out = torch.empty(a["q"].shape[0], hq, 128, device="cuda")
        items.append(eb.attn_fp8_item(dev["q"], dev["kc"], dev["vc"], dev["ks"], dev["vs"],
                                      dev["tree_k"], dev["tree_v"], mask, out, S))
        keep.append((dev, mask, out))
    ws = eb.eagle_tree_attn_fp8_batched(items, hq, hkv, 128, device=torch.device("cuda"))
    torch.cuda.synchronize()
    assert eb.workspace_error(ws) == expect
    return [k[2].cpu().numpy() for k in keep]


@pytest.mark.parametrize("m,hq,hkv,S", [
    (60, 32, 8, 2048),     # llama-3-8b layer shape
    (60, 28, 4, 8192),     # qwen2-7b layer shape, 8K
    (45, 8, 1, 4099),      # MQA, ragged prefix (last page partial)
    (16, 8, 2, 0),         # no prefix: tree keys only
    (100, 16, 4, 257),     # two tree chunks
    (256, 8, 2, 1000),     # two full tree chunks after eight pages
    (60, 8, 1, 40000),     # one kv head: many prefix splits
    (24, 16, 2, 12345),    # a few prefix splits, ragged last page
])
def test_fp8_prefix_matches_the_oracle(m, hq, hkv, S):
    a, ref = _problem(m, hq, hkv, S, seed=m + S)
    out = _run([(a, ref, S)], hq, hkv)[0]
    err = max_abs(out, _oracle(a, ref, S))
    assert err <= ATTN_TOL, err
    record_attn_error(f"fp8 prefix m{m} {hq}/{hkv} S{S}", err)


def test_fp8_batched_ragged_items_with_different_scales():
    # several sequences in one launch, prefixes of different lengths, one of
    # them with keys 40x larger (its page scales differ by the same factor:
    # scores concentrate on a few keys, so the bf16-weight bound applies
    # there), one with keys 20x smaller
    probs = []
    for b, (S, sk) in enumerate([(700, 1.0), (3000, 40.0), (128, 1.0), (1500, 0.05)]):
        a, ref = _problem(60, 32, 8, S, seed=100 + b, scale_k=sk)
        probs.append((a, ref, S, sk))
    outs = _run([p[:3] for p in probs], 32, 8)
    for (a, ref, S, sk), out in zip(probs, outs):
        err = max_abs(out, _oracle(a, ref, S))
        values = np.concatenate([dequantize_cache(a["vc"].numpy(), a["vs"].double().numpy()).ravel(),
                                 a["tree_v"].float().numpy().ravel()])
        tol = peaked_tol(values) if sk > 1.0 else ATTN_TOL
        assert err <= tol, (S, sk, err, tol)


def test_fp8_reports_a_query_outside_the_fp16_range():
    # the prefix's products are formed from an fp16 copy of the query: an
    # element above 65504 in magnitude is reported (detail 61), not rounded
    a, ref = _problem(16, 8, 2, 300, seed=5)
    a["q"][3, 1, 7] = 1.0e5
    _run([(a, ref, 300)], 8, 2, expect=(eb.EAGLE_ERR_DEVICE_ASSERT, 61))


def test_fp8_reports_a_value_scale_outside_the_fp16_range():
    # P carries the page's value scale in fp16: a scale above 65504 is
    # reported (detail 62)
    a, ref = _problem(16, 8, 2, 300, seed=6)
    a["vs"][1, 2] = 1.0e5
    _run([(a, ref, 300)], 8, 2, expect=(eb.EAGLE_ERR_DEVICE_ASSERT, 62))


def test_fp8_rejects_other_head_dims():
    a, ref = _problem(8, 4, 2, 256, seed=1)
    dev = {k: v.cuda() for k, v in a.items()}
    mask = torch.from_numpy(ref["mask"].view(np.int64).reshape(-1).copy()).cuda()
    out = torch.empty(8, 4, 128, device="cuda")
    it = eb.attn_fp8_item(dev["q"], dev["kc"], dev["vc"], dev["ks"], dev["vs"], dev["tree_k"],
                          dev["tree_v"], mask, out, 256)
    with pytest.raises(eb.EagleError) as e:
        eb.eagle_tree_attn_fp8_batched([it], 4, 2, 64, ws=eb.workspace(1 << 20))
    assert e.value.status == 2
