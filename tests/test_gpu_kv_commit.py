"""GPU parity of eagle_kv_commit / eagle_kv_commit_batched against the
oracle (bit-exact: the commit moves bytes), through the C ABI, including the
chain tree build -> verify -> commit on the c2 workload and the device-side
bounds checks."""

import numpy as np
import pytest
import torch

from eagle_speculative_decoding_verify_gb300 import binding as eb
from eagle_speculative_decoding_verify_gb300 import workloads as wl
from oracle.kv_commit import kv_commit
from oracle.tree_build import build_draft_tree
from tests.parity import to_device_rows

pytestmark = pytest.mark.gpu


def _path(parents, last):
    chain = []
    while last >= 0:
        chain.append(int(last))
        last = int(parents[last])
    return chain[::-1]


def _tree(seed, k=4, D=5, m=40, V=300):
    rng = np.random.default_rng(seed)
    R = 1 + (D - 1) * k
    logits = (rng.standard_normal((R, V)) * 3).astype(np.float32)
    return build_draft_tree(logits, k, D, m, 0)


def _caches(seed, Hkv, cap, d, m, dtype):
    g = torch.Generator().manual_seed(seed)
    r = lambda *s: torch.randn(*s, generator=g).to(dtype)
    return r(Hkv, cap, d), r(Hkv, cap, d), r(m, Hkv, d), r(m, Hkv, d)


def _run_one(kc, vc, tk, tv, path, S, dev="cuda"):
    acc = torch.zeros(tk.shape[0], dtype=torch.int32)
    acc[: len(path)] = torch.tensor(path, dtype=torch.int32)
    n = torch.tensor([len(path) - 1], dtype=torch.int32)
    kd, vd = kc.to(dev), vc.to(dev)
    ws = eb.workspace(eb.eagle_kv_commit_workspace_size())
    eb.eagle_kv_commit(kd, vd, tk.to(dev), tv.to(dev), acc.to(dev), n.to(dev), S, ws=ws)
    assert eb.workspace_error(ws) == (0, 0)
    return kd.cpu(), vd.cpu()


def _as_np(t):
    return t.view(torch.int16).numpy() if t.dtype == torch.bfloat16 else t.numpy()


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32])
@pytest.mark.parametrize("Hkv,d,S", [(4, 128, 1000), (8, 64, 0), (1, 128, 4099), (2, 8, 5)])
def test_paths_match_the_oracle(dtype, Hkv, d, S):
    t = _tree(Hkv + d + S)
    m = t["m"]
    kc, vc, tk, tv = _caches(S + d, Hkv, S + m + 3, d, m, dtype)
    for last in (0, m - 1, m // 2, int(np.argmax(t["depth"]))):
        path = _path(t["parents"], last)
        kg, vg = _run_one(kc, vc, tk, tv, path, S)
        ko, vo, _ = kv_commit(_as_np(kc), _as_np(vc), S, _as_np(tk), _as_np(tv), path, len(path) - 1)
        assert np.array_equal(_as_np(kg), ko) and np.array_equal(_as_np(vg), vo)


def test_verify_then_commit_c2():
    w = wl.WORKLOADS["c2"]
    draft = wl.draft_logits(w).cuda()
    tree = eb.eagle_tree_build(draft, w.top_k, w.depth, w.total_tokens, wl.root_token(w))
    parents = tree.parents.cpu().numpy()
    tokens = tree.tokens.cpu().numpy()
    target = wl.target_logits(w, parents, tokens)
    acc, n, bonus = eb.eagle_tree_verify(to_device_rows(target), tree,
                                         eb.sampling(False, 0.7, 50, 0.9), 1234, 0)
    a = wl.attention_inputs(w, device="cpu")
    S = w.prefix
    cap = S + w.total_tokens
    kc = torch.zeros(w.n_kv_heads, cap, w.head_dim, dtype=a["k_cache"].dtype)
    vc = torch.zeros_like(kc)
    kc[:, :S] = a["k_cache"]
    vc[:, :S] = a["v_cache"]
    kd, vd = kc.cuda(), vc.cuda()
    ws = eb.workspace(eb.eagle_kv_commit_workspace_size())
    eb.eagle_kv_commit(kd, vd, a["tree_k"].cuda(), a["tree_v"].cuda(), acc, n, S, ws=ws)
    assert eb.workspace_error(ws) == (0, 0)
    path = acc.cpu().numpy()
    nn = int(n.item())
    assert path[0] == 0 and all(parents[path[i]] == path[i - 1] for i in range(1, nn + 1))
    ko, vo, new_len = kv_commit(_as_np(kc), _as_np(vc), S, _as_np(a["tree_k"]),
                                _as_np(a["tree_v"]), path, nn)
    assert new_len == S + nn + 1
    assert np.array_equal(_as_np(kd.cpu()), ko) and np.array_equal(_as_np(vd.cpu()), vo)


def test_batched_layers_and_ragged_paths():
    t = _tree(3, k=5, D=6, m=60, V=500)
    m, Hkv, d = t["m"], 8, 128
    items, host, dev_bufs = [], [], []
    for layer in range(20):
        S = 64 * layer + (layer % 3)
        kc, vc, tk, tv = _caches(100 + layer, Hkv, S + m, d, m, torch.bfloat16)
        path = _path(t["parents"], (7 * layer) % m)
        acc = torch.zeros(m, dtype=torch.int32)
        acc[: len(path)] = torch.tensor(path, dtype=torch.int32)
        n = torch.tensor([len(path) - 1], dtype=torch.int32)
        bufs = [x.cuda() for x in (kc, vc, tk, tv, acc, n)]
        dev_bufs.append(bufs)
        host.append((kc, vc, tk, tv, path, S))
        items.append(eb.kv_item(*bufs, S))
    ws = eb.workspace(eb.eagle_kv_commit_workspace_size())
    eb.eagle_kv_commit_batched(items, Hkv, d, eb.EAGLE_BF16, ws=ws)
    assert eb.workspace_error(ws) == (0, 0)
    for (kc, vc, tk, tv, path, S), bufs in zip(host, dev_bufs):
        ko, vo, _ = kv_commit(_as_np(kc), _as_np(vc), S, _as_np(tk), _as_np(tv), path, len(path) - 1)
        assert np.array_equal(_as_np(bufs[0].cpu()), ko) and np.array_equal(_as_np(bufs[1].cpu()), vo)


def test_device_values_out_of_range_are_reported_and_skipped():
    m, Hkv, d, S = 8, 2, 64, 4
    kc, vc, tk, tv = _caches(7, Hkv, S + 3, d, m, torch.bfloat16)
    ws = eb.workspace(eb.eagle_kv_commit_workspace_size())
    # n_accepted too large for the cache capacity (3 free rows): nothing is written
    kd, vd = kc.cuda(), vc.cuda()
    acc = torch.tensor([0, 1, 2, 3, 4, 5, 6, 7], dtype=torch.int32, device="cuda")
    eb.eagle_kv_commit(kd, vd, tk.cuda(), tv.cuda(), acc, torch.tensor([5], dtype=torch.int32,
                       device="cuda"), S, ws=ws)
    st, _ = eb.workspace_error(ws)
    assert st == eb.EAGLE_ERR_DEVICE_ASSERT
    assert torch.equal(kd.cpu(), kc) and torch.equal(vd.cpu(), vc)
    # an accepted id outside the tree: that row is skipped, the others are written
    ws = eb.workspace(eb.eagle_kv_commit_workspace_size())
    kd, vd = kc.cuda(), vc.cuda()
    acc = torch.tensor([0, 99, 3, 0, 0, 0, 0, 0], dtype=torch.int32, device="cuda")
    eb.eagle_kv_commit(kd, vd, tk.cuda(), tv.cuda(), acc, torch.tensor([2], dtype=torch.int32,
                       device="cuda"), S, ws=ws)
    st, _ = eb.workspace_error(ws)
    assert st == eb.EAGLE_ERR_DEVICE_ASSERT
    kg = kd.cpu()
    assert torch.equal(kg[:, S], tk[0]) and torch.equal(kg[:, S + 1], kc[:, S + 1])
    assert torch.equal(kg[:, S + 2], tk[3])


def test_rejects_bad_arguments():
    m, Hkv, S = 4, 2, 2
    kc, vc, tk, tv = _caches(1, Hkv, S + m, 4, m, torch.bfloat16)   # head_dim 4: 8-byte rows
    acc = torch.zeros(m, dtype=torch.int32, device="cuda")
    n = torch.zeros(1, dtype=torch.int32, device="cuda")
    with pytest.raises(eb.EagleError):
        eb.eagle_kv_commit(kc.cuda(), vc.cuda(), tk.cuda(), tv.cuda(), acc, n, S)
