"""GPU parity of eagle_tree_verify against the oracle (bit-exact accepted
path and bonus token; near ties reported), through the C ABI."""

import numpy as np
import pytest
import torch

from eagle_speculative_decoding_verify_gb300 import binding as eb
from eagle_speculative_decoding_verify_gb300 import workloads as wl
from oracle.tree_build import build_draft_tree
from oracle.verify import verify_tree
from tests.parity import path_matches, to_device_rows

pytestmark = pytest.mark.gpu


def _case(key, item=0):
    w = wl.WORKLOADS[key]
    ref = build_draft_tree(wl.draft_logits(w, item).numpy(), w.top_k, w.depth, w.total_tokens,
                           wl.root_token(w, item))
    target = wl.target_logits(w, ref["parents"], ref["tokens"], item)
    return w, ref, target


def _verify(target, ref, greedy=True, T=1.0, top_k=0, top_p=1.0, seed=0, step=0):
    tree = eb.Tree.from_arrays(ref["parents"], ref["tokens"])
    acc, n, bonus = eb.eagle_tree_verify(to_device_rows(target), tree,
                                         eb.sampling(greedy, T, top_k, top_p), seed, step)
    torch.cuda.synchronize()
    return acc.cpu().numpy(), int(n.item()), int(bonus.item())


@pytest.mark.parametrize("key", ["c0", "c1", "c3"])
def test_greedy_workloads(key):
    w, ref, target = _case(key)
    v = verify_tree(target.numpy(), ref["parents"], ref["tokens"])
    acc, n, bonus = _verify(target, ref)
    path_matches(acc, n, bonus, v, key, ref["parents"], ref["tokens"], target.numpy(),
                 (1, 1.0, 0, 1.0))


def test_greedy_forced_full_chain():
    w, ref, target = _case("c1")
    target = target.clone()
    # force every node's argmax onto its first child: the walk accepts the
    # whole first-child chain
    kids = {}
    for i in range(1, ref["m"]):
        kids.setdefault(int(ref["parents"][i]), []).append(i)
    for p, cs in kids.items():
        target[p, int(ref["tokens"][cs[0]])] = 100.0
    v = verify_tree(target.numpy(), ref["parents"], ref["tokens"])
    acc, n, bonus = _verify(target, ref)
    chain = 0       # length of the first-child chain from the root
    node = 0
    while node in kids:
        node = kids[node][0]
        chain += 1
    assert n == chain
    path_matches(acc, n, bonus, v, "forced chain", ref["parents"], ref["tokens"], target.numpy(),
                 (1, 1.0, 0, 1.0))


@pytest.mark.parametrize("seed", range(8))
def test_sampling_topk_topp_qwen7b(seed):
    w, ref, target = _case("c2")
    _, T, k, p = w.sampling_of(0)
    v = verify_tree(target.numpy(), ref["parents"], ref["tokens"], greedy=False, temperature=T,
                    top_k=k, top_p=p, seed=seed, step=seed * 7)
    acc, n, bonus = _verify(target, ref, False, T, k, p, seed, seed * 7)
    path_matches(acc, n, bonus, v, f"seed{seed}", ref["parents"], ref["tokens"], target.numpy(),
                 (0, T, k, p))


@pytest.mark.parametrize("seed", range(6))
def test_sampling_full_vocab(seed):
    w, ref, target = _case("c4", item=8)
    v = verify_tree(target.numpy(), ref["parents"], ref["tokens"], greedy=False, temperature=1.0,
                    seed=seed, step=3)
    acc, n, bonus = _verify(target, ref, False, 1.0, 0, 1.0, seed, 3)
    path_matches(acc, n, bonus, v, f"full seed{seed}", ref["parents"], ref["tokens"],
                 target.numpy(), (0, 1.0, 0, 1.0))


@pytest.mark.parametrize("T,k,p", [(0.5, 1, 1.0), (1.3, 64, 1.0), (0.9, 7, 0.5), (2.0, 0, 1.0)])
def test_sampling_variants_rejections(T, k, p):
    # flat rows so that children get rejected and residual draws happen
    w = wl.WORKLOADS["c0"]
    ref = build_draft_tree(wl.draft_logits(w).numpy(), w.top_k, w.depth, w.total_tokens, 5)
    g = torch.Generator().manual_seed(17)
    target = torch.randn(w.total_tokens, 5003, generator=g) * 0.7
    for seed in range(12):
        v = verify_tree(target.numpy(), ref["parents"], ref["tokens"], greedy=False,
                        temperature=T, top_k=k, top_p=p, seed=seed, step=1)
        acc, n, bonus = _verify(target, ref, False, T, k, p, seed, 1)
        path_matches(acc, n, bonus, v, f"T{T} k{k} p{p} seed{seed}", ref["parents"],
                     ref["tokens"], target.numpy(), (0, T, k, p))


def test_batched_ragged16_mixed_modes():
    w = wl.WORKLOADS["c4"]
    refs, targets, trees, params = [], [], [], []
    for b in range(w.items):
        _, ref, target = _case("c4", b)
        refs.append(ref)
        targets.append(target)
        trees.append(eb.Tree.from_arrays(ref["parents"], ref["tokens"]))
        gr, T, k, p = w.sampling_of(b)
        params.append(eb.sampling(gr, T, k, p))
    seeds = [1000 + b for b in range(w.items)]
    acc, n, bonus = eb.eagle_tree_verify_batched([t.cuda() for t in targets], trees, params,
                                                 seeds, step=5)
    torch.cuda.synchronize()
    for b in range(w.items):
        gr, T, k, p = w.sampling_of(b)
        v = verify_tree(targets[b].numpy(), refs[b]["parents"], refs[b]["tokens"], greedy=bool(gr),
                        temperature=T, top_k=k, top_p=p, seed=seeds[b], step=5)
        path_matches(acc[b].cpu().numpy(), int(n[b]), int(bonus[b]), v, f"item{b}",
                     refs[b]["parents"], refs[b]["tokens"], targets[b].numpy(), (gr, T, k, p))


def test_single_node_tree():
    g = torch.Generator().manual_seed(3)
    target = torch.randn(1, 3000, generator=g)
    ref = dict(parents=np.array([-1]), tokens=np.array([7]))
    acc, n, bonus = _verify(target, ref)
    assert n == 0 and bonus == int(torch.argmax(target[0]))


# Nucleus over the whole vocabulary (top_p < 1, top_k = 0): the kept set is
# cut by the library's radix select over exact fixed-point masses.
@pytest.mark.parametrize("T,p,scale,vocab", [(1.0, 0.9, 0.7, 5003), (0.7, 0.5, 1.0, 5003),
                                             (1.3, 0.99, 0.5, 12288), (1.0, 0.3, 3.0, 1000)])
def test_nucleus_full_vocab_flat_rows(T, p, scale, vocab):
    w = wl.WORKLOADS["c0"]
    ref = build_draft_tree(wl.draft_logits(w).numpy(), w.top_k, w.depth, w.total_tokens, 5)
    g = torch.Generator().manual_seed(23)
    target = torch.randn(w.total_tokens, vocab, generator=g) * scale
    for seed in range(10):
        v = verify_tree(target.numpy(), ref["parents"], ref["tokens"], greedy=False,
                        temperature=T, top_k=0, top_p=p, seed=seed, step=2)
        acc, n, bonus = _verify(target, ref, False, T, 0, p, seed, 2)
        path_matches(acc, n, bonus, v, f"nucleus T{T} p{p} seed{seed}", ref["parents"],
                     ref["tokens"], target.numpy(), (0, T, 0, p))


@pytest.mark.parametrize("seed", range(3))
def test_nucleus_full_vocab_qwen7b(seed):
    w, ref, target = _case("c2")
    v = verify_tree(target.numpy(), ref["parents"], ref["tokens"], greedy=False, temperature=0.7,
                    top_k=0, top_p=0.9, seed=seed, step=4)
    acc, n, bonus = _verify(target, ref, False, 0.7, 0, 0.9, seed, 4)
    path_matches(acc, n, bonus, v, f"nucleus c2 seed{seed}", ref["parents"], ref["tokens"],
                 target.numpy(), (0, 0.7, 0, 0.9))


def test_nucleus_full_vocab_tied_logits():
    # logits on a grid of 1/8: hundreds of tokens share each value, so the
    # crossing value is shared and the cut falls between equal logits
    # (token ids ascending decide)
    w = wl.WORKLOADS["c0"]
    ref = build_draft_tree(wl.draft_logits(w).numpy(), w.top_k, w.depth, w.total_tokens, 5)
    g = torch.Generator().manual_seed(29)
    target = torch.round(torch.randn(w.total_tokens, 7001, generator=g) * 8.0) / 8.0
    for p in (0.25, 0.6, 0.95):
        for seed in range(6):
            v = verify_tree(target.numpy(), ref["parents"], ref["tokens"], greedy=False,
                            temperature=1.0, top_k=0, top_p=p, seed=seed, step=9)
            acc, n, bonus = _verify(target, ref, False, 1.0, 0, p, seed, 9)
            path_matches(acc, n, bonus, v, f"tied p{p} seed{seed}", ref["parents"],
                         ref["tokens"], target.numpy(), (0, 1.0, 0, p))


# Sampling over target rows built to stress the row stream's top-k (a single
# lane holding a row's best entries, 100 exact copies of a row's maximum, the
# best entries in the unaligned tail of a row, one lane with a raised element
# in every slot): the verify kernel's second pass reloads its threads'
# candidate slots, or for a lane with more qualifying slots than it records
# every qualifying slot of its warp, ahead of absorbing them, which these
# rows exercise at the tie rules' edges.
@pytest.mark.parametrize("kind,V,k,p", [
    ("one_lane", 40000, 50, 1.0),
    ("one_lane", 152064, 2, 1.0),
    ("duplicates", 30000, 50, 1.0),
    ("duplicates", 152064, 64, 0.9),
    ("tail", 5003, 64, 1.0),
    ("tail", 152063, 16, 0.95),
    ("slots", 152064, 50, 1.0),
    ("slots", 152064, 8, 0.9),
])
def test_sampling_on_adversarial_target_rows(kind, V, k, p):
    from tests.test_gpu_build import _adversarial
    g = torch.Generator().manual_seed(V + k)
    draft = torch.randn(51, V, generator=g) * 2.0
    ref = build_draft_tree(draft.numpy(), 10, 6, 60, 3)
    target = _adversarial(kind, 60, V, k, 17)
    for seed in range(2):
        v = verify_tree(target.numpy(), ref["parents"], ref["tokens"], greedy=False,
                        temperature=1.0, top_k=k, top_p=p, seed=seed, step=3)
        acc, n, bonus = _verify(target, ref, False, 1.0, k, p, seed, 3)
        path_matches(acc, n, bonus, v, f"{kind} V{V} k{k} seed{seed}", ref["parents"],
                     ref["tokens"], target.numpy(), (0, 1.0, k, p))
