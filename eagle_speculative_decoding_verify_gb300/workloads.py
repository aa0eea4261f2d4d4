"""Seeded synthetic workloads for one EAGLE-2 verify step.

This module only draws random inputs with the shapes, sizes and value
distributions of the five reference workloads; it holds none of the method's
arithmetic (no softmax, no top-k, no tree building, no attention).  Both the
CUDA path and the fp64 oracle read the tensors it returns.

Workloads (sizes from the method's target configurations):
  tiny      vocab 1000, top_k 4, depth 3, 16 tree tokens; 4 q / 2 kv heads,
            d 64, fp32 Q/K/V ~ N(0,1), prefix 128; greedy.
  llama8b   vocab 128256, top_k 10, depth 6, 60 tree tokens; 32 q / 8 kv
            heads, d 128, bf16 KV ~ N(0,1), prefix 2048; greedy.
  qwen7b    vocab 152064, same tree; 28 q / 4 kv heads, d 128, bf16, prefix
            8192; sampling T 0.7, top_k 50, top_p 0.9.
  long32    llama8b shapes, prefix 32768, 32 independent layers of KV (layer
            seed = seed*100 + layer); greedy.
  ragged16  16 sequences, each its own tree and logits, prefix lengths uniform
            in [512, 16384]; 64 q / 8 kv heads, d 128, bf16; greedy on
            sequences 0-7, sampling at T 1.0 (no top_k / top_p) on 8-15.

Draft logits: every drafted row is N(0, sigma^2) with sigma drawn per row
from {1, 3, 6}.  Target logits: N(0, 4) (sigma 2) plus +8 on one token per
row: for a node with children, the token of its first child with probability
0.8, otherwise a uniformly drawn token; for a leaf, a uniformly drawn token.
Tensors that the GPU reads in bf16 are rounded once (round-to-nearest-even)
here, so both sides see identical values.
"""

from dataclasses import dataclass

import torch


@dataclass(frozen=True)
class Workload:
    key: str
    name: str
    vocab: int
    top_k: int
    depth: int
    total_tokens: int
    n_q_heads: int
    n_kv_heads: int
    head_dim: int
    prefix: int                 # prefix length (ragged: upper bound)
    dtype: str                  # "f32" or "bf16" for Q/K/V
    seed: int
    items: int = 1              # independent sequences
    layers: int = 1             # independent KV layers sharing one tree
    ragged_min: int = 0         # ragged prefix lower bound (0 = fixed)
    sampling: tuple = ()        # per-item (greedy, temperature, top_k, top_p)

    @property
    def n_rows(self):
        return 1 + (self.depth - 1) * self.top_k

    @property
    def n_candidates(self):
        return self.top_k + (self.depth - 1) * self.top_k * self.top_k

    def sampling_of(self, item):
        return self.sampling[item % len(self.sampling)]


GREEDY = (1, 1.0, 0, 1.0)

WORKLOADS = {
    "c0": Workload("c0", "tiny", 1000, 4, 3, 16, 4, 2, 64, 128, "f32", 7,
                   sampling=(GREEDY,)),
    "c1": Workload("c1", "llama8b", 128256, 10, 6, 60, 32, 8, 128, 2048, "bf16", 1007,
                   sampling=(GREEDY,)),
    "c2": Workload("c2", "qwen7b", 152064, 10, 6, 60, 28, 4, 128, 8192, "bf16", 2007,
                   sampling=((0, 0.7, 50, 0.9),)),
    "c3": Workload("c3", "long32", 128256, 10, 6, 60, 32, 8, 128, 32768, "bf16", 3007,
                   layers=32, sampling=(GREEDY,)),
    "c4": Workload("c4", "ragged16", 128256, 10, 6, 60, 64, 8, 128, 16384, "bf16", 4007,
                   items=16, ragged_min=512,
                   sampling=tuple([GREEDY] * 8 + [(0, 1.0, 0, 1.0)] * 8)),
}

# stream tags: every tensor gets its own generator so generation order and
# shapes of other tensors never change it
_TAG = dict(sigma=1, draft=2, root=3, q=4, k=5, v=6, tree_k=7, tree_v=8,
            target=9, bump=10, ragged=11)


def _gen(seed, tag, item=0, device="cpu"):
    g = torch.Generator(device=device)
    g.manual_seed((int(seed) * 1_000_003 + _TAG[tag] * 10_007 + int(item) * 101) % (2 ** 62))
    return g


def _normal(shape, g, device):
    return torch.randn(shape, generator=g, device=device, dtype=torch.float32)


def prefix_lengths(w):
    """Prefix length of every item (ragged workloads draw them uniformly)."""
    if not w.ragged_min:
        return [w.prefix] * w.items
    g = _gen(w.seed, "ragged")
    return torch.randint(w.ragged_min, w.prefix + 1, (w.items,), generator=g).tolist()


def root_token(w, item=0):
    g = _gen(w.seed, "root", item)
    return int(torch.randint(0, w.vocab, (1,), generator=g).item())


def draft_logits(w, item=0, device="cpu", rows=None):
    """fp32 [R, V]: row r ~ N(0, sigma_r^2), sigma_r uniform over {1, 3, 6}."""
    R = w.n_rows if rows is None else rows
    choices = torch.tensor([1.0, 3.0, 6.0])
    g_sigma = _gen(w.seed, "sigma", item)
    sigma = choices[torch.randint(0, 3, (R,), generator=g_sigma)]
    x = _normal((R, w.vocab), _gen(w.seed, "draft", item, device), device)
    return x * sigma.to(device)[:, None]


def _as_qkv(x, w):
    return x.to(torch.bfloat16) if w.dtype == "bf16" else x


def attention_inputs(w, item=0, layer=0, device="cpu", prefix=None):
    """q [m, Hq, d]; k/v cache [Hkv, S, d]; tree k/v [m, Hkv, d] -- N(0,1),
    bf16-rounded for bf16 workloads."""
    S = w.prefix if prefix is None else prefix
    m, d = w.total_tokens, w.head_dim
    s = w.seed * 100 + layer if w.layers > 1 else w.seed
    return dict(
        q=_as_qkv(_normal((m, w.n_q_heads, d), _gen(s, "q", item, device), device), w),
        k_cache=_as_qkv(_normal((w.n_kv_heads, S, d), _gen(s, "k", item, device), device), w),
        v_cache=_as_qkv(_normal((w.n_kv_heads, S, d), _gen(s, "v", item, device), device), w),
        tree_k=_as_qkv(_normal((m, w.n_kv_heads, d), _gen(s, "tree_k", item, device), device), w),
        tree_v=_as_qkv(_normal((m, w.n_kv_heads, d), _gen(s, "tree_v", item, device), device), w),
    )


def fp8_kv(cache, page=128):
    """A key or value cache [Hkv, S, d] stored as E4M3 codes with one fp32
    scale per (kv head, page of `page` tokens), as a cache writer would store
    it: scale = the page's largest magnitude / 448, code = the value / scale
    rounded by PyTorch's float8_e4m3fn conversion.  Returns (uint8 codes
    [Hkv, S, d], float32 scales [Hkv, ceil(S / page)])."""
    x = cache.to(torch.float32)
    hkv, S, d = x.shape
    n = (S + page - 1) // page
    pad = torch.zeros(hkv, n * page, d, dtype=torch.float32, device=x.device)
    pad[:, :S] = x
    amax = pad.view(hkv, n, page * d).abs().amax(dim=2)
    scales = torch.where(amax > 0, amax / 448.0, torch.ones_like(amax))
    codes = (pad.view(hkv, n, page, d) / scales[:, :, None, None]).to(torch.float8_e4m3fn)
    return codes.view(torch.uint8).reshape(hkv, n * page, d)[:, :S].contiguous(), scales


def target_logits(w, parents, tokens, item=0, device="cpu"):
    """fp32 [m, V]: N(0, 4) plus +8 at the first child's token (p = 0.8) or
    at a uniformly drawn token (otherwise, and always for leaves)."""
    parents = [int(p) for p in parents]
    tokens = [int(t) for t in tokens]
    m = len(parents)
    x = 2.0 * _normal((m, w.vocab), _gen(w.seed, "target", item, device), device)
    g = _gen(w.seed, "bump", item)
    coin = torch.rand((m,), generator=g)
    rand_tok = torch.randint(0, w.vocab, (m,), generator=g)
    first_child = [-1] * m
    for i in range(m - 1, 0, -1):          # lowest node index wins
        first_child[parents[i]] = i
    where = []
    for i in range(m):
        if first_child[i] >= 0 and float(coin[i]) < 0.8:
            where.append(tokens[first_child[i]])
        else:
            where.append(int(rand_tok[i]))
    idx = torch.tensor(where, dtype=torch.long, device=x.device)
    x[torch.arange(m, device=x.device), idx] += 8.0
    return x
