"""Thin Python binding of the C ABI in include/eagle.h (argument marshalling
only: every step of the path runs in the library's CUDA kernels).

The functions carry the C names.  Tensors are torch tensors on the current
CUDA device; workspaces are uint8 tensors that the binding allocates
zero-filled when the caller passes none.  If the library is missing the
first call raises: there is no fallback path.
"""

import ctypes
import os

import torch

LIB_PATH = os.path.join(os.path.dirname(os.path.abspath(__file__)), "libeagle.so")

EAGLE_OK = 0
EAGLE_ERR_WORKSPACE_TOO_SMALL = 3
EAGLE_ERR_TIMEOUT = 5
EAGLE_ERR_DEVICE_ASSERT = 6
STATUS_NAMES = {0: "ok", 1: "invalid argument", 2: "unsupported shape",
                3: "workspace too small", 4: "CUDA error", 5: "device wait timed out",
                6: "device invariant violated"}
EAGLE_F32 = 0
EAGLE_BF16 = 1
EAGLE_NOALLOC_SCRATCH_BYTES = 16 * 1024   # include/eagle.h
EAGLE_KV_PAGE_TOKENS = 128
MAX_TOP_K = 64
MAX_DEPTH = 16
MAX_CANDIDATES = 2048
MAX_TREE = 256
MAX_BATCH = 32


class EagleError(RuntimeError):
    def __init__(self, status, what):
        super().__init__(f"{what}: {STATUS_NAMES.get(status, status)} ({status})")
        self.status = status


class CTree(ctypes.Structure):
    _fields_ = [("parents", ctypes.c_void_p), ("tokens", ctypes.c_void_p),
                ("depth", ctypes.c_void_p), ("pos", ctypes.c_void_p),
                ("mask", ctypes.c_void_p), ("values", ctypes.c_void_p),
                ("m", ctypes.c_int32), ("mask_words", ctypes.c_int32)]


class CSampling(ctypes.Structure):
    _fields_ = [("greedy", ctypes.c_int32), ("temperature", ctypes.c_float),
                ("top_k", ctypes.c_int32), ("top_p", ctypes.c_float)]


class CAttnItem(ctypes.Structure):
    _fields_ = [("q", ctypes.c_void_p), ("k_cache", ctypes.c_void_p),
                ("v_cache", ctypes.c_void_p), ("tree_k", ctypes.c_void_p),
                ("tree_v", ctypes.c_void_p), ("mask", ctypes.c_void_p),
                ("out", ctypes.c_void_p), ("cache_head_stride", ctypes.c_int64),
                ("prefix_len", ctypes.c_int32), ("m", ctypes.c_int32)]


class CAttnPagedItem(ctypes.Structure):
    _fields_ = [("q", ctypes.c_void_p), ("k_pool", ctypes.c_void_p), ("v_pool", ctypes.c_void_p),
                ("block_table", ctypes.c_void_p), ("tree_k", ctypes.c_void_p),
                ("tree_v", ctypes.c_void_p), ("mask", ctypes.c_void_p), ("out", ctypes.c_void_p),
                ("pool_head_stride", ctypes.c_int64), ("prefix_len", ctypes.c_int32),
                ("m", ctypes.c_int32)]


class CAttnFp8Item(ctypes.Structure):
    _fields_ = [("q", ctypes.c_void_p), ("k_cache", ctypes.c_void_p), ("v_cache", ctypes.c_void_p),
                ("k_scale", ctypes.c_void_p), ("v_scale", ctypes.c_void_p),
                ("tree_k", ctypes.c_void_p), ("tree_v", ctypes.c_void_p), ("mask", ctypes.c_void_p),
                ("out", ctypes.c_void_p), ("cache_head_stride", ctypes.c_int64),
                ("scale_head_stride", ctypes.c_int64), ("prefix_len", ctypes.c_int32),
                ("m", ctypes.c_int32)]


class CTreePolicy(ctypes.Structure):
    _fields_ = [("kind", ctypes.c_int32), ("width", ctypes.c_int32), ("depth", ctypes.c_int32),
                ("reserved", ctypes.c_int32), ("tau", ctypes.c_double)]


EAGLE_POLICY_STATIC, EAGLE_POLICY_CHAINS, EAGLE_POLICY_CONFIDENCE = 0, 1, 2


class CKvItem(ctypes.Structure):
    _fields_ = [("k_cache", ctypes.c_void_p), ("v_cache", ctypes.c_void_p),
                ("tree_k", ctypes.c_void_p), ("tree_v", ctypes.c_void_p),
                ("accepted", ctypes.c_void_p), ("n_accepted", ctypes.c_void_p),
                ("cache_head_stride", ctypes.c_int64), ("prefix_len", ctypes.c_int32),
                ("m", ctypes.c_int32)]


_P = ctypes.c_void_p
_I32 = ctypes.c_int32
_I64 = ctypes.c_int64
_U64 = ctypes.c_uint64
_SZ = ctypes.c_size_t
_F = ctypes.c_float

EXPORTS = {
    "eagle_status_string": (ctypes.c_char_p, [_I32]),
    "eagle_version": (_I32, []),
    "eagle_build_id": (ctypes.c_char_p, []),
    "eagle_tree_build_noalloc_error": (_I32, [_P, ctypes.POINTER(_I32), ctypes.POINTER(_I32)]),
    "eagle_workspace_init": (_I32, [_P, _SZ, _P]),
    "eagle_workspace_error": (_I32, [_P, _P, ctypes.POINTER(_I32), ctypes.POINTER(_I32)]),
    "eagle_tree_build_workspace_size": (_SZ, [_I32, _I32, _I32, _I32, _I32, _I32]),
    "eagle_tree_build": (_I32, [_P, _I64, _I32, _I32, _I32, _I32, _I32, _I32, CTree, _P, _SZ, _P]),
    "eagle_tree_build_batched": (_I32, [_I32, _P, _I64, _I32, _I32, _I32, _I32, _I32, _P, _P,
                                        _P, _SZ, _P]),
    "eagle_tree_build_noalloc": (_I32, [_P, _I64, _I32, _I32, _I32, _I32, _I32, _I32, CTree,
                                        _P]),
    "eagle_tree_attn_workspace_size": (_SZ, [_I32, _I32, _I32, _I32, _I32, _I32]),
    "eagle_tree_attn": (_I32, [_P, _P, _P, _I64, _P, _P, _P, _I32, _I32, _I32, _I32, _I32, _I32,
                               _F, _P, _P, _SZ, _P]),
    "eagle_tree_attn_batched_workspace_size": (_SZ, [_P, _I32, _I32, _I32, _I32, _I32]),
    "eagle_tree_attn_num_launches": (_I32, [_P, _I32, _I32, _I32, _I32, _I32]),
    "eagle_tree_attn_batched": (_I32, [_P, _I32, _I32, _I32, _I32, _I32, _F, _P, _SZ, _P]),
    "eagle_tree_verify_workspace_size": (_SZ, [_I32, _I32, _I32]),
    "eagle_tree_verify": (_I32, [_P, _I64, _I32, CTree, ctypes.POINTER(CSampling), _U64, _U64,
                                 _P, _P, _P, _P, _SZ, _P]),
    "eagle_tree_verify_batched": (_I32, [_I32, _P, _I64, _I32, _P, _P, _P, _U64, _P, _P, _P,
                                         _P, _SZ, _P]),
    "eagle_tree_attn_paged_workspace_size": (_SZ, [_P, _I32, _I32, _I32, _I32]),
    "eagle_tree_attn_paged_batched": (_I32, [_P, _I32, _I32, _I32, _I32, _F, _P, _SZ, _P]),
    "eagle_tree_attn_fp8_workspace_size": (_SZ, [_P, _I32, _I32, _I32, _I32]),
    "eagle_tree_attn_fp8_batched": (_I32, [_P, _I32, _I32, _I32, _I32, _F, _P, _SZ, _P]),
    "eagle_tree_state_bytes": (_SZ, [_I32, _I32]),
    "eagle_tree_expand_workspace_size": (_SZ, [_I32, _I32]),
    "eagle_tree_expand": (_I32, [_P, _I64, _I32, _I32, _I32, _I32, _P, _P, _P, _SZ, _P]),
    "eagle_tree_finalize": (_I32, [_P, _I32, _I32, _I32, _I32, CTree, _P, _SZ, _P]),
    "eagle_tree_policy_workspace_size": (_SZ, [_I32, ctypes.POINTER(CTreePolicy), _I32]),
    "eagle_tree_build_policy": (_I32, [_P, _I64, _I32, _I32, ctypes.POINTER(CTreePolicy), _I32,
                                       _I32, CTree, _P, _P, _SZ, _P]),
    "eagle_kv_commit_workspace_size": (_SZ, []),
    "eagle_kv_commit": (_I32, [_P, _P, _I64, _I32, _P, _P, _I32, _I32, _I32, _I32, _P, _P, _P,
                               _SZ, _P]),
    "eagle_kv_commit_batched": (_I32, [_P, _I32, _I32, _I32, _I32, _P, _SZ, _P]),
}

_lib = None


def lib():
    """The loaded C library (raises if it was not built)."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(f"{LIB_PATH} is missing: build it first "
                               "(python -c 'import __graft_entry__ as g; g.build()')")
        handle = ctypes.CDLL(LIB_PATH)
        for name, (res, args) in EXPORTS.items():
            fn = getattr(handle, name)
            fn.restype = res
            fn.argtypes = args
        from . import _build
        built = handle.eagle_build_id().decode()
        if os.path.isdir(_build.CSRC) and built != _build.source_hash():
            raise RuntimeError(f"{LIB_PATH} was built from other sources (build id {built}, "
                               f"sources {_build.source_hash()}): rebuild it "
                               "(python -c 'import __graft_entry__ as g; g.build()')")
        _lib = handle
    return _lib


def build_id():
    """Hash of the sources the loaded library was built from."""
    return lib().eagle_build_id().decode()


def _check(status, what):
    if status != EAGLE_OK:
        raise EagleError(status, what)


def _stream(stream):
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream)


def _on(t):
    """Make t's device current for the call (the library works on the current
    device, and its default stream is that device's current stream)."""
    return torch.cuda.device(t.device if isinstance(t, torch.Tensor) else t)


def _ptr(t):
    return ctypes.c_void_p(t.data_ptr()) if t is not None else ctypes.c_void_p(0)


def workspace(nbytes, device=None):
    """Zero-filled uint8 workspace of at least nbytes (256-byte aligned)."""
    return torch.zeros(max(int(nbytes), 256), dtype=torch.uint8,
                       device=device or torch.device("cuda"))


def eagle_workspace_init(ws, stream=None):
    """Zero-fill a workspace on the stream (what every call's workspace needs
    once, and again after a recorded device error)."""
    _check(lib().eagle_workspace_init(_ptr(ws), ws.numel() * ws.element_size(), _stream(stream)),
           "eagle_workspace_init")


def workspace_test_hook(ws, no_copies=False, wait_us=0):
    """Set the workspace header's test hook (words 2 and 3): with no_copies the
    attention kernel's producers issue no copy, so every consumer wait runs out
    after wait_us microseconds and the call records EAGLE_ERR_TIMEOUT.  Test use
    only; eagle_workspace_init clears it."""
    hdr = ws[:16].view(torch.int32)
    hdr[2] = 1 if no_copies else 0
    hdr[3] = int(wait_us)


def workspace_error(ws, stream=None):
    st, detail = _I32(0), _I32(0)
    _check(lib().eagle_workspace_error(_ptr(ws), _stream(stream), ctypes.byref(st),
                                       ctypes.byref(detail)), "eagle_workspace_error")
    return st.value, detail.value


class Tree:
    """Device arrays of one draft tree (see eagle_tree in include/eagle.h)."""

    def __init__(self, m, device=None, with_values=True):
        dev = device or torch.device("cuda")
        self.m = int(m)
        self.mask_words = (self.m + 63) // 64
        self.parents = torch.empty(self.m, dtype=torch.int32, device=dev)
        self.tokens = torch.empty(self.m, dtype=torch.int32, device=dev)
        self.depth = torch.empty(self.m, dtype=torch.int32, device=dev)
        self.pos = torch.empty(self.m, dtype=torch.int32, device=dev)
        self.mask = torch.empty(self.m * self.mask_words, dtype=torch.int64, device=dev)
        self.values = torch.empty(self.m, dtype=torch.float64, device=dev) if with_values else None

    def c(self):
        return CTree(self.parents.data_ptr(), self.tokens.data_ptr(), self.depth.data_ptr(),
                     self.pos.data_ptr(), self.mask.data_ptr(),
                     self.values.data_ptr() if self.values is not None else 0,
                     self.m, self.mask_words)

    @staticmethod
    def from_arrays(parents, tokens, device=None):
        """Tree with given parents/tokens (other arrays left unset)."""
        parents = torch.as_tensor(parents, dtype=torch.int32)
        t = Tree(parents.numel(), device, with_values=False)
        t.parents.copy_(parents)
        t.tokens.copy_(torch.as_tensor(tokens, dtype=torch.int32))
        return t

    def mask_u64(self):
        """mask as a host numpy uint64 array [m, mask_words]."""
        return self.mask.cpu().numpy().view("uint64").reshape(self.m, self.mask_words)


# ------------------------------------------------------------------ build
def eagle_tree_build_workspace_size(n_items, n_rows, vocab, top_k, depth, total_tokens):
    return lib().eagle_tree_build_workspace_size(n_items, n_rows, vocab, top_k, depth,
                                                 total_tokens)


def eagle_tree_build(draft_logits, top_k, depth, total_tokens, root_token, out=None, ws=None,
                     stream=None):
    """draft_logits: fp32 CUDA tensor [n_rows, vocab] (row stride may exceed vocab)."""
    n_rows, vocab = draft_logits.shape
    out = out or Tree(total_tokens, draft_logits.device)
    if ws is None:
        ws = workspace(eagle_tree_build_workspace_size(1, n_rows, vocab, top_k, depth,
                                                       total_tokens), draft_logits.device)
    with _on(draft_logits):
        _check(lib().eagle_tree_build(_ptr(draft_logits), draft_logits.stride(0), n_rows, vocab,
                                      top_k, depth, total_tokens, int(root_token), out.c(), _ptr(ws),
                                      ws.numel(), _stream(stream)), "eagle_tree_build")
    return out


def tree_policy(kind, width, depth, tau=2.0):
    return CTreePolicy(int(kind), int(width), int(depth), 0, float(tau))


def eagle_tree_policy_workspace_size(vocab, policy, total_tokens):
    return lib().eagle_tree_policy_workspace_size(int(vocab), ctypes.byref(policy),
                                                  int(total_tokens))


def eagle_tree_build_policy(draft_logits, policy, total_tokens, root_token, out=None,
                            n_nodes=None, ws=None, stream=None):
    """draft_logits: fp32 CUDA tensor [n_rows, vocab]; policy: tree_policy(...).
    Returns (tree with total_tokens node slots, device int32 [1] tree size)."""
    n_rows, vocab = draft_logits.shape
    dev = draft_logits.device
    out = out or Tree(total_tokens, dev, with_values=False)
    n_nodes = n_nodes if n_nodes is not None else torch.zeros(1, dtype=torch.int32, device=dev)
    if ws is None:
        ws = workspace(eagle_tree_policy_workspace_size(vocab, policy, total_tokens), dev)
    with _on(draft_logits):
        _check(lib().eagle_tree_build_policy(_ptr(draft_logits), draft_logits.stride(0), n_rows,
                                             vocab, ctypes.byref(policy), total_tokens,
                                             int(root_token), out.c(), _ptr(n_nodes), _ptr(ws),
                                             ws.numel(), _stream(stream)), "eagle_tree_build_policy")
    return out, n_nodes


def eagle_tree_build_noalloc(draft_logits, top_k, depth, total_tokens, root_token, out=None,
                             stream=None):
    """eagle_tree_build on the library's fixed static scratch (no workspace);
    calls on one device must not overlap on the GPU."""
    n_rows, vocab = draft_logits.shape
    out = out or Tree(total_tokens, draft_logits.device)
    with _on(draft_logits):
        _check(lib().eagle_tree_build_noalloc(_ptr(draft_logits), draft_logits.stride(0), n_rows,
                                              vocab, top_k, depth, total_tokens, int(root_token),
                                              out.c(), _stream(stream)), "eagle_tree_build_noalloc")
    return out


def eagle_tree_build_noalloc_error(stream=None):
    """(status, detail) of the static scratch's error word after the last
    eagle_tree_build_noalloc call on the current device (synchronises)."""
    st, detail = _I32(0), _I32(0)
    _check(lib().eagle_tree_build_noalloc_error(_stream(stream), ctypes.byref(st),
                                                ctypes.byref(detail)),
           "eagle_tree_build_noalloc_error")
    return st.value, detail.value


def eagle_tree_build_batched(draft_logits, top_k, depth, total_tokens, root_tokens, outs=None,
                             ws=None, stream=None):
    """draft_logits: list of fp32 CUDA tensors [n_rows, vocab], same shape/stride."""
    n = len(draft_logits)
    n_rows, vocab = draft_logits[0].shape
    outs = outs or [Tree(total_tokens, draft_logits[0].device) for _ in range(n)]
    if ws is None:
        ws = workspace(eagle_tree_build_workspace_size(n, n_rows, vocab, top_k, depth,
                                                       total_tokens), draft_logits[0].device)
    ptrs = (ctypes.c_void_p * n)(*[t.data_ptr() for t in draft_logits])
    roots = (ctypes.c_int32 * n)(*[int(r) for r in root_tokens])
    trees = (CTree * n)(*[o.c() for o in outs])
    with _on(draft_logits[0]):
        _check(lib().eagle_tree_build_batched(n, ptrs, draft_logits[0].stride(0), n_rows, vocab,
                                              top_k, depth, total_tokens, roots, trees, _ptr(ws),
                                              ws.numel(), _stream(stream)),
               "eagle_tree_build_batched")
    return outs


# -------------------------------------------------------------- attention
def _dtype_code(t):
    if t.dtype == torch.float32:
        return EAGLE_F32
    if t.dtype == torch.bfloat16:
        return EAGLE_BF16
    raise TypeError(f"unsupported dtype {t.dtype}")


def attn_item(q, k_cache, v_cache, tree_k, tree_v, mask, out, prefix_len=None):
    """C item for one attention problem (k/v cache [Hkv, cap, d])."""
    S = k_cache.shape[1] if prefix_len is None else int(prefix_len)
    return CAttnItem(q.data_ptr(), k_cache.data_ptr(), v_cache.data_ptr(), tree_k.data_ptr(),
                     tree_v.data_ptr(), mask.data_ptr(), out.data_ptr(), k_cache.stride(0), S,
                     q.shape[0])


def eagle_tree_attn_workspace_size(m, n_q_heads, n_kv_heads, head_dim, prefix_len, dtype):
    return lib().eagle_tree_attn_workspace_size(m, n_q_heads, n_kv_heads, head_dim, prefix_len,
                                                dtype)


def eagle_tree_attn(q, k_cache, v_cache, tree_k, tree_v, mask, prefix_len=None, scale=0.0,
                    out=None, ws=None, stream=None):
    """q [m, Hq, d]; k/v_cache [Hkv, cap, d]; tree_k/v [m, Hkv, d]; mask int64 [m * W].
    Returns fp32 [m, Hq, d]."""
    m, hq, d = q.shape
    hkv = k_cache.shape[0]
    S = k_cache.shape[1] if prefix_len is None else int(prefix_len)
    dt = _dtype_code(q)
    out = out if out is not None else torch.empty(m, hq, d, dtype=torch.float32, device=q.device)
    if ws is None:
        ws = workspace(eagle_tree_attn_workspace_size(m, hq, hkv, d, S, dt), q.device)
    with _on(q):
        _check(lib().eagle_tree_attn(_ptr(q), _ptr(k_cache), _ptr(v_cache), k_cache.stride(0),
                                     _ptr(tree_k), _ptr(tree_v), _ptr(mask), m, hq, hkv, d, S, dt,
                                     float(scale), _ptr(out), _ptr(ws), ws.numel(), _stream(stream)),
               "eagle_tree_attn")
    return out


def eagle_tree_attn_batched_workspace_size(items, n_q_heads, n_kv_heads, head_dim, dtype):
    arr = (CAttnItem * len(items))(*items)
    return lib().eagle_tree_attn_batched_workspace_size(arr, len(items), n_q_heads, n_kv_heads,
                                                        head_dim, dtype)


def eagle_tree_attn_num_launches(items, n_q_heads, n_kv_heads, head_dim, dtype):
    arr = (CAttnItem * len(items))(*items)
    return lib().eagle_tree_attn_num_launches(arr, len(items), n_q_heads, n_kv_heads, head_dim,
                                              dtype)


def eagle_tree_attn_batched(items, n_q_heads, n_kv_heads, head_dim, dtype, scale=0.0, ws=None,
                            stream=None, device=None):
    """items: list of CAttnItem (see attn_item)."""
    arr = (CAttnItem * len(items))(*items)
    if ws is None:
        ws = workspace(eagle_tree_attn_batched_workspace_size(items, n_q_heads, n_kv_heads,
                                                              head_dim, dtype), device)
    _check(lib().eagle_tree_attn_batched(arr, len(items), n_q_heads, n_kv_heads, head_dim,
                                         dtype, float(scale), _ptr(ws), ws.numel(),
                                         _stream(stream)), "eagle_tree_attn_batched")


# ----------------------------------------------------------------- verify
def eagle_tree_verify_workspace_size(n_items, m, vocab):
    return lib().eagle_tree_verify_workspace_size(n_items, m, vocab)


def sampling(greedy=True, temperature=1.0, top_k=0, top_p=1.0):
    return CSampling(int(bool(greedy)), float(temperature), int(top_k), float(top_p))


def eagle_tree_verify(target_logits, tree, params=None, seed=0, step=0, accepted=None,
                      n_accepted=None, bonus_token=None, ws=None, stream=None):
    """target_logits fp32 [m, vocab].  Returns (accepted [m], n_accepted [1], bonus [1])
    as int32 CUDA tensors."""
    m, vocab = target_logits.shape
    dev = target_logits.device
    params = params or sampling()
    accepted = accepted if accepted is not None else torch.full((m,), -1, dtype=torch.int32,
                                                                device=dev)
    n_accepted = n_accepted if n_accepted is not None else torch.zeros(1, dtype=torch.int32,
                                                                       device=dev)
    bonus_token = bonus_token if bonus_token is not None else torch.zeros(1, dtype=torch.int32,
                                                                          device=dev)
    if ws is None:
        ws = workspace(eagle_tree_verify_workspace_size(1, m, vocab), dev)
    with _on(target_logits):
        _check(lib().eagle_tree_verify(_ptr(target_logits), target_logits.stride(0), vocab, tree.c(),
                                       ctypes.byref(params), seed, step, _ptr(accepted),
                                       _ptr(n_accepted), _ptr(bonus_token), _ptr(ws), ws.numel(),
                                       _stream(stream)), "eagle_tree_verify")
    return accepted, n_accepted, bonus_token


def eagle_tree_verify_batched(target_logits, trees, params, seeds, step=0, accepted=None,
                              n_accepted=None, bonus_tokens=None, ws=None, stream=None):
    n = len(target_logits)
    m, vocab = target_logits[0].shape
    dev = target_logits[0].device
    accepted = accepted or [torch.full((m,), -1, dtype=torch.int32, device=dev) for _ in range(n)]
    n_accepted = n_accepted if n_accepted is not None else torch.zeros(n, dtype=torch.int32,
                                                                       device=dev)
    bonus_tokens = bonus_tokens if bonus_tokens is not None else torch.zeros(n, dtype=torch.int32,
                                                                             device=dev)
    if ws is None:
        ws = workspace(eagle_tree_verify_workspace_size(n, m, vocab), dev)
    lp = (ctypes.c_void_p * n)(*[t.data_ptr() for t in target_logits])
    tr = (CTree * n)(*[t.c() for t in trees])
    pa = (CSampling * n)(*params)
    sd = (ctypes.c_uint64 * n)(*[int(s) for s in seeds])
    ac = (ctypes.c_void_p * n)(*[a.data_ptr() for a in accepted])
    with _on(target_logits[0]):
        _check(lib().eagle_tree_verify_batched(n, lp, target_logits[0].stride(0), vocab, tr, pa, sd,
                                               step, ac, _ptr(n_accepted), _ptr(bonus_tokens),
                                               _ptr(ws), ws.numel(), _stream(stream)),
               "eagle_tree_verify_batched")
    return accepted, n_accepted, bonus_tokens


# ----------------------------------------------------------------- KV commit
def eagle_kv_commit_workspace_size():
    return lib().eagle_kv_commit_workspace_size()


def kv_item(k_cache, v_cache, tree_k, tree_v, accepted, n_accepted, prefix_len):
    """C item for one commit (k/v cache [Hkv, cap, d], rows contiguous)."""
    return CKvItem(k_cache.data_ptr(), v_cache.data_ptr(), tree_k.data_ptr(), tree_v.data_ptr(),
                   accepted.data_ptr(), n_accepted.data_ptr(), k_cache.stride(0),
                   int(prefix_len), tree_k.shape[0])


def eagle_kv_commit(k_cache, v_cache, tree_k, tree_v, accepted, n_accepted, prefix_len, ws=None,
                    stream=None):
    """Append the accepted path (node ids ``accepted``, *n_accepted + 1 of them,
    both device int32) of tree_k/v [m, Hkv, d] to k/v_cache [Hkv, cap, d] at
    rows prefix_len ..; returns nothing (the caches are updated in place)."""
    hkv, _, d = k_cache.shape
    if ws is None:
        ws = workspace(eagle_kv_commit_workspace_size(), k_cache.device)
    with _on(k_cache):
        _check(lib().eagle_kv_commit(_ptr(k_cache), _ptr(v_cache), k_cache.stride(0), int(prefix_len),
                                     _ptr(tree_k), _ptr(tree_v), tree_k.shape[0], hkv, d,
                                     _dtype_code(k_cache), _ptr(accepted), _ptr(n_accepted), _ptr(ws),
                                     ws.numel(), _stream(stream)), "eagle_kv_commit")


def eagle_kv_commit_batched(items, n_kv_heads, head_dim, dtype, ws=None, stream=None, device=None):
    """items: list of CKvItem (see kv_item)."""
    arr = (CKvItem * len(items))(*items)
    if ws is None:
        ws = workspace(eagle_kv_commit_workspace_size(), device)
    _check(lib().eagle_kv_commit_batched(arr, len(items), n_kv_heads, head_dim, dtype, _ptr(ws),
                                         ws.numel(), _stream(stream)), "eagle_kv_commit_batched")


# ----------------------------------------------------------- incremental build
class TreeGrowth:
    """Device state of one drafting round of eagle_tree_expand calls."""

    def __init__(self, top_k, depth, vocab, device=None):
        dev = device or torch.device("cuda")
        self.top_k, self.depth, self.vocab = int(top_k), int(depth), int(vocab)
        self.state = torch.zeros(max(int(lib().eagle_tree_state_bytes(top_k, depth)), 16),
                                 dtype=torch.uint8, device=dev)
        self.ws = workspace(lib().eagle_tree_expand_workspace_size(top_k, vocab), dev)
        self.frontier = torch.zeros(2, top_k, dtype=torch.int32, device=dev)

    def expand(self, rows, level, stream=None):
        """rows: fp32 [1 or top_k, V] with a row stride that is a multiple of 4.
        Returns the new frontier (device int32 [2, top_k]: tokens, parent slots)."""
        with _on(rows):
            _check(lib().eagle_tree_expand(_ptr(rows), rows.stride(0), rows.shape[1], self.top_k,
                                           self.depth, int(level), _ptr(self.state),
                                           _ptr(self.frontier), _ptr(self.ws), self.ws.numel(),
                                           _stream(stream)), "eagle_tree_expand")
        return self.frontier

    def finalize(self, total_tokens, root_token, out=None, stream=None):
        out = out or Tree(total_tokens, self.state.device)
        with _on(self.state):
            _check(lib().eagle_tree_finalize(_ptr(self.state), self.top_k, self.depth,
                                             int(total_tokens), int(root_token), out.c(),
                                             _ptr(self.ws), self.ws.numel(), _stream(stream)),
                   "eagle_tree_finalize")
        return out


# ----------------------------------------------------------- paged prefix
def attn_paged_item(q, k_pool, v_pool, block_table, tree_k, tree_v, mask, out, prefix_len):
    """C item for one attention problem over a paged prefix (pools [Hkv, rows, d],
    block_table device int32 page ids of the prefix's 128-token pages)."""
    return CAttnPagedItem(q.data_ptr(), k_pool.data_ptr(), v_pool.data_ptr(),
                          block_table.data_ptr(), tree_k.data_ptr(), tree_v.data_ptr(),
                          mask.data_ptr(), out.data_ptr(), k_pool.stride(0), int(prefix_len),
                          q.shape[0])


def eagle_tree_attn_paged_batched(items, n_q_heads, n_kv_heads, head_dim, scale=0.0, ws=None,
                                  stream=None, device=None):
    """items: list of CAttnPagedItem (see attn_paged_item)."""
    arr = (CAttnPagedItem * len(items))(*items)
    if ws is None:
        ws = workspace(lib().eagle_tree_attn_paged_workspace_size(arr, len(items), n_q_heads,
                                                                  n_kv_heads, head_dim), device)
    _check(lib().eagle_tree_attn_paged_batched(arr, len(items), n_q_heads, n_kv_heads, head_dim,
                                               float(scale), _ptr(ws), ws.numel(),
                                               _stream(stream)), "eagle_tree_attn_paged_batched")
    return ws


# ------------------------------------------------------------- E4M3 prefix
def attn_fp8_item(q, k_codes, v_codes, k_scale, v_scale, tree_k, tree_v, mask, out,
                  prefix_len=None):
    """C item for one attention problem over an E4M3 prefix cache: codes uint8
    [Hkv, cap, d], scales float32 [Hkv, pages] (one per 128-token page)."""
    S = k_codes.shape[1] if prefix_len is None else int(prefix_len)
    return CAttnFp8Item(q.data_ptr(), k_codes.data_ptr(), v_codes.data_ptr(), k_scale.data_ptr(),
                        v_scale.data_ptr(), tree_k.data_ptr(), tree_v.data_ptr(), mask.data_ptr(),
                        out.data_ptr(), k_codes.stride(0), k_scale.stride(0), S, q.shape[0])


def eagle_tree_attn_fp8_batched(items, n_q_heads, n_kv_heads, head_dim, scale=0.0, ws=None,
                                stream=None, device=None):
    """items: list of CAttnFp8Item (see attn_fp8_item)."""
    arr = (CAttnFp8Item * len(items))(*items)
    if ws is None:
        ws = workspace(lib().eagle_tree_attn_fp8_workspace_size(arr, len(items), n_q_heads,
                                                                n_kv_heads, head_dim), device)
    _check(lib().eagle_tree_attn_fp8_batched(arr, len(items), n_q_heads, n_kv_heads, head_dim,
                                             float(scale), _ptr(ws), ws.numel(), _stream(stream)),
           "eagle_tree_attn_fp8_batched")
    return ws
