"""Host-only checks of the C ABI: the library loads, exports every symbol
declared in include/eagle.h, and rejects bad arguments on the host before
touching the GPU (no compute calls here: this runs without a GPU)."""

import ctypes
import os
import re

import pytest

from eagle_speculative_decoding_verify_gb300 import binding as eb

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "eagle.h")


def _declared():
    text = open(HEADER).read()
    return sorted(set(re.findall(r"^\s*(?:const\s+char\s*\*|eagle_status|size_t|int32_t)\s+"
                                 r"(eagle_\w+)\s*\(", text, re.M)))


@pytest.fixture(scope="module")
def lib():
    import __graft_entry__
    __graft_entry__.build()
    return eb.lib()


def test_every_declared_symbol_is_exported(lib):
    names = _declared()
    assert len(names) >= 14
    for n in names:
        assert hasattr(lib, n), n
    assert set(names) <= set(eb.EXPORTS), set(names) - set(eb.EXPORTS)


def test_build_id_is_the_hash_of_the_sources(lib):
    from eagle_speculative_decoding_verify_gb300 import _build
    bid = lib.eagle_build_id().decode()
    assert len(bid) == 16 and bid == _build.source_hash()
    assert _build.up_to_date()


def test_status_strings_and_version(lib):
    assert lib.eagle_version() >= 1
    for code in range(7):
        assert lib.eagle_status_string(code).decode()
    assert lib.eagle_status_string(99) == b"unknown status"


def test_workspace_sizes_are_host_only_and_positive(lib):
    assert eb.eagle_tree_build_workspace_size(1, 51, 128256, 10, 6, 60) > 0
    assert eb.eagle_tree_verify_workspace_size(16, 60, 128256) > 0
    assert eb.eagle_tree_attn_workspace_size(60, 28, 4, 128, 8192, eb.EAGLE_BF16) >= 256
    a = eb.eagle_tree_build_workspace_size(2, 51, 128256, 10, 6, 60)
    b = eb.eagle_tree_build_workspace_size(1, 51, 128256, 10, 6, 60)
    assert a > b


def _fake_tree(m=16):
    fake = 1 << 20   # never dereferenced: validation fails first
    return eb.CTree(fake, fake, fake, fake, fake, 0, m, (m + 63) // 64)


@pytest.mark.parametrize("kwargs,status", [
    (dict(logits=0), 1),                          # null logits
    (dict(top_k=0), 1),
    (dict(top_k=65), 2),                          # above the library limit
    (dict(depth=17), 2),
    (dict(total_tokens=300), 2),
    (dict(row_stride=1001), 1),                   # not a multiple of 4
    (dict(n_rows=3), 1),                          # fewer rows than the tree needs
    (dict(ws_bytes=64), 3),                       # workspace too small
])
def test_build_rejects_bad_arguments_before_launch(lib, kwargs, status):
    args = dict(logits=1 << 20, row_stride=1000, n_rows=9, vocab=1000, top_k=4, depth=3,
                total_tokens=16, ws_bytes=1 << 30)
    args.update(kwargs)
    st = lib.eagle_tree_build(ctypes.c_void_p(args["logits"]), args["row_stride"], args["n_rows"],
                              args["vocab"], args["top_k"], args["depth"], args["total_tokens"], 0,
                              _fake_tree(args["total_tokens"]), ctypes.c_void_p(1 << 21),
                              args["ws_bytes"], None)
    assert st == status


def test_verify_rejects_bad_sampling(lib):
    fake = ctypes.c_void_p(1 << 20)
    for samp, status in [(eb.sampling(False, 0.0), 1), (eb.sampling(False, 1.0, 65), 2),
                         (eb.sampling(False, 1.0, 0, 1.5), 1), (eb.sampling(False, 1.0, 0, 0.0), 1)]:
        st = lib.eagle_tree_verify(fake, 1000, 1000, _fake_tree(), ctypes.byref(samp), 0, 0, fake,
                                   fake, fake, ctypes.c_void_p(1 << 21), 1 << 30, None)
        assert st == status
    # a nucleus over the whole vocabulary is limited to 4032 tiles of 1024 tokens
    big = 4081 * 1024
    samp = eb.sampling(False, 1.0, 0, 0.9)
    st = lib.eagle_tree_verify(fake, big, big, _fake_tree(), ctypes.byref(samp), 0, 0, fake,
                               fake, fake, ctypes.c_void_p(1 << 21), 1 << 40, None)
    assert st == 2


def test_attn_rejects_bad_arguments(lib):
    fake = 1 << 20
    base = dict(m=16, hq=4, hkv=2, d=64, S=128, dtype=eb.EAGLE_BF16, stride=128 * 64)
    cases = [(dict(hq=5), 1), (dict(d=256), 2), (dict(m=0), 1), (dict(m=300), 2),
             (dict(stride=100 * 64), 1), (dict(dtype=7), 1)]
    for over, status in cases:
        a = dict(base, **over)
        st = lib.eagle_tree_attn(fake, fake, fake, a["stride"], fake, fake, fake, a["m"], a["hq"],
                                 a["hkv"], a["d"], a["S"], a["dtype"], 0.0, fake,
                                 ctypes.c_void_p(1 << 21), 1 << 30, None)
        assert st == status, over


def test_new_workspace_and_state_sizes_are_host_only(lib):
    assert lib.eagle_kv_commit_workspace_size() >= 16
    a = lib.eagle_tree_state_bytes(10, 6)
    assert a > 0 and a % 16 == 0
    assert lib.eagle_tree_state_bytes(10, 7) > a        # more candidates, more state
    assert lib.eagle_tree_state_bytes(0, 6) == 0
    # the row stream keeps per-CTA candidate buffers: the size grows with top_k, not the vocabulary
    assert lib.eagle_tree_expand_workspace_size(10, 128256) >= 256
    assert lib.eagle_tree_expand_workspace_size(64, 128256) > lib.eagle_tree_expand_workspace_size(4, 128256)


_FAKE = 1 << 20
_FAKE_WS = 1 << 21


@pytest.mark.parametrize("over,status", [
    (dict(k_cache=0), 1),                        # null cache
    (dict(k_cache=_FAKE + 8), 1),                # cache not 16-byte aligned
    (dict(m=0), 1),
    (dict(prefix_len=-1), 1),
    (dict(stride=100), 1),                       # head stride not a multiple of d
    (dict(stride=32), 1),                        # head stride below one row
    (dict(d=4), 2),                              # a row of 8 bytes cannot be copied in 16-byte units
    (dict(dtype=7), 1),
    (dict(ws_bytes=8), 1),
])
def test_kv_commit_rejects_bad_arguments(lib, over, status):
    a = dict(k_cache=_FAKE, stride=64 * 64, prefix_len=5, m=9, hkv=2, d=64, dtype=eb.EAGLE_BF16,
             ws_bytes=1 << 12)
    a.update(over)
    st = lib.eagle_kv_commit(ctypes.c_void_p(a["k_cache"]), ctypes.c_void_p(_FAKE), a["stride"],
                             a["prefix_len"], ctypes.c_void_p(_FAKE), ctypes.c_void_p(_FAKE), a["m"],
                             a["hkv"], a["d"], a["dtype"], ctypes.c_void_p(_FAKE),
                             ctypes.c_void_p(_FAKE), ctypes.c_void_p(_FAKE_WS), a["ws_bytes"], None)
    assert st == status, over


def test_kv_commit_batched_checks_every_item(lib):
    good = eb.CKvItem(_FAKE, _FAKE, _FAKE, _FAKE, _FAKE, _FAKE, 64 * 64, 5, 9)
    bad = eb.CKvItem(_FAKE, _FAKE, _FAKE, 0, _FAKE, _FAKE, 64 * 64, 5, 9)   # null tree_v
    arr = (eb.CKvItem * 3)(good, good, bad)
    st = lib.eagle_kv_commit_batched(arr, 3, 2, 64, eb.EAGLE_BF16, ctypes.c_void_p(_FAKE_WS), 1 << 12,
                                     None)
    assert st == 1
    assert lib.eagle_kv_commit_batched(arr, 0, 2, 64, eb.EAGLE_BF16, ctypes.c_void_p(_FAKE_WS),
                                       1 << 12, None) == 1


@pytest.mark.parametrize("over,status", [
    (dict(rows=0), 1),
    (dict(level=3), 1),                          # level must be below depth
    (dict(level=-1), 1),
    (dict(top_k=65), 2),
    (dict(top_k=1001), 2),                       # more children than the vocabulary
    (dict(depth=17), 2),
    (dict(row_stride=1002), 1),                  # not a multiple of 4
    (dict(row_stride=996), 1),                   # shorter than a row
    (dict(ws_bytes=64), 3),
])
def test_tree_expand_rejects_bad_arguments(lib, over, status):
    a = dict(rows=_FAKE, row_stride=1000, vocab=1000, top_k=4, depth=3, level=0, ws_bytes=1 << 30)
    a.update(over)
    st = lib.eagle_tree_expand(ctypes.c_void_p(a["rows"]), a["row_stride"], a["vocab"], a["top_k"],
                               a["depth"], a["level"], ctypes.c_void_p(_FAKE), None,
                               ctypes.c_void_p(_FAKE_WS), a["ws_bytes"], None)
    assert st == status, over


@pytest.mark.parametrize("over,status", [
    (dict(state=0), 1),
    (dict(top_k=0), 1),
    (dict(total_tokens=38), 2),                  # above 1 + the 4 + 2*16 candidates of top_k 4, depth 3
    (dict(total_tokens=300), 2),                 # above the tree limit
    (dict(out_m=8), 1),                          # output arrays sized for another tree
    (dict(ws_bytes=4), 1),
])
def test_tree_finalize_rejects_bad_arguments(lib, over, status):
    a = dict(state=_FAKE, top_k=4, depth=3, total_tokens=10, out_m=None, ws_bytes=1 << 12)
    a.update(over)
    out = _fake_tree(a["out_m"] or a["total_tokens"])
    st = lib.eagle_tree_finalize(ctypes.c_void_p(a["state"]), a["top_k"], a["depth"],
                                 a["total_tokens"], 7, out, ctypes.c_void_p(_FAKE_WS), a["ws_bytes"],
                                 None)
    assert st == status, over


def _paged(**over):
    f = dict(q=_FAKE, k_pool=_FAKE, v_pool=_FAKE, block_table=_FAKE, tree_k=_FAKE, tree_v=_FAKE,
             mask=_FAKE, out=_FAKE, pool_head_stride=4 * 128 * 64, prefix_len=300, m=16)
    f.update(over)
    return eb.CAttnPagedItem(**f)


@pytest.mark.parametrize("item,shape,status", [
    (dict(m=0), {}, 1),
    (dict(m=300), {}, 2),
    (dict(block_table=0), {}, 1),                # a prefix needs a page table
    (dict(k_pool=_FAKE + 4), {}, 1),             # pool not 16-byte aligned
    (dict(pool_head_stride=100 * 64), {}, 1),    # fewer rows per head than one page
    (dict(q=0), {}, 1),
    (dict(), dict(hq=5), 1),                     # query heads not a multiple of KV heads
    (dict(), dict(d=96), 2),                     # head size the kernel does not take
])
def test_attn_paged_rejects_bad_arguments(lib, item, shape, status):
    s = dict(hq=4, hkv=2, d=64)
    s.update(shape)
    arr = (eb.CAttnPagedItem * 2)(_paged(), _paged(**item))
    st = lib.eagle_tree_attn_paged_batched(arr, 2, s["hq"], s["hkv"], s["d"], 0.125,
                                           ctypes.c_void_p(_FAKE_WS), 1 << 30, None)
    assert st == status, (item, shape)
    assert lib.eagle_tree_attn_paged_workspace_size(arr, 2, s["hq"], s["hkv"], s["d"]) == 0


def test_attn_paged_without_prefix_needs_no_pool(lib):
    arr = (eb.CAttnPagedItem * 1)(_paged(k_pool=0, v_pool=0, block_table=0, prefix_len=0))
    assert lib.eagle_tree_attn_paged_workspace_size(arr, 1, 4, 2, 64) >= 256


@pytest.mark.parametrize("pol,m,n_rows,status", [
    (dict(kind=0, width=2, depth=3), 14, 7, 1),        # static tree of 15 nodes, not 14
    (dict(kind=0, width=2, depth=3), 15, 6, 1),        # 7 inner nodes need 7 rows
    (dict(kind=0, width=2, depth=8), 511, 255, 2),     # past the tree limit
    (dict(kind=0, width=65, depth=1), 66, 1, 2),       # width above the top-k limit
    (dict(kind=1, width=3, depth=0), 1, 1, 1),         # chains need depth >= 1
    (dict(kind=1, width=3, depth=4), 12, 10, 1),       # chains of 13 nodes, not 12
    (dict(kind=1, width=3, depth=4), 13, 9, 1),        # 10 rows needed
    (dict(kind=2, width=1, depth=7, tau=2.0), 20, 19, 1),   # confidence width >= 2
    (dict(kind=2, width=9, depth=7, tau=2.0), 20, 19, 2),   # ... and <= 8
    (dict(kind=2, width=4, depth=7, tau=0.0), 20, 19, 1),   # tau > 0
    (dict(kind=2, width=4, depth=7, tau=float("inf")), 20, 19, 1),
    (dict(kind=2, width=4, depth=7, tau=2.0), 20, 18, 1),   # m - 1 rows needed
    (dict(kind=3, width=4, depth=7, tau=2.0), 20, 19, 1),   # unknown policy
])
def test_policy_build_rejects_bad_arguments(lib, pol, m, n_rows, status):
    p = eb.tree_policy(pol["kind"], pol["width"], pol["depth"], pol.get("tau", 2.0))
    st = lib.eagle_tree_build_policy(ctypes.c_void_p(_FAKE), 1000, n_rows, 1000, ctypes.byref(p),
                                     m, 0, _fake_tree(m), None, ctypes.c_void_p(_FAKE_WS), 1 << 30,
                                     None)
    assert st == status, (pol, m, n_rows)


def test_policy_workspace_sizes(lib):
    ok = eb.tree_policy(eb.EAGLE_POLICY_CONFIDENCE, 4, 7, 2.0)
    assert eb.eagle_tree_policy_workspace_size(152064, ok, 60) > 0
    bad = eb.tree_policy(eb.EAGLE_POLICY_STATIC, 2, 3)
    assert eb.eagle_tree_policy_workspace_size(1000, bad, 14) == 0
    assert eb.eagle_tree_policy_workspace_size(1000, bad, 15) > 0
