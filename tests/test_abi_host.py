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
    for samp, status in [(eb.sampling(False, 0.0), 1), (eb.sampling(False, 1.0, 0, 0.9), 2),
                         (eb.sampling(False, 1.0, 65), 2), (eb.sampling(False, 1.0, 0, 1.5), 1)]:
        st = lib.eagle_tree_verify(fake, 1000, 1000, _fake_tree(), ctypes.byref(samp), 0, 0, fake,
                                   fake, fake, ctypes.c_void_p(1 << 21), 1 << 30, None)
        assert st == status


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
