"""Pins for the oracle's counter-based generator (Philox4x32-10).

The oracle's Philox is checked against an independent implementation of the
same published generator (the one inside the triton package, run by its CPU
interpreter in a child process) on random counters and keys, and its
uniforms are checked for uniformity and 24-bit exactness.
"""

import json
import os
import subprocess
import sys
import textwrap

import numpy as np
import pytest
from scipy import stats

from oracle import philox

pytestmark = pytest.mark.filterwarnings("ignore::DeprecationWarning")

_CHILD = textwrap.dedent(r"""
    import json, os, sys
    os.environ["TRITON_INTERPRET"] = "1"
    import torch, triton, triton.language as tl

    @triton.jit
    def run(c0p, c1p, c2p, c3p, out, seed, N: tl.constexpr):
        i = tl.arange(0, N)
        a, b, c, d = tl.philox(seed, tl.load(c0p + i), tl.load(c1p + i),
                               tl.load(c2p + i), tl.load(c3p + i))
        tl.store(out + 4 * i + 0, a)
        tl.store(out + 4 * i + 1, b)
        tl.store(out + 4 * i + 2, c)
        tl.store(out + 4 * i + 3, d)

    cases = json.loads(sys.stdin.read())
    res = []
    for seed, ctrs in cases:
        cs = [torch.tensor([c[w] for c in ctrs], dtype=torch.int64).to(torch.int32) for w in range(4)]
        cs = [c.view(torch.uint32) if hasattr(torch, "uint32") else c for c in cs]
        out = torch.zeros(4 * len(ctrs), dtype=torch.int32)
        run[(1,)](*cs, out, seed, N=len(ctrs))
        res.append([(int(v) & 0xffffffff) for v in out.tolist()])
    print(json.dumps(res))
""")


def test_philox_matches_independent_implementation():
    pytest.importorskip("triton")
    rng = np.random.default_rng(1234)
    cases = []
    for _ in range(4):
        seed = int(rng.integers(0, 2 ** 63))
        ctrs = [[int(x) for x in rng.integers(0, 2 ** 32, size=4)] for _ in range(16)]
        cases.append([seed, ctrs])
    env = dict(os.environ, TRITON_INTERPRET="1")
    proc = subprocess.run([sys.executable, "-c", _CHILD], input=json.dumps(cases),
                          capture_output=True, text=True, env=env, timeout=600)
    if proc.returncode != 0:
        pytest.skip("triton interpreter unavailable: " + proc.stderr.strip()[-300:])
    theirs = json.loads(proc.stdout.strip().splitlines()[-1])
    for (seed, ctrs), words in zip(cases, theirs):
        for n, ctr in enumerate(ctrs):
            mine = philox.philox4x32_10(ctr, (seed & 0xFFFFFFFF, seed >> 32))
            assert list(mine) == words[4 * n:4 * n + 4], (seed, ctr)


def test_uniforms_are_24_bit_and_uniform():
    us = np.array([philox.uniform(99, 3, node, child)
                   for node in range(200) for child in range(64)])
    scaled = us * 2 ** 24
    assert np.all(scaled == np.floor(scaled)) and us.min() >= 0.0 and us.max() < 1.0
    counts, _ = np.histogram(us, bins=64, range=(0.0, 1.0))
    assert stats.chisquare(counts).pvalue > 1e-3
    assert stats.kstest(us, "uniform").pvalue > 1e-3


def test_key_and_counter_words_all_matter():
    base = philox.uniform(5, 7, 11, 13)
    variants = [philox.uniform(5 + (1 << 40), 7, 11, 13), philox.uniform(5, 7 + (1 << 33), 11, 13),
                philox.uniform(6, 7, 11, 13), philox.uniform(5, 8, 11, 13),
                philox.uniform(5, 7, 12, 13), philox.uniform(5, 7, 11, 14),
                philox.uniform(5, 7, 11, philox.RESIDUAL_CHILD)]
    assert all(v != base for v in variants)
