"""The policy kernel's breadth-first walk (csrc/eagle_policy.cuh, plain C++)
compiled for the host and compared with the oracle's tree-shape policies on
random rows, ties and every policy parameter.  The records fed to it are the
rows' best entries in (value desc, token asc) order, as the row stream
delivers them; GPU parity of the whole kernel is in test_gpu_tree_policy.py."""

import math
import os
import shutil
import subprocess

import numpy as np
import pytest

from oracle.tree_policies import candidate_chains, confidence_tree, static_tree, static_tree_size

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
CSRC = os.path.join(ROOT, "eagle_speculative_decoding_verify_gb300", "csrc")


@pytest.fixture(scope="module")
def walk(tmp_path_factory):
    cxx = shutil.which("g++")
    if cxx is None:
        pytest.skip("no host C++ compiler")
    exe = str(tmp_path_factory.mktemp("walk") / "policy_walk")
    subprocess.run([cxx, "-O2", "-std=c++17", "-I", CSRC,
                    os.path.join(ROOT, "tests", "host", "policy_walk_main.cpp"), "-o", exe],
                   check=True)
    return exe


def _run(exe, kind, x, width, depth, ln_tau, m_cap, root, rows, K, ks):
    top = np.argsort(-x[:rows].astype(np.float64), axis=1, kind="stable")[:, :K]
    lines = [f"{kind} {width} {depth} {float(ln_tau).hex()} {m_cap} {root} {rows} {ks} {K}"]
    lines += [f"{float(x[0, t]).hex()} {t}" for t in top[0, :K]]
    lines += [f"{float(x[r, top[r, c]]).hex()} {top[r, c]}" for r in range(rows) for c in range(ks)]
    out = subprocess.run([exe], input="\n".join(lines) + "\n", capture_output=True, text=True,
                         check=True).stdout.split("\n")
    m, short = map(int, out[0].split())
    return m, short, np.array([list(map(int, ln.split())) for ln in out[1:1 + m]])


def test_walk_matches_the_oracle(walk):
    rng = np.random.default_rng(2024)
    for trial in range(240):
        V = int(rng.integers(8, 300))
        x = (rng.standard_normal((260, V)) * rng.choice([0.2, 0.7, 2.0, 5.0])).astype(np.float32)
        if trial % 5 == 0:
            x = (np.round(x * 2) / 2).astype(np.float32)   # many exact ties
        root = int(rng.integers(0, V))
        kind = trial % 3
        if kind == 0:
            w = int(rng.integers(1, min(6, V) + 1))
            D = int(rng.integers(0, 5))
            while static_tree_size(w, D) > 256:
                D -= 1
            ref = static_tree(x, w, D, root)
            rows = max(1, static_tree_size(w, D - 1) if D else 1)
            got = _run(walk, 0, x, w, D, 0.0, ref["m"], root, rows, w, w)
        elif kind == 1:
            w = int(rng.integers(1, min(10, V) + 1))
            D = int(rng.integers(1, 8))
            ref = candidate_chains(x, w, D, root)
            got = _run(walk, 1, x, w, D, 0.0, ref["m"], root, 1 + w * (D - 1), w, 1)
        else:
            w = int(rng.integers(2, min(8, V) + 1))
            D = int(rng.integers(0, 9))
            tau = float(rng.choice([0.5, 1.0, 1.5, 2.0, 3.0, 10.0, 1e30]))
            m_cap = int(rng.integers(1, 257))
            ref = confidence_tree(x, tau, m_cap, root, max_depth=D, max_branch=w)
            got = _run(walk, 2, x, w, D, math.log(tau), m_cap, root, max(1, m_cap - 1), w, w)
        m, short, arr = got
        assert short == 0 and m == ref["m"], (trial, kind, m, ref["m"])
        np.testing.assert_array_equal(arr[:, 0], ref["parents"], err_msg=f"trial {trial}")
        np.testing.assert_array_equal(arr[:, 1], ref["tokens"], err_msg=f"trial {trial}")
        np.testing.assert_array_equal(arr[:, 2], ref["depth"], err_msg=f"trial {trial}")
