"""Writes the stored expected values under tests/golden/ from the oracle only.

Run from the repository root:  python tests/golden/make_golden.py
The pages print no worked example, so every stored value here is produced by
the oracle (``oracle/``) on a seeded synthetic input; the tests re-derive them
to catch regressions and the GPU tests may compare against them.
"""

import json
import os
import sys

import numpy as np

ROOT = os.path.dirname(os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
sys.path.insert(0, ROOT)

from eagle_speculative_decoding_verify_gb300 import workloads as wl  # noqa: E402
from oracle.tree_build import build_draft_tree  # noqa: E402
from oracle.tree_attn import tree_attention  # noqa: E402
from oracle.verify import verify_tree  # noqa: E402


def tiny_case():
    w = wl.WORKLOADS["c0"]
    draft = wl.draft_logits(w).numpy()
    root = wl.root_token(w)
    t = build_draft_tree(draft, w.top_k, w.depth, w.total_tokens, root)
    target = wl.target_logits(w, t["parents"], t["tokens"]).numpy()
    v = verify_tree(target, t["parents"], t["tokens"])
    a = wl.attention_inputs(w)
    o = tree_attention(*(a[n].double().numpy() for n in ("q", "k_cache", "v_cache", "tree_k", "tree_v")),
                       t["mask"], w.prefix)
    return dict(
        workload="c0 tiny: vocab 1000, top_k 4, depth 3, 16 tokens, 4/2 heads, d 64, prefix 128",
        root_token=root,
        parents=t["parents"].tolist(), tokens=t["tokens"].tolist(), depth=t["depth"].tolist(),
        mask=[[f"{int(x):016x}" for x in row] for row in t["mask"]],
        values=t["values"].tolist(),
        path=v["path"], n_accepted=v["n_accepted"], bonus=v["bonus"],
        attn_row_sums=o.sum(axis=2).tolist(),
        near_ties=t["log"].summary() + v["log"].summary(),
    )


if __name__ == "__main__":
    out = os.path.join(os.path.dirname(os.path.abspath(__file__)), "tiny_step.json")
    with open(out, "w") as f:
        json.dump(tiny_case(), f, indent=1)
    print("wrote", out)
