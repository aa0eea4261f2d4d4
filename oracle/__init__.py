"""Plain fp64 CPU oracle for one EAGLE-2 verify step.

TEST INFRASTRUCTURE ONLY.  Nothing on the product path imports this package:
only the tests, the smoke check and the timed CPU baseline of the bench may
use it.  It shares no code with the CUDA library (no kernels, tables, helpers
or constants); the only thing both sides consume is the seeded input
generator, which holds none of the method's arithmetic.

Every function follows the definitions on the source pages and cites them by
page title and section:

* "EAGLE-2: Feature-Level Speculative Decoding Guide" (blog post) --
  "The Recurrent Feature Drafting Step" (next-token distribution is the
  softmax of the LM-head logits), "Context-Aware Dynamic Tree Construction"
  and "Single-Pass Tree Verification" (ancestor-only tree attention mask,
  root-to-leaf acceptance walk, lossless output).
* "Support Eagle-3 Speculative Decoding in llama.cpp" (discussion thread) --
  the reply that describes the dynamic tree as valued by draft confidence,
  expanded per step and pruned at the end of drafting, and the acceptance /
  rejection (speculative sampling) strategy for draft tokens.
* "EAGLE-2 Speculative Decoding Support for llama.cpp - Phase 1" (PR text) --
  "Performance Notes": mixed sampling = temperature + top_k + top_p.

Precision: fp64 throughout.  Decisions taken on derived floating-point values
(node values, acceptance tests, nucleus cut, inverse-CDF threshold) record
their margin; a margin within 1e-6 relative is a near tie that is reported,
not silently passed (see ``near_tie``).

Pins: every function is checked in ``tests/test_oracle_*.py`` against facts
fixed independently of this code (hand-worked examples, closed forms, brute
force, library routines, an external Philox implementation).
"""

from . import philox, near_tie, tree_build, tree_attn, verify, kv_commit, kv_fp8  # noqa: F401
