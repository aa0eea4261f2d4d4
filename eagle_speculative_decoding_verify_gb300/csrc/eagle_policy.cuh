// Breadth-first walk of the tree-shape policies over per-row top-K records.
//
// Sources: "Support Eagle-3 Speculative Decoding in llama.cpp", the reply on
// PR #3624 (static expansion: n candidates at every decoding step) and the
// proposal of batched candidate sequences; "EAGLE-2: Feature-Level
// Speculative Decoding Guide", "Context-Aware Dynamic Tree Construction in
// EAGLE-2" (confidence C = P(y1) / P(y2): above tau a chain, otherwise 2 to 4
// branches; chains up to 7 deep).
//
// Nodes are numbered breadth-first (depth, then parent, then the child's rank
// in its parent's row) and draft row i is node i's draft output.  Static
// tree: every node above depth D gets its row's n best tokens.  Chains: the
// root gets row 0's n best, every chain then grows by its last node's best
// token until depth D.  Confidence: a node above the maximum depth gets one
// child when l1 - l2 > ln tau, else its row's b best tokens with b the number
// of tokens within a factor tau of the best (at least 2, at most the width);
// nodes are expanded in order while the tree has fewer than m_cap nodes.
// Ties were already broken by the records (value desc, token id asc); ln tau
// and the logit gaps are compared in fp64, where the gap of two fp32 logits is
// exact.
//
// Plain C++ on purpose: the same function runs in one thread of the policy
// kernel and compiles for the host.
#pragma once

#include <stdint.h>

#ifdef __CUDACC__
#define EAGLE_HD __host__ __device__
#else
#define EAGLE_HD
#endif

namespace eagle {

enum : int { kPolicyStatic = 0, kPolicyChains = 1, kPolicyConfidence = 2 };

struct PolicyWalk {
  int kind, width, depth;   // depth: static / chains depth, confidence maximum depth
  double ln_tau;
  int m_cap;                // node slots (root included)
  int root_token;
  int n_rows;               // rows available: a node at or past it is not expanded
  int ks;                   // entries kept per row in rv / ri (row 0 also in root_*)
};

// Row r's entry c (value desc, token asc); row 0 keeps all K entries apart.
struct PolicyRows {
  const float* root_v;
  const int* root_i;
  const float* rv;
  const int* ri;
};

EAGLE_HD inline float policy_val(const PolicyWalk& P, const PolicyRows& R, int r, int c) {
  return r == 0 ? R.root_v[c] : R.rv[r * P.ks + c];
}
EAGLE_HD inline int policy_tok(const PolicyWalk& P, const PolicyRows& R, int r, int c) {
  return r == 0 ? R.root_i[c] : R.ri[r * P.ks + c];
}

// Fills par / tok / dep for nodes 0 .. n-1 and returns n (<= m_cap).  Sets
// *short_rows when a node it would expand has no row (the host rules this out).
EAGLE_HD inline int policy_walk(const PolicyWalk& P, const PolicyRows& R, int* par, int* tok,
                                int* dep, int* short_rows) {
  int m = 1;
  par[0] = -1;
  tok[0] = P.root_token;
  dep[0] = 0;
  *short_rows = 0;
  auto add = [&](int parent, int token) {
    par[m] = parent;
    tok[m] = token;
    dep[m] = dep[parent] + 1;
    ++m;
  };
  if (P.kind == kPolicyStatic) {
    for (int i = 0; i < m && m < P.m_cap; ++i) {
      if (dep[i] >= P.depth) continue;
      if (i >= P.n_rows) {
        *short_rows = 1;
        break;
      }
      for (int c = 0; c < P.width && m < P.m_cap; ++c) add(i, policy_tok(P, R, i, c));
    }
  } else if (P.kind == kPolicyChains) {
    if (P.depth >= 1)
      for (int c = 0; c < P.width && m < P.m_cap; ++c) add(0, policy_tok(P, R, 0, c));
    for (int d = 2; d <= P.depth; ++d)
      for (int j = 0; j < P.width && m < P.m_cap; ++j) {
        const int p = 1 + (d - 2) * P.width + j;   // chain j's node at depth d - 1
        if (p >= P.n_rows) {
          *short_rows = 1;
          return m;
        }
        add(p, policy_tok(P, R, p, 0));
      }
  } else {
    for (int i = 0; i < m && m < P.m_cap; ++i) {
      if (dep[i] >= P.depth) continue;
      if (i >= P.n_rows) {
        *short_rows = 1;
        break;
      }
      const double best = static_cast<double>(policy_val(P, R, i, 0));
      int b = 1;
      if (!(best - static_cast<double>(policy_val(P, R, i, 1)) > P.ln_tau)) {
        b = 2;
        while (b < P.width && best - static_cast<double>(policy_val(P, R, i, b)) <= P.ln_tau) ++b;
      }
      for (int c = 0; c < b && m < P.m_cap; ++c) add(i, policy_tok(P, R, i, c));
    }
  }
  return m;
}

}  // namespace eagle
