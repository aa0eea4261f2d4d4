// Test harness: runs the policy kernel's breadth-first walk (eagle_policy.cuh,
// plain C++) on the host.  Reads one case from stdin -- the walk parameters,
// then row 0's K entries and every row's ks entries as "hexfloat token"
// pairs in (value desc, token asc) order -- and prints "n short_rows" and
// then "parent token depth" per node.
#include <cstdio>
#include <vector>

#include "eagle_policy.cuh"

int main() {
  eagle::PolicyWalk P;
  int K = 0;
  if (scanf("%d %d %d %la %d %d %d %d %d", &P.kind, &P.width, &P.depth, &P.ln_tau, &P.m_cap,
            &P.root_token, &P.n_rows, &P.ks, &K) != 9)
    return 1;
  std::vector<float> root_v(K), rv(static_cast<size_t>(P.n_rows) * P.ks);
  std::vector<int> root_i(K), ri(rv.size());
  for (int c = 0; c < K; ++c)
    if (scanf("%a %d", &root_v[c], &root_i[c]) != 2) return 1;
  for (size_t e = 0; e < rv.size(); ++e)
    if (scanf("%a %d", &rv[e], &ri[e]) != 2) return 1;
  const eagle::PolicyRows R{root_v.data(), root_i.data(), rv.data(), ri.data()};
  std::vector<int> par(256), tok(256), dep(256);
  int short_rows = 0;
  const int m = eagle::policy_walk(P, R, par.data(), tok.data(), dep.data(), &short_rows);
  printf("%d %d\n", m, short_rows);
  for (int i = 0; i < m; ++i) printf("%d %d %d\n", par[i], tok[i], dep[i]);
  return 0;
}
