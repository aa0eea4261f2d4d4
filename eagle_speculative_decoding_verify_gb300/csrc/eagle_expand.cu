// eagle_tree_expand / eagle_tree_finalize: the tree of eagle_tree_build,
// grown one depth per call as the drafting loop produces the draft rows of
// the current frontier.
//
// Source: "Support Eagle-3 Speculative Decoding in llama.cpp", reply on the
// dynamic tree (the draft tree is valued by draft confidence, expanded step
// by step and pruned at the end of drafting); "EAGLE-2: Feature-Level
// Speculative Decoding Guide", "The Recurrent Feature Drafting Step" (the
// draft model runs once per step on the tokens just drafted, so the rows of
// depth l + 1 exist only after the frontier of depth l is known) and
// "Context-Aware Dynamic Tree Construction".
//
// Per call (level L = 0 .. depth - 1): one HBM pass over the call's rows
// (the root's row for L = 0, else the top_k rows of the current frontier in
// frontier-slot order) with the row stream of the one-shot build (top_k and
// logsumexp per row), then in the CTA whose row arrives last: the values of
// the depth-(L+1) candidates (parent value + log-probability), their ranks
// within the depth (value desc, candidate index asc) and the next frontier
// (the top_k of the depth), kept in a caller-owned device state.  The same
// fp64 arithmetic and order as the one-shot build, so the trees are
// identical.  eagle_tree_finalize then takes the final top-(m-1) cut over all
// depths and writes the tree arrays (one CTA).
#include "eagle_stream_host.h"

namespace eagle {

// Device state of a growing tree with C candidates (16-byte aligned arrays):
// key[C] order keys of the fp64 values | tok[C] | par[C] (parent candidate,
// -1 at depth 1) | srt[C] (candidates of each depth, best first) | lrank[C]
// (rank within the depth) | frontier[kKMax] | levels done
struct TreeState {
  uint64_t* key;
  int* tok;
  int* par;
  int* srt;
  int* lrank;
  int* frontier;
  int* levels;
};

__host__ __device__ inline size_t tree_state_bytes_for(int C) {
  return align_up(8 * static_cast<size_t>(C), 16) + 4 * align_up(4 * static_cast<size_t>(C), 16) +
         align_up(4 * static_cast<size_t>(kKMax), 16) + 16;
}

inline TreeState tree_state_view(void* base, int C) {
  char* p = static_cast<char*>(base);
  TreeState T;
  T.key = reinterpret_cast<uint64_t*>(p);
  p += align_up(8 * static_cast<size_t>(C), 16);
  T.tok = reinterpret_cast<int*>(p);
  p += align_up(4 * static_cast<size_t>(C), 16);
  T.par = reinterpret_cast<int*>(p);
  p += align_up(4 * static_cast<size_t>(C), 16);
  T.srt = reinterpret_cast<int*>(p);
  p += align_up(4 * static_cast<size_t>(C), 16);
  T.lrank = reinterpret_cast<int*>(p);
  p += align_up(4 * static_cast<size_t>(C), 16);
  T.frontier = reinterpret_cast<int*>(p);
  p += align_up(4 * static_cast<size_t>(kKMax), 16);
  T.levels = reinterpret_cast<int*>(p);
  return T;
}

struct ExpandArgs {
  RowStream rs;
  TreeState st;
  int top_k, depth, level;
  int warm_stream;      // 1: a stream code warm-up cluster follows the rows' (long rows)
  int32_t* front_out;   // [2][top_k]: tokens and parent slots of the new frontier, or null
};

// The level's candidates, ranks and next frontier (the CTA whose row arrived
// last; the other rows' records are visible through the item counter).
static __device__ __noinline__ void expand_level(const ExpandArgs& A, StreamSmem& S) {
  const int tid = threadIdx.x;
  const int k = A.top_k, L = A.level;
  const TreeState& T = A.st;
  if (L > 0 && *reinterpret_cast<volatile int*>(T.levels) != L) {   // calls out of order
    if (tid == 0) record_error(A.rs.err, kDevAssert, 50);
    return;
  }
  const int n = L == 0 ? 1 : k;                  // rows of this call
  const int rb = rec_bytes(A.rs.rec_k);
  char* rows = A.rs.rows;
  // scratch over the (idle) ring: row logsumexp, row top-k, the level's keys
  double* lse = reinterpret_cast<double*>(S.ring);               // [kKMax]
  float* rv = reinterpret_cast<float*>(lse + kKMax);              // [kKMax * kKMax]
  int* ri = reinterpret_cast<int*>(rv + kKMax * kKMax);           // [kKMax * kKMax]
  uint64_t* lk = reinterpret_cast<uint64_t*>(ri + kKMax * kKMax); // [kKMax * kKMax]
  int* nf = reinterpret_cast<int*>(lk + kKMax * kKMax);           // [kKMax] next frontier
  int* pf = nf + kKMax;                                            // [kKMax] frontier slots
  uint64_t* pkey = reinterpret_cast<uint64_t*>(pf + kKMax);       // [kKMax] their keys
  // the frontier and its keys load beside the row records (not after them)
  if (L > 0 && tid >= kThreads - k) {
    const int sl = tid - (kThreads - k);
    const int pa = T.frontier[sl];
    pf[sl] = pa;
    pkey[sl] = T.key[pa];
  }
  for (int r = tid; r < n; r += kThreads)   // each row's leader put its logsumexp in the record
    lse[r] = reinterpret_cast<const volatile RecHead*>(rows + r * rb)->sum;
  for (int e = tid; e < n * k; e += kThreads) {
    const int r = e / k, c = e - r * k;
    rv[e] = __ldcg(rec_val(rows + r * rb) + c);
    ri[e] = __ldcg(rec_idx(rows + r * rb, A.rs.rec_k) + c);
  }
  __syncthreads();
  // candidates of depth L + 1: the root's top-k, or the children (in draft
  // rank order) of every frontier slot of depth L
  const int cnt = L == 0 ? k : k * k;
  const int base = L == 0 ? 0 : k + (L - 1) * k * k;
  for (int e = tid; e < cnt; e += kThreads) {
    uint64_t key;
    int pa;
    if (L == 0) {
      key = order_key(static_cast<double>(rv[e]) - lse[0]);
      pa = -1;
    } else {
      const int s = e / k, c = e - s * k;
      pa = pf[s];
      key = order_key(key_value(pkey[s]) + (static_cast<double>(rv[s * k + c]) - lse[s]));
    }
    lk[e] = key;
    T.key[base + e] = key;
    T.tok[base + e] = ri[e];
    T.par[base + e] = pa;
  }
  __syncthreads();
  // rank within the depth by counting; the best top_k form the next frontier
  for (int e = tid; e < cnt; e += kThreads) {
    const uint64_t kv = lk[e];
    int r = 0;
    for (int f = 0; f < cnt; ++f) {
      const uint64_t o = lk[f];
      r += ((o > kv) | ((o == kv) & (f < e))) ? 1 : 0;
    }
    T.srt[base + r] = base + e;
    T.lrank[base + e] = r;
    if (r < k) nf[r] = e;
  }
  __syncthreads();
  if (tid < k) {
    const int e = nf[tid];
    T.frontier[tid] = base + e;
    if (A.front_out) {
      A.front_out[tid] = ri[e];
      A.front_out[k + tid] = L == 0 ? 0 : e / k;
    }
  }
  // the next call reads the state after this kernel has completed
  if (tid == 0) *T.levels = L + 1;
}

// Grid: the rows' clusters, then (long rows: stream_warm_up) one cluster that
// streams the short warm-up row through the same code at launch (see
// warm_row_job): after an L2 flush the first launch of a round would
// otherwise fetch that code from HBM in every row's cluster at once.
__global__ void __launch_bounds__(kThreads, 2) expand_kernel(const __grid_constant__ ExpandArgs A) {
  extern __shared__ __align__(128) char smem_raw[];
  StreamSmem& S = *reinterpret_cast<StreamSmem*>(smem_raw);
  const int PC = A.rs.ctas_per_row;
  const int64_t rows = static_cast<int64_t>(A.rs.n_items) * A.rs.rows_per_item;
  const int64_t cl = blockIdx.x / PC;
  const int rank = static_cast<int>(blockIdx.x - cl * PC);
  pdl_trigger();
  const bool warm = cl >= rows;   // (only when warm_stream)
  if (!warm) pdl_wait();          // the warm-up touches no caller memory
  const RowJob R = warm ? warm_row_job(A.rs, rank) : row_job(A.rs, cl, rank);
  const RowCtx cx = stream_row(R, S);
  if (!cx.leader || warm) return;
  // the row's logsumexp replaces the record's sum, here in parallel over the
  // rows, as in the one-shot build (the sum holds the max's own term 1, so its
  // log is >= 0, kept so through the rounding of log_d)
  if (threadIdx.x == 0)
    reinterpret_cast<RecHead*>(R.rec)->sum =
        static_cast<double>(S.rmax) + fmax(0.0, log_d(S.rsum));
  if (item_arrive(A.rs, S, cx.item)) expand_level(A, S);
}

static_assert(kScratchBytes >= 8 * kKMax + (4 + 4 + 8) * kKMax * kKMax + (4 + 4 + 8) * kKMax,
              "expand scratch must fit in the stream's shared memory");

struct FinalArgs {
  TreeState st;
  eagle_tree out;
  int top_k, depth, total_tokens, n_cand, root_token;
  int32_t* err;
};

__device__ __forceinline__ int depth_of(int a, int k) { return a < k ? 1 : 2 + (a - k) / (k * k); }

// The final top-(m-1) cut over all depths and the tree arrays (one CTA).
__global__ void __launch_bounds__(kThreads) finalize_kernel(const __grid_constant__ FinalArgs A) {
  __shared__ uint64_t skey[EAGLE_MAX_CANDIDATES];
  __shared__ int sidx[EAGLE_MAX_CANDIDATES];
  __shared__ int node[EAGLE_MAX_CANDIDATES];
  __shared__ int npar[EAGLE_MAX_TREE];
  __shared__ int warp_tot[kWarps];
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int k = A.top_k, D = A.depth, m = A.total_tokens, C = A.n_cand;
  const int kk = k * k;
  const TreeState& T = A.st;
  const eagle_tree out = A.out;
  pdl_trigger();   // one CTA
  pdl_wait();
  if (*reinterpret_cast<volatile int*>(T.levels) != D) {   // not every depth expanded
    if (tid == 0) record_error(A.err, kDevAssert, 51);
    return;
  }
  // a candidate is kept iff fewer than need = m - 1 candidates come before it:
  // its rank in its own depth plus, for every other depth, the entries before
  // it (binary search over that depth's keys in sorted order, keys and
  // candidate ids both in shared memory: a probe that waited on a global load
  // would cost an L2 round trip)
  for (int i = tid; i < C; i += kThreads) {
    const int c = T.srt[i];
    sidx[i] = c;
    skey[i] = T.key[c];
  }
  __syncthreads();
  const int need = m - 1;
  for (int a = tid; a < C; a += kThreads) {
    const int la = a < k ? 0 : 1 + (a - k) / kk;
    int rank = T.lrank[a];
    const uint64_t kv = T.key[a];
    for (int l = 0; l < D && rank < need; ++l) {
      if (l == la) continue;
      const int lb = l == 0 ? 0 : k + (l - 1) * kk;
      int lo = 0, hi = l == 0 ? k : kk;
      while (lo < hi) {
        const int mid = (lo + hi) >> 1;
        const uint64_t o = skey[lb + mid];
        const bool go = (o > kv) | ((o == kv) & (sidx[lb + mid] < a));
        lo = go ? mid + 1 : lo;
        hi = go ? hi : mid;
      }
      rank += lo;
    }
    node[a] = rank < need ? 1 : 0;
  }
  __syncthreads();
  // node ids: 1 + exclusive count of kept candidates before it
  const int per = (C + kThreads - 1) / kThreads;
  const int a0 = tid * per, a1 = min(C, a0 + per);
  int local = 0;
  for (int a = a0; a < a1; ++a) local += node[a];
  int incl = local;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int y = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += y;
  }
  if (lane == 31) warp_tot[warp] = incl;
  __syncthreads();
  int off = 0, total = 0;
  for (int w = 0; w < kWarps; ++w) {
    if (w < warp) off += warp_tot[w];
    total += warp_tot[w];
  }
  off += incl - local;
  for (int a = a0; a < a1; ++a) node[a] = node[a] ? 1 + off++ : 0;
  __syncthreads();
  if (tid == 0 && total != (need > 0 ? min(need, C) : 0)) record_error(A.err, kDevAssert, 52);
  if (tid == 0) {
    out.parents[0] = -1;
    out.tokens[0] = A.root_token;
    out.depth[0] = 0;
    out.pos[0] = 0;
    if (out.values) out.values[0] = 0.0;
    npar[0] = -1;
  }
  for (int a = tid; a < C; a += kThreads) {
    const int nd = node[a];
    if (!nd) continue;
    int pn = 0;
    if (T.par[a] >= 0) {
      pn = node[T.par[a]];
      if (pn == 0) record_error(A.err, kDevAssert, 53);   // kept set not ancestor-closed
    }
    const int dep = depth_of(a, k);
    out.parents[nd] = pn;
    out.tokens[nd] = T.tok[a];
    out.depth[nd] = dep;
    out.pos[nd] = dep;
    if (out.values) out.values[nd] = key_value(T.key[a]);
    npar[nd] = pn;
  }
  __syncthreads();
  // ancestor masks by walking parents (at most depth + 1 steps)
  const int W = out.mask_words;
  for (int nd = tid; nd < m; nd += kThreads) {
    uint64_t w0 = 0, w1 = 0, w2 = 0, w3 = 0;
    int q = nd;
    for (int guard = 0; q >= 0 && guard <= EAGLE_MAX_DEPTH + 1; ++guard) {
      const uint64_t bit = 1ull << (q & 63);
      const int wi = q >> 6;
      w0 |= wi == 0 ? bit : 0ull;
      w1 |= wi == 1 ? bit : 0ull;
      w2 |= wi == 2 ? bit : 0ull;
      w3 |= wi == 3 ? bit : 0ull;
      q = npar[q];
    }
    uint64_t* dst = out.mask + static_cast<int64_t>(nd) * W;
    dst[0] = w0;
    if (W > 1) dst[1] = w1;
    if (W > 2) dst[2] = w2;
    if (W > 3) dst[3] = w3;
  }
}

static int64_t n_candidates(int top_k, int depth) {
  return top_k + static_cast<int64_t>(depth - 1) * top_k * top_k;
}

}  // namespace eagle

using namespace eagle;

extern "C" size_t eagle_tree_state_bytes(int32_t top_k, int32_t depth) {
  if (top_k < 1 || depth < 1) return 0;
  return tree_state_bytes_for(static_cast<int>(n_candidates(top_k, depth)));
}

extern "C" size_t eagle_tree_expand_workspace_size(int32_t top_k, int32_t vocab) {
  if (top_k < 1 || vocab < 1) return kWsHeader;
  return stream_layout(1, top_k, vocab, top_k, false, false).total;
}

extern "C" eagle_status eagle_tree_expand(const float* rows, int64_t row_stride, int32_t vocab,
                                          int32_t top_k, int32_t depth, int32_t level,
                                          void* state, int32_t* frontier_out, void* ws,
                                          size_t ws_bytes, eagle_stream stream) {
  EAGLE_CHECK_ARG(rows && state && ws && aligned16(rows) && aligned16(state));
  EAGLE_CHECK_ARG(vocab >= 1 && top_k >= 1 && depth >= 1 && level >= 0 && level < depth);
  EAGLE_CHECK_SHAPE(top_k <= kKMax && top_k <= vocab && depth <= EAGLE_MAX_DEPTH);
  EAGLE_CHECK_SHAPE(n_candidates(top_k, depth) <= EAGLE_MAX_CANDIDATES);
  EAGLE_CHECK_ARG(row_stride >= vocab && row_stride % 4 == 0);
  const int n_rows = level == 0 ? 1 : top_k;
  const StreamLayout L = stream_layout(1, n_rows, vocab, top_k, false, false);
  if (ws_bytes < L.total) return EAGLE_ERR_WORKSPACE_TOO_SMALL;
  ExpandArgs A;
  memset(&A, 0, sizeof(A));
  const int occ = stream_ctas_per_sm(expand_kernel);
  if (occ <= 0) return EAGLE_ERR_CUDA;
  const int ctas = stream_ctas_per_row(expand_kernel, L, occ, 1);
  if (ctas <= 0) return EAGLE_ERR_CUDA;
  fill_stream(A.rs, L, static_cast<char*>(ws), 1, n_rows, vocab, row_stride, ctas, false);
  A.rs.base[0] = rows;
  A.rs.exp_scale[0] = 1.0f;
  A.rs.topk[0] = static_cast<int16_t>(top_k);
  A.rs.flags[0] = kWantSum;
  A.st = tree_state_view(state, static_cast<int>(n_candidates(top_k, depth)));
  A.top_k = top_k;
  A.depth = depth;
  A.level = level;
  A.front_out = frontier_out;
  A.warm_stream = stream_warm_up(L.tiles_per_row, ctas) ? 1 : 0;
  return launch_stream(expand_kernel, A, L.n_rows + A.warm_stream, ctas,
                       reinterpret_cast<cudaStream_t>(stream));
}

extern "C" eagle_status eagle_tree_finalize(const void* state, int32_t top_k, int32_t depth,
                                            int32_t total_tokens, int32_t root_token,
                                            eagle_tree out, void* ws, size_t ws_bytes,
                                            eagle_stream stream) {
  EAGLE_CHECK_ARG(state && ws && aligned16(state) && ws_bytes >= kWsHeader);
  EAGLE_CHECK_ARG(top_k >= 1 && depth >= 1 && total_tokens >= 1);
  EAGLE_CHECK_SHAPE(top_k <= kKMax && depth <= EAGLE_MAX_DEPTH);
  const int64_t C = n_candidates(top_k, depth);
  EAGLE_CHECK_SHAPE(C <= EAGLE_MAX_CANDIDATES);
  EAGLE_CHECK_SHAPE(total_tokens <= EAGLE_MAX_TREE && total_tokens <= 1 + C);
  EAGLE_CHECK_ARG(out.parents && out.tokens && out.depth && out.pos && out.mask);
  EAGLE_CHECK_ARG(out.m == total_tokens && out.mask_words == (total_tokens + 63) / 64);
  FinalArgs A;
  memset(&A, 0, sizeof(A));
  A.st = tree_state_view(const_cast<void*>(state), static_cast<int>(C));
  A.out = out;
  A.top_k = top_k;
  A.depth = depth;
  A.total_tokens = total_tokens;
  A.n_cand = static_cast<int>(C);
  A.root_token = root_token;
  A.err = static_cast<int32_t*>(ws);
  if (launch_pdl(finalize_kernel, dim3(1), dim3(kThreads), 0,
                 reinterpret_cast<cudaStream_t>(stream), A) != cudaSuccess) {
    (void)cudaGetLastError();
    return EAGLE_ERR_CUDA;
  }
  return launch_status();
}
