// eagle_tree_build_policy: draft logits -> a tree of a fixed-shape or
// confidence-ratio policy (static tree, batched candidate chains, confidence
// ratio; see eagle_policy.cuh for the rules and their sources), one launch.
//
// Phase 1 (the row stream of eagle_rowstream.cuh): one HBM pass over the rows
// the policy can read -> each row's best K logits and tokens (K = the
// policy's width, no sums).  Phase 2 (the CTA whose row arrives last): the
// records are gathered into shared memory, one thread walks the policy
// breadth-first, and the block writes the node arrays and ancestor masks.
#include <cmath>

#include "eagle_policy.cuh"
#include "eagle_stream_host.h"

namespace eagle {

constexpr int kPolicyMaxConfWidth = 8;   // confidence policy: branches per node
static_assert(EAGLE_POLICY_STATIC == kPolicyStatic && EAGLE_POLICY_CHAINS == kPolicyChains &&
                  EAGLE_POLICY_CONFIDENCE == kPolicyConfidence,
              "policy kinds of the header and of the walk");

struct PolicyArgs {
  RowStream rs;
  PolicyWalk walk;
  eagle_tree out;
  int32_t* n_nodes;   // optional
};

static __device__ __noinline__ void assemble_policy(const PolicyArgs& A, StreamSmem& S) {
  const int tid = threadIdx.x;
  const int K = A.rs.rec_k;
  const int rb = rec_bytes(K);
  const int R = A.rs.rows_per_item;
  const PolicyWalk& W = A.walk;
  const char* rows = A.rs.rows;

  // scratch carved from the idle ring (16-byte aligned pieces; <= 20 KB)
  char* p = reinterpret_cast<char*>(S.ring);
  auto carve = [&p](size_t bytes) {
    char* q = p;
    p += align_up(bytes, 16);
    return q;
  };
  float* root_v = reinterpret_cast<float*>(carve(sizeof(float) * K));
  int* root_i = reinterpret_cast<int*>(carve(sizeof(int) * K));
  float* rv = reinterpret_cast<float*>(carve(sizeof(float) * R * W.ks));
  int* ri = reinterpret_cast<int*>(carve(sizeof(int) * R * W.ks));
  int* par = reinterpret_cast<int*>(carve(sizeof(int) * EAGLE_MAX_TREE));
  int* tok = reinterpret_cast<int*>(carve(sizeof(int) * EAGLE_MAX_TREE));
  int* dep = reinterpret_cast<int*>(carve(sizeof(int) * EAGLE_MAX_TREE));
  int* nn = reinterpret_cast<int*>(carve(sizeof(int) * 4));

  for (int c = tid; c < K; c += kThreads) {
    root_v[c] = __ldcg(rec_val(const_cast<char*>(rows)) + c);
    root_i[c] = __ldcg(rec_idx(const_cast<char*>(rows), K) + c);
  }
  for (int e = tid; e < R * W.ks; e += kThreads) {
    const int r = e / W.ks, c = e - r * W.ks;
    char* rec = const_cast<char*>(rows) + static_cast<int64_t>(r) * rb;
    rv[e] = __ldcg(rec_val(rec) + c);
    ri[e] = __ldcg(rec_idx(rec, K) + c);
  }
  __syncthreads();
  if (tid == 0) {
    PolicyRows rr;
    rr.root_v = root_v;
    rr.root_i = root_i;
    rr.rv = rv;
    rr.ri = ri;
    int short_rows = 0;
    nn[0] = policy_walk(W, rr, par, tok, dep, &short_rows);
    if (short_rows) record_error(A.rs.err, kDevAssert, 70);
  }
  __syncthreads();
  const int m = nn[0];
  const eagle_tree out = A.out;
  // node arrays; slots past the tree's size: parent -1, token -1, depth 0, no mask bits
  for (int i = tid; i < out.m; i += kThreads) {
    const bool in = i < m;
    out.parents[i] = in ? par[i] : -1;
    out.tokens[i] = in ? tok[i] : -1;
    out.depth[i] = in ? dep[i] : 0;
    out.pos[i] = in ? dep[i] : 0;
  }
  const int MW = out.mask_words;
  for (int i = tid; i < out.m; i += kThreads) {
    uint64_t w0 = 0, w1 = 0, w2 = 0, w3 = 0;
    if (i < m) {
      int q = i;
      for (int guard = 0; q >= 0 && guard < EAGLE_MAX_TREE; ++guard) {
        const uint64_t bit = 1ull << (q & 63);
        const int wi = q >> 6;
        w0 |= wi == 0 ? bit : 0ull;
        w1 |= wi == 1 ? bit : 0ull;
        w2 |= wi == 2 ? bit : 0ull;
        w3 |= wi == 3 ? bit : 0ull;
        q = par[q];
      }
    }
    uint64_t* dst = out.mask + static_cast<int64_t>(i) * MW;
    dst[0] = w0;
    if (MW > 1) dst[1] = w1;
    if (MW > 2) dst[2] = w2;
    if (MW > 3) dst[3] = w3;
  }
  if (tid == 0 && A.n_nodes) *A.n_nodes = m;
}

__global__ void __launch_bounds__(kThreads, 2) policy_kernel(const __grid_constant__ PolicyArgs A) {
  extern __shared__ __align__(128) char smem_raw[];
  StreamSmem& S = *reinterpret_cast<StreamSmem*>(smem_raw);
  const int PC = A.rs.ctas_per_row;
  pdl_trigger();
  pdl_wait();
  const RowCtx cx = stream_row(row_job(A.rs, blockIdx.x / PC, static_cast<int>(blockIdx.x % PC)), S);
  if (!cx.leader) return;
  if (item_arrive(A.rs, S, cx.item)) assemble_policy(A, S);
}

static_assert(kScratchBytes >= 8 * 64 + 8 * EAGLE_MAX_TREE * kPolicyMaxConfWidth +
                                   12 * EAGLE_MAX_TREE + 16 * 8,
              "policy scratch must fit in the stream's shared memory");

// Tree size, rows read, record width K and entries kept per row of a policy;
// EAGLE_OK or the status that rejects it.
struct PolicyShape {
  int m, rows, K, ks;
};

static eagle_status policy_shape(const eagle_tree_policy* pol, int32_t vocab,
                                 int32_t total_tokens, PolicyShape* sh) {
  EAGLE_CHECK_ARG(pol != nullptr && vocab >= 1 && total_tokens >= 1);
  EAGLE_CHECK_SHAPE(total_tokens <= EAGLE_MAX_TREE);
  const int w = pol->width, D = pol->depth;
  if (pol->kind == EAGLE_POLICY_STATIC) {
    EAGLE_CHECK_ARG(w >= 1 && D >= 0);
    EAGLE_CHECK_SHAPE(w <= kKMax && w <= vocab);
    // full w-ary tree: 1 + w + ... + w^D nodes, 1 + ... + w^(D-1) of them expanded
    int64_t level = 1, nodes = 1, internal = 0;
    for (int d = 0; d < D; ++d) {
      internal += level;
      level *= w;
      nodes += level;
      EAGLE_CHECK_SHAPE(nodes <= EAGLE_MAX_TREE);
    }
    EAGLE_CHECK_ARG(nodes == total_tokens);
    sh->m = static_cast<int>(nodes);
    sh->rows = internal > 0 ? static_cast<int>(internal) : 1;
    sh->K = w;
    sh->ks = w;
  } else if (pol->kind == EAGLE_POLICY_CHAINS) {
    EAGLE_CHECK_ARG(w >= 1 && D >= 1);
    EAGLE_CHECK_SHAPE(w <= kKMax && w <= vocab);
    EAGLE_CHECK_SHAPE(static_cast<int64_t>(w) * D + 1 <= EAGLE_MAX_TREE);
    EAGLE_CHECK_ARG(1 + w * D == total_tokens);
    sh->m = total_tokens;
    sh->rows = 1 + w * (D - 1);
    sh->K = w;
    sh->ks = 1;
  } else if (pol->kind == EAGLE_POLICY_CONFIDENCE) {
    EAGLE_CHECK_ARG(w >= 2 && D >= 0 && std::isfinite(pol->tau) && pol->tau > 0.0);
    EAGLE_CHECK_SHAPE(w <= kPolicyMaxConfWidth && w <= vocab);
    sh->m = total_tokens;
    sh->rows = total_tokens > 1 ? total_tokens - 1 : 1;   // every node that can expand
    sh->K = w;
    sh->ks = w;
  } else {
    return EAGLE_ERR_INVALID_ARG;
  }
  return EAGLE_OK;
}

}  // namespace eagle

using namespace eagle;

extern "C" size_t eagle_tree_policy_workspace_size(int32_t vocab, const eagle_tree_policy* policy,
                                                   int32_t total_tokens) {
  PolicyShape sh;
  if (policy_shape(policy, vocab, total_tokens, &sh) != EAGLE_OK) return 0;
  return stream_layout(1, sh.rows, vocab, sh.K, false, false).total;
}

extern "C" eagle_status eagle_tree_build_policy(const float* draft_logits, int64_t row_stride,
                                                int32_t n_rows, int32_t vocab,
                                                const eagle_tree_policy* policy,
                                                int32_t total_tokens, int32_t root_token,
                                                eagle_tree out, int32_t* n_nodes, void* ws,
                                                size_t ws_bytes, eagle_stream stream) {
  EAGLE_CHECK_ARG(draft_logits && aligned16(draft_logits) && ws && aligned16(ws));
  EAGLE_CHECK_ARG(vocab >= 1 && n_rows >= 1 && row_stride >= vocab && row_stride % 4 == 0);
  PolicyShape sh;
  const eagle_status st = policy_shape(policy, vocab, total_tokens, &sh);
  if (st != EAGLE_OK) return st;
  EAGLE_CHECK_ARG(n_rows >= sh.rows);
  EAGLE_CHECK_ARG(out.parents && out.tokens && out.depth && out.pos && out.mask);
  EAGLE_CHECK_ARG(out.m == total_tokens && out.mask_words == (total_tokens + 63) / 64);
  const StreamLayout L = stream_layout(1, sh.rows, vocab, sh.K, false, false);
  if (ws_bytes < L.total) return EAGLE_ERR_WORKSPACE_TOO_SMALL;

  PolicyArgs A;
  memset(&A, 0, sizeof(A));
  const int occ = stream_ctas_per_sm(policy_kernel);
  if (occ <= 0) return EAGLE_ERR_CUDA;
  const int ctas = stream_ctas_per_row(policy_kernel, L, occ);
  if (ctas <= 0) return EAGLE_ERR_CUDA;
  fill_stream(A.rs, L, static_cast<char*>(ws), 1, sh.rows, vocab, row_stride, ctas, false);
  A.rs.base[0] = draft_logits;
  A.rs.exp_scale[0] = 1.0f;
  A.rs.topk[0] = static_cast<int16_t>(sh.K);
  A.rs.flags[0] = 0;
  A.walk.kind = policy->kind;
  A.walk.width = policy->width;
  A.walk.depth = policy->depth;
  A.walk.ln_tau = policy->kind == EAGLE_POLICY_CONFIDENCE ? std::log(policy->tau) : 0.0;
  A.walk.m_cap = sh.m;
  A.walk.root_token = root_token;
  A.walk.n_rows = sh.rows;
  A.walk.ks = sh.ks;
  A.out = out;
  A.n_nodes = n_nodes;
  return launch_stream(policy_kernel, A, L.n_rows, ctas, reinterpret_cast<cudaStream_t>(stream));
}
