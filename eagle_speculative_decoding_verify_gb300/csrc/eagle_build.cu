// eagle_tree_build: draft logits -> dynamic draft tree, one fused launch.
//
// Sources: "EAGLE-2: Feature-Level Speculative Decoding Guide", "The
// Recurrent Feature Drafting Step" (draft distribution = softmax of the
// LM-head logits; its listing takes the top candidates of that softmax) and
// "Context-Aware Dynamic Tree Construction"; "Support Eagle-3 Speculative
// Decoding in llama.cpp", reply on the dynamic tree (node value = draft
// confidence, tree grown per drafting step and pruned at the end).
//
// Phase 1 (one cluster per row, eagle_rowstream.cuh): one HBM pass over the
// R draft rows -> per row the top_k (value desc, token id asc) and logsumexp.
// Phase 2 (the CTA whose row of an item arrives last): candidate values
// value = parent value + (logit - logsumexp), in fp64; the best m-1 kept
// level by level as one sorted list, merged with each level's children by
// counting (order-preserving 64-bit keys, ties -> lower candidate index); a
// candidate's slot in its level's frontier is its rank among that level's
// kept entries; node ids by rank in candidate order; ancestor mask by
// walking parent pointers (depth <= 16).
#include <cuda.h>
#include <cudaTypedefs.h>

#include <mutex>

#include "eagle_stream_host.h"

namespace eagle {

struct BuildArgs {
  RowStream rs;
  int top_k, depth, total_tokens, n_cand;
  int root_token[kMaxItems];
  eagle_tree out[kMaxItems];
  int warm_stream;  // 1: a stream code warm-up cluster follows the rows' (long rows)
};

// One tree assembly: the item's R row records and its outputs.
struct TreeJob {
  char* rows;        // R records of rec_bytes(rec_k) bytes
  eagle_tree out;
  int32_t* err;
  int rec_k, top_k, depth, total_tokens, n_cand, root_token;
};

// Scratch of the assembly's code warm-up (library-owned, see warm_row_job):
// error word, 3 records of a top-2 row, parents / tokens / depth / pos of 4
// nodes, 4 mask words.
constexpr int kWarmK = 2;
constexpr size_t kWarmBytes = 256;
static_assert(16 + 3 * rec_bytes(kWarmK) + 4 * 16 + 8 * 4 <= kWarmBytes, "warm-up scratch");
static __device__ __align__(16) char g_warm_tree[kWarmBytes];

__device__ __forceinline__ int cand_depth(int a, int k) { return a < k ? 1 : 2 + (a - k) / (k * k); }

// (key, candidate) a before (key, candidate) b: larger value first, then the
// lower candidate index.
__device__ __forceinline__ bool cand_before(uint64_t ka, int ia, uint64_t kb, int ib) {
  return (ka > kb) | ((ka == kb) & (ia < ib));
}

// The tree assembly (all threads of one CTA).  Candidate a of level 1 is
// entry a of row 0; candidate a = k + (l-2) k^2 + s k + c of level l >= 2 is
// entry c of row 1 + (l-2) k + s, the row drafted from the s-th best of level
// l-1 (its slot s): candidate a is row entry a, with offset w = logit -
// logsumexp <= 0 of its row (each row's leader has put the logsumexp, at
// least the row's max, in the record), so a child's value never exceeds its
// parent's and it comes after its parent in (value desc, candidate asc).
//
// The result is the best need = m-1 candidates, kept level by level as a
// sorted list B (the best need of the levels so far; B is a prefix of their
// order).  A candidate of level l+1 can enter B only if its parent is in B:
// otherwise the parent, and so the child, comes after B's last entry.  And a
// candidate of level l in B has every candidate of level l before it in B,
// so its rank in level l -- its slot, if below k -- is the number of level-l
// entries of B before it.  Per level:
//   children: every (B entry of level l with level rank s < k, c < k) gives
//     candidate base + s k + c, value = parent value + w; it is kept (list Y)
//     if it comes before B's last entry (or B is not yet full);
//   merge: a Y entry's place in B u Y = (Y entries before it) + (B entries
//     before it), a B entry's = its place + (Y entries before it), by
//     counting; places below need form the new B, the Y entries with their
//     level rank = the Y entries before them.
// Node ids: 1 + the number of selected candidates of lower index.
static __device__ __noinline__ void assemble_tree(const TreeJob J, StreamSmem& S) {
  const int tid = threadIdx.x;
  const int k = J.top_k, D = J.depth, m = J.total_tokens, C = J.n_cand;
  const int kk = k * k;
  const int rk = J.rec_k;
  const int rb = rec_bytes(rk);
  const int need = m - 1;
  char* rows = J.rows;
  const eagle_tree out = J.out;

  // scratch carved from the (now idle) ring; every array starts on a 16-byte
  // boundary (about 32 C + 18 KB bytes)
  char* p = reinterpret_cast<char*>(S.ring);
  auto carve = [&p](size_t bytes) {
    char* q = p;
    p += align_up(bytes, 16);
    return q;
  };
  double* w = reinterpret_cast<double*>(carve(sizeof(double) * C));      // logit - logsumexp
  int* tok = reinterpret_cast<int*>(carve(sizeof(int) * C));
  int* node = reinterpret_cast<int*>(carve(sizeof(int) * C));
  uint64_t* ykey = reinterpret_cast<uint64_t*>(carve(sizeof(uint64_t) * C));  // list Y
  int* ycand = reinterpret_cast<int*>(carve(sizeof(int) * C));
  int* ypar = reinterpret_cast<int*>(carve(sizeof(int) * C));
  constexpr int T = EAGLE_MAX_TREE;
  uint64_t* bkey = reinterpret_cast<uint64_t*>(carve(sizeof(uint64_t) * 2 * T));  // list B, x2
  int* bcand = reinterpret_cast<int*>(carve(sizeof(int) * 2 * T));
  int* bpar = reinterpret_cast<int*>(carve(sizeof(int) * 2 * T));
  int* blr = reinterpret_cast<int*>(carve(sizeof(int) * 2 * T));   // level << 16 | level rank
  int* npar = reinterpret_cast<int*>(carve(sizeof(int) * T));
  int* ny = reinterpret_cast<int*>(carve(sizeof(int) * 2));        // |Y|, by level parity

  // every candidate's offset and token; level 1 (row 0's top-k, in order)
  // is the first B
  for (int a = tid; a < C; a += kThreads) {
    const int r = a / k, c = a - r * k;
    char* rec = rows + r * rb;
    const double lse = __ldcg(&reinterpret_cast<const RecHead*>(rec)->sum);
    const double wa = static_cast<double>(__ldcg(rec_val(rec) + c)) - lse;
    w[a] = wa;
    tok[a] = __ldcg(rec_idx(rec, rk) + c);
    node[a] = 0;
    if (a < k && a < need) {
      bkey[a] = order_key(wa);
      bcand[a] = a;
      bpar[a] = -1;
      blr[a] = (1 << 16) | a;
    }
  }
  if (tid < 2) ny[tid] = 0;
  int nb = k < need ? k : need;   // |B|
  int cur = 0;                    // which half of the B arrays holds it
  __syncthreads();

  for (int l = 1; l < D && need > 0; ++l) {
    const int nbase = k + (l - 1) * kk;    // level l+1
    const uint64_t* bk = bkey + cur * T;
    const int* bc = bcand + cur * T;
    const int* bl = blr + cur * T;
    int* cnt_y = ny + (l & 1);
    const bool full = nb == need;
    const uint64_t tk = full ? bk[nb - 1] : 0ull;
    const int tc = full ? bc[nb - 1] : 0;
    // children of B's level-l entries of level rank < k that come before
    // B's last entry
    for (int t = tid; t < nb * k; t += kThreads) {
      const int i = t / k, c = t - i * k;
      const int lr = bl[i];
      if ((lr >> 16) != l || (lr & 0xffff) >= k) continue;
      const int a = nbase + (lr & 0xffff) * k + c;
      const uint64_t kv = order_key(key_value(bk[i]) + w[a]);
      if (full && !cand_before(kv, a, tk, tc)) continue;
      const int y = atomicAdd(cnt_y, 1);
      ykey[y] = kv;
      ycand[y] = a;
      ypar[y] = bc[i];
    }
    __syncthreads();
    const int n_y = *cnt_y;
    if (tid == 0) ny[(l + 1) & 1] = 0;     // the next level's counter
    // merge: tpc threads per entry (a power of two), every thread of a warp
    // reading the same list entries (broadcast)
    const int ne = n_y + nb;
    int tpc = ne > 0 ? kThreads / ne : 1;
    tpc = tpc >= 8 ? 8 : tpc >= 4 ? 4 : tpc >= 2 ? 2 : 1;
    const int sub = tid & (tpc - 1);
    const int stride = kThreads / tpc;
    uint64_t* nk = bkey + (cur ^ 1) * T;
    int* nc = bcand + (cur ^ 1) * T;
    int* np = bpar + (cur ^ 1) * T;
    int* nl = blr + (cur ^ 1) * T;
    const int* bp = bpar + cur * T;
    for (int e0 = 0; e0 < ne; e0 += stride) {
      const int e = e0 + tid / tpc;
      uint64_t kv = 0;
      int a = 0, before_y = 0, before_b = 0;
      if (e < ne) {
        kv = e < n_y ? ykey[e] : bk[e - n_y];
        a = e < n_y ? ycand[e] : bc[e - n_y];
        // unrolled: a thread's shared loads go out together, not one per
        // dependent round
#pragma unroll 4
        for (int f = sub; f < n_y; f += tpc) before_y += cand_before(ykey[f], ycand[f], kv, a) ? 1 : 0;
        if (e < n_y) {
#pragma unroll 4
          for (int f = sub; f < nb; f += tpc) before_b += cand_before(bk[f], bc[f], kv, a) ? 1 : 0;
        }
      }
      for (int o = tpc >> 1; o; o >>= 1) {
        before_y += __shfl_xor_sync(0xffffffffu, before_y, o);
        before_b += __shfl_xor_sync(0xffffffffu, before_b, o);
      }
      if (e < ne && sub == 0) {
        if (e < n_y) {
          const int pos = before_y + before_b;
          if (pos < need) {
            nk[pos] = kv;
            nc[pos] = a;
            np[pos] = ypar[e];
            nl[pos] = ((l + 1) << 16) | before_y;
          }
        } else {
          const int i = e - n_y;
          const int pos = i + before_y;
          if (pos < need) {
            nk[pos] = kv;
            nc[pos] = a;
            np[pos] = bp[i];
            nl[pos] = bl[i];
          }
        }
      }
    }
    nb = nb + n_y < need ? nb + n_y : need;
    cur ^= 1;
    __syncthreads();
  }
  const uint64_t* sk = bkey + cur * T;   // the selected candidates, best first
  const int* sel = bcand + cur * T;
  const int* spar = bpar + cur * T;
  if (tid == 0 && nb != (need > 0 ? need : 0)) record_error(J.err, kDevAssert, 10);

  // node ids: selected candidates numbered 1.. in candidate order
  for (int i = tid; i < nb; i += kThreads) {
    const int a = sel[i];
    int before_a = 0;
#pragma unroll 8
    for (int q = 0; q < nb; ++q) before_a += sel[q] < a ? 1 : 0;
    node[a] = 1 + before_a;
  }
  __syncthreads();

  // node arrays
  if (tid == 0) {
    out.parents[0] = -1;
    out.tokens[0] = J.root_token;
    out.depth[0] = 0;
    out.pos[0] = 0;
    if (out.values) out.values[0] = 0.0;
    npar[0] = -1;
  }
  for (int i = tid; i < nb; i += kThreads) {
    const int a = sel[i];
    const int n = node[a];
    int pn = 0;
    if (spar[i] >= 0) {
      pn = node[spar[i]];
      if (pn == 0) record_error(J.err, kDevAssert, 11);  // kept set not ancestor-closed
    }
    const int dep = cand_depth(a, k);
    out.parents[n] = pn;
    out.tokens[n] = tok[a];
    out.depth[n] = dep;
    out.pos[n] = dep;
    if (out.values) out.values[n] = key_value(sk[i]);
    npar[n] = pn;
  }
  __syncthreads();
  const int W = out.mask_words;
  for (int n = tid; n < m; n += kThreads) {
    uint64_t w0 = 0, w1 = 0, w2 = 0, w3 = 0;
    int q = n;
    for (int guard = 0; q >= 0 && guard <= EAGLE_MAX_DEPTH + 1; ++guard) {
      const uint64_t bit = 1ull << (q & 63);
      const int wi = q >> 6;
      w0 |= wi == 0 ? bit : 0ull;
      w1 |= wi == 1 ? bit : 0ull;
      w2 |= wi == 2 ? bit : 0ull;
      w3 |= wi == 3 ? bit : 0ull;
      q = npar[q];
    }
    uint64_t* dst = out.mask + static_cast<int64_t>(n) * W;
    dst[0] = w0;
    if (W > 1) dst[1] = w1;
    if (W > 2) dst[2] = w2;
    if (W > 3) dst[3] = w3;
  }
  __syncthreads();
}

// Code warm-up.  The tree assembly runs once per item, in one CTA, after the
// item's last row; when the L2 holds other data (as it does between decode
// steps, after the target model's forward pass) each first use of a stretch
// of its code is an instruction fetch from HBM, several microseconds in all.
// The first CTA of one extra cluster runs the same function at launch, on a
// tree of its own (three top-2 rows, depth 2, four nodes) in the library's
// g_warm_tree, so that the code is in L2 when the real assembly needs it.  It
// reads and writes nothing else (no caller memory: it runs before the
// launch's dependency wait) and has its own error word.
static __device__ __noinline__ void warm_assembly(StreamSmem& S) {
  char* warm = g_warm_tree;
  const int rb = rec_bytes(kWarmK);
  char* rows = warm + 16;
  int32_t* ints = reinterpret_cast<int32_t*>(rows + 3 * rb);
  const int t = threadIdx.x;
  if (t == 0) *reinterpret_cast<int32_t*>(warm) = 0;
  if (t < 3) {
    char* rec = rows + t * rb;
    RecHead* h = reinterpret_cast<RecHead*>(rec);
    h->sum = 1.0;   // stands for the row's logsumexp (any finite value)
    h->max = 0.f;
    h->count = kWarmK;
    rec_val(rec)[0] = 0.f;
    rec_val(rec)[1] = -1.f;
    rec_idx(rec, kWarmK)[0] = 2 * t;
    rec_idx(rec, kWarmK)[1] = 2 * t + 1;
  }
  __threadfence();
  __syncthreads();
  TreeJob J;
  J.rows = rows;
  J.out.parents = ints;
  J.out.tokens = ints + 4;
  J.out.depth = ints + 8;
  J.out.pos = ints + 12;
  J.out.mask = reinterpret_cast<uint64_t*>(ints + 16);
  J.out.values = nullptr;
  J.out.m = 4;
  J.out.mask_words = 1;
  J.err = reinterpret_cast<int32_t*>(warm);
  J.rec_k = kWarmK;
  J.top_k = kWarmK;
  J.depth = 2;
  J.total_tokens = 4;
  J.n_cand = kWarmK + kWarmK * kWarmK;
  J.root_token = 0;
  assemble_tree(J, S);
}

// Grid: the rows' clusters, then the clusters for the code warm-ups: (long
// rows: stream_warm_up) one that streams the short warm-up row (see
// warm_row_job), then one whose first CTA runs the tree assembly on its own
// tree at launch.
__global__ void __launch_bounds__(kThreads, 2) build_kernel(const __grid_constant__ BuildArgs A) {
  extern __shared__ __align__(128) char smem_raw[];
  StreamSmem& S = *reinterpret_cast<StreamSmem*>(smem_raw);
  const int PC = A.rs.ctas_per_row;
  const int64_t rows = static_cast<int64_t>(A.rs.n_items) * A.rs.rows_per_item;
  const int64_t cl = blockIdx.x / PC;
  const int rank = static_cast<int>(blockIdx.x - cl * PC);
  pdl_trigger();
  if (cl >= rows + A.warm_stream) {
    if (rank == 0) warm_assembly(S);
    return;
  }
  const bool warm = cl == rows;   // (only when warm_stream)
  if (!warm) pdl_wait();          // the warm-ups touch no caller memory
  const RowJob R = warm ? warm_row_job(A.rs, rank) : row_job(A.rs, cl, rank);
  const RowCtx cx = stream_row(R, S);
  if (!cx.leader || warm) return;
  // the row's logsumexp replaces the record's sum (the tree assembly needs
  // only that; one fp64 log per row, here, in parallel over the rows).  The
  // sum holds the max's own term 1, so its log is >= 0: kept so through the
  // rounding of log_d, which makes every offset logit - logsumexp <= 0
  if (threadIdx.x == 0)
    reinterpret_cast<RecHead*>(R.rec)->sum =
        static_cast<double>(S.rmax) + fmax(0.0, log_d(S.rsum));   // sum >= 1: log >= 0
  if (!item_arrive(A.rs, S, cx.item)) return;
  const int rb = rec_bytes(A.rs.rec_k);
  TreeJob J;
  J.rows = A.rs.rows + static_cast<int64_t>(cx.item) * A.rs.rows_per_item * rb;
  J.out = A.out[cx.item];
  J.err = A.rs.err;
  J.rec_k = A.rs.rec_k;
  J.top_k = A.top_k;
  J.depth = A.depth;
  J.total_tokens = A.total_tokens;
  J.n_cand = A.n_cand;
  J.root_token = A.root_token[cx.item];
  assemble_tree(J, S);
}

// tree assembly scratch (R = 1 + (depth-1) top_k <= 256 whenever C <= 2048)
static_assert(kScratchBytes >= (2 * 8 + 4 * 4) * EAGLE_MAX_CANDIDATES +
                                   (2 * 8 + 3 * 2 * 4 + 4) * EAGLE_MAX_TREE + 16 * 16,
              "tree assembly scratch must fit in the stream's shared memory");

static eagle_status build_impl(int32_t n_items, const float* const* logits, int64_t row_stride,
                               int32_t n_rows, int32_t vocab, int32_t top_k, int32_t depth,
                               int32_t total_tokens, const int32_t* roots,
                               const eagle_tree* outs, void* ws, size_t ws_bytes,
                               cudaStream_t stream) {
  EAGLE_CHECK_ARG(logits && roots && outs && ws);
  EAGLE_CHECK_ARG(n_items >= 1 && vocab >= 1 && n_rows >= 1 && top_k >= 1 && depth >= 1 &&
                  total_tokens >= 1);
  EAGLE_CHECK_SHAPE(n_items <= kMaxItems);
  EAGLE_CHECK_SHAPE(top_k <= kKMax && top_k <= vocab && depth <= EAGLE_MAX_DEPTH);
  const int64_t C = top_k + static_cast<int64_t>(depth - 1) * top_k * top_k;
  EAGLE_CHECK_SHAPE(C <= EAGLE_MAX_CANDIDATES);
  EAGLE_CHECK_SHAPE(total_tokens <= EAGLE_MAX_TREE && total_tokens <= 1 + C);
  const int R = 1 + (depth - 1) * top_k;
  EAGLE_CHECK_ARG(n_rows >= R);
  EAGLE_CHECK_ARG(row_stride >= vocab && row_stride % 4 == 0);
  for (int i = 0; i < n_items; ++i) {
    EAGLE_CHECK_ARG(logits[i] && aligned16(logits[i]));
    const eagle_tree& t = outs[i];
    EAGLE_CHECK_ARG(t.parents && t.tokens && t.depth && t.pos && t.mask);
    EAGLE_CHECK_ARG(t.m == total_tokens && t.mask_words == (total_tokens + 63) / 64);
  }
  const StreamLayout L = stream_layout(n_items, R, vocab, top_k, false, false);
  if (ws_bytes < L.total) return EAGLE_ERR_WORKSPACE_TOO_SMALL;

  BuildArgs A;
  memset(&A, 0, sizeof(A));
  const int occ = stream_ctas_per_sm(build_kernel);
  if (occ <= 0) return EAGLE_ERR_CUDA;
  const int ctas = stream_ctas_per_row(build_kernel, L, occ, 2);
  if (ctas <= 0) return EAGLE_ERR_CUDA;
  fill_stream(A.rs, L, static_cast<char*>(ws), n_items, R, vocab, row_stride, ctas, false);
  for (int i = 0; i < n_items; ++i) {
    A.rs.base[i] = logits[i];
    A.rs.exp_scale[i] = 1.0f;
    A.rs.topk[i] = static_cast<int16_t>(top_k);
    A.rs.flags[i] = kWantSum;
    A.root_token[i] = roots[i];
    A.out[i] = outs[i];
  }
  A.top_k = top_k;
  A.depth = depth;
  A.total_tokens = total_tokens;
  A.n_cand = static_cast<int>(C);
  A.warm_stream = stream_warm_up(L.tiles_per_row, ctas) ? 1 : 0;
  return launch_stream(build_kernel, A, L.n_rows + 1 + A.warm_stream, ctas, stream);
}

// Scratch of the allocation-free entry point: fixed size, static device
// memory of this library, shared by every call on a device.
static __device__ __align__(256) unsigned char g_noalloc_scratch[EAGLE_NOALLOC_SCRATCH_BYTES];

constexpr int kMaxDevices = 64;

// Unique id of the calling thread's current CUDA context (cuCtxGetId, reached
// through the runtime's driver entry-point query, so the library does not
// link the driver library itself); 0 when there is no current context yet or
// the query is unavailable.  The id is never reused within a process, so a
// context created after cudaDeviceReset, or a separate driver-API context on
// the same device, gets a new one.
static unsigned long long current_context_id() {
  static PFN_cuCtxGetCurrent_v4000 get_current = nullptr;
  static PFN_cuCtxGetId_v12000 get_id = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &p, 4000, cudaEnableDefault, &q) ==
            cudaSuccess && q == cudaDriverEntryPointSuccess)
      get_current = reinterpret_cast<PFN_cuCtxGetCurrent_v4000>(p);
    p = nullptr;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess && q == cudaDriverEntryPointSuccess)
      get_id = reinterpret_cast<PFN_cuCtxGetId_v12000>(p);
  });
  if (!get_current || !get_id) return 0;
  CUcontext ctx = nullptr;
  unsigned long long id = 0;
  if (get_current(&ctx) != CUDA_SUCCESS || !ctx) return 0;
  if (get_id(ctx, &id) != CUDA_SUCCESS) return 0;
  return id;
}

// Device address of g_noalloc_scratch in the current context.  The symbol's
// address belongs to the library's module as loaded in one context, so it is
// looked up with cudaGetSymbolAddress once per (device, context) -- on the
// first call in a context, with that device current -- and cached under the
// context's id; when the id cannot be read, it is looked up on every call.
static eagle_status noalloc_scratch(void** out) {
  static std::mutex mu;
  static void* addr[kMaxDevices] = {};
  static unsigned long long ctx_of[kMaxDevices] = {};
  int dev = 0;
  EAGLE_CUDA(cudaGetDevice(&dev));
  if (dev < 0 || dev >= kMaxDevices) return EAGLE_ERR_UNSUPPORTED_SHAPE;
  std::lock_guard<std::mutex> lock(mu);
  unsigned long long ctx = current_context_id();
  if (ctx != 0 && ctx_of[dev] == ctx && addr[dev]) {
    *out = addr[dev];
    return EAGLE_OK;
  }
  void* p = nullptr;
  EAGLE_CUDA(cudaGetSymbolAddress(&p, g_noalloc_scratch));
  if (!p || !aligned16(p)) return EAGLE_ERR_CUDA;
  ctx = current_context_id();   // the lookup made the device's context current
  addr[dev] = p;
  ctx_of[dev] = ctx;
  *out = p;
  return EAGLE_OK;
}

}  // namespace eagle

using namespace eagle;

extern "C" size_t eagle_tree_build_workspace_size(int32_t n_items, int32_t n_rows, int32_t vocab,
                                                  int32_t top_k, int32_t depth,
                                                  int32_t total_tokens) {
  (void)n_rows;
  (void)total_tokens;
  if (n_items < 1 || vocab < 1 || top_k < 1 || depth < 1) return 0;
  const int R = 1 + (depth - 1) * top_k;
  return stream_layout(n_items, R, vocab, top_k, false, false).total;
}

extern "C" eagle_status eagle_tree_build(const float* draft_logits, int64_t row_stride,
                                         int32_t n_rows, int32_t vocab, int32_t top_k,
                                         int32_t depth, int32_t total_tokens,
                                         int32_t root_token, eagle_tree out, void* ws,
                                         size_t ws_bytes, eagle_stream stream) {
  return build_impl(1, &draft_logits, row_stride, n_rows, vocab, top_k, depth, total_tokens,
                    &root_token, &out, ws, ws_bytes, reinterpret_cast<cudaStream_t>(stream));
}

extern "C" eagle_status eagle_tree_build_batched(int32_t n_items,
                                                 const float* const* draft_logits,
                                                 int64_t row_stride, int32_t n_rows,
                                                 int32_t vocab, int32_t top_k, int32_t depth,
                                                 int32_t total_tokens,
                                                 const int32_t* root_tokens,
                                                 const eagle_tree* outs, void* ws,
                                                 size_t ws_bytes, eagle_stream stream) {
  return build_impl(n_items, draft_logits, row_stride, n_rows, vocab, top_k, depth,
                    total_tokens, root_tokens, outs, ws, ws_bytes,
                    reinterpret_cast<cudaStream_t>(stream));
}

extern "C" eagle_status eagle_tree_build_noalloc(const float* draft_logits, int64_t row_stride,
                                                 int32_t n_rows, int32_t vocab, int32_t top_k,
                                                 int32_t depth, int32_t total_tokens,
                                                 int32_t root_token, eagle_tree out,
                                                 eagle_stream stream) {
  // the checks build_impl makes, made here first so that a bad argument
  // enqueues nothing (not even the scratch clear)
  EAGLE_CHECK_ARG(draft_logits && aligned16(draft_logits));
  EAGLE_CHECK_ARG(vocab >= 1 && n_rows >= 1 && top_k >= 1 && depth >= 1 && total_tokens >= 1);
  EAGLE_CHECK_SHAPE(top_k <= kKMax && top_k <= vocab && depth <= EAGLE_MAX_DEPTH);
  const int64_t C = top_k + static_cast<int64_t>(depth - 1) * top_k * top_k;
  EAGLE_CHECK_SHAPE(C <= EAGLE_MAX_CANDIDATES);
  EAGLE_CHECK_SHAPE(total_tokens <= EAGLE_MAX_TREE && total_tokens <= 1 + C);
  const int R = 1 + (depth - 1) * top_k;
  EAGLE_CHECK_ARG(n_rows >= R);
  EAGLE_CHECK_ARG(row_stride >= vocab && row_stride % 4 == 0);
  EAGLE_CHECK_ARG(out.parents && out.tokens && out.depth && out.pos && out.mask);
  EAGLE_CHECK_ARG(out.m == total_tokens && out.mask_words == (total_tokens + 63) / 64);
  const StreamLayout L = stream_layout(1, R, vocab, top_k, false, false);
  if (L.total > EAGLE_NOALLOC_SCRATCH_BYTES) return EAGLE_ERR_WORKSPACE_TOO_SMALL;
  void* ws = nullptr;
  const eagle_status st = noalloc_scratch(&ws);
  if (st != EAGLE_OK) return st;
  const cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  // header (error word) and the per-item arrival counters must start at
  // zero; the row records behind them are written before they are read
  EAGLE_CUDA(cudaMemsetAsync(ws, 0, L.off_rows, s));
  return build_impl(1, &draft_logits, row_stride, n_rows, vocab, top_k, depth, total_tokens,
                    &root_token, &out, ws, EAGLE_NOALLOC_SCRATCH_BYTES, s);
}

extern "C" eagle_status eagle_tree_build_noalloc_error(eagle_stream stream, int32_t* status,
                                                       int32_t* detail) {
  EAGLE_CHECK_ARG(status != nullptr);
  void* ws = nullptr;
  const eagle_status st = noalloc_scratch(&ws);
  if (st != EAGLE_OK) return st;
  return eagle_workspace_error(ws, stream, status, detail);
}
