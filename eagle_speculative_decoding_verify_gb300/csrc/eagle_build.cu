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
// value = parent value + (logit - logsumexp), in fp64; per depth the top_k
// frontier; the final best m-1 -- both by ranks across the sorted child lists
// (binary search on order-preserving 64-bit keys, ties -> lower candidate
// index); node ids by a block scan; ancestor mask by walking parent pointers
// (depth <= 16).
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
  char* warm;   // kWarmBytes of workspace for the code warm-up's own tree
};

// One tree assembly: the item's R row records and its outputs.
struct TreeJob {
  char* rows;        // R records of rec_bytes(rec_k) bytes
  eagle_tree out;
  int32_t* err;
  int rec_k, top_k, depth, total_tokens, n_cand, root_token;
};

// Workspace of the code warm-up: error word, 3 records of a top-2 row,
// parents / tokens / depth / pos of 4 nodes, 4 mask words.
constexpr int kWarmK = 2;
constexpr size_t kWarmBytes = 256;
static_assert(16 + 3 * rec_bytes(kWarmK) + 4 * 16 + 8 * 4 <= kWarmBytes, "warm-up workspace");

__device__ __forceinline__ int cand_depth(int a, int k) { return a < k ? 1 : 2 + (a - k) / (k * k); }

// Block-wide exclusive scan of per-thread counts (blockDim == kThreads).
static __device__ __noinline__ int block_excl_scan(int v, int* warp_tot, int& total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  int incl = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int y = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += y;
  }
  if (lane == 31) warp_tot[warp] = incl;
  __syncthreads();
  int off = 0;
  total = 0;
  for (int w = 0; w < kWarps; ++w) {
    if (w < warp) off += warp_tot[w];
    total += warp_tot[w];
  }
  __syncthreads();
  return off + incl - v;
}

static __device__ __noinline__ void assemble_tree(const TreeJob J, StreamSmem& S) {
  const int tid = threadIdx.x, lane = tid & 31;
  const int k = J.top_k, D = J.depth, m = J.total_tokens, C = J.n_cand;
  const int R = 1 + (D - 1) * k;
  const int kk = k * k;
  const int rk = J.rec_k;
  const int rb = rec_bytes(rk);
  char* rows = J.rows;
  const eagle_tree out = J.out;

  // scratch carved from the (now idle) ring and warp buffers; every array
  // starts on a 16-byte boundary (<= 77 KB for C <= 2048; R k = C)
  char* p = reinterpret_cast<char*>(S.ring);
  auto carve = [&p](size_t bytes) {
    char* q = p;
    p += align_up(bytes, 16);
    return q;
  };
  uint64_t* key = reinterpret_cast<uint64_t*>(carve(sizeof(uint64_t) * C));  // value as order key
  double* lse = reinterpret_cast<double*>(carve(sizeof(double) * R));
  float* rv = reinterpret_cast<float*>(carve(sizeof(float) * C));   // row top-k logits
  int* ri = reinterpret_cast<int*>(carve(sizeof(int) * C));         // row top-k tokens
  int* tok = reinterpret_cast<int*>(carve(sizeof(int) * C));
  int* par = reinterpret_cast<int*>(carve(sizeof(int) * C));
  int* srt = reinterpret_cast<int*>(carve(sizeof(int) * C));    // candidates of each level, best first
  int* lrank = reinterpret_cast<int*>(carve(sizeof(int) * C));  // rank of a candidate in its level
  int* node = reinterpret_cast<int*>(carve(sizeof(int) * C));
  int* npar = reinterpret_cast<int*>(carve(sizeof(int) * EAGLE_MAX_TREE));
  int* fr = reinterpret_cast<int*>(carve(sizeof(int) * 2 * kKMax));  // frontiers, by depth parity
  int* warp_tot = reinterpret_cast<int*>(carve(sizeof(int) * EAGLE_MAX_DEPTH));

  // every row's statistics in one pass: logsumexp, top-k logits and tokens
  for (int r = tid; r < R; r += kThreads) {
    const volatile RecHead* h = reinterpret_cast<volatile RecHead*>(rows + r * rb);
    lse[r] = static_cast<double>(h->max) + log_d(h->sum);
  }
  for (int e = tid; e < C; e += kThreads) {
    const int r = e / k, c = e - r * k;
    rv[e] = __ldcg(rec_val(rows + r * rb) + c);
    ri[e] = __ldcg(rec_idx(rows + r * rb, rk) + c);
  }
  __syncthreads();

  // Candidates are compared on (value desc, candidate index asc), values as
  // order-preserving integer keys.  Level 1 = candidates 0..k-1 (the root's
  // top_k, already in order); level j >= 2 = candidates k + (j-2) k^2 ..
  // + k^2 - 1, ranked by counting with every thread of a warp reading the
  // same keys (broadcast, no bank conflicts).
  for (int c = tid; c < k; c += kThreads) {
    key[c] = order_key(static_cast<double>(rv[c]) - lse[0]);
    tok[c] = ri[c];
    par[c] = -1;
    fr[c] = c;
    srt[c] = c;
    lrank[c] = c;
  }
  __syncthreads();

  // threads per candidate for the level ranks: a power of two <= 8
  int tpc = kThreads / kk;
  tpc = tpc >= 8 ? 8 : tpc >= 4 ? 4 : tpc >= 2 ? 2 : 1;
  const int sub = tid & (tpc - 1);
  const int stride = kThreads / tpc;
  int base = k;   // first candidate of the level being built
  for (int l = 1; l < D; ++l) {
    const int* fcur = fr + ((l - 1) & 1) * kKMax;
    int* fnext = fr + (l & 1) * kKMax;
    for (int e = tid; e < kk; e += kThreads) {
      const int s = e / k, c = e - s * k;
      const int r = 1 + (l - 1) * k + s;
      const int a = base + e;
      const int pa = fcur[s];
      key[a] = order_key(key_value(key[pa]) + (static_cast<double>(rv[r * k + c]) - lse[r]));
      tok[a] = ri[r * k + c];
      par[a] = pa;
    }
    __syncthreads();
    // full rank of every candidate within the level (tpc threads each)
    const uint64_t* lk = key + base;
    for (int e0 = 0; e0 < kk; e0 += stride) {
      const int e = e0 + tid / tpc;
      int cnt = 0;
      if (e < kk) {
        const uint64_t kv = lk[e];
#pragma unroll 4
        for (int f = sub; f < kk; f += tpc) {
          const uint64_t o = lk[f];
          cnt += ((o > kv) | ((o == kv) & (f < e))) ? 1 : 0;
        }
      }
      for (int o = tpc >> 1; o; o >>= 1) cnt += __shfl_xor_sync(0xffffffffu, cnt, o);
      if (e < kk && sub == 0) {
        srt[base + cnt] = base + e;
        lrank[base + e] = cnt;
        if (cnt < k && l + 1 < D) fnext[cnt] = base + e;
      }
    }
    __syncthreads();
    base += kk;
  }

  // final rerank: the best need = m-1 of the C candidates.  The global rank
  // of a candidate is its rank in its own level plus, for every other level,
  // the number of that level's entries before it (a binary search over the
  // level's keys in sorted order, materialised over the row top-k scratch,
  // which is no longer needed); it is kept if that rank is below need.
  // Every candidate is ranked independently, all in parallel.
  uint64_t* skey = reinterpret_cast<uint64_t*>(rv);   // rv and ri are contiguous: 8 C bytes
  for (int i = tid; i < C; i += kThreads) skey[i] = key[srt[i]];
  __syncthreads();
  const int need = m - 1;
  for (int a = tid; a < C; a += kThreads) {
    const int la = a < k ? 0 : 1 + (a - k) / kk;
    int rank = lrank[a];
    const uint64_t kv = key[a];
    for (int l = 0; l < D && rank < need; ++l) {
      if (l == la) continue;
      const int lb = l == 0 ? 0 : k + (l - 1) * kk;
      int lo = 0, hi = l == 0 ? k : kk;   // entries of level l before (kv, a)
      while (lo < hi) {
        const int mid = (lo + hi) >> 1;
        const uint64_t o = skey[lb + mid];
        const bool go = (o > kv) | ((o == kv) & (srt[lb + mid] < a));
        lo = go ? mid + 1 : lo;
        hi = go ? hi : mid;
      }
      rank += lo;
    }
    node[a] = rank < need ? 1 : 0;
  }
  __syncthreads();
  const int per = (C + kThreads - 1) / kThreads;
  const int a0 = tid * per, a1 = min(C, a0 + per);
  int cnt_local = 0;
  for (int a = a0; a < a1; ++a) cnt_local += node[a];

  // selection flags in candidate order -> node ids (1 + exclusive count)
  int total = 0;
  int off = block_excl_scan(cnt_local, warp_tot, total);
  for (int a = a0; a < a1; ++a) {
    if (node[a]) node[a] = 1 + off++;
    else node[a] = 0;
  }
  __syncthreads();
  if (tid == 0 && total != (need > 0 ? min(need, C) : 0)) record_error(J.err, kDevAssert, 10);
  (void)lane;

  // node arrays
  if (tid == 0) {
    out.parents[0] = -1;
    out.tokens[0] = J.root_token;
    out.depth[0] = 0;
    out.pos[0] = 0;
    if (out.values) out.values[0] = 0.0;
    npar[0] = -1;
  }
  for (int a = tid; a < C; a += kThreads) {
    const int n = node[a];
    if (!n) continue;
    int pn = 0;
    if (par[a] >= 0) {
      pn = node[par[a]];
      if (pn == 0) {
        record_error(J.err, kDevAssert, 11);  // kept set not ancestor-closed
        pn = 0;
      }
    }
    const int dep = cand_depth(a, k);
    out.parents[n] = pn;
    out.tokens[n] = tok[a];
    out.depth[n] = dep;
    out.pos[n] = dep;
    if (out.values) out.values[n] = key_value(key[a]);
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
// tree of its own (three top-2 rows, depth 2, four nodes) in kWarmBytes of
// workspace, so that the code is in L2 when the real assembly needs it.  It
// reads and writes nothing else and has its own error word.
static __device__ __noinline__ void warm_assembly(char* warm, StreamSmem& S) {
  const int rb = rec_bytes(kWarmK);
  char* rows = warm + 16;
  int32_t* ints = reinterpret_cast<int32_t*>(rows + 3 * rb);
  const int t = threadIdx.x;
  if (t == 0) *reinterpret_cast<int32_t*>(warm) = 0;
  if (t < 3) {
    char* rec = rows + t * rb;
    RecHead* h = reinterpret_cast<RecHead*>(rec);
    h->sum = 2.0;
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

// Grid: the rows' clusters, then one more cluster for the code warm-up.
__global__ void __launch_bounds__(kThreads, 2) build_kernel(const __grid_constant__ BuildArgs A) {
  extern __shared__ __align__(128) char smem_raw[];
  StreamSmem& S = *reinterpret_cast<StreamSmem*>(smem_raw);
  const int64_t row_ctas =
      static_cast<int64_t>(A.rs.n_items) * A.rs.rows_per_item * A.rs.ctas_per_row;
  if (blockIdx.x >= row_ctas) {
    if (blockIdx.x == row_ctas) warm_assembly(A.warm, S);
    return;
  }
  const RowCtx cx = stream_row(A.rs, S);
  if (!cx.leader) return;
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
static_assert(kScratchBytes >= (8 + 4 * 7) * EAGLE_MAX_CANDIDATES + 8 * 256 +
                                   4 * (EAGLE_MAX_TREE + 2 * kKMax + kWarps) + 16 * 16,
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
  if (ws_bytes < L.total + kWarmBytes) return EAGLE_ERR_WORKSPACE_TOO_SMALL;

  BuildArgs A;
  memset(&A, 0, sizeof(A));
  const int occ = stream_ctas_per_sm(build_kernel);
  if (occ <= 0) return EAGLE_ERR_CUDA;
  const int ctas = stream_ctas_per_row(build_kernel, L, occ);
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
  A.warm = static_cast<char*>(ws) + L.total;
  return launch_stream(build_kernel, A, L.n_rows + 1, ctas, stream);
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
  return stream_layout(n_items, R, vocab, top_k, false, false).total + kWarmBytes;
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
  if (L.total + kWarmBytes > EAGLE_NOALLOC_SCRATCH_BYTES) return EAGLE_ERR_WORKSPACE_TOO_SMALL;
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
