/*
 * eagle.h -- C ABI of the GB300 (sm_103a) library for the hot path of one
 * EAGLE-2 speculative-decoding verify step:
 *
 *   eagle_tree_build   draft logits            -> dynamic draft tree
 *   eagle_tree_attn    tree queries + KV cache -> tree-masked attention output
 *   eagle_tree_verify  target logits + tree    -> accepted path + bonus token
 *
 * Sources (page title and section):
 *   [blog]  "EAGLE-2: Feature-Level Speculative Decoding Guide":
 *           "The Recurrent Feature Drafting Step" (draft distribution =
 *           softmax of LM-head logits), "Context-Aware Dynamic Tree
 *           Construction", "Single-Pass Tree Verification" (ancestor-only
 *           tree mask, root-to-leaf acceptance, lossless output).
 *   [disc]  "Support Eagle-3 Speculative Decoding in llama.cpp": reply on the
 *           dynamic tree (valued by draft confidence, pruned at the end of
 *           drafting), the acceptance / rejection strategy, and the reply on
 *           KV caches (target keeps the accepted context).
 *   [pr]    "EAGLE-2 Speculative Decoding Support for llama.cpp - Phase 1",
 *           "Performance Notes": mixed sampling = temperature + top_k + top_p.
 *
 * Conventions for every entry point:
 *   - All tensor pointers are DEVICE pointers unless marked "host".  The
 *     caller owns every buffer, including the workspace `ws`; the library
 *     allocates nothing and keeps no global state (one exception: the
 *     fixed static scratch of eagle_tree_build_noalloc).
 *   - Work is enqueued on `stream` (a cudaStream_t; NULL = legacy default
 *     stream); nothing synchronises with the host.  Calls on one stream run
 *     in order; two calls that share a workspace must not overlap.
 *   - Arguments are validated on the host before anything is launched; on a
 *     bad argument nothing is enqueued.  Launch failures return
 *     EAGLE_ERR_CUDA.  Device-side problems (a bounded wait that ran out, a
 *     violated invariant) do not fail the call: they are recorded in the
 *     workspace's error word, read with eagle_workspace_error().
 *   - Workspaces must be zero-filled once before first use (for example with
 *     eagle_workspace_init); every successful call leaves its workspace
 *     ready for the next call.  After a recorded device error, re-initialise.
 *     A workspace starts with a 256-byte header: int32 words 0 and 1 are the
 *     device error word and its detail; words 2 and 3 are a test hook that
 *     must stay zero in normal use (for the head_dim 128 tensor-core
 *     attention: word 2 = 1 makes its producers issue no copy, so that every
 *     consumer wait runs out; word 3 = that wait's limit in microseconds,
 *     0 = the default 2 s) -- how the tests make a bounded device wait
 *     expire without a fault.
 *   - Floating-point inputs must be finite (no NaN / +-inf).
 */
#ifndef EAGLE_H
#define EAGLE_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Same type as cudaStream_t. */
typedef struct CUstream_st* eagle_stream;

typedef enum {
  EAGLE_OK = 0,
  EAGLE_ERR_INVALID_ARG = 1,         /* null pointer, negative size, bad stride/alignment   */
  EAGLE_ERR_UNSUPPORTED_SHAPE = 2,   /* valid but outside the library's limits (below)      */
  EAGLE_ERR_WORKSPACE_TOO_SMALL = 3, /* ws_bytes < the matching *_workspace_size()          */
  EAGLE_ERR_CUDA = 4,                /* a CUDA runtime call or launch failed                 */
  EAGLE_ERR_TIMEOUT = 5,             /* device error word: a bounded wait expired            */
  EAGLE_ERR_DEVICE_ASSERT = 6        /* device error word: an internal invariant was broken  */
} eagle_status;

typedef enum { EAGLE_F32 = 0, EAGLE_BF16 = 1 } eagle_dtype;

/* Library limits (EAGLE_ERR_UNSUPPORTED_SHAPE beyond them). */
#define EAGLE_MAX_TOP_K 64        /* draft top_k and sampling top_k             */
#define EAGLE_MAX_DEPTH 16
#define EAGLE_MAX_CANDIDATES 2048 /* C = top_k + (depth-1)*top_k^2             */
#define EAGLE_MAX_TREE 256        /* m = total_tokens                          */
#define EAGLE_MAX_BATCH 32        /* items per batched build / verify call     */

/*
 * Draft tree, one per sequence ([blog] "Context-Aware Dynamic Tree
 * Construction" and "Single-Pass Tree Verification").  All arrays are device
 * arrays of length m (mask: m * mask_words words), written by
 * eagle_tree_build and read by eagle_tree_verify.
 *   node 0 is the root (parents[0] = -1, tokens[0] = root token, depth 0);
 *   nodes 1..m-1 are the selected draft candidates in candidate order, so
 *   parents[i] < i and siblings appear in draft-rank order;
 *   mask[i*mask_words + w] bit b  <=>  node 64*w+b is node i or an ancestor;
 *   pos[i] = depth[i] (the caller adds its prefix length);
 *   values[i] = cumulative draft log-probability of node i (optional, may be
 *   NULL; 0 for the root).
 */
typedef struct {
  int32_t*  parents;
  int32_t*  tokens;
  int32_t*  depth;
  int32_t*  pos;
  uint64_t* mask;
  double*   values;
  int32_t   m;          /* total_tokens, root included */
  int32_t   mask_words; /* must equal (m + 63) / 64    */
} eagle_tree;

/* Target sampling parameters ([pr] "Performance Notes").  greedy != 0 walks
 * by argmax and ignores the rest.  Otherwise: logits / temperature (> 0),
 * keep the top_k largest (0 = all, at most EAGLE_MAX_TOP_K), softmax, then
 * nucleus top_p in (0, 1] (the shortest prefix in probability order, ties ->
 * lower token id, whose mass reaches top_p, the crossing token kept; with
 * top_k = 0 over the whole vocabulary, at most 4032 tiles of 1024 tokens),
 * renormalise. */
typedef struct {
  int32_t greedy;
  float   temperature;
  int32_t top_k;
  float   top_p;
} eagle_sampling;

const char* eagle_status_string(eagle_status status);
int32_t eagle_version(void);

/* Hash (16 hex digits) of the sources and compiler flags the library was
 * built from; a build tool compares it with the sources on disk to tell a
 * stale binary from a current one.  Static string, never NULL. */
const char* eagle_build_id(void);

/* Zero-fill a workspace (cudaMemsetAsync on `stream`). */
eagle_status eagle_workspace_init(void* ws, size_t ws_bytes, eagle_stream stream);

/* Synchronise `stream`, then read the workspace's device error word into
 * *status (EAGLE_OK, EAGLE_ERR_TIMEOUT or EAGLE_ERR_DEVICE_ASSERT) and
 * *detail (where it happened).  Debug / test use: it blocks the host. */
eagle_status eagle_workspace_error(const void* ws, eagle_stream stream,
                                   int32_t* status, int32_t* detail);

/* ------------------------------------------------------------------------
 * eagle_tree_build -- [blog] "The Recurrent Feature Drafting Step" and
 * "Context-Aware Dynamic Tree Construction"; [disc] reply on the dynamic
 * tree (value = draft confidence, grow per step, prune at the end).
 *
 * draft_logits: fp32 [n_rows][row_stride] row-major, 16-byte aligned,
 *   row_stride % 4 == 0, row_stride >= vocab.  n_rows >= R where
 *   R = 1 + (depth-1)*top_k.  Row 0 belongs to the root; the draft row of
 *   the j-th node of the depth-l frontier is 1 + (l-1)*top_k + j.
 * Per row: log-probabilities = logit - logsumexp(row) (draft temperature 1)
 * and the top_k tokens (ties -> lower token id).  Node value = parent value +
 * log-probability (root 0).  Depth-1 candidates are the root's top_k; at
 * each depth l = 2..depth-1 the frontier is the top_k candidates of depth l
 * by value (ties -> lower candidate index), ordered best first, and each
 * frontier node is expanded by its row's top_k.  The tree keeps the root plus
 * the best total_tokens-1 candidates overall (ties -> lower candidate index);
 * the kept set is closed under ancestors because values never increase
 * along a path.
 * Limits: 1 <= top_k <= min(64, vocab); 1 <= depth <= 16;
 *   C = top_k + (depth-1)*top_k^2 <= 2048; 1 <= total_tokens <= min(1+C, 256).
 * out: device arrays sized for m = total_tokens; out.m must equal
 *   total_tokens and out.mask_words (m+63)/64.
 * ws: at least eagle_tree_build_workspace_size(1, n_rows, vocab, top_k,
 *   depth, total_tokens) bytes, zero-filled before first use.
 * ------------------------------------------------------------------------ */
size_t eagle_tree_build_workspace_size(int32_t n_items, int32_t n_rows, int32_t vocab,
                                       int32_t top_k, int32_t depth, int32_t total_tokens);

eagle_status eagle_tree_build(const float* draft_logits, int64_t row_stride,
                              int32_t n_rows, int32_t vocab, int32_t top_k,
                              int32_t depth, int32_t total_tokens, int32_t root_token,
                              eagle_tree out, void* ws, size_t ws_bytes,
                              eagle_stream stream);

/* n_items independent sequences in one launch: draft_logits (host array of
 * n_items device pointers, same row_stride / n_rows / vocab), root_tokens
 * (host array), outs (host array of n_items trees, same total_tokens). */
eagle_status eagle_tree_build_batched(int32_t n_items, const float* const* draft_logits,
                                      int64_t row_stride, int32_t n_rows, int32_t vocab,
                                      int32_t top_k, int32_t depth, int32_t total_tokens,
                                      const int32_t* root_tokens, const eagle_tree* outs,
                                      void* ws, size_t ws_bytes, eagle_stream stream);

/* ------------------------------------------------------------------------
 * eagle_tree_build_noalloc -- the pages have no counterpart: this is a
 * deployment variant of eagle_tree_build for callers that cannot hand the
 * library device memory (no allocator reachable at the call site, or a
 * runtime that forbids allocation while it runs).  Same computation, same
 * arguments and same output as eagle_tree_build, without `ws`.
 *
 * Scratch: a fixed array of EAGLE_NOALLOC_SCRATCH_BYTES in the library's own
 * static device memory (one per device) -- the one piece of global state in
 * the library.  Its device address is looked up (cudaGetSymbolAddress) on
 * the first call in each CUDA context, with that context's device current,
 * and cached under the context's unique id, so a context created later (after
 * cudaDeviceReset, or a separate driver-API context) gets its own lookup;
 * make that first call before any stream capture.  The stream must belong to
 * the calling thread's current context.  The call allocates nothing (no
 * cudaMalloc / cudaFree / allocating library routine); it clears the
 * scratch's header and counters on `stream` before its launch, so stale
 * contents from an earlier call (even one that recorded a device error) do
 * not matter.  Every call on a device shares that array: calls that overlap
 * on the GPU (different streams without ordering, or concurrent host
 * threads) race and give undefined results.  Device-side errors are recorded
 * in the shared scratch's error word: eagle_tree_build_noalloc_error reads
 * the last call's.
 * Limit: the workspace of the shape,
 *   eagle_tree_build_workspace_size(1, n_rows, vocab, top_k, depth, m),
 *   must fit in EAGLE_NOALLOC_SCRATCH_BYTES; larger shapes return
 *   EAGLE_ERR_WORKSPACE_TOO_SMALL before anything is enqueued.  The size
 *   is about 0.7 KB + R * (16 + 8*top_k, rounded up to 16) bytes, R = 1 +
 *   (depth-1)*top_k rows: every shape with top_k <= 10 fits; e.g. top_k
 *   12, depth 13 does not (16,896 bytes).
 * ------------------------------------------------------------------------ */
#define EAGLE_NOALLOC_SCRATCH_BYTES (16u * 1024u)

eagle_status eagle_tree_build_noalloc(const float* draft_logits, int64_t row_stride,
                                      int32_t n_rows, int32_t vocab, int32_t top_k,
                                      int32_t depth, int32_t total_tokens, int32_t root_token,
                                      eagle_tree out, eagle_stream stream);

/* Synchronise `stream`, then read the error word of the static scratch as
 * eagle_workspace_error does for a workspace: the device-side status of the
 * last eagle_tree_build_noalloc call on the current device (EAGLE_OK,
 * EAGLE_ERR_TIMEOUT or EAGLE_ERR_DEVICE_ASSERT).  Allocates nothing. */
eagle_status eagle_tree_build_noalloc_error(eagle_stream stream, int32_t* status,
                                            int32_t* detail);

/* ------------------------------------------------------------------------
 * eagle_tree_build_policy -- tree shapes other than the dynamic top-k tree:
 *   [disc] reply on PR #3624 (a static tree: n candidate tokens taken at
 *   every decoding step) and the proposal of batched candidate sequences;
 *   [blog] "Context-Aware Dynamic Tree Construction in EAGLE-2" (confidence
 *   C = P(y1) / P(y2); above tau a linear chain, otherwise 2 to 4 branches).
 *
 * Nodes are numbered breadth-first (by depth, then parent, then the child's
 * rank in its parent's row), node 0 = the root (token root_token), pos =
 * depth, and draft row i (row i of draft_logits) is node i's draft output.
 *   EAGLE_POLICY_STATIC      every node above depth `depth` gets the `width`
 *                            best tokens of its row (a full width-ary tree);
 *                            total_tokens must be 1 + width + ... + width^depth;
 *                            rows read: the 1 + ... + width^(depth-1) inner nodes.
 *   EAGLE_POLICY_CHAINS      the root gets row 0's `width` best tokens; every
 *                            chain then grows by its last node's best token
 *                            to depth `depth` (>= 1); total_tokens must be
 *                            1 + width*depth; rows read: 1 + width*(depth-1)
 *                            (chain j's node at depth d is node 1+(d-1)*width+j).
 *   EAGLE_POLICY_CONFIDENCE  breadth-first; a node above depth `depth` whose
 *                            row has l1 - l2 > ln(tau) gets one child (its best
 *                            token), otherwise the b best tokens, b = the count
 *                            of tokens with l1 - l <= ln(tau) (2 <= b <= width,
 *                            width 2..8); children are added while the tree
 *                            has fewer than total_tokens nodes, so the tree
 *                            may come out smaller; rows read: total_tokens - 1.
 * Ties go to the lower token id; the logit gaps and ln(tau) are compared in
 * double precision (the gap of two float logits is exact there).
 *
 * draft_logits: float [n_rows][row_stride], 16-byte aligned, row_stride >= vocab,
 *               a multiple of 4; n_rows >= the rows the policy reads.
 * policy:       host pointer.
 * out:          out.m == total_tokens (the node slots); slots past the tree's
 *               size get parent -1, token -1, depth 0, pos 0 and no mask bits;
 *               out.values is not written.
 * n_nodes:      optional device int32: the tree's size (<= total_tokens).
 *               The tree can go to eagle_tree_attn / eagle_tree_verify with
 *               all total_tokens slots: a padded slot is nobody's child, so
 *               the walk never accepts it, and it sees no tree keys, so its
 *               attention output is unspecified (it has no keys at all when
 *               prefix_len is 0).
 * ws:           eagle_tree_policy_workspace_size(vocab, policy, total_tokens)
 *               bytes (0 = the policy or the sizes are rejected).
 * Errors: EAGLE_ERR_INVALID_ARG for a bad pointer, stride, policy field or a
 * total_tokens that does not match a static / chains shape;
 * EAGLE_ERR_UNSUPPORTED_SHAPE past EAGLE_MAX_TREE nodes, a width above
 * EAGLE_MAX_TOP_K (8 for the confidence policy) or above vocab.
 * ------------------------------------------------------------------------ */
#define EAGLE_POLICY_STATIC 0
#define EAGLE_POLICY_CHAINS 1
#define EAGLE_POLICY_CONFIDENCE 2

typedef struct {
  int32_t kind;    /* EAGLE_POLICY_*                                         */
  int32_t width;   /* static: children per node; chains: number of chains;   */
                   /* confidence: most branches per node (2..8)             */
  int32_t depth;   /* static / chains: depth; confidence: maximum depth      */
  int32_t reserved;
  double  tau;     /* confidence threshold (> 0); ignored by the others      */
} eagle_tree_policy;

size_t eagle_tree_policy_workspace_size(int32_t vocab, const eagle_tree_policy* policy,
                                        int32_t total_tokens);

eagle_status eagle_tree_build_policy(const float* draft_logits, int64_t row_stride,
                                     int32_t n_rows, int32_t vocab,
                                     const eagle_tree_policy* policy, int32_t total_tokens,
                                     int32_t root_token, eagle_tree out, int32_t* n_nodes,
                                     void* ws, size_t ws_bytes, eagle_stream stream);

/* ------------------------------------------------------------------------
 * eagle_tree_attn -- [blog] "Single-Pass Tree Verification" (a tree token
 * attends to its ancestors and itself, never to other branches) over the
 * target's KV cache of the accepted prefix ([disc] reply on KV caches).
 *
 *   out[i][h] = sum_j softmax_j(scale * q[i][h] . k_j) v_j,
 *   j over the prefix keys of kv head h / (n_q_heads / n_kv_heads) plus the
 *   tree keys t with mask bit (i, t) set.
 *
 * q:        [m][n_q_heads][head_dim]
 * k_cache,
 * v_cache:  [n_kv_heads][cache_head_stride] -- head h starts at
 *           h*cache_head_stride elements; its rows (one per prefix token,
 *           head_dim elements each) are contiguous; rows 0..prefix_len-1
 *           are read.  cache_head_stride >= prefix_len*head_dim, multiple
 *           of 8 elements; the pointers 16-byte aligned.
 * tree_k,
 * tree_v:   [m][n_kv_heads][head_dim]: keys / values of the tree tokens.
 * mask:     [m][(m+63)/64] ancestor bitmask (as written by eagle_tree_build).
 * out:      fp32 [m][n_q_heads][head_dim].
 * dtype:    element type of q / caches / tree k,v: EAGLE_BF16 (tensor-core
 *           path, head_dim 64 or 128) or EAGLE_F32 (CUDA-core path, head_dim
 *           <= 128, multiple of 4).
 * scale:    0 selects 1/sqrt(head_dim).
 * Limits: 1 <= m <= 256; n_q_heads % n_kv_heads == 0; prefix_len >= 0.
 * ------------------------------------------------------------------------ */
size_t eagle_tree_attn_workspace_size(int32_t m, int32_t n_q_heads, int32_t n_kv_heads,
                                      int32_t head_dim, int32_t prefix_len,
                                      eagle_dtype dtype);

eagle_status eagle_tree_attn(const void* q, const void* k_cache, const void* v_cache,
                             int64_t cache_head_stride, const void* tree_k,
                             const void* tree_v, const uint64_t* mask, int32_t m,
                             int32_t n_q_heads, int32_t n_kv_heads, int32_t head_dim,
                             int32_t prefix_len, eagle_dtype dtype, float scale,
                             float* out, void* ws, size_t ws_bytes, eagle_stream stream);

/* One independent attention problem per item (a layer, or a sequence of a
 * ragged batch), all in one launch.  Same head counts, head_dim and dtype for
 * every item; each item has its own pointers, m, prefix_len and cache stride. */
typedef struct {
  const void*     q;
  const void*     k_cache;
  const void*     v_cache;
  const void*     tree_k;
  const void*     tree_v;
  const uint64_t* mask;
  float*          out;
  int64_t         cache_head_stride;
  int32_t         prefix_len;
  int32_t         m;
} eagle_attn_item;

/* items: host array; only m and prefix_len are read here. */
size_t eagle_tree_attn_batched_workspace_size(const eagle_attn_item* items, int32_t n_items,
                                              int32_t n_q_heads, int32_t n_kv_heads,
                                              int32_t head_dim, eagle_dtype dtype);

/* Number of kernels one eagle_tree_attn_batched call with these items
 * launches (host-side planning only; items: host array, only m and
 * prefix_len are read). */
int32_t eagle_tree_attn_num_launches(const eagle_attn_item* items, int32_t n_items,
                                     int32_t n_q_heads, int32_t n_kv_heads, int32_t head_dim,
                                     eagle_dtype dtype);

eagle_status eagle_tree_attn_batched(const eagle_attn_item* items, int32_t n_items,
                                     int32_t n_q_heads, int32_t n_kv_heads, int32_t head_dim,
                                     eagle_dtype dtype, float scale,
                                     void* ws, size_t ws_bytes, eagle_stream stream);

/* Paged prefix cache (serving: the cache lives in a shared pool; [blog]
 * production section).  Fixed pages of EAGLE_KV_PAGE_TOKENS tokens: page j
 * of an item (its prefix tokens 128 j .. 128 j + 127) is pool rows
 * block_table[j] * 128 .. + 127 of every kv head.
 *
 * k_pool,
 * v_pool:          [n_kv_heads][pool_head_stride]; each head's rows (head_dim
 *                  elements each) are contiguous; pool_head_stride a multiple
 *                  of head_dim and of 8, at least one page; 16-byte aligned.
 * block_table:     device int32 [ceil(prefix_len / 128)] page ids; an id
 *                  outside the pool is recorded as EAGLE_ERR_DEVICE_ASSERT in
 *                  the workspace error word (page 0 is read instead).
 * Everything else as for eagle_tree_attn_batched; bf16 only, head_dim 64 or
 * 128 (the tensor-core path). */
#define EAGLE_KV_PAGE_TOKENS 128

typedef struct {
  const void*     q;
  const void*     k_pool;
  const void*     v_pool;
  const int32_t*  block_table;
  const void*     tree_k;
  const void*     tree_v;
  const uint64_t* mask;
  float*          out;
  int64_t         pool_head_stride;
  int32_t         prefix_len;
  int32_t         m;
} eagle_attn_paged_item;

size_t eagle_tree_attn_paged_workspace_size(const eagle_attn_paged_item* items,
                                            int32_t n_items, int32_t n_q_heads,
                                            int32_t n_kv_heads, int32_t head_dim);

eagle_status eagle_tree_attn_paged_batched(const eagle_attn_paged_item* items, int32_t n_items,
                                           int32_t n_q_heads, int32_t n_kv_heads,
                                           int32_t head_dim, float scale, void* ws,
                                           size_t ws_bytes, eagle_stream stream);

/* FP8 prefix cache (serving: half the bytes of a bf16 cache in the shared
 * pool; [blog] production section).  The pages give no number format; this
 * library reads it as E4M3 codes (1 sign, 4 exponent bits with bias 7, 3
 * mantissa bits; subnormals m * 2^-9; the code S.1111.111 is not a number;
 * largest magnitude 448) with one fp32 scale per (kv head, 128-token page):
 * prefix element = decode(code) * scale.  The tree's own keys / values are
 * bf16 (they are not cached yet when the tree is verified).
 *
 * k_cache,
 * v_cache:           uint8 E4M3 codes [n_kv_heads][cache_head_stride]; each
 *                    head's rows (head_dim codes each) contiguous; stride a
 *                    multiple of 16, at least prefix_len * head_dim; 16-byte
 *                    aligned.
 * k_scale, v_scale:  fp32 [n_kv_heads][scale_head_stride]: entry p of head h
 *                    scales prefix tokens 128 p .. 128 p + 127 of that head;
 *                    scale_head_stride >= ceil(prefix_len / 128).
 * q, tree_k, tree_v: bf16 as for eagle_tree_attn; out fp32.
 * The prefix's products run on fp16 tensor-core operands (codes widened
 * exactly; the query as fp16, exact for magnitudes in [2^-14, 65504];
 * softmax weights times the page's value scale as fp16): a query element
 * above 65504 in magnitude is reported as EAGLE_ERR_DEVICE_ASSERT with
 * detail 61, a value scale above 65504 with detail 62 (outputs then
 * unspecified).
 * head_dim 128 only (EAGLE_ERR_UNSUPPORTED_SHAPE otherwise); everything else
 * as for eagle_tree_attn_batched. */
typedef struct {
  const void*     q;
  const uint8_t*  k_cache;
  const uint8_t*  v_cache;
  const float*    k_scale;
  const float*    v_scale;
  const void*     tree_k;
  const void*     tree_v;
  const uint64_t* mask;
  float*          out;
  int64_t         cache_head_stride;
  int64_t         scale_head_stride;
  int32_t         prefix_len;
  int32_t         m;
} eagle_attn_fp8_item;

size_t eagle_tree_attn_fp8_workspace_size(const eagle_attn_fp8_item* items, int32_t n_items,
                                          int32_t n_q_heads, int32_t n_kv_heads,
                                          int32_t head_dim);

eagle_status eagle_tree_attn_fp8_batched(const eagle_attn_fp8_item* items, int32_t n_items,
                                         int32_t n_q_heads, int32_t n_kv_heads,
                                         int32_t head_dim, float scale, void* ws,
                                         size_t ws_bytes, eagle_stream stream);

/* ------------------------------------------------------------------------
 * eagle_tree_verify -- [blog] "Single-Pass Tree Verification" (walk from the
 * root, accept matching tokens until the first discrepancy; lossless) and
 * [disc] proposal (acceptance / rejection by speculative sampling).
 *
 * target_logits: fp32 [tree.m][row_stride] (16-byte aligned, row_stride % 4
 *   == 0); row i predicts the token that follows node i.
 * tree: as written by eagle_tree_build (parents, tokens and m are read).
 * params (host): greedy -> follow the argmax (ties -> lower id); the bonus
 *   token is the argmax at the last accepted node.  Sampling -> recursive
 *   speculative sampling over the children of the current node in node
 *   order with one-hot draft distributions: u_j = U(seed, step, node, j);
 *   accept child j iff u_j * (1 - rho) < p(token_j), else rho += p(token_j);
 *   with no child accepted (or at a leaf) the bonus token is the first token
 *   (ids ascending, rejected tokens removed) whose cumulative p exceeds
 *   U(seed, step, node, 0xffffffff) * (1 - rho).  U is Philox4x32-10 with
 *   key (seed lo, seed hi), counter (step lo, step hi, node, child), u =
 *   (word0 >> 8) * 2^-24.
 * accepted: device int32 [tree.m]: node ids of the accepted path starting
 *   with the root (entries past *n_accepted + 1 are left untouched).
 * n_accepted, bonus_token: device int32 scalars (accepted draft tokens,
 *   0..depth; the token to emit after them).
 * ------------------------------------------------------------------------ */
size_t eagle_tree_verify_workspace_size(int32_t n_items, int32_t m, int32_t vocab);

eagle_status eagle_tree_verify(const float* target_logits, int64_t row_stride, int32_t vocab,
                               eagle_tree tree, const eagle_sampling* params,
                               uint64_t seed, uint64_t step, int32_t* accepted,
                               int32_t* n_accepted, int32_t* bonus_token,
                               void* ws, size_t ws_bytes, eagle_stream stream);

/* n_items sequences (same m, row_stride, vocab) in one launch.  Host arrays:
 * target_logits, trees, params, seeds, accepted (device pointers each).
 * n_accepted, bonus_tokens: device int32 [n_items]. */
eagle_status eagle_tree_verify_batched(int32_t n_items, const float* const* target_logits,
                                       int64_t row_stride, int32_t vocab,
                                       const eagle_tree* trees, const eagle_sampling* params,
                                       const uint64_t* seeds, uint64_t step,
                                       int32_t* const* accepted, int32_t* n_accepted,
                                       int32_t* bonus_tokens,
                                       void* ws, size_t ws_bytes, eagle_stream stream);

/* ------------------------------------------------------------------------
 * eagle_tree_expand / eagle_tree_finalize -- the tree of eagle_tree_build,
 * grown one depth per call as the drafting loop produces the draft rows
 * ([blog] "The Recurrent Feature Drafting Step": the draft model runs on the
 * tokens just drafted, so the rows of depth l + 1 exist only once the
 * frontier of depth l is known; [disc] reply on the dynamic tree: expanded
 * step by step, pruned at the end of drafting).
 *
 * Call eagle_tree_expand for level = 0, 1, .., depth - 1 in order, then
 * eagle_tree_finalize; the result equals eagle_tree_build on the same rows
 * (level 0: the root's row; level l: row j = the draft row of frontier slot
 * j of depth l, j = 0 .. top_k - 1, i.e. draft rows 1 + (l-1) top_k + j of
 * the one-shot build).
 *
 * rows:         fp32 [1 or top_k][row_stride] (16-byte aligned, row_stride
 *               % 4 == 0).
 * state:        caller-owned device buffer of eagle_tree_state_bytes(top_k,
 *               depth) bytes (16-byte aligned) holding the growing tree
 *               between the calls of one drafting round (no host copy).
 * frontier_out: device int32 [2][top_k] or null: the new frontier (the
 *               top_k candidates of depth level + 1, best first): their
 *               tokens, then the frontier slot of their parent at depth level
 *               (0 at level 0) -- what the drafting loop feeds to its next
 *               draft-model pass.
 * ws:           eagle_tree_expand_workspace_size(top_k, vocab) bytes for the
 *               expand calls; at least 256 bytes (its error word) for
 *               finalize.
 * Errors: as eagle_tree_build; calls out of order (a level before the
 * previous one, finalize before depth levels) are recorded as
 * EAGLE_ERR_DEVICE_ASSERT in the workspace error word and write nothing.
 * ------------------------------------------------------------------------ */
size_t eagle_tree_state_bytes(int32_t top_k, int32_t depth);

size_t eagle_tree_expand_workspace_size(int32_t top_k, int32_t vocab);

eagle_status eagle_tree_expand(const float* rows, int64_t row_stride, int32_t vocab,
                               int32_t top_k, int32_t depth, int32_t level, void* state,
                               int32_t* frontier_out, void* ws, size_t ws_bytes,
                               eagle_stream stream);

eagle_status eagle_tree_finalize(const void* state, int32_t top_k, int32_t depth,
                                 int32_t total_tokens, int32_t root_token, eagle_tree out,
                                 void* ws, size_t ws_bytes, eagle_stream stream);

/* ------------------------------------------------------------------------
 * eagle_kv_commit -- [disc] reply on KV caches (the target model keeps the
 * KV cache of accepted tokens only) and [blog] "Single-Pass Tree
 * Verification" (the tree's keys / values come from one target pass; the
 * accepted tokens form a root-to-node path).  Appends the accepted path to
 * the prefix cache, for every kv head h and i = 0 .. *n_accepted:
 *
 *   k_cache[h][prefix_len + i][:] = tree_k[accepted[i]][h][:]   (same for v)
 *
 * The root is node 0 of the tree and has keys / values like every tree
 * token, so *n_accepted + 1 rows are written and the new prefix length is
 * prefix_len + *n_accepted + 1.  No other cache row is touched.
 *
 * k_cache,
 * v_cache:   [n_kv_heads][cache_head_stride] as for eagle_tree_attn; the
 *            head stride is also the capacity (cache_head_stride / head_dim
 *            rows), a multiple of head_dim; 16-byte aligned.
 * tree_k,
 * tree_v:    [m][n_kv_heads][head_dim] (16-byte aligned).
 * accepted:  device int32, node ids of the accepted path starting with the
 *            root; n_accepted: device int32 scalar (both as written by
 *            eagle_tree_verify; read on the device, no host synchronisation).
 * dtype:     EAGLE_BF16 or EAGLE_F32; head_dim * element size a multiple of
 *            16 bytes.
 * ws:        at least eagle_kv_commit_workspace_size() bytes (its error word).
 * Errors: bad arguments -> EAGLE_ERR_INVALID_ARG / UNSUPPORTED_SHAPE before
 * any launch.  A device value out of range (*n_accepted outside [0, m), the
 * committed rows past the capacity, an accepted id outside [0, m)) is
 * recorded as EAGLE_ERR_DEVICE_ASSERT in the workspace error word and the
 * affected rows are not written.
 * ------------------------------------------------------------------------ */
size_t eagle_kv_commit_workspace_size(void);

eagle_status eagle_kv_commit(void* k_cache, void* v_cache, int64_t cache_head_stride,
                             int32_t prefix_len, const void* tree_k, const void* tree_v,
                             int32_t m, int32_t n_kv_heads, int32_t head_dim, eagle_dtype dtype,
                             const int32_t* accepted, const int32_t* n_accepted,
                             void* ws, size_t ws_bytes, eagle_stream stream);

/* One commit per item (a layer of the target, or a sequence of a batch), all
 * in one launch per 64 items; same head count, head_dim and dtype. */
typedef struct {
  void*          k_cache;
  void*          v_cache;
  const void*    tree_k;
  const void*    tree_v;
  const int32_t* accepted;
  const int32_t* n_accepted;
  int64_t        cache_head_stride;
  int32_t        prefix_len;
  int32_t        m;
} eagle_kv_item;

eagle_status eagle_kv_commit_batched(const eagle_kv_item* items, int32_t n_items,
                                     int32_t n_kv_heads, int32_t head_dim, eagle_dtype dtype,
                                     void* ws, size_t ws_bytes, eagle_stream stream);

#ifdef __cplusplus
}
#endif

#endif /* EAGLE_H */
