// eagle_kv_commit / eagle_kv_commit_batched: append the accepted path's keys
// and values to the target's KV cache.
//
// Source: "Support Eagle-3 Speculative Decoding in llama.cpp", reply on KV
// caches (the target keeps the KV cache of accepted tokens only);
// "EAGLE-2: Feature-Level Speculative Decoding Guide", "Single-Pass Tree
// Verification" (the tree's keys and values come from one target pass; the
// accepted tokens are a root-to-node path).
//
// For item b, kv head h and i = 0 .. n (n = *n_accepted, read on the device):
//   k_cache[h][prefix_len + i][:] = tree_k[accepted[i]][h][:]   (same for v)
// A pure gather / scatter of (n + 1) rows per head: one block per (item, kv
// head), 16-byte vector copies, every device-side value bounds-checked
// before it is used (a bad one is recorded in the workspace error word and
// its row is skipped).
#include "eagle_common.cuh"
#include "eagle_host.h"

namespace eagle {

constexpr int kKvMaxItems = 64;     // items per launch (pointers live in the params)
constexpr int kKvThreads = 128;

struct KvItem {
  uint8_t* k_cache;
  uint8_t* v_cache;
  const uint8_t* tree_k;
  const uint8_t* tree_v;
  const int32_t* accepted;
  const int32_t* n_accepted;
  int64_t head_bytes;   // cache head stride in bytes
  int32_t prefix_len, m, cap_rows;
};

struct KvParams {
  KvItem items[kKvMaxItems];
  int n_kv_heads, row_bytes;   // row_bytes = head_dim * element size (multiple of 16)
  int32_t* err;
};

__global__ void __launch_bounds__(kKvThreads) kv_commit_kernel(const __grid_constant__ KvParams P) {
  pdl_trigger();   // dependent launch: see pdl_attribute
  pdl_wait();
  const int item = blockIdx.x / P.n_kv_heads;
  const int h = blockIdx.x - item * P.n_kv_heads;
  const KvItem& it = P.items[item];
  const int n = *it.n_accepted;
  if (n < 0 || n >= it.m || it.prefix_len + n + 1 > it.cap_rows) {
    if (threadIdx.x == 0 && h == 0) record_error(P.err, kDevAssert, 40);
    return;
  }
  const int vec_per_row = P.row_bytes / 16;
  const int rows = n + 1;
  // one 16-byte vector per thread and step, over (row, vector) pairs, for K then V
  for (int e = threadIdx.x; e < 2 * rows * vec_per_row; e += kKvThreads) {
    const int kv = e / (rows * vec_per_row);
    const int r = e - kv * rows * vec_per_row;
    const int i = r / vec_per_row, c = r - i * vec_per_row;
    const int node = __ldg(it.accepted + i);
    if (node < 0 || node >= it.m) {
      if (c == 0 && kv == 0 && h == 0) record_error(P.err, kDevAssert, 41);
      continue;
    }
    const uint8_t* src = (kv ? it.tree_v : it.tree_k) +
                         (static_cast<int64_t>(node) * P.n_kv_heads + h) * P.row_bytes;
    uint8_t* dst = (kv ? it.v_cache : it.k_cache) + h * it.head_bytes +
                   static_cast<int64_t>(it.prefix_len + i) * P.row_bytes;
    reinterpret_cast<int4*>(dst)[c] = __ldg(reinterpret_cast<const int4*>(src) + c);
  }
}

static eagle_status commit_impl(const eagle_kv_item* items, int32_t n_items, int32_t n_kv_heads,
                                int32_t head_dim, eagle_dtype dtype, void* ws, size_t ws_bytes,
                                cudaStream_t stream) {
  EAGLE_CHECK_ARG(items && n_items >= 1 && n_kv_heads >= 1 && head_dim >= 1 && ws);
  EAGLE_CHECK_ARG(dtype == EAGLE_BF16 || dtype == EAGLE_F32);
  EAGLE_CHECK_ARG(ws_bytes >= kWsHeader && aligned16(ws));
  const int esize = dtype == EAGLE_BF16 ? 2 : 4;
  const int64_t row_bytes = static_cast<int64_t>(head_dim) * esize;
  EAGLE_CHECK_SHAPE(row_bytes % 16 == 0 && row_bytes <= (1 << 20));
  for (int b = 0; b < n_items; ++b) {
    const eagle_kv_item& x = items[b];
    EAGLE_CHECK_ARG(x.k_cache && x.v_cache && x.tree_k && x.tree_v && x.accepted && x.n_accepted);
    EAGLE_CHECK_ARG(aligned16(x.k_cache) && aligned16(x.v_cache) && aligned16(x.tree_k) &&
                    aligned16(x.tree_v));
    EAGLE_CHECK_ARG(x.m >= 1 && x.prefix_len >= 0 && x.cache_head_stride >= head_dim &&
                    x.cache_head_stride % head_dim == 0 && (x.cache_head_stride * esize) % 16 == 0);
    EAGLE_CHECK_ARG(x.cache_head_stride / head_dim <= INT32_MAX);
  }
  for (int b0 = 0; b0 < n_items; b0 += kKvMaxItems) {
    const int nb = n_items - b0 < kKvMaxItems ? n_items - b0 : kKvMaxItems;
    KvParams P;
    memset(&P, 0, sizeof(P));
    for (int b = 0; b < nb; ++b) {
      const eagle_kv_item& x = items[b0 + b];
      KvItem& k = P.items[b];
      k.k_cache = static_cast<uint8_t*>(x.k_cache);
      k.v_cache = static_cast<uint8_t*>(x.v_cache);
      k.tree_k = static_cast<const uint8_t*>(x.tree_k);
      k.tree_v = static_cast<const uint8_t*>(x.tree_v);
      k.accepted = x.accepted;
      k.n_accepted = x.n_accepted;
      k.head_bytes = x.cache_head_stride * esize;
      k.prefix_len = x.prefix_len;
      k.m = x.m;
      k.cap_rows = static_cast<int32_t>(x.cache_head_stride / head_dim);
    }
    P.n_kv_heads = n_kv_heads;
    P.row_bytes = static_cast<int>(row_bytes);
    P.err = static_cast<int32_t*>(ws);
    EAGLE_CUDA(launch_pdl(kv_commit_kernel, dim3(static_cast<unsigned>(nb * n_kv_heads)),
                          dim3(kKvThreads), 0, stream, P));
    const eagle_status st = launch_status();
    if (st != EAGLE_OK) return st;
  }
  return EAGLE_OK;
}

}  // namespace eagle

using namespace eagle;

extern "C" size_t eagle_kv_commit_workspace_size(void) { return kWsHeader; }

extern "C" eagle_status eagle_kv_commit(void* k_cache, void* v_cache, int64_t cache_head_stride,
                                        int32_t prefix_len, const void* tree_k, const void* tree_v,
                                        int32_t m, int32_t n_kv_heads, int32_t head_dim,
                                        eagle_dtype dtype, const int32_t* accepted,
                                        const int32_t* n_accepted, void* ws, size_t ws_bytes,
                                        eagle_stream stream) {
  eagle_kv_item x;
  x.k_cache = k_cache;
  x.v_cache = v_cache;
  x.tree_k = tree_k;
  x.tree_v = tree_v;
  x.accepted = accepted;
  x.n_accepted = n_accepted;
  x.cache_head_stride = cache_head_stride;
  x.prefix_len = prefix_len;
  x.m = m;
  return commit_impl(&x, 1, n_kv_heads, head_dim, dtype, ws, ws_bytes,
                     reinterpret_cast<cudaStream_t>(stream));
}

extern "C" eagle_status eagle_kv_commit_batched(const eagle_kv_item* items, int32_t n_items,
                                                int32_t n_kv_heads, int32_t head_dim,
                                                eagle_dtype dtype, void* ws, size_t ws_bytes,
                                                eagle_stream stream) {
  return commit_impl(items, n_items, n_kv_heads, head_dim, dtype, ws, ws_bytes,
                     reinterpret_cast<cudaStream_t>(stream));
}
