// Launch plan shared by the attention kernels (CUDA-core path, merge, and the
// tcgen05 tensor-core path).
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include "eagle_common.cuh"

namespace eagle {

constexpr int kAttnMaxItems = 32;  // items per launch (more are chunked)
// SM count the split plans assume when no device can be queried (a
// workspace-size query on a host without a GPU); otherwise the plan fills the
// current device's SMs, and workspace sizes cover both plans.
constexpr int kPlanSMs = 152;

inline int plan_sms() {
  int dev = 0, n = 0;
  if (cudaGetDevice(&dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n < 1) {
    (void)cudaGetLastError();
    return kPlanSMs;
  }
  return n;
}

// Floats per (row, split) partial: head_dim outputs, then max (log2 units)
// and sum, padded to a 16-byte multiple.
__host__ __device__ constexpr int part_stride(int head_dim) { return head_dim + 4; }

struct AttnItemDev {
  const void* q;
  const void* k_cache;
  const void* v_cache;
  const void* tree_k;
  const void* tree_v;
  const uint64_t* mask;
  float* out;
  int64_t cache_head_stride;
  int32_t prefix_len;
  int32_t m;
};

struct AttnPlan {
  AttnItemDev items[kAttnMaxItems];
  int splits[kAttnMaxItems];
  int unit_start[kAttnMaxItems + 1];     // first CTA of each item
  int64_t row_start[kAttnMaxItems + 1];  // first output row (query x q head)
  int64_t part_start[kAttnMaxItems];     // first partial float of each item
  int64_t part_floats;
  int n_items, n_q_heads, n_kv_heads, head_dim;
  float scale;
  int32_t* err;
  float* partials;
};

// Launch the split merge (eagle_attn.cu) for a plan whose partials are set.
eagle_status launch_attn_merge(const AttnPlan& P, cudaStream_t stream);

// tensor-core path (eagle_attn_tc.cu)
bool tc_supported(int head_dim);
size_t attn_tc_ws_size(const eagle_attn_item* items, int n, int hq, int hkv, int d, int sms);
int attn_tc_num_launches(const eagle_attn_item* items, int n, int hq, int hkv, int d, int sms);
eagle_status attn_tc_launch(const eagle_attn_item* items, int n, int hq, int hkv, int d,
                            float scale, void* ws, size_t ws_bytes, cudaStream_t stream, int sms);

}  // namespace eagle
