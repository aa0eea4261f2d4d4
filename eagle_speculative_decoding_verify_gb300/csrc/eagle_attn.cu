// eagle_tree_attn: tree-masked GQA attention of the m tree tokens over the
// committed prefix KV cache plus the tree's own keys and values.
//
// Source: "EAGLE-2: Feature-Level Speculative Decoding Guide", "Single-Pass
// Tree Verification" (one target pass over the whole tree; a token sees its
// ancestors and itself, never another branch); "Support Eagle-3 Speculative
// Decoding in llama.cpp", reply on KV caches (the target keeps the KV cache of
// the accepted context).
//
// Split-KV (flash-decoding) plan: the prefix of every (item, kv head) is cut
// into splits; each split produces an unnormalised partial (o, max, sum) per
// query row and a merge kernel combines them with the log-sum-exp rule.  The
// tree keys go with the last split and are filtered by the ancestor mask.
//
// This file holds the CUDA-core path (fp32 inputs, or any head_dim), the
// merge kernel and the host entry points; the bf16 tensor-core path
// (tcgen05 + TMA) lives in eagle_attn_tc.cu.
#include <cuda_bf16.h>

#include "eagle_attn.h"
#include "eagle_host.h"

namespace eagle {

template <typename T>
__device__ __forceinline__ float to_f(T x);
template <>
__device__ __forceinline__ float to_f<float>(float x) { return x; }
template <>
__device__ __forceinline__ float to_f<__nv_bfloat16>(__nv_bfloat16 x) { return __bfloat162float(x); }

// One CTA = (item, kv head, query i, split).  The split's keys go through
// shared memory in chunks of kSimtKeys: fp32 rows by 16-byte asynchronous
// copies all issued at once (bf16 rows widened through registers), key rows
// padded to d + 4 floats so that 16-byte reads of different rows by the
// lanes of a quarter-warp fall on different banks.  The group's q vectors
// (pre-scaled) sit in shared memory.  Warp w handles q heads w, w+4, ... of
// the group; per 32-key step every lane scores its own key (float4 dot
// products, four independent sums), the warp forms the online-softmax update,
// the 32 weights go through shared memory, and lanes own head_dim columns
// lane, lane+32, ... of the output.
constexpr int kSimtKeys = 64;
constexpr int kSimtHeadsPerWarp = 8;   // group size g <= 32

__device__ __forceinline__ void cp_async16(void* dst, const void* src) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(smem_addr(dst)), "l"(src)
               : "memory");
}

template <typename T>
__global__ void __launch_bounds__(128) attn_simt_kernel(const __grid_constant__ AttnPlan P) {
  pdl_trigger();   // let a dependent launch of the next kernel start (see pdl_attribute)
  extern __shared__ __align__(16) float simt_smem[];
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  int item = 0;
  while (item + 1 < P.n_items && static_cast<int>(blockIdx.x) >= P.unit_start[item + 1]) ++item;
  const AttnItemDev& it = P.items[item];
  const int splits = P.splits[item];
  int u = blockIdx.x - P.unit_start[item];
  const int split = u % splits;
  u /= splits;
  const int i = u % it.m;
  const int kvh = u / it.m;
  const int d = P.head_dim, g = P.n_q_heads / P.n_kv_heads;
  const int E = (d + 31) / 32;
  const int ks = d + 4;                      // padded key row stride (floats, 16-byte rows)
  float* Ks = simt_smem;                     // [kSimtKeys][d + 4]
  float* Vs = Ks + kSimtKeys * ks;           // [kSimtKeys][d]
  float* Qs = Vs + kSimtKeys * d;            // [g][d], pre-scaled
  float* Ps = Qs + 32 * d;                   // [4 warps][32] weights of a step
  const int span = (it.prefix_len + splits - 1) / splits;
  const int j0 = min(it.prefix_len, split * span), j1 = min(it.prefix_len, j0 + span);
  const bool with_tree = (split == splits - 1);
  const int W = (it.m + 63) / 64;
  const float qscale = P.scale * 1.4426950408889634f;
  const T* kc = static_cast<const T*>(it.k_cache) + static_cast<int64_t>(kvh) * it.cache_head_stride;
  const T* vc = static_cast<const T*>(it.v_cache) + static_cast<int64_t>(kvh) * it.cache_head_stride;
  const T* tk = static_cast<const T*>(it.tree_k);
  const T* tv = static_cast<const T*>(it.tree_v);
  const uint64_t* mrow = it.mask + static_cast<int64_t>(i) * W;

  const T* qg = static_cast<const T*>(it.q) + (static_cast<int64_t>(i) * P.n_q_heads + kvh * g) * d;
  for (int x = threadIdx.x; x < g * d; x += blockDim.x) Qs[x] = to_f(__ldg(qg + x)) * qscale;

  float o[kSimtHeadsPerWarp][4], mx[kSimtHeadsPerWarp], l[kSimtHeadsPerWarp];
#pragma unroll
  for (int a = 0; a < kSimtHeadsPerWarp; ++a) {
    mx[a] = -INFINITY;
    l[a] = 0.f;
#pragma unroll
    for (int r = 0; r < 4; ++r) o[a][r] = 0.f;
  }

  // n keys whose rows start at element offsets row(k) (k < n) into K / V
  auto stage = [&](int n, auto row, const T* ksrc, const T* vsrc) {
    if constexpr (sizeof(T) == 4) {
      const int q4 = d / 4;
      for (int x = threadIdx.x; x < n * q4; x += blockDim.x) {
        const int k = x / q4, c = x - k * q4;
        const int64_t gi = row(k) + 4 * c;
        cp_async16(Ks + k * ks + 4 * c, ksrc + gi);
        cp_async16(Vs + k * d + 4 * c, vsrc + gi);
      }
      cp_async_commit();
      cp_async_wait_all();
    } else {
      for (int x = threadIdx.x; x < n * d; x += blockDim.x) {
        const int k = x / d, e = x - k * d;
        const int64_t gi = row(k) + e;
        Ks[k * ks + e] = to_f(__ldg(ksrc + gi));
        Vs[k * d + e] = to_f(__ldg(vsrc + gi));
      }
    }
  };

  // one chunk of n keys in shared memory; bit k of valid: key k counts
  auto consume = [&](int n, uint64_t valid) {
    for (int sub = 0; sub < n; sub += 32) {
      const int kk = sub + lane;
      const bool ok = kk < n && ((valid >> (kk & 63)) & 1ull);
      const float4* kr = reinterpret_cast<const float4*>(Ks + (kk < n ? kk : 0) * ks);
#pragma unroll
      for (int a = 0; a < kSimtHeadsPerWarp; ++a) {
        const int hl = warp + 4 * a;
        if (hl >= g) break;
        const float4* qr = reinterpret_cast<const float4*>(Qs + hl * d);
        float s4[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll 4
        for (int c = 0; c < d / 4; ++c) {
          const float4 qv = qr[c], kv = kr[c];
          s4[0] = fmaf(qv.x, kv.x, s4[0]);
          s4[1] = fmaf(qv.y, kv.y, s4[1]);
          s4[2] = fmaf(qv.z, kv.z, s4[2]);
          s4[3] = fmaf(qv.w, kv.w, s4[3]);
        }
        const float sc = ok ? (s4[0] + s4[1]) + (s4[2] + s4[3]) : -INFINITY;
        const float m_new = fmaxf(mx[a], warp_max(sc));
        if (m_new == -INFINITY) continue;   // nothing visible yet
        const float c0 = exp2f(mx[a] - m_new);
        const float p = ok ? exp2f(sc - m_new) : 0.f;
        float ps = p;
#pragma unroll
        for (int off = 16; off; off >>= 1) ps += __shfl_xor_sync(0xffffffffu, ps, off);
        l[a] = l[a] * c0 + ps;
        mx[a] = m_new;
        Ps[warp * 32 + lane] = p;
        __syncwarp();
        const int nk = min(32, n - sub);
#pragma unroll
        for (int r = 0; r < 4; ++r) {
          const int e = r * 32 + lane;
          if (r >= E || e >= d) break;
          float acc0 = o[a][r] * c0, acc1 = 0.f;
#pragma unroll 8
          for (int k = 0; k < 32; k += 2) {
            if (k < nk) acc0 = fmaf(Ps[warp * 32 + k], Vs[(sub + k) * d + e], acc0);
            if (k + 1 < nk) acc1 = fmaf(Ps[warp * 32 + k + 1], Vs[(sub + k + 1) * d + e], acc1);
          }
          o[a][r] = acc0 + acc1;
        }
        __syncwarp();
      }
    }
  };

  // prefix keys of this split
  for (int c0 = j0; c0 < j1; c0 += kSimtKeys) {
    const int n = min(kSimtKeys, j1 - c0);
    __syncthreads();   // the previous chunk is consumed (and Qs written, the first time)
    stage(n, [&](int k) { return static_cast<int64_t>(c0 + k) * d; }, kc, vc);
    __syncthreads();
    consume(n, ~0ull);
  }
  // tree keys (last split): the ancestor mask decides which count
  if (with_tree) {
    for (int c0 = 0; c0 < it.m; c0 += kSimtKeys) {
      const int n = min(kSimtKeys, it.m - c0);
      __syncthreads();
      stage(n, [&](int k) { return (static_cast<int64_t>(c0 + k) * P.n_kv_heads + kvh) * d; },
            tk, tv);
      __syncthreads();
      consume(n, mrow[c0 >> 6]);   // c0 is a multiple of 64: one mask word per chunk
    }
  }

#pragma unroll
  for (int a = 0; a < kSimtHeadsPerWarp; ++a) {
    const int hl = warp + 4 * a;
    if (hl >= g) break;
    const int64_t row = static_cast<int64_t>(i) * P.n_q_heads + kvh * g + hl;
    if (splits == 1) {
      const float inv = l[a] > 0.f ? 1.f / l[a] : 0.f;
#pragma unroll
      for (int r = 0; r < 4; ++r) {
        const int e = r * 32 + lane;
        if (r < E && e < d) it.out[row * d + e] = o[a][r] * inv;
      }
    } else {
      float* part = P.partials + P.part_start[item] +
                    (row * splits + split) * static_cast<int64_t>(part_stride(d));
#pragma unroll
      for (int r = 0; r < 4; ++r) {
        const int e = r * 32 + lane;
        if (r < E && e < d) part[e] = o[a][r];
      }
      if (lane == 0) {
        part[d] = mx[a];
        part[d + 1] = l[a];
      }
    }
  }
}

static size_t simt_smem_bytes(int d) {
  return sizeof(float) * (kSimtKeys * (2 * d + 4) + 32 * d + 4 * 32);
}

// Combine split partials: out = sum_s 2^(m_s - M) o_s / sum_s 2^(m_s - M) l_s
// (maxima are in log2 units).  One warp per (item, query row, q head).
__global__ void __launch_bounds__(128) attn_merge_kernel(const __grid_constant__ AttnPlan P) {
  pdl_trigger();   // let a dependent launch of the next kernel start (see pdl_attribute)
  const int lane = threadIdx.x & 31;
  const int64_t wid = static_cast<int64_t>(blockIdx.x) * 4 + (threadIdx.x >> 5);
  int item = 0;
  while (item + 1 < P.n_items && wid >= P.row_start[item + 1]) ++item;
  const AttnItemDev& it = P.items[item];
  const int64_t row = wid - P.row_start[item];
  if (row >= static_cast<int64_t>(it.m) * P.n_q_heads) return;
  const int splits = P.splits[item];
  if (splits == 1) return;
  const int d = P.head_dim;
  const int ps = part_stride(d);
  const float* part = P.partials + P.part_start[item] + row * splits * static_cast<int64_t>(ps);
  float M = -INFINITY;
  for (int s = 0; s < splits; ++s) M = fmaxf(M, __ldcg(part + s * ps + d));
  float L = 0.f;
  for (int s = 0; s < splits; ++s) {
    const float ms = __ldcg(part + s * ps + d);
    if (ms != -INFINITY) L += exp2f(ms - M) * __ldcg(part + s * ps + d + 1);
  }
  const float inv = L > 0.f ? 1.f / L : 0.f;
  for (int e = lane; e < d; e += 32) {
    float acc = 0.f;
    for (int s = 0; s < splits; ++s) {
      const float ms = __ldcg(part + s * ps + d);
      if (ms != -INFINITY) acc += exp2f(ms - M) * __ldcg(part + s * ps + e);
    }
    it.out[row * d + e] = acc * inv;
  }
}

// ------------------------------------------------------------------ host
eagle_status launch_attn_merge(const AttnPlan& P, cudaStream_t stream) {
  const int64_t rows = P.row_start[P.n_items];
  attn_merge_kernel<<<static_cast<int>((rows + 3) / 4), 128, 0, stream>>>(P);
  return launch_status();
}

static eagle_status validate(const eagle_attn_item* items, int n, int hq, int hkv, int d,
                             eagle_dtype dtype) {
  EAGLE_CHECK_ARG(items && n >= 1);
  EAGLE_CHECK_ARG(hq >= 1 && hkv >= 1 && hq % hkv == 0 && d >= 1);
  EAGLE_CHECK_ARG(dtype == EAGLE_F32 || dtype == EAGLE_BF16);
  EAGLE_CHECK_SHAPE(d <= 128 && d % 4 == 0);
  // the CUDA-core path (fp32, or a head_dim without tensor-core support)
  // handles groups of up to 32 q heads per kv head
  EAGLE_CHECK_SHAPE((dtype == EAGLE_BF16 && (d == 64 || d == 128)) || hq / hkv <= 32);
  for (int b = 0; b < n; ++b) {
    const eagle_attn_item& it = items[b];
    EAGLE_CHECK_ARG(it.m >= 1 && it.prefix_len >= 0);
    EAGLE_CHECK_SHAPE(it.m <= EAGLE_MAX_TREE);
    EAGLE_CHECK_ARG(it.q && it.tree_k && it.tree_v && it.mask && it.out);
    EAGLE_CHECK_ARG(it.prefix_len == 0 || (it.k_cache && it.v_cache));
    EAGLE_CHECK_ARG(it.cache_head_stride >= static_cast<int64_t>(it.prefix_len) * d);
    EAGLE_CHECK_ARG(it.cache_head_stride % 8 == 0);
    EAGLE_CHECK_ARG(aligned16(it.q) && aligned16(it.tree_k) && aligned16(it.tree_v) &&
                    aligned16(it.out));
    EAGLE_CHECK_ARG(it.prefix_len == 0 || (aligned16(it.k_cache) && aligned16(it.v_cache)));
  }
  return EAGLE_OK;
}

// SIMT plan: splits per item so that the grid covers the GPU a few times.
static void plan_simt(AttnPlan& P, const eagle_attn_item* items, int n, int hq, int hkv, int d,
                      float scale, int sms) {
  memset(&P, 0, sizeof(P));
  P.n_items = n;
  P.n_q_heads = hq;
  P.n_kv_heads = hkv;
  P.head_dim = d;
  P.scale = scale != 0.f ? scale : 1.0f / sqrtf(static_cast<float>(d));
  int64_t base = 0;
  for (int b = 0; b < n; ++b) base += static_cast<int64_t>(hkv) * items[b].m;
  const int64_t target = static_cast<int64_t>(sms) * 8;
  int64_t units = 0, rows = 0, part = 0;
  for (int b = 0; b < n; ++b) {
    const eagle_attn_item& it = items[b];
    int splits = static_cast<int>((target + base - 1) / (base > 0 ? base : 1));
    const int max_splits = (it.prefix_len + 127) / 128;
    if (splits > max_splits) splits = max_splits;
    if (splits < 1) splits = 1;
    P.splits[b] = splits;
    P.unit_start[b] = static_cast<int>(units);
    P.row_start[b] = rows;
    P.part_start[b] = part;
    units += static_cast<int64_t>(hkv) * it.m * splits;
    rows += static_cast<int64_t>(it.m) * hq;
    if (splits > 1) part += static_cast<int64_t>(it.m) * hq * splits * part_stride(d);
    AttnItemDev& di = P.items[b];
    di.q = it.q;
    di.k_cache = it.k_cache;
    di.v_cache = it.v_cache;
    di.tree_k = it.tree_k;
    di.tree_v = it.tree_v;
    di.mask = it.mask;
    di.out = it.out;
    di.cache_head_stride = it.cache_head_stride;
    di.prefix_len = it.prefix_len;
    di.m = it.m;
  }
  P.unit_start[n] = static_cast<int>(units);
  P.row_start[n] = rows;
  P.part_floats = part;
}

static size_t simt_ws(const AttnPlan& P) {
  return align_up(kWsHeader + sizeof(float) * static_cast<size_t>(P.part_floats), 256);
}

static eagle_status attn_batched_impl(const eagle_attn_item* items, int32_t n, int32_t hq,
                                      int32_t hkv, int32_t d, eagle_dtype dtype, float scale,
                                      void* ws, size_t ws_bytes, cudaStream_t stream) {
  eagle_status st = validate(items, n, hq, hkv, d, dtype);
  if (st != EAGLE_OK) return st;
  EAGLE_CHECK_ARG(ws != nullptr);
  const int sms = plan_sms();
  for (int b0 = 0; b0 < n; b0 += kAttnMaxItems) {
    const int nb = (n - b0) < kAttnMaxItems ? (n - b0) : kAttnMaxItems;
    if (dtype == EAGLE_BF16 && tc_supported(d)) {
      st = attn_tc_launch(items + b0, nb, hq, hkv, d, scale, ws, ws_bytes, stream, sms);
      if (st != EAGLE_OK) return st;
      continue;
    }
    AttnPlan P;
    plan_simt(P, items + b0, nb, hq, hkv, d, scale, sms);
    if (ws_bytes < simt_ws(P)) return EAGLE_ERR_WORKSPACE_TOO_SMALL;
    P.err = static_cast<int32_t*>(ws);
    P.partials = reinterpret_cast<float*>(static_cast<char*>(ws) + kWsHeader);
    const int grid = P.unit_start[nb];
    const size_t smem = simt_smem_bytes(d);
    if (dtype == EAGLE_F32) {
      EAGLE_CUDA(cudaFuncSetAttribute(attn_simt_kernel<float>,
                                      cudaFuncAttributeMaxDynamicSharedMemorySize,
                                      static_cast<int>(smem)));
      attn_simt_kernel<float><<<grid, 128, smem, stream>>>(P);
    } else {
      EAGLE_CUDA(cudaFuncSetAttribute(attn_simt_kernel<__nv_bfloat16>,
                                      cudaFuncAttributeMaxDynamicSharedMemorySize,
                                      static_cast<int>(smem)));
      attn_simt_kernel<__nv_bfloat16><<<grid, 128, smem, stream>>>(P);
    }
    if ((st = launch_status()) != EAGLE_OK) return st;
    if (P.part_floats > 0 && (st = launch_attn_merge(P, stream)) != EAGLE_OK) return st;
  }
  return EAGLE_OK;
}

static size_t attn_ws_size(const eagle_attn_item* items, int32_t n, int32_t hq, int32_t hkv,
                           int32_t d, eagle_dtype dtype) {
  if (!items || n < 1 || hq < 1 || hkv < 1 || d < 1) return 0;
  size_t need = kWsHeader;
  // large enough for the plan of the current device and for the default one
  for (const int sms : {kPlanSMs, plan_sms()})
    for (int b0 = 0; b0 < n; b0 += kAttnMaxItems) {
      const int nb = (n - b0) < kAttnMaxItems ? (n - b0) : kAttnMaxItems;
      size_t s;
      if (dtype == EAGLE_BF16 && tc_supported(d)) {
        s = attn_tc_ws_size(items + b0, nb, hq, hkv, d, sms);
      } else {
        AttnPlan P;
        plan_simt(P, items + b0, nb, hq, hkv, d, 0.f, sms);
        s = simt_ws(P);
      }
      if (s > need) need = s;
    }
  return need;
}

static int32_t attn_num_launches(const eagle_attn_item* items, int32_t n, int32_t hq,
                                 int32_t hkv, int32_t d, eagle_dtype dtype) {
  if (!items || n < 1 || hq < 1 || hkv < 1 || d < 1) return 0;
  int32_t count = 0;
  for (int b0 = 0; b0 < n; b0 += kAttnMaxItems) {
    const int nb = (n - b0) < kAttnMaxItems ? (n - b0) : kAttnMaxItems;
    if (dtype == EAGLE_BF16 && tc_supported(d)) {
      count += attn_tc_num_launches(items + b0, nb, hq, hkv, d, plan_sms());
    } else {
      AttnPlan P;
      plan_simt(P, items + b0, nb, hq, hkv, d, 0.f, plan_sms());
      count += 1 + (P.part_floats > 0 ? 1 : 0);
    }
  }
  return count;
}

}  // namespace eagle

using namespace eagle;

extern "C" int32_t eagle_tree_attn_num_launches(const eagle_attn_item* items, int32_t n_items,
                                                int32_t n_q_heads, int32_t n_kv_heads,
                                                int32_t head_dim, eagle_dtype dtype) {
  return attn_num_launches(items, n_items, n_q_heads, n_kv_heads, head_dim, dtype);
}

extern "C" size_t eagle_tree_attn_batched_workspace_size(const eagle_attn_item* items,
                                                         int32_t n_items, int32_t n_q_heads,
                                                         int32_t n_kv_heads, int32_t head_dim,
                                                         eagle_dtype dtype) {
  return attn_ws_size(items, n_items, n_q_heads, n_kv_heads, head_dim, dtype);
}

extern "C" size_t eagle_tree_attn_workspace_size(int32_t m, int32_t n_q_heads,
                                                 int32_t n_kv_heads, int32_t head_dim,
                                                 int32_t prefix_len, eagle_dtype dtype) {
  eagle_attn_item it;
  memset(&it, 0, sizeof(it));
  it.m = m;
  it.prefix_len = prefix_len;
  return attn_ws_size(&it, 1, n_q_heads, n_kv_heads, head_dim, dtype);
}

extern "C" eagle_status eagle_tree_attn_batched(const eagle_attn_item* items, int32_t n_items,
                                                int32_t n_q_heads, int32_t n_kv_heads,
                                                int32_t head_dim, eagle_dtype dtype, float scale,
                                                void* ws, size_t ws_bytes,
                                                eagle_stream stream) {
  return attn_batched_impl(items, n_items, n_q_heads, n_kv_heads, head_dim, dtype, scale, ws,
                           ws_bytes, reinterpret_cast<cudaStream_t>(stream));
}

extern "C" eagle_status eagle_tree_attn(const void* q, const void* k_cache, const void* v_cache,
                                        int64_t cache_head_stride, const void* tree_k,
                                        const void* tree_v, const uint64_t* mask, int32_t m,
                                        int32_t n_q_heads, int32_t n_kv_heads, int32_t head_dim,
                                        int32_t prefix_len, eagle_dtype dtype, float scale,
                                        float* out, void* ws, size_t ws_bytes,
                                        eagle_stream stream) {
  eagle_attn_item it;
  it.q = q;
  it.k_cache = k_cache;
  it.v_cache = v_cache;
  it.tree_k = tree_k;
  it.tree_v = tree_v;
  it.mask = mask;
  it.out = out;
  it.cache_head_stride = cache_head_stride;
  it.prefix_len = prefix_len;
  it.m = m;
  return attn_batched_impl(&it, 1, n_q_heads, n_kv_heads, head_dim, dtype, scale, ws, ws_bytes,
                           reinterpret_cast<cudaStream_t>(stream));
}
