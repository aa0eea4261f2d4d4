// Tensor-core path of eagle_tree_attn for bf16 Q/K/V (head_dim 64 or 128).
//
// Source: "EAGLE-2: Feature-Level Speculative Decoding Guide", "Single-Pass
// Tree Verification" (one target pass over the tree; a token attends to its
// ancestors and itself only) over the target's prefix KV cache.
//
// The m tree queries of one KV head times its g query heads form the M
// dimension (row R = i*g + head-in-group), so the g heads that share a KV
// head share every K/V byte.  One CTA = (item, kv head, pair of 128-row
// query tiles, split).  Splits 0..n-2 each take a contiguous span of prefix
// chunks (128 keys); the last split takes the tree keys only (a CTA of its
// own, so the masked chunk with its two P fills is off the prefix critical
// path).  Warp-specialised:
//   warp 0      TMA producer: K and V chunks into a 5-slot ring of
//               128-byte-swizzled shared-memory tiles.
//   warp 1      tensor-memory owner and MMA issuer: S_t = Q_t K^T (M 128,
//               N 128, K = head_dim, A and B from shared memory) and
//               O_t += P_t V (M 128, N = head_dim, K 128, A = P from tensor
//               memory) with tcgen05.mma kind::f16, fp32 accumulators in
//               tensor memory (S_0, S_1, O_0, O_1 = 512 columns).  The MMAs
//               of a thread run in issue order, so PV_t(j) has read P_t(j)
//               before S_t(j+1) overwrites those columns, and the completion
//               of S_t(j+1) implies that of PV_t(j).
//   warps 4-7   softmax for tile 0, warps 8-11 for tile 1: one thread per
//   / 8-11      query row reads its S row from tensor memory, applies scale,
//               the prefix bound and the ancestor mask, updates the running
//               max / sum (O rescaled in tensor memory only when the max
//               grows by more than 2^8) and writes P as bf16 over the S
//               columns it has read (32 keys -> 16 columns); for tree keys
//               (few, possibly dominant) the bf16 rounding residual goes to
//               the next 16 columns and a second MMA adds it, so that O
//               accumulates P to ~2^-17.
// The epilogue writes the normalised row (one split) or an unnormalised
// partial (o, max, sum) that attn_tc_merge_kernel combines.  Every mbarrier
// wait is bounded; on a timeout the CTA records the error, drains its own
// copies and MMAs, frees tensor memory and returns.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_bf16.h>

#include <algorithm>
#include <mutex>

#include "eagle_attn.h"
#include "eagle_host.h"
#include "eagle_tc.cuh"

namespace eagle {

constexpr int kTcMaxItems = 16;     // items per launch (tensor maps live in the params)
constexpr int kTcThreads = 384;     // 12 warps
constexpr int kChunk = 128;         // keys per K/V chunk
constexpr int kSlots = 5;           // K/V ring depth
constexpr uint32_t kTmemCols = 512;

struct TcItem {
  const __nv_bfloat16* q;
  float* out;
  const uint64_t* mask;
  int m, prefix_len, splits, tile_pairs, unit_start;
  int64_t part_start;   // first partial unit of the item (units of 256 rows)
};

struct TcParams {
  CUtensorMap kmap[kTcMaxItems];
  CUtensorMap vmap[kTcMaxItems];
  CUtensorMap tkmap[kTcMaxItems];
  CUtensorMap tvmap[kTcMaxItems];
  TcItem items[kTcMaxItems];
  int n_items, hq, hkv, g, span_chunks, total_units;
  float scale_log2;
  float* part_o;     // [unit][256 rows][D]
  float2* part_ml;   // [unit][256 rows] (max in log2 units, sum)
  int32_t* err;
};

template <int D>
struct TcSmem {
  static constexpr int kTileBytes = 128 * D * 2;      // one 128-row bf16 tile of width D
  static constexpr int kQ = 0;
  static constexpr int kRing = kQ + 2 * kTileBytes;
  static constexpr int kBars = kRing + kSlots * kTileBytes;
  static constexpr int kBytes = kBars + 256;
  static constexpr int kAlloc = kBytes + 1024;        // slack for 1024-byte alignment
};
static_assert(TcSmem<128>::kAlloc <= 232448, "shared memory of the tensor-core kernel");

__device__ __forceinline__ bool bounded_wait(uint64_t* bar, uint32_t parity, int32_t* err,
                                             volatile int* abort_flag, int where) {
  if (*abort_flag) return false;
  if (mbar_wait(bar, parity)) return true;
  record_error(err, kDevTimeout, where);
  *abort_flag = 1;
  return false;
}

template <int D>
__global__ void __launch_bounds__(kTcThreads, 1) attn_tc_kernel(const __grid_constant__ TcParams P) {
  using L = TcSmem<D>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + L::kBars);
  uint64_t* empty = full + kSlots;
  uint64_t* s_full = empty + kSlots;    // [2]
  uint64_t* p_full = s_full + 2;        // [2]
  uint64_t* o_done = p_full + 2;        // [2]
  uint64_t* drain = o_done + 2;         // [1]
  uint64_t* q_ready = drain + 1;        // [1] Q tiles written (8 softmax warps)
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(q_ready + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;

  // ---- work unit
  int item = 0;
  while (item + 1 < P.n_items && static_cast<int>(blockIdx.x) >= P.items[item + 1].unit_start)
    ++item;
  const TcItem& it = P.items[item];
  int u = blockIdx.x - it.unit_start;
  const int split = u % it.splits;
  u /= it.splits;
  const int tp = u % it.tile_pairs;
  const int kvh = u / it.tile_pairs;
  const int g = P.g;
  const int M = it.m * g;
  const int n_tiles = (M - 256 * tp) > 128 ? 2 : 1;
  const bool tree_split = split == it.splits - 1;
  const int split_start = split * P.span_chunks * kChunk;
  const int split_end = tree_split ? 0 : min(it.prefix_len, split_start + P.span_chunks * kChunk);
  const int n_pref = split_end > split_start ? (split_end - split_start + kChunk - 1) / kChunk : 0;
  const int n_chunks = n_pref + (tree_split ? (it.m + kChunk - 1) / kChunk : 0);

  if (tid == 0) {
    for (int s = 0; s < kSlots; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    for (int t = 0; t < 2; ++t) {
      mbar_init(&s_full[t], 1);
      mbar_init(&p_full[t], 4);   // one arrival per softmax warp
      mbar_init(&o_done[t], 1);
    }
    mbar_init(drain, 1);
    mbar_init(q_ready, 8);
    *abort_flag = 0;
    fence_barrier_init();
  }
  if (warp == 1) {
    tmem_alloc(tmem_slot, kTmemCols);
    tmem_relinquish();
  }
  if (warp == 0 && lane == 0) {
    tma_prefetch_map(&P.kmap[item]);
    tma_prefetch_map(&P.vmap[item]);
    tma_prefetch_map(&P.tkmap[item]);
    tma_prefetch_map(&P.tvmap[item]);
  }

  tc_fence_before();
  __syncthreads();   // barriers initialised, tensor memory allocated
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const uint32_t tmem_S = tmem;               // S_t at column 128 t (P_t aliases it)
  const uint32_t tmem_O = tmem + 256;         // O_t at column 256 + D t

  // ---- Q tiles -> shared memory (128-byte swizzle), mask rows -> registers;
  // the producer is already streaming K/V meanwhile
  const int wg = warp >= 4 ? (warp - 4) >> 2 : -1;   // softmax warpgroup = query tile
  const int row = (warp & 3) * 32 + lane;            // row within the tile = TMEM lane
  const int R = 256 * tp + 128 * (wg < 0 ? 0 : wg) + row;
  if (wg >= 0) {
    uint8_t* qt = smem + L::kQ + wg * L::kTileBytes;
    const bool valid = R < M;
    const int qi = valid ? R / g : 0;
    const int hl = valid ? R - qi * g : 0;
    const int4* src = reinterpret_cast<const int4*>(
        it.q + (static_cast<int64_t>(qi) * P.hq + kvh * g + hl) * D);
    int4 qv[D / 8];
#pragma unroll
    for (int c = 0; c < D / 8; ++c) qv[c] = valid ? __ldg(src + c) : make_int4(0, 0, 0, 0);
#pragma unroll
    for (int c = 0; c < D / 8; ++c) {   // 16-byte chunks of the row
      const int half = c >> 3, cc = c & 7;
      *reinterpret_cast<int4*>(qt + half * (128 * 128) + row * 128 + ((cc ^ (row & 7)) << 4)) = qv[c];
    }
    fence_proxy_async_smem();
    __syncwarp();
    if (lane == 0) mbar_arrive(q_ready);
  }

  if (warp == 0) {
    // ================================================================ TMA producer
    if (lane == 0) {
      constexpr uint32_t kBytesChunk = static_cast<uint32_t>(L::kTileBytes);
      int issued = 0;
      for (int n = 0; n < 2 * n_chunks; ++n) {
        const int slot = n % kSlots, use = n / kSlots;
        if (use > 0 && !bounded_wait(&empty[slot], (use - 1) & 1, P.err, abort_flag, 20)) break;
        const int j = n >> 1;
        const bool is_v = n & 1;
        uint8_t* dst = smem + L::kRing + slot * L::kTileBytes;
        mbar_arrive_expect_tx(&full[slot], kBytesChunk);
        if (j < n_pref) {
          const CUtensorMap* map = is_v ? &P.vmap[item] : &P.kmap[item];
          const int y = split_start + j * kChunk;
#pragma unroll
          for (int h = 0; h < D / 64; ++h) tma_load_3d(dst + h * 128 * 128, map, 64 * h, y, kvh, &full[slot]);
        } else {
          const CUtensorMap* map = is_v ? &P.tvmap[item] : &P.tkmap[item];
          const int z = (j - n_pref) * kChunk;
#pragma unroll
          for (int h = 0; h < D / 64; ++h) tma_load_3d(dst + h * 128 * 128, map, 64 * h, kvh, z, &full[slot]);
        }
        issued = n + 1;
      }
      // make sure no copy of ours is still landing when the CTA leaves
      for (int n = (issued > kSlots ? issued - kSlots : 0); n < issued; ++n)
        mbar_wait(&full[n % kSlots], (n / kSlots) & 1, 200000000ull);
    }
  } else if (warp == 1) {
    // ================================================================ MMA issuer
    if (lane == 0) {
      constexpr uint32_t idesc_s = idesc_bf16_f32(128, kChunk, false);
      constexpr uint32_t idesc_o = idesc_bf16_f32(128, D, true);
      const uint32_t q_base = smem_addr(smem + L::kQ);
      const uint32_t ring_base = smem_addr(smem + L::kRing);
      auto issue_s = [&](int t, int slot) {   // S_t = Q_t K^T
        const uint32_t qa = q_base + t * L::kTileBytes;
        const uint32_t kb = ring_base + slot * L::kTileBytes;
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint32_t off = (kk >> 2) * (128 * 128) + (kk & 3) * 32;
          mma_bf16(tmem_S + 128 * t, smem_desc_sw128(qa + off, 16, 1024),
                   smem_desc_sw128(kb + off, 16, 1024), idesc_s, kk > 0);
        }
      };
      auto issue_pv = [&](int t, int slot, int fill, bool acc) {   // O_t += P_t V
        // keys 16kk.. : columns 32 (kk/2) + 16 fill + 8 (kk%2) of S_t (bf16 pairs)
        const uint32_t pa = tmem_S + 128 * t + 16 * fill;
        const uint32_t vb = ring_base + slot * L::kTileBytes;
#pragma unroll
        for (int kk = 0; kk < kChunk / 16; ++kk)
          mma_bf16_ta(tmem_O + D * t, pa + 32 * (kk >> 1) + 8 * (kk & 1),
                      smem_desc_sw128(vb + kk * 2048, 128 * 128, 1024), idesc_o, (acc || kk > 0));
      };
      bool ok = n_chunks > 0 && bounded_wait(q_ready, 0, P.err, abort_flag, 29) &&
                bounded_wait(&full[0], 0, P.err, abort_flag, 30);
      if (ok) {
        tc_fence_after();
        for (int t = 0; t < n_tiles; ++t) {
          issue_s(t, 0);
          mma_commit(&s_full[t]);
        }
        mma_commit(&empty[0]);
      }
      for (int j = 0; ok && j < n_chunks; ++j) {
        const int nv = 2 * j + 1, nk = 2 * j + 2;
        const int vslot = nv % kSlots, kslot = nk % kSlots;
        const int nf = j < n_pref ? 1 : 2;   // tree keys: P = hi + lo
        if (!bounded_wait(&full[vslot], (nv / kSlots) & 1, P.err, abort_flag, 31)) break;
        tc_fence_after();
        const bool more = j + 1 < n_chunks;
        for (int t = 0; t < n_tiles; ++t) {
          if (!bounded_wait(&p_full[t], j & 1, P.err, abort_flag, 32)) { ok = false; break; }
          tc_fence_after();
          for (int f = 0; f < nf; ++f) issue_pv(t, vslot, f, j > 0 || f > 0);
          mma_commit(&o_done[t]);
          if (more) {
            if (t == 0) {
              if (!bounded_wait(&full[kslot], (nk / kSlots) & 1, P.err, abort_flag, 33)) { ok = false; break; }
              tc_fence_after();
            }
            issue_s(t, kslot);
            mma_commit(&s_full[t]);
          }
        }
        if (!ok) break;
        if (more) mma_commit(&empty[kslot]);
        mma_commit(&empty[vslot]);
      }
      // every MMA of this CTA has completed once `drain` flips
      mma_commit(drain);
      mbar_wait(drain, 0, 200000000ull);
    }
  } else if (wg >= 0 && wg < n_tiles) {
    // ================================================================ softmax
    const int t = wg;
    const uint32_t lane_off = static_cast<uint32_t>((warp & 3) * 32) << 16;
    const uint32_t s_addr = tmem_S + 128 * t + lane_off;
    const uint32_t o_addr = tmem_O + D * t + lane_off;
    const float sl2 = P.scale_log2;
    float m_run = -INFINITY, l_run = 0.f;
    bool ok = true;
    for (int j = 0; j < n_chunks; ++j) {
      // S_t(j) done implies PV_t(j-1) done: P and O may be touched
      if (!bounded_wait(&s_full[t], j & 1, P.err, abort_flag, 40)) { ok = false; break; }
      tc_fence_after();
      // key validity: only the last prefix chunk of a split and the tree
      // chunks need a mask
      const bool pref = j < n_pref;
      const int nvalid = pref ? min(kChunk, split_end - (split_start + j * kChunk)) : 0;
      const bool masked = !pref || nvalid < kChunk;
      const int t0 = pref ? 0 : (j - n_pref) * kChunk;
      // ancestor mask words of this row for the chunk's 128 tree keys
      uint64_t wlo = ~0ull, whi = ~0ull;
      if (!pref) {
        wlo = whi = 0ull;
        if (R < M) {
          const int W = (it.m + 63) >> 6;
          const uint64_t* mr = it.mask + static_cast<int64_t>(R / g) * W + (t0 >> 6);
          wlo = __ldg(mr);
          if ((t0 >> 6) + 1 < W) whi = __ldg(mr + 1);
        }
      }
      const int nt = pref ? nvalid : it.m - t0;   // keys present in this chunk
      // load 64 columns of S (two 32-column loads, one wait); mask if needed
      auto load64 = [&](int half, float (&v)[64]) {
        uint32_t ra[32], rb[32];
        tmem_ld32(s_addr + 64 * half, ra);
        tmem_ld32(s_addr + 64 * half + 32, rb);
        tmem_wait_ld();
#pragma unroll
        for (int e = 0; e < 32; ++e) {
          v[e] = __uint_as_float(ra[e]);
          v[32 + e] = __uint_as_float(rb[e]);
        }
        if (masked) {
          const uint64_t w = half ? whi : wlo;
#pragma unroll
          for (int e = 0; e < 64; ++e) {
            const int c = 64 * half + e;
            const bool vis = c < nt && (pref || ((w >> e) & 1ull));
            if (!vis) v[e] = -INFINITY;
          }
        }
      };
      float mx = -INFINITY;
#pragma unroll 1
      for (int half = 0; half < 2; ++half) {
        float v[64];
        load64(half, v);
        float m8[8];
#pragma unroll
        for (int a = 0; a < 8; ++a) m8[a] = v[a];
#pragma unroll
        for (int e = 8; e < 64; ++e) m8[e & 7] = fmaxf(m8[e & 7], v[e]);
        mx = fmaxf(mx, fmaxf(fmaxf(fmaxf(m8[0], m8[1]), fmaxf(m8[2], m8[3])),
                             fmaxf(fmaxf(m8[4], m8[5]), fmaxf(m8[6], m8[7]))));
      }
      mx *= sl2;   // scale > 0: max of the scaled row
      const float m_new = fmaxf(m_run, mx);
      const bool grow = (j == 0) || (m_new > m_run + 8.0f);
      if (j > 0 && __any_sync(0xffffffffu, grow)) {
        const float f = grow ? ex2(m_run - m_new) : 1.0f;
#pragma unroll 1
        for (int c = 0; c < D / 32; ++c) {
          uint32_t r[32];
          tmem_ld32(o_addr + 32 * c, r);
          tmem_wait_ld();
#pragma unroll
          for (int e = 0; e < 32; ++e) r[e] = __float_as_uint(__uint_as_float(r[e]) * f);
          tmem_st32(o_addr + 32 * c, r);
        }
        if (grow) l_run *= f;
      }
      if (grow) m_run = m_new;
      const float mref = (m_run == -INFINITY) ? 0.f : m_run;
      // P = 2^(s sl2 - m) in bf16 over the S columns just read: keys
      // 32q..32q+31 -> columns 32q..32q+15 (key pairs per column); tree
      // chunks write the rounding residual to columns 32q+16..32q+31.
      float ls[4] = {0.f, 0.f, 0.f, 0.f};
      if (!masked) {
        // full prefix chunk: the next quarter's S load is in flight while
        // this one is computed
        auto fill = [&](int q, const uint32_t (&ra)[32]) {
          uint32_t hi[16];
#pragma unroll
          for (int e = 0; e < 16; ++e) {
            const float p0 = ex2(fmaf(__uint_as_float(ra[2 * e]), sl2, -mref));
            const float p1 = ex2(fmaf(__uint_as_float(ra[2 * e + 1]), sl2, -mref));
            ls[e & 3] += p0 + p1;
            hi[e] = pack_bf16x2(p0, p1);
          }
          tmem_st16(s_addr + 32 * q, hi);
        };
        uint32_t qa[32], qb[32];
        tmem_ld32(s_addr, qa);
        tmem_wait_ld();
        tmem_ld32(s_addr + 32, qb);
        fill(0, qa);
        tmem_wait_ld();
        tmem_ld32(s_addr + 64, qa);
        fill(1, qb);
        tmem_wait_ld();
        tmem_ld32(s_addr + 96, qb);
        fill(2, qa);
        tmem_wait_ld();
        fill(3, qb);
      } else {
        // masked chunk (tree keys, or the ragged end of a split): invisible
        // keys get P = 0; tree keys also get the bf16 rounding residual
#pragma unroll 1
        for (int q = 0; q < 4; ++q) {
          uint32_t ra[32];
          tmem_ld32(s_addr + 32 * q, ra);
          tmem_wait_ld();
          const uint64_t w = q < 2 ? wlo : whi;
          uint32_t hi[16], lo[16];
#pragma unroll
          for (int e = 0; e < 16; ++e) {
            float s0 = __uint_as_float(ra[2 * e]), s1 = __uint_as_float(ra[2 * e + 1]);
            const int c0 = 32 * q + 2 * e;
            const int b0 = (32 * (q & 1)) + 2 * e;   // bit of key c0 in its mask word
            if (!(c0 < nt && (pref || ((w >> b0) & 1ull)))) s0 = -INFINITY;
            if (!(c0 + 1 < nt && (pref || ((w >> (b0 + 1)) & 1ull)))) s1 = -INFINITY;
            const float p0 = ex2(fmaf(s0, sl2, -mref));
            const float p1 = ex2(fmaf(s1, sl2, -mref));
            ls[e & 3] += p0 + p1;
            hi[e] = pack_bf16x2(p0, p1);
            const float r0 = p0 - __uint_as_float(hi[e] << 16);
            const float r1 = p1 - __uint_as_float(hi[e] & 0xffff0000u);
            lo[e] = pack_bf16x2(r0, r1);
          }
          tmem_st16(s_addr + 32 * q, hi);
          if (!pref) tmem_st16(s_addr + 32 * q + 16, lo);
        }
      }
      l_run += (ls[0] + ls[1]) + (ls[2] + ls[3]);
      tmem_wait_st();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&p_full[t]);
    }
    // ---- epilogue: the last PV of this tile
    if (ok && n_chunks > 0 && bounded_wait(&o_done[t], (n_chunks - 1) & 1, P.err, abort_flag, 42)) {
      tc_fence_after();
      const bool valid = R < M;
      const int qi = valid ? R / g : 0, hl = valid ? R - qi * g : 0;
      const int64_t orow = static_cast<int64_t>(qi) * P.hq + kvh * g + hl;
      const float inv = l_run > 0.f ? 1.f / l_run : 0.f;
      const int64_t punit = it.part_start + static_cast<int64_t>(kvh * it.tile_pairs + tp) * it.splits + split;
      float* po = P.part_o + (punit * 256 + (R - 256 * tp)) * D;
#pragma unroll 1
      for (int c = 0; c < D / 32; ++c) {
        uint32_t r[32];
        tmem_ld32(o_addr + 32 * c, r);
        tmem_wait_ld();
        if (!valid) continue;
        float4* dst = reinterpret_cast<float4*>((it.splits == 1 ? it.out + orow * D : po) + 32 * c);
        const float sc = it.splits == 1 ? inv : 1.f;
#pragma unroll
        for (int e = 0; e < 8; ++e)
          dst[e] = make_float4(__uint_as_float(r[4 * e]) * sc, __uint_as_float(r[4 * e + 1]) * sc,
                               __uint_as_float(r[4 * e + 2]) * sc, __uint_as_float(r[4 * e + 3]) * sc);
      }
      if (valid && it.splits > 1) P.part_ml[punit * 256 + (R - 256 * tp)] = make_float2(m_run, l_run);
    }
  }

  // ---- teardown: tensor memory is freed by the warp that allocated it
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 1) tmem_dealloc(tmem, kTmemCols);
}

// Split merge: one thread per (row, 4 output columns) of every 256-row tile
// pair of every kv head, online over the splits (running max in log2 units);
// partial and output rows are read and written as contiguous float4 runs.
struct TcMergeParams {
  TcItem items[kTcMaxItems];
  int block_start[kTcMaxItems + 1];   // first block of each item
  int n_items, hq, hkv, g;
  const float* part_o;
  const float2* part_ml;
};

template <int D>
__global__ void __launch_bounds__(256) attn_tc_merge_kernel(const __grid_constant__ TcMergeParams P) {
  constexpr int kCols4 = D / 4;                 // threads per row
  constexpr int kRows = 256 / kCols4;           // rows per block
  int item = 0;
  while (item + 1 < P.n_items && static_cast<int>(blockIdx.x) >= P.block_start[item + 1]) ++item;
  const TcItem& it = P.items[item];
  const int S = it.splits;
  const int b = blockIdx.x - P.block_start[item];
  const int blocks_per_pair = 256 / kRows;
  const int pair = b / blocks_per_pair;         // kvh * tile_pairs + tp
  const int kvh = pair / it.tile_pairs, tp = pair - kvh * it.tile_pairs;
  const int r = (b - pair * blocks_per_pair) * kRows + threadIdx.x / kCols4;   // row in the pair
  const int c4 = threadIdx.x % kCols4;
  const int Rg = 256 * tp + r;
  if (Rg >= it.m * P.g) return;
  const int64_t u0 = it.part_start + static_cast<int64_t>(pair) * S;
  float mx = -INFINITY, l = 0.f;
  float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll 4
  for (int s = 0; s < S; ++s) {
    const float2 ml = __ldcg(P.part_ml + (u0 + s) * 256 + r);
    const float4 o = __ldcg(reinterpret_cast<const float4*>(P.part_o + ((u0 + s) * 256 + r) * D) + c4);
    const float mn = fmaxf(mx, ml.x);
    const float a = mx == -INFINITY ? 0.f : ex2(mx - mn);
    const float w = ml.x == -INFINITY ? 0.f : ex2(ml.x - mn);
    acc = make_float4(acc.x * a + w * o.x, acc.y * a + w * o.y, acc.z * a + w * o.z,
                      acc.w * a + w * o.w);
    l = l * a + w * ml.y;
    mx = mn;
  }
  const float inv = l > 0.f ? 1.f / l : 0.f;
  const int qi = Rg / P.g, hl = Rg - qi * P.g;
  reinterpret_cast<float4*>(it.out + (static_cast<int64_t>(qi) * P.hq + kvh * P.g + hl) * D)[c4] =
      make_float4(acc.x * inv, acc.y * inv, acc.z * inv, acc.w * inv);
}

// ------------------------------------------------------------------ host
static PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  });
  return fn;
}

// 3-D bf16 tensor map with a (64 x rows_box x 1) box, 128-byte swizzle.
static bool encode_3d(CUtensorMap* map, const void* base, uint64_t d0, uint64_t d1, uint64_t d2,
                      uint64_t stride1_bytes, uint64_t stride2_bytes, uint32_t box1,
                      uint32_t box2) {
  auto fn = encode_fn();
  if (!fn) return false;
  cuuint64_t dims[3] = {d0, d1 ? d1 : 1, d2 ? d2 : 1};
  cuuint64_t strides[2] = {stride1_bytes, stride2_bytes};
  cuuint32_t box[3] = {64, box1, box2};
  cuuint32_t estr[3] = {1, 1, 1};
  return fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides, box,
            estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

bool tc_supported(int head_dim) { return head_dim == 64 || head_dim == 128; }

struct TcPlan {
  int span;
  int splits[kTcMaxItems];
  int tile_pairs[kTcMaxItems];
  int units;
  int64_t part_units;   // 256-row partial blocks
};

// Splits per (kv head, tile pair): ceil(prefix chunks / span) prefix splits
// plus one tree split.  The span minimises waves x (span + 2) -- the +2 for a
// CTA's fixed work (Q tiles, epilogue) -- plus a small charge per CTA for its
// partial's write and read.
static TcPlan plan_tc(const eagle_attn_item* items, int n, int hq, int hkv, int d) {
  TcPlan T;
  memset(&T, 0, sizeof(T));
  const int g = hq / hkv;
  int max_nc = 1;
  for (int b = 0; b < n; ++b) {
    T.tile_pairs[b] = (items[b].m * g + 255) / 256;
    max_nc = std::max(max_nc, (items[b].prefix_len + kChunk - 1) / kChunk);
  }
  double best_cost = -1.0;
  for (int span = 1; span <= max_nc; ++span) {
    int64_t total = 0;
    for (int b = 0; b < n; ++b) {
      const int nc = (items[b].prefix_len + kChunk - 1) / kChunk;
      total += static_cast<int64_t>(hkv) * T.tile_pairs[b] * ((nc + span - 1) / span + 1);
    }
    const int64_t waves = (total + kPlanSMs - 1) / kPlanSMs;
    const double cost = static_cast<double>(waves * (span + 2)) + 0.05 * static_cast<double>(total);
    if (best_cost < 0.0 || cost <= best_cost) {
      best_cost = cost;
      T.span = span;
    }
  }
  int64_t units = 0, part = 0;
  for (int b = 0; b < n; ++b) {
    const int nc = (items[b].prefix_len + kChunk - 1) / kChunk;
    T.splits[b] = (nc + T.span - 1) / T.span + 1;
    units += static_cast<int64_t>(hkv) * T.tile_pairs[b] * T.splits[b];
    if (T.splits[b] > 1) part += static_cast<int64_t>(hkv) * T.tile_pairs[b] * T.splits[b];
  }
  T.units = static_cast<int>(units);
  T.part_units = part;
  (void)d;
  return T;
}

static size_t part_bytes(const TcPlan& T, int d) {
  return align_up(sizeof(float) * static_cast<size_t>(T.part_units) * 256 * d, 256) +
         align_up(sizeof(float2) * static_cast<size_t>(T.part_units) * 256, 256);
}

int attn_tc_num_launches(const eagle_attn_item* items, int n, int hq, int hkv, int d) {
  int count = 0;
  for (int b0 = 0; b0 < n; b0 += kTcMaxItems) {
    const int nb = std::min(kTcMaxItems, n - b0);
    const TcPlan T = plan_tc(items + b0, nb, hq, hkv, d);
    count += 1 + (T.part_units > 0 ? 1 : 0);
  }
  return count;
}

size_t attn_tc_ws_size(const eagle_attn_item* items, int n, int hq, int hkv, int d, int) {
  size_t need = kWsHeader;
  for (int b0 = 0; b0 < n; b0 += kTcMaxItems) {
    const int nb = std::min(kTcMaxItems, n - b0);
    const TcPlan T = plan_tc(items + b0, nb, hq, hkv, d);
    need = std::max(need, kWsHeader + part_bytes(T, d));
  }
  return need;
}

template <int D>
static eagle_status launch_d(const eagle_attn_item* items, int n, int hq, int hkv, float scale,
                             void* ws, size_t ws_bytes, cudaStream_t stream) {
  static_assert(sizeof(TcParams) < 32000, "kernel parameter block too large");
  for (int b0 = 0; b0 < n; b0 += kTcMaxItems) {
    const int nb = std::min(kTcMaxItems, n - b0);
    const eagle_attn_item* its = items + b0;
    const TcPlan T = plan_tc(its, nb, hq, hkv, D);
    if (ws_bytes < kWsHeader + part_bytes(T, D)) return EAGLE_ERR_WORKSPACE_TOO_SMALL;
    TcParams P;
    memset(&P, 0, sizeof(P));
    int64_t units = 0, part = 0;
    for (int b = 0; b < nb; ++b) {
      const eagle_attn_item& x = its[b];
      const uint64_t S = static_cast<uint64_t>(x.prefix_len);
      const void* kbase = x.prefix_len ? x.k_cache : x.tree_k;
      const void* vbase = x.prefix_len ? x.v_cache : x.tree_v;
      const uint64_t hs = static_cast<uint64_t>(x.cache_head_stride) * 2;
      if (!encode_3d(&P.kmap[b], kbase, D, S, hkv, D * 2, x.prefix_len ? hs : D * 2, kChunk, 1) ||
          !encode_3d(&P.vmap[b], vbase, D, S, hkv, D * 2, x.prefix_len ? hs : D * 2, kChunk, 1) ||
          !encode_3d(&P.tkmap[b], x.tree_k, D, hkv, x.m, D * 2, static_cast<uint64_t>(hkv) * D * 2, 1, kChunk) ||
          !encode_3d(&P.tvmap[b], x.tree_v, D, hkv, x.m, D * 2, static_cast<uint64_t>(hkv) * D * 2, 1, kChunk))
        return EAGLE_ERR_CUDA;
      TcItem& ti = P.items[b];
      ti.q = static_cast<const __nv_bfloat16*>(x.q);
      ti.out = x.out;
      ti.mask = x.mask;
      ti.m = x.m;
      ti.prefix_len = x.prefix_len;
      ti.splits = T.splits[b];
      ti.tile_pairs = T.tile_pairs[b];
      ti.unit_start = static_cast<int>(units);
      ti.part_start = part;
      units += static_cast<int64_t>(hkv) * T.tile_pairs[b] * T.splits[b];
      if (T.splits[b] > 1) part += static_cast<int64_t>(hkv) * T.tile_pairs[b] * T.splits[b];
    }
    P.n_items = nb;
    P.hq = hq;
    P.hkv = hkv;
    P.g = hq / hkv;
    P.span_chunks = T.span;
    P.total_units = static_cast<int>(units);
    P.scale_log2 = (scale != 0.f ? scale : 1.0f / sqrtf(static_cast<float>(D))) * 1.4426950408889634f;
    P.err = static_cast<int32_t*>(ws);
    char* pbase = static_cast<char*>(ws) + kWsHeader;
    P.part_o = reinterpret_cast<float*>(pbase);
    P.part_ml = reinterpret_cast<float2*>(
        pbase + align_up(sizeof(float) * static_cast<size_t>(T.part_units) * 256 * D, 256));
    const size_t smem = TcSmem<D>::kAlloc;
    EAGLE_CUDA(cudaFuncSetAttribute(attn_tc_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                    static_cast<int>(smem)));
    attn_tc_kernel<D><<<static_cast<unsigned>(units), kTcThreads, smem, stream>>>(P);
    eagle_status st = launch_status();
    if (st != EAGLE_OK) return st;
    if (part > 0) {
      TcMergeParams MP;
      memset(&MP, 0, sizeof(MP));
      constexpr int kRows = 256 / (D / 4);
      int blocks = 0;
      for (int b = 0; b < nb; ++b) {
        MP.items[b] = P.items[b];
        MP.block_start[b] = blocks;
        if (P.items[b].splits > 1) blocks += hkv * P.items[b].tile_pairs * (256 / kRows);
      }
      MP.block_start[nb] = blocks;
      MP.n_items = nb;
      MP.hq = hq;
      MP.hkv = hkv;
      MP.g = hq / hkv;
      MP.part_o = P.part_o;
      MP.part_ml = P.part_ml;
      attn_tc_merge_kernel<D><<<blocks, 256, 0, stream>>>(MP);
      if ((st = launch_status()) != EAGLE_OK) return st;
    }
  }
  return EAGLE_OK;
}

eagle_status attn_tc_launch(const eagle_attn_item* items, int n, int hq, int hkv, int d,
                            float scale, void* ws, size_t ws_bytes, cudaStream_t stream, int) {
  if (d == 128) return launch_d<128>(items, n, hq, hkv, scale, ws, ws_bytes, stream);
  if (d == 64) return launch_d<64>(items, n, hq, hkv, scale, ws, ws_bytes, stream);
  return EAGLE_ERR_UNSUPPORTED_SHAPE;
}

}  // namespace eagle
