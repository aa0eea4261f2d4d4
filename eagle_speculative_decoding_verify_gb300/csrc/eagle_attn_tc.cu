// Tensor-core path of eagle_tree_attn for bf16 Q/K/V: head_dim 128 runs the
// 2-SM kernel (attn2_kernel, a cluster of two CTAs per work unit, tcgen05
// .cta_group::2), head_dim 64 the 1-SM kernel below (attn_tc_kernel).  An
// E4M3 prefix cache (eagle_tree_attn_fp8_batched, head_dim 128) runs the
// 1-SM kernel with its prefix chunks widened to fp16 in shared memory and
// those splits' MMAs on fp16 operands (see TcSmem and the converter warps).
//
// Source: "EAGLE-2: Feature-Level Speculative Decoding Guide", "Single-Pass
// Tree Verification" (one target pass over the tree; a token attends to its
// ancestors and itself only) over the target's prefix KV cache.
//
// Both kernels stack the m tree queries of one KV head times its g query
// heads into the M dimension (row R = i*g + head-in-group), so the g heads
// that share a KV head share every K/V byte, and every K/V chunk a work unit
// streams serves two 128-row query tiles.
//
// 1-SM kernel (head_dim 64).  One CTA = (item, kv head, pair of 128-row
// query tiles, split).  Splits 0..n-2 each take a contiguous span of prefix
// chunks (128 keys); the last split takes the tree keys only.
// Warp-specialised:
//   warp 0      TMA producer: K and V chunks (K0 V0 K1 V1 ..., the order the
//               MMAs consume them) into a 5-slot ring of 128-byte-swizzled
//               shared-memory tiles; the first five are issued by the thread
//               that initialises the barriers, before the CTA-wide barrier.
//   warp 1      tensor-memory owner and MMA issuer: S_t = Q_t K^T (M 128,
//               N 128, K = head_dim, A and B from shared memory) and
//               O_t += P_t V (M 128, N = head_dim, K 128, A = P from tensor
//               memory) with tcgen05.mma kind::f16, fp32 accumulators in
//               tensor memory (O_0, O_1, S_0, S_1: 4 x 128 columns).  Per
//               chunk j it issues PV_0(j), S_0(j+1), PV_1(j), S_1(j+1), so
//               the tensor core works for one tile while the other tile's
//               softmax runs (ping-pong).  The MMAs of a thread run in issue
//               order, so PV_t(j) has read P_t(j) before S_t(j+1)
//               overwrites those columns.
//   warps 4-7   softmax of tile 0, warps 8-11 of tile 1: one thread per
//   / 8-11      query row (= TMEM lane) over the chunk's 128 keys, in two
//               passes over tensor memory (row maximum, then P) so that 64
//               values at a time sit in registers; scale, prefix bound and
//               ancestor mask applied; running max / sum with O rescaled in
//               tensor memory only when the max grows by more than 2^8; P
//               written as bf16 over the S columns just read (32 keys -> 16
//               columns); for tree keys (few, possibly dominant) the bf16
//               rounding residual goes to the next 16 columns and a second
//               MMA adds it, so that O accumulates P to ~2^-17.
// Barriers are kept per query tile; every tile barrier completes once per
// chunk and no parity wait is ever two phases away from its barrier.  The
// epilogue writes the normalised row (one split) or an unnormalised partial
// (o, max, sum) that attn_tc_merge_kernel combines.  Every mbarrier wait is
// bounded; on a timeout the CTA records the error, drains its own copies and
// MMAs, frees tensor memory and returns.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_bf16.h>

#include <algorithm>
#include <mutex>
#include <vector>

#include "eagle_attn.h"
#include "eagle_host.h"
#include "eagle_tc.cuh"

namespace eagle {

constexpr int kTcMaxItems = 32;     // items per launch (tensor maps live in the params)
constexpr int kTcThreads = 384;     // 12 warps
constexpr int kChunk = 128;         // keys per K/V chunk
constexpr int kSlots = 5;           // K/V ring depth
constexpr uint32_t kTmemCols = 512;

struct TcItem {
  const __nv_bfloat16* q;
  float* out;
  const uint64_t* mask;
  int m, prefix_len, splits, tiles, pairs, unit_start;
  int64_t part_start;   // first partial unit of the item (units of 128 rows)
  int cnt_start;        // first split-arrival counter of the item (2-SM kernel)
  const int32_t* table; // paged prefix: pool page of every 128-token page (null: contiguous)
  int pool_pages;       // pages in the pool (the table's entries must lie below)
  const float* kscale;  // E4M3 prefix cache: scale of every (kv head, 128-token page)
  const float* vscale;
  int64_t sstride;      // scales between kv heads
};

struct TcParams {
  CUtensorMap kmap[kTcMaxItems];
  CUtensorMap vmap[kTcMaxItems];
  CUtensorMap tkmap[kTcMaxItems];
  CUtensorMap tvmap[kTcMaxItems];
  TcItem items[kTcMaxItems];
  int n_items, hq, hkv, g, span_chunks, total_units;
  float scale_log2;
  float* part_o;     // [unit][D][128 rows]
  float2* part_ml;   // [unit][128 rows] (max in log2 units, sum)
  int32_t* counters; // [item][kv head][tile] splits arrived (2-SM kernel; left at zero)
  int fuse_merge;    // 2-SM kernel: the last split of a tile merges (else a merge kernel runs)
  int32_t* err;
};

// F8: the prefix comes from an E4M3 cache -- a chunk's codes land (TMA) in
// the upper half of its ring slot, where two warps widen them in place.
template <int D, bool F8 = false>
struct TcSmem {
  static constexpr int kQTileBytes = 128 * D * 2;       // one 128-row 16-bit query tile
  static constexpr int kKvBytes = kChunk * D * 2;       // one K or V chunk (128 keys)
  static constexpr int kBoxBytes = kChunk * 128;        // 128 rows x 64 elements (128 B)
  static constexpr int kCodeBytes = kChunk * D;         // one E4M3 chunk
  static constexpr int kCodeOff = kKvBytes - kCodeBytes;   // its place in the slot
  static constexpr int kQ = 0;                          // the CTA's two query tiles
  static constexpr int kRing = kQ + 2 * kQTileBytes;
  static constexpr int kBars = kRing + kSlots * kKvBytes;
  static constexpr int kBytes = kBars + 256;
  static constexpr int kAlloc = kBytes + 1024;        // slack for 1024-byte alignment
};
static_assert(TcSmem<128>::kAlloc <= 232448, "shared memory of the tensor-core kernel");
static_assert(TcSmem<128, true>::kAlloc <= 232448, "shared memory of the E4M3 kernel");

// 16 E4M3 codes -> 16 fp16 (exact: every E4M3 value is an fp16 value; one
// conversion per pair of codes); the first code lands in the low half of
// out[0]
__device__ __forceinline__ void e4m3x16_to_f16(const uint4 in, uint32_t (&out)[8]) {
  const uint32_t w[4] = {in.x, in.y, in.z, in.w};
#pragma unroll
  for (int q = 0; q < 4; ++q) {
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      const uint16_t pair = static_cast<uint16_t>(w[q] >> (16 * h));
      asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(out[2 * q + h]) : "h"(pair));
    }
  }
}

// Bounded wait whose outcome is the same for the whole warp (tcgen05.ld/st
// after it must be executed by all 32 lanes).
__device__ __forceinline__ bool bounded_wait(uint64_t* bar, uint32_t parity, int32_t* err,
                                             volatile int* abort_flag, int where,
                                             uint64_t limit_ns = 2000000000ull) {
  if (mbar_try_wait(bar, parity)) return true;   // fast path: phase already complete
  bool ok = !*abort_flag && mbar_wait(bar, parity, limit_ns);
  if (!ok && !*abort_flag) {
    record_error(err, kDevTimeout, where);
    *abort_flag = 1;
  }
  return ok;
}

template <int D, bool F8>
__global__ void __launch_bounds__(kTcThreads, 1) attn_tc_kernel(const __grid_constant__ TcParams P) {
  pdl_trigger();   // let a dependent launch of the next kernel start (see pdl_attribute)
  using L = TcSmem<D, F8>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + L::kBars);
  uint64_t* empty = full + kSlots;
  uint64_t* s_full = empty + kSlots;    // [query tile]
  uint64_t* p_full = s_full + 2;        // [query tile]
  uint64_t* o_done = p_full + 2;        // [query tile]: that tile's PV done
  uint64_t* drain = o_done + 2;         // [1]
  uint64_t* q_ready = drain + 1;        // [1] both Q tiles written (8 softmax warps)
  uint64_t* full8 = q_ready + 1;        // [slot] E4M3 codes landed (F8)
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(full8 + kSlots);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;

  // ---- work unit: (item, kv head, pair of 128-row query tiles, split)
  int item = 0;
  while (item + 1 < P.n_items && static_cast<int>(blockIdx.x) >= P.items[item + 1].unit_start)
    ++item;
  const TcItem& it = P.items[item];
  int u = blockIdx.x - it.unit_start;
  const int split = u % it.splits;
  u /= it.splits;
  const int tp = u % it.pairs;
  const int kvh = u / it.pairs;
  const int g = P.g;
  const int M = it.m * g;
  const int ntile = min(2, it.tiles - 2 * tp);   // query tiles of this CTA: 1 or 2
  const bool tree_split = split == it.splits - 1;
  const int split_start = split * P.span_chunks * kChunk;
  const int split_end = tree_split ? 0 : min(it.prefix_len, split_start + P.span_chunks * kChunk);
  const int n_pref = split_end > split_start ? (split_end - split_start + kChunk - 1) / kChunk : 0;
  const int n_chunks = n_pref + (tree_split ? (it.m + kChunk - 1) / kChunk : 0);

  // ring item n: K of chunk n/2 (n even) or V (n odd), into slot n % kSlots;
  // the MMAs consume them in this order
  auto issue_kv = [&](int n) {
    const int slot = n % kSlots;
    const int j = n >> 1;
    const bool is_v = n & 1;
    uint8_t* dst = smem + L::kRing + slot * L::kKvBytes;
    mbar_arrive_expect_tx(&full[slot], static_cast<uint32_t>(L::kKvBytes));
    if (j < n_pref) {
      const CUtensorMap* map = is_v ? &P.vmap[item] : &P.kmap[item];
      int y = split_start + j * kChunk;
      if (it.table) {   // paged prefix: a chunk is one page (a bad id reads page 0, reported)
        int page = __ldg(it.table + split_start / kChunk + j);
        if (page < 0 || page >= it.pool_pages) {
          record_error(P.err, kDevAssert, 60);
          page = 0;
        }
        y = page * kChunk;
      }
#pragma unroll
      for (int h = 0; h < D / 64; ++h) tma_load_3d(dst + h * L::kBoxBytes, map, 64 * h, y, kvh, &full[slot]);
    } else {
      const CUtensorMap* map = is_v ? &P.tvmap[item] : &P.tkmap[item];
      const int z = (j - n_pref) * kChunk;
#pragma unroll
      for (int h = 0; h < D / 64; ++h) tma_load_3d(dst + h * L::kBoxBytes, map, 64 * h, kvh, z, &full[slot]);
    }
  };

  // E4M3 prefix (F8): item n of a prefix split is staged as codes, then
  // widened to fp16 into ring slot n % kSlots by the converter warps.  A
  // prefix split holds only prefix chunks and a tree split only tree chunks,
  // so a staged split runs every MMA on fp16 operands (its query tiles are
  // written as fp16, P is fp16) and the tree split stays bf16.
  const bool staged = F8 && !tree_split;
  auto issue_stage = [&](int n) {
    const int slot = n % kSlots;
    const int j = n >> 1;
    const CUtensorMap* map = (n & 1) ? &P.vmap[item] : &P.kmap[item];
    mbar_arrive_expect_tx(&full8[slot], static_cast<uint32_t>(L::kCodeBytes));
    tma_load_3d(smem + L::kRing + slot * L::kKvBytes + L::kCodeOff, map, 0, split_start + j * kChunk,
                kvh, &full8[slot]);
  };

  if (tid == 0) {
    for (int s = 0; s < kSlots; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    for (int s = 0; F8 && s < kSlots; ++s) mbar_init(&full8[s], 1);
    for (int t = 0; t < 2; ++t) {
      mbar_init(&s_full[t], 1);
      mbar_init(&p_full[t], 4);   // one arrival per warp of the tile's warpgroup
      mbar_init(&o_done[t], 1);
    }
    mbar_init(drain, 1);
    mbar_init(q_ready, 8);
    *abort_flag = 0;
    fence_barrier_init();
    // the producer (this thread) starts streaming before the CTA-wide barrier
    if (staged) {
      for (int n = 0; n < kSlots && n < 2 * n_chunks; ++n) issue_stage(n);
    } else {
      for (int n = 0; n < kSlots && n < 2 * n_chunks; ++n) issue_kv(n);
    }
  }
  if (warp == 1) {
    tmem_alloc(tmem_slot, kTmemCols);
    tmem_relinquish();
  }

  tc_fence_before();
  __syncthreads();   // barriers initialised, tensor memory allocated
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  // tensor memory: O of tile t in columns 128 t .., S (then P) of tile t in 256 + 128 t ..

  // ---- softmax warpgroup t (warps 4-7: tile 0, warps 8-11: tile 1), one
  // thread per query row (= TMEM lane); it first writes its Q row into the
  // tile (128-byte swizzle) while the producer already streams K/V
  const int t = warp >= 8 ? 1 : 0;
  const int row = (warp & 3) * 32 + lane;
  const int R = 256 * tp + 128 * t + row;
  const bool row_valid = t < ntile && R < M;
  if (warp >= 4) {
    uint8_t* qt = smem + L::kQ + t * L::kQTileBytes;
    const int qi = row_valid ? R / g : 0;
    const int hl = row_valid ? R - qi * g : 0;
    const int4* src = reinterpret_cast<const int4*>(it.q + (static_cast<int64_t>(qi) * P.hq + kvh * g + hl) * D);
#pragma unroll
    for (int half = 0; half < 2; ++half) {
      int4 qv[D / 16];
#pragma unroll
      for (int c = 0; c < D / 16; ++c)
        qv[c] = row_valid ? __ldg(src + half * (D / 16) + c) : make_int4(0, 0, 0, 0);
#pragma unroll
      for (int c = 0; c < D / 16; ++c) {   // 16-byte chunks of the row
        const int cg = half * (D / 16) + c;
        const int box = cg >> 3, cc = cg & 7;
        int4 x = qv[c];
        if (staged) {
          // fp16 (exact for magnitudes in [2^-14, 65504], the rest within
          // 2^-25); a larger element is reported
          const uint32_t w[4] = {static_cast<uint32_t>(x.x), static_cast<uint32_t>(x.y),
                                 static_cast<uint32_t>(x.z), static_cast<uint32_t>(x.w)};
          uint32_t h16[4];
          bool big = false;
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const float lo = __uint_as_float(w[e] << 16), hi = __uint_as_float(w[e] & 0xffff0000u);
            big |= fmaxf(fabsf(lo), fabsf(hi)) > 65504.f;
            h16[e] = pack_f16x2(lo, hi);
          }
          if (big) record_error(P.err, kDevAssert, 61);
          x = make_int4(static_cast<int>(h16[0]), static_cast<int>(h16[1]), static_cast<int>(h16[2]),
                        static_cast<int>(h16[3]));
        }
        *reinterpret_cast<int4*>(qt + box * (128 * 128) + row * 128 + ((cc ^ (row & 7)) << 4)) = x;
      }
    }
    fence_proxy_async_smem();
    __syncwarp();
    if (lane == 0) mbar_arrive(q_ready);
  }

  if (warp == 0) {
    // ================================================================ TMA producer
    if (lane == 0 && staged) {
      int issued = kSlots < 2 * n_chunks ? kSlots : 2 * n_chunks;   // the prologue's
      for (int n = issued; n < 2 * n_chunks; ++n) {
        const int slot = n % kSlots, use = n / kSlots;
        if (!bounded_wait(&empty[slot], (use - 1) & 1, P.err, abort_flag, 21)) break;
        issue_stage(n);
        issued = n + 1;
      }
      // make sure no copy of ours is still landing when the CTA leaves
      for (int n = (issued > kSlots ? issued - kSlots : 0); n < issued; ++n)
        mbar_wait(&full8[n % kSlots], (n / kSlots) & 1, 200000000ull);
    } else if (lane == 0) {
      int issued = kSlots < 2 * n_chunks ? kSlots : 2 * n_chunks;   // the prologue's
      for (int n = issued; n < 2 * n_chunks; ++n) {
        const int slot = n % kSlots, use = n / kSlots;
        if (!bounded_wait(&empty[slot], (use - 1) & 1, P.err, abort_flag, 20)) break;
        issue_kv(n);
        issued = n + 1;
      }
      // make sure no copy of ours is still landing when the CTA leaves
      for (int n = (issued > kSlots ? issued - kSlots : 0); n < issued; ++n)
        mbar_wait(&full[n % kSlots], (n / kSlots) & 1, 200000000ull);
    }
  } else if (staged && (warp == 2 || warp == 3)) {
    // ================================================================ E4M3 -> fp16
    // item n: the codes [128 keys][D codes] in the upper half of ring slot
    // n % kSlots -> fp16 in the whole slot, in the layout a 16-bit TMA would
    // have written (boxes of 64 columns, 128-byte rows, 128-byte swizzle).
    // Every code of the chunk is read into registers before the first store
    // (a named barrier between), since the stores cover the codes.  Both
    // warps run every item and meet at the barriers, also after a wait ran
    // out.
    const int ct = tid - 64;   // 0..63
    constexpr int kPer = kChunk * D / 16 / 64;   // pieces (16 codes) per converter thread
    bool live = true;
    for (int n = 0; n < 2 * n_chunks; ++n) {
      const int slot = n % kSlots;
      live = live && __all_sync(0xffffffffu, bounded_wait(&full8[slot], (n / kSlots) & 1, P.err,
                                                          abort_flag, 22));
      uint8_t* dst = smem + L::kRing + slot * L::kKvBytes;
      // piece pc = 16 codes at byte 16 pc of the codes (key pc / (D / 16),
      // columns 16 (pc % (D / 16)) ..)
      uint4 in[kPer];
      if (live) {
#pragma unroll
        for (int i = 0; i < kPer; ++i)
          in[i] = *reinterpret_cast<const uint4*>(dst + L::kCodeOff + 16 * (ct + 64 * i));
      }
      named_sync(2, 64);
      if (live) {
#pragma unroll
        for (int i = 0; i < kPer; ++i) {
          const int pc = ct + 64 * i;
          const int r = pc / (D / 16), pp = pc - r * (D / 16);
          uint32_t o[8];
          e4m3x16_to_f16(in[i], o);
          const int col = 16 * pp, box = col >> 6, cc = (col & 63) >> 3;
          uint8_t* rowp = dst + box * L::kBoxBytes + r * 128;
          *reinterpret_cast<uint4*>(rowp + ((cc ^ (r & 7)) << 4)) = make_uint4(o[0], o[1], o[2], o[3]);
          *reinterpret_cast<uint4*>(rowp + (((cc + 1) ^ (r & 7)) << 4)) = make_uint4(o[4], o[5], o[6], o[7]);
        }
        fence_proxy_async_smem();
      }
      named_sync(2, 64);
      if (ct == 0 && live) mbar_arrive(&full[slot]);
    }
  } else if (warp == 1) {
    // ================================================================ MMA issuer
    // per chunk j: PV_0(j), S_0(j+1), PV_1(j), S_1(j+1) -- while the tensor
    // core works for one tile, the other tile's softmax runs
    if (lane == 0) {
      // a staged (E4M3 prefix) split: fp16 operands throughout
      const uint32_t idesc_s = staged ? idesc_f16_f32(128, kChunk, false) : idesc_bf16_f32(128, kChunk, false);
      const uint32_t idesc_o = staged ? idesc_f16_f32(128, D, true) : idesc_bf16_f32(128, D, true);
      const uint32_t q_base = smem_addr(smem + L::kQ);
      const uint32_t ring_base = smem_addr(smem + L::kRing);
      // descriptors built once; a k-step adds its byte offset / 16 to the
      // start-address field (no carry: shared memory is < 256 KB)
      const uint64_t qdesc0 = smem_desc_sw128(q_base, 16, 1024);
      const uint64_t kdesc0 = smem_desc_sw128(ring_base, 16, 1024);
      const uint64_t vdesc0 = smem_desc_sw128(ring_base, L::kBoxBytes, 1024);
      auto issue_s = [&](int tt, int slot) {   // S_t = Q_t K^T
        const uint64_t qd = qdesc0 + static_cast<uint64_t>((tt * L::kQTileBytes) >> 4);
        const uint64_t kd = kdesc0 + static_cast<uint64_t>((slot * L::kKvBytes) >> 4);
        const uint32_t dst = tmem + 256 + 128 * tt;
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk)
          mma_bf16(dst, qd + (((kk >> 2) * (128 * 128) + (kk & 3) * 32) >> 4),
                   kd + (((kk >> 2) * L::kBoxBytes + (kk & 3) * 32) >> 4), idesc_s, kk > 0);
      };
      // O_t += P_t V: key 16kk.. sits in columns 32 (kk/2) + 16 fill + 8 (kk%2)
      // of tile t's S columns (bf16 pairs)
      auto issue_pv = [&](int tt, int slot, int fill, bool acc) {
        const uint32_t pa = tmem + 256 + 128 * tt + 16 * fill;
        const uint64_t vd = vdesc0 + static_cast<uint64_t>((slot * L::kKvBytes) >> 4);
#pragma unroll
        for (int kk = 0; kk < kChunk / 16; ++kk)
          mma_bf16_ta(tmem + 128 * tt, pa + 32 * (kk >> 1) + 8 * (kk & 1), vd + ((kk * 2048) >> 4), idesc_o,
                      (acc || kk > 0));
      };
      bool ok = n_chunks > 0 && bounded_wait(q_ready, 0, P.err, abort_flag, 29) &&
                bounded_wait(&full[0], 0, P.err, abort_flag, 30);
      if (ok) {   // S of chunk 0 for every tile
        tc_fence_after();
        for (int tt = 0; tt < ntile; ++tt) {
          issue_s(tt, 0);
          mma_commit(&s_full[tt]);
        }
        mma_commit(&empty[0]);
      }
      for (int j = 0; ok && j < n_chunks; ++j) {
        const int nv = 2 * j + 1, nk = 2 * j + 2;   // ring items of V_j and K_j+1
        const int vslot = nv % kSlots, kslot = nk % kSlots;
        const bool more = j + 1 < n_chunks;
        const int nf = j < n_pref ? 1 : 2;   // tree keys: P = hi + lo
        if (!bounded_wait(&full[vslot], (nv / kSlots) & 1, P.err, abort_flag, 31)) break;
        for (int tt = 0; ok && tt < ntile; ++tt) {
          if (!bounded_wait(&p_full[tt], j & 1, P.err, abort_flag, 32)) { ok = false; break; }
          tc_fence_after();
          for (int f = 0; f < nf; ++f) issue_pv(tt, vslot, f, j > 0 || f > 0);
          mma_commit(&o_done[tt]);
          if (more) {   // S_t(j+1) overwrites P_t(j): issued after PV_t(j), so in order
            if (tt == 0 && !bounded_wait(&full[kslot], (nk / kSlots) & 1, P.err, abort_flag, 33)) {
              ok = false;
              break;
            }
            issue_s(tt, kslot);
            mma_commit(&s_full[tt]);
          }
        }
        if (!ok) break;
        mma_commit(&empty[vslot]);
        if (more) mma_commit(&empty[kslot]);
      }
      // every MMA of this CTA has completed once `drain` flips
      mma_commit(drain);
      mbar_wait(drain, 0, 200000000ull);
    }
  } else if (warp >= 4 && t < ntile) {
    // ================================================================ softmax
    const uint32_t lane_off = static_cast<uint32_t>((warp & 3) * 32) << 16;
    const uint32_t o_addr = tmem + 128 * t + lane_off;          // O of this row, D columns
    const uint32_t s_addr = tmem + 256 + 128 * t + lane_off;    // S / P of this row, 128 keys
    const float sl2 = P.scale_log2;
    const int W = (it.m + 63) >> 6;
    const int64_t mrow = R < M ? static_cast<int64_t>(R / g) * W : -1;
    float m_run = -INFINITY, l_run = 0.f;
    bool ok = true;
    for (int j = 0; j < n_chunks; ++j) {
      ok = __all_sync(0xffffffffu, bounded_wait(&s_full[t], j & 1, P.err, abort_flag, 40));
      if (!ok) break;
      tc_fence_after();
      // key validity: only the last prefix chunk of a split and the tree
      // chunks need a mask (key count, ancestor words for tree keys)
      const bool pref = j < n_pref;
      // E4M3 prefix chunk: S carries the page's key scale, P (fp16: a value
      // scale above 65504 is reported) the value scale
      float sl2j = sl2, svj = 1.f;
      if (staged) {
        const int64_t pg = static_cast<int64_t>(kvh) * it.sstride + split_start / kChunk + j;
        sl2j = sl2 * __ldg(it.kscale + pg);
        svj = __ldg(it.vscale + pg);
        if (svj > 65504.f && row == 0) record_error(P.err, kDevAssert, 62);
      }
      const int t0 = pref ? 0 : (j - n_pref) * kChunk;
      const int nvalid = pref ? min(kChunk, split_end - (split_start + j * kChunk)) : min(kChunk, it.m - t0);
      const bool masked = !pref || nvalid < kChunk;
      uint64_t w0 = ~0ull, w1 = ~0ull;
      if (!pref) {
        const int wi = t0 >> 6;
        w0 = (mrow >= 0 && wi < W) ? __ldg(it.mask + mrow + wi) : 0ull;
        w1 = (mrow >= 0 && wi + 1 < W) ? __ldg(it.mask + mrow + wi + 1) : 0ull;
      }
      // 64 keys (half h of the chunk) from tensor memory, masked
      auto load64 = [&](int h, float (&v)[64]) {
        uint32_t ra[32], rb[32];
        tmem_ld32(s_addr + 64 * h, ra);
        tmem_ld32(s_addr + 64 * h + 32, rb);
        tmem_wait_ld();
#pragma unroll
        for (int e = 0; e < 32; ++e) {
          v[e] = __uint_as_float(ra[e]);
          v[32 + e] = __uint_as_float(rb[e]);
        }
        if (masked) {
          const uint64_t w = h ? w1 : w0;
#pragma unroll
          for (int e = 0; e < 64; ++e)
            if (!((64 * h + e < nvalid) & static_cast<bool>((w >> e) & 1ull))) v[e] = -INFINITY;
        }
      };
      float v[64];
      // pass 1: the row's maximum over the chunk
      float mx = -INFINITY;
#pragma unroll 1
      for (int h = 0; h < 2; ++h) {
        load64(h, v);
        float m8[8];
#pragma unroll
        for (int a = 0; a < 8; ++a) m8[a] = v[a];
#pragma unroll
        for (int e = 8; e < 64; ++e) m8[e & 7] = fmaxf(m8[e & 7], v[e]);
        mx = fmaxf(mx, fmaxf(fmaxf(fmaxf(m8[0], m8[1]), fmaxf(m8[2], m8[3])),
                             fmaxf(fmaxf(m8[4], m8[5]), fmaxf(m8[6], m8[7]))));
      }
      mx *= sl2j;   // scale > 0
      const float m_new = fmaxf(m_run, mx);
      const bool grow = (j == 0) || (m_new > m_run + 8.0f);
      if (j > 0 && __any_sync(0xffffffffu, grow)) {
        // O is rescaled once this tile's previous PV has landed
        ok = __all_sync(0xffffffffu, bounded_wait(&o_done[t], (j - 1) & 1, P.err, abort_flag, 41));
        if (!ok) break;
        tc_fence_after();
        const float f = grow ? ex2(m_run - m_new) : 1.0f;
#pragma unroll 1
        for (int c = 0; c < D / 16; ++c) {
          uint32_t r[16];
          tmem_ld16(o_addr + 16 * c, r);
          tmem_wait_ld();
#pragma unroll
          for (int e = 0; e < 16; ++e) r[e] = __float_as_uint(__uint_as_float(r[e]) * f);
          tmem_st16(o_addr + 16 * c, r);
        }
        if (grow) l_run *= f;
      }
      if (grow) m_run = m_new;
      const float mref = (m_run == -INFINITY) ? 0.f : m_run;
      // pass 2: P = 2^(s sl2 - m) in bf16 over the S columns just read: keys
      // 32q..32q+31 -> columns 32q..32q+15 (key pairs); tree chunks write the
      // rounding residual to columns 32q+16..32q+31
      float ls[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll 1
      for (int h = 0; h < 2; ++h) {
        load64(h, v);
#pragma unroll
        for (int q = 0; q < 2; ++q) {
          uint32_t hi[16], lo[16];
#pragma unroll
          for (int e = 0; e < 16; ++e) {
            const float p0 = ex2(fmaf(v[32 * q + 2 * e], sl2j, -mref));
            const float p1 = ex2(fmaf(v[32 * q + 2 * e + 1], sl2j, -mref));
            hi[e] = staged ? pack_f16x2(p0 * svj, p1 * svj) : pack_bf16x2(p0, p1);
            // the row sum takes the weights the MMA uses: the bf16-rounded
            // ones for bf16 prefix keys (a dominant key's rounding then
            // cancels in the normalisation), hi + lo ~ p for tree keys, p for
            // E4M3 prefix keys (fp16 weights, 2^-11 relative)
            ls[e & 3] += (pref && !staged)
                             ? __uint_as_float(hi[e] << 16) + __uint_as_float(hi[e] & 0xffff0000u)
                             : p0 + p1;
            if (!pref) {
              const float r0 = p0 - __uint_as_float(hi[e] << 16);
              const float r1 = p1 - __uint_as_float(hi[e] & 0xffff0000u);
              lo[e] = pack_bf16x2(r0, r1);
            }
          }
          tmem_st16(s_addr + 64 * h + 32 * q, hi);
          if (!pref) tmem_st16(s_addr + 64 * h + 32 * q + 16, lo);
        }
      }
      l_run += (ls[0] + ls[1]) + (ls[2] + ls[3]);
      tmem_wait_st();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&p_full[t]);
    }
    // ---- epilogue: this row's O, normalised (one split) or as a partial
    ok = ok && n_chunks > 0 &&
         __all_sync(0xffffffffu, bounded_wait(&o_done[t], (n_chunks - 1) & 1, P.err, abort_flag, 42));
    tc_fence_after();
    if (ok) {
      const int qi = row_valid ? R / g : 0, hl = row_valid ? R - qi * g : 0;
      const int64_t orow = static_cast<int64_t>(qi) * P.hq + kvh * g + hl;
      const float inv = l_run > 0.f ? 1.f / l_run : 0.f;
      const int64_t punit =
          it.part_start + static_cast<int64_t>(kvh * it.tiles + 2 * tp + t) * it.splits + split;
      float* po = P.part_o + punit * D * 128 + row;   // column c at po + 128 c: a warp's
#pragma unroll 1                                     // store covers 32 consecutive rows
      for (int c = 0; c < D / 32; ++c) {
        uint32_t r[32];
        tmem_ld32(o_addr + 32 * c, r);
        tmem_wait_ld();
        if (!row_valid) continue;
        if (it.splits == 1) {
          float4* dst = reinterpret_cast<float4*>(it.out + orow * D + 32 * c);
#pragma unroll
          for (int e = 0; e < 8; ++e)
            dst[e] = make_float4(__uint_as_float(r[4 * e]) * inv, __uint_as_float(r[4 * e + 1]) * inv,
                                 __uint_as_float(r[4 * e + 2]) * inv, __uint_as_float(r[4 * e + 3]) * inv);
        } else {
#pragma unroll
          for (int e = 0; e < 32; ++e) po[(32 * c + e) * 128] = __uint_as_float(r[e]);
        }
      }
      if (row_valid && it.splits > 1) P.part_ml[punit * 128 + row] = make_float2(m_run, l_run);
    }
  }

  // ---- teardown: tensor memory is freed by the warp that allocated it
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 1) tmem_dealloc(tmem, kTmemCols);
}

// ======================================================== 2-SM form (d 128)
// One cluster of two CTAs = (item, kv head, pair of 128-row query tiles,
// split); CTA r holds query tile 2 tp + r (128 rows) in its shared and tensor
// memory.  The tensor cores of the pair work as one (tcgen05 .cta_group::2,
// M = 256): for S = Q K^T each CTA holds 64 of a chunk's 128 keys (B split by
// N), for O += P V each CTA holds 64 of the 128 value columns, so every CTA
// loads half of each K / V chunk and every K / V byte still serves 256 rows.
// Per CTA, tensor memory holds O (128 columns) and S / P triple-buffered
// (3 x 128 columns): S of chunk j+3 is issued as soon as PV(j) is done, so
// the tensor core has the next chunks' S queued and the softmax does not
// wait for it; each MMA instruction keeps the tensor core busy for 64 cycles
// per SM (N 128).
// Warps per CTA: 0 TMA producer (its half of every chunk, completion on the
// even CTA's barrier), 1 tensor-memory owner and, in the even CTA, the PV
// issuer, 2 (even CTA) the S issuer; 4-7 and 8-11 softmax over keys 0-63 /
// 64-127 of each chunk, one thread per query row, the two halves' row maxima
// exchanged through shared memory at a named barrier.
// A split covers a contiguous range of the item's chunk list (prefix chunks,
// then the tree chunks), so the tree keys ride with the last split.
constexpr int k2Threads = 384;
constexpr int k2Slots = 10;                  // ring items (one CTA's half of a K or V chunk)
constexpr int k2Bufs = 3;                    // S / P buffers
constexpr uint32_t k2TmemCols = 512;         // O 128 + S 3 x 128

struct Sm2 {
  static constexpr int kQBytes = 128 * 128 * 2;   // one 128-row bf16 query tile (2 boxes)
  static constexpr int kItem = 64 * 128 * 2;      // half of a K or V chunk: 16 KB
  static constexpr int kQ = 0;
  static constexpr int kRing = kQ + kQBytes;
  static constexpr int kXch = kRing + k2Slots * kItem;   // [2][2][128] maxima, [2][128] sums
  static constexpr int kBars = kXch + 4096;
  static constexpr int kBytes = kBars + 512;
  static constexpr int kAlloc = kBytes + 1024;
};
static_assert(Sm2::kAlloc <= 232448, "shared memory of the 2-SM kernel");

__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(k2Threads, 1)
    attn2_kernel(const __grid_constant__ TcParams P) {
  pdl_trigger();   // let a dependent launch of the next kernel start (see pdl_attribute)
  constexpr int D = 128;
  using L = Sm2;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + L::kBars);   // [slot] (even CTA's)
  uint64_t* empty = full + k2Slots;     // [slot] (each CTA: its producer may refill)
  uint64_t* s_full = empty + k2Slots;   // [buffer] (each CTA)
  uint64_t* o_done = s_full + k2Bufs;   // [buffer]: PV of a chunk of that buffer done
  uint64_t* p_full = o_done + k2Bufs;   // [buffer] (even CTA's): 16 softmax warps
  uint64_t* q_ready = p_full + k2Bufs;  // [1] (even CTA's): 8 warps wrote Q
  uint64_t* drain = q_ready + 1;        // [2]: each issuer's MMAs all done
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(drain + 2);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  float* xch = reinterpret_cast<float*>(smem + L::kXch);   // [parity][wg][row] maxima, at 512: [wg][row] sums

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const uint32_t rank = pair2::cta_rank();
  // the workspace header's test hook: a short wait limit, and producers that
  // issue nothing (both zero in normal use)
  const WsHeader* hdr = reinterpret_cast<const WsHeader*>(P.err);
  const int32_t test_flags = hdr->test_flags;
  const uint64_t wait_ns =
      hdr->test_wait_us > 0 ? 1000ull * static_cast<uint64_t>(hdr->test_wait_us) : 2000000000ull;

  // ---- work unit: (item, kv head, pair of query tiles, split)
  const int unit = blockIdx.x >> 1;
  int item = 0;
  while (item + 1 < P.n_items && unit >= P.items[item + 1].unit_start) ++item;
  const TcItem& it = P.items[item];
  int u = unit - it.unit_start;
  const int split = u % it.splits;
  u /= it.splits;
  const int tp = u % it.pairs;
  const int kvh = u / it.pairs;
  const int g = P.g;
  const int M = it.m * g;
  const int tile = 2 * tp + static_cast<int>(rank);
  // chunk list of the item: nc prefix chunks, then the tree chunks; this
  // split covers entries [v0, v1)
  const int nc = (it.prefix_len + kChunk - 1) / kChunk;
  const int nv = nc + (it.m + kChunk - 1) / kChunk;
  const int v0 = split * P.span_chunks;
  const int v1 = min(nv, v0 + P.span_chunks);
  const int n_chunks = max(0, v1 - v0);

  // ring item n: K (n even) or V (n odd) of chunk n >> 1, this CTA's half
  auto issue_kv = [&](int n, uint32_t full_leader) {
    const int slot = n % k2Slots;
    const int j = n >> 1;
    const bool is_v = n & 1;
    uint8_t* dst = smem + L::kRing + slot * L::kItem;
    const int v = v0 + j;
    if (v < nc) {
      int y = v * kChunk;
      if (it.table) {   // paged prefix: a chunk is one page (a bad id reads page 0, reported)
        int page = __ldg(it.table + v);
        if (page < 0 || page >= it.pool_pages) {
          record_error(P.err, kDevAssert, 60);
          page = 0;
        }
        y = page * kChunk;
      }
      if (is_v) {
        pair2::tma_load_3d(dst, &P.vmap[item], 64 * rank, y, kvh, full_leader);
      } else {
#pragma unroll
        for (int h = 0; h < 2; ++h)
          pair2::tma_load_3d(dst + h * 8192, &P.kmap[item], 64 * h, y + 64 * rank, kvh, full_leader);
      }
    } else {
      const int z = (v - nc) * kChunk;
      if (is_v) {
        pair2::tma_load_3d(dst, &P.tvmap[item], 64 * rank, kvh, z, full_leader);
      } else {
#pragma unroll
        for (int h = 0; h < 2; ++h)
          pair2::tma_load_3d(dst + h * 8192, &P.tkmap[item], 64 * h, kvh, z + 64 * rank, full_leader);
      }
    }
  };

  if (tid == 0) {
    for (int s = 0; s < k2Slots; ++s) {
      mbar_init(&full[s], 1);   // the even CTA's producer arrives with both halves' bytes
      mbar_init(&empty[s], 1);
    }
    for (int b = 0; b < k2Bufs; ++b) {
      mbar_init(&s_full[b], 1);
      mbar_init(&o_done[b], 1);
      mbar_init(&p_full[b], 16);
    }
    mbar_init(q_ready, 8);
    mbar_init(&drain[0], 1);
    mbar_init(&drain[1], 1);
    *abort_flag = 0;
    fence_barrier_init();
  }
  if (warp == 1) {
    pair2::tmem_alloc(tmem_slot, k2TmemCols);
    pair2::tmem_relinquish();
  }
  tc_fence_before();
  pair2::cluster_sync();   // both CTAs' barriers initialised, tensor memory allocated
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  // tensor memory (each CTA): O in columns 0..127, S / P buffer b in 128 + 128 b ..

  const int wg = warp >= 8 ? 1 : 0;          // softmax warpgroup: keys 64 wg .. of a chunk
  const int row = (warp & 3) * 32 + lane;
  const int R = 256 * tp + 128 * static_cast<int>(rank) + row;
  const bool row_valid = tile < it.tiles && R < M;
  if (warp >= 4 && warp < 8) {
    // warpgroup 0 writes this CTA's Q tile (128-byte swizzle) while the
    // producer streams K / V
    const int qi = row_valid ? R / g : 0;
    const int hl = row_valid ? R - qi * g : 0;
    const int4* src = reinterpret_cast<const int4*>(it.q + (static_cast<int64_t>(qi) * P.hq + kvh * g + hl) * D);
#pragma unroll
    for (int half = 0; half < 2; ++half) {
      int4 qv[D / 16];
#pragma unroll
      for (int c = 0; c < D / 16; ++c)
        qv[c] = row_valid ? __ldg(src + half * (D / 16) + c) : make_int4(0, 0, 0, 0);
#pragma unroll
      for (int c = 0; c < D / 16; ++c) {
        const int cg = half * (D / 16) + c;
        const int box = cg >> 3, cc = cg & 7;
        *reinterpret_cast<int4*>(smem + L::kQ + box * (128 * 128) + row * 128 + ((cc ^ (row & 7)) << 4)) = qv[c];
      }
    }
    fence_proxy_async_smem();
    __syncwarp();
    if (lane == 0) pair2::arrive_cluster(pair2::map_to(smem_addr(q_ready), 0));
  }

  if (warp == 0) {
    // ================================================================ TMA producer
    if (lane == 0) {
      const int n_items = (test_flags & kTestNoCopies) ? 0 : 2 * n_chunks;
      for (int n = 0; n < n_items; ++n) {
        const int slot = n % k2Slots, use = n / k2Slots;
        if (use > 0 && !bounded_wait(&empty[slot], (use - 1) & 1, P.err, abort_flag, 20, wait_ns)) break;
        if (rank == 0) mbar_arrive_expect_tx(&full[slot], 2u * L::kItem);
        issue_kv(n, pair2::map_to(smem_addr(&full[slot]), 0));
      }
    }
    __syncwarp();
  } else if ((warp == 1 || warp == 2) && rank == 0) {
    // ================================================================ MMA issuers (even CTA)
    // Two threads issue, so that one MMA stream's instruction issue never
    // waits behind the other's: warp 2 issues S(j) = Q K_j^T into buffer
    // j % 3 once PV(j-3), the last reader of that buffer, has completed;
    // warp 1 issues O += P(j) V_j once the softmax has written P(j).
    if (lane == 0) {
      const uint32_t ring_base = smem_addr(smem + L::kRing);
      auto slot_of = [](int n) { return n % k2Slots; };
      auto full_parity = [](int n) { return static_cast<uint32_t>((n / k2Slots) & 1); };
      if (warp == 2) {
        constexpr uint32_t idesc_s = idesc_bf16_f32(256, kChunk, false);
        const uint64_t qdesc0 = smem_desc_sw128(smem_addr(smem + L::kQ), 16, 1024);
        const uint64_t kdesc0 = smem_desc_sw128(ring_base, 16, 1024);
        bool ok = n_chunks > 0 && bounded_wait(q_ready, 0, P.err, abort_flag, 29, wait_ns);
        for (int j = 0; ok && j < n_chunks; ++j) {
          const int b = j % k2Bufs, nki = 2 * j;
          if ((j >= k2Bufs &&
               !bounded_wait(&o_done[b], ((j - k2Bufs) / k2Bufs) & 1, P.err, abort_flag, 34, wait_ns)) ||
              !bounded_wait(&full[slot_of(nki)], full_parity(nki), P.err, abort_flag, 33, wait_ns))
            break;
          tc_fence_after();
          const uint64_t kd = kdesc0 + static_cast<uint64_t>((slot_of(nki) * L::kItem) >> 4);
          const uint32_t dst = tmem + 128 + 128 * b;
#pragma unroll
          for (int kk = 0; kk < D / 16; ++kk)
            pair2::mma_bf16(dst, qdesc0 + (((kk >> 2) * (128 * 128) + (kk & 3) * 32) >> 4),
                            kd + (((kk >> 2) * 8192 + (kk & 3) * 32) >> 4), idesc_s, kk > 0);
          pair2::commit_both(&s_full[b]);
          pair2::commit_both(&empty[slot_of(nki)]);
        }
        pair2::commit_local(&drain[1]);
        mbar_wait(&drain[1], 0, 200000000ull);
      } else {
        constexpr uint32_t idesc_o = idesc_bf16_f32(256, D, true);
        const uint64_t vdesc0 = smem_desc_sw128(ring_base, 8192, 1024);
        for (int j = 0; j < n_chunks; ++j) {
          const int b = j % k2Bufs, nvi = 2 * j + 1;
          const int nf = v0 + j < nc ? 1 : 2;   // tree keys: P = hi + lo
          if (!bounded_wait(&full[slot_of(nvi)], full_parity(nvi), P.err, abort_flag, 31, wait_ns) ||
              !bounded_wait(&p_full[b], (j / k2Bufs) & 1, P.err, abort_flag, 32, wait_ns))
            break;
          tc_fence_after();
          // keys 16kk.. of the chunk in columns 8kk.. of the buffer (bf16
          // pairs), the tree chunks' residual fill 64 columns further
          const uint64_t vd = vdesc0 + static_cast<uint64_t>((slot_of(nvi) * L::kItem) >> 4);
          for (int f = 0; f < nf; ++f) {
            const uint32_t pa = tmem + 128 + 128 * b + 64 * f;
#pragma unroll
            for (int kk = 0; kk < kChunk / 16; ++kk)
              pair2::mma_bf16_ta(tmem, pa + 8 * kk, vd + ((kk * 2048) >> 4), idesc_o,
                                 (j > 0 || f > 0 || kk > 0));
          }
          pair2::commit_both(&o_done[b]);
          pair2::commit_both(&empty[slot_of(nvi)]);
        }
        pair2::commit_local(&drain[0]);
        mbar_wait(&drain[0], 0, 200000000ull);
      }
    }
    __syncwarp();
  } else if (warp >= 4) {
    // ================================================================ softmax
    // Every softmax thread runs all n_chunks iterations and meets its
    // partner warpgroup at the named barrier in each; after a wait that ran
    // out (`live` false) the iterations skip their work.
    const uint32_t lane_off = static_cast<uint32_t>((warp & 3) * 32) << 16;
    const uint32_t o_addr = tmem + lane_off + 64 * wg;   // this warpgroup's 64 O columns
    const uint32_t s_addr = tmem + 128 + lane_off;       // S / P buffers of this row
    const uint32_t p_full_leader = pair2::map_to(smem_addr(p_full), 0);
    const float sl2 = P.scale_log2;
    const uint64_t sl2x2 = f32x2(sl2, sl2);
    const int W = (it.m + 63) >> 6;
    const int64_t mrow = row_valid ? static_cast<int64_t>(R / g) * W : -1;
    float m_run = -INFINITY, l_run = 0.f;
    bool live = n_chunks > 0;
    for (int j = 0; j < n_chunks; ++j) {
      const int b = j % k2Bufs;
      const uint32_t sb = s_addr + 128 * b;
      live = live && __all_sync(0xffffffffu, bounded_wait(&s_full[b], (j / k2Bufs) & 1, P.err, abort_flag, 40, wait_ns));
      // keys 64 wg .. 64 wg + 63 of the chunk; only the prefix's last chunk
      // and the tree chunks need a mask (key count, ancestor word)
      const int v = v0 + j;
      const bool pref = v < nc;
      float x[64];
      float mx = -INFINITY;
      if (live) {
        tc_fence_after();
        const int k0 = (pref ? v : v - nc) * kChunk + 64 * wg;
        const int nvalid = min(64, (pref ? it.prefix_len : it.m) - k0);
        uint32_t ra[32], rb[32];
        tmem_ld32(sb + 64 * wg, ra);
        tmem_ld32(sb + 64 * wg + 32, rb);
        tmem_wait_ld();
#pragma unroll
        for (int c = 0; c < 32; ++c) {
          x[c] = __uint_as_float(ra[c]);
          x[32 + c] = __uint_as_float(rb[c]);
        }
        if (!pref || nvalid < 64) {
          uint64_t wbits = ~0ull;
          if (!pref) wbits = (mrow >= 0 && nvalid > 0) ? __ldg(it.mask + mrow + (k0 >> 6)) : 0ull;
#pragma unroll
          for (int c = 0; c < 64; ++c)
            if (!((c < nvalid) & static_cast<bool>((wbits >> c) & 1ull))) x[c] = -INFINITY;
        }
        float m8[8];
#pragma unroll
        for (int a = 0; a < 8; ++a) m8[a] = fmax3(x[a], x[a + 8], x[a + 16]);
#pragma unroll
        for (int a = 0; a < 8; ++a) m8[a] = fmax3(m8[a], x[a + 24], x[a + 32]);
#pragma unroll
        for (int a = 0; a < 8; ++a) m8[a] = fmax3(m8[a], x[a + 40], x[a + 48]);
#pragma unroll
        for (int a = 0; a < 8; ++a) m8[a] = fmaxf(m8[a], x[a + 56]);
        mx = fmax3(fmax3(m8[0], m8[1], m8[2]), fmax3(m8[3], m8[4], m8[5]), fmaxf(m8[6], m8[7]));
      }
      // the other warpgroup's maximum of this row (both have their S values
      // in registers by now, so P may overwrite any of the buffer after this)
      xch[((j & 1) * 2 + wg) * 128 + row] = mx;
      named_sync(1, 256);
      if (!live) continue;
      mx = sl2 * fmaxf(mx, xch[((j & 1) * 2 + (1 - wg)) * 128 + row]);   // scale > 0
      const float m_new = fmaxf(m_run, mx);
      const bool grow = (j == 0) || (m_new > m_run + 8.0f);
      if (j > 0 && __any_sync(0xffffffffu, grow)) {
        // O is rescaled once the previous PV has landed.  S(j) was issued
        // after PV(j-3) completed, so PV(j-3) is done here while PV(j-2),
        // PV(j-1) may not be: one barrier per buffer keeps this wait within
        // one phase.
        live = __all_sync(0xffffffffu, bounded_wait(&o_done[(j - 1) % k2Bufs], ((j - 1) / k2Bufs) & 1,
                                                    P.err, abort_flag, 41, wait_ns));
        if (!live) continue;
        tc_fence_after();
        const float f = grow ? ex2(m_run - m_new) : 1.0f;
#pragma unroll 1
        for (int c = 0; c < 4; ++c) {
          uint32_t r[16];
          tmem_ld16(o_addr + 16 * c, r);
          tmem_wait_ld();
#pragma unroll
          for (int e = 0; e < 16; ++e) r[e] = __float_as_uint(__uint_as_float(r[e]) * f);
          tmem_st16(o_addr + 16 * c, r);
        }
        if (grow) l_run *= f;
      }
      if (grow) m_run = m_new;
      const float mref = (m_run == -INFINITY) ? 0.f : m_run;
      const uint64_t nm2 = f32x2(-mref, -mref);
      // P = 2^(s sl2 - m) as bf16 pairs: keys 2c, 2c+1 of the chunk -> column
      // c (this warpgroup: columns 32 wg ..); tree chunks put the rounding
      // residual 64 columns further
      uint32_t hi[32];
      uint64_t ls2[4] = {0ull, 0ull, 0ull, 0ull};
#pragma unroll
      for (int c = 0; c < 32; ++c) {
        float a0, a1;
        f32x2_split(fma_x2(f32x2(x[2 * c], x[2 * c + 1]), sl2x2, nm2), a0, a1);
        const float p0 = ex2(a0), p1 = ex2(a1);
        const uint64_t pp = f32x2(p0, p1);
        ls2[c & 3] = c < 4 ? pp : add_x2(ls2[c & 3], pp);
        hi[c] = pack_bf16x2(p0, p1);
        if (!pref) {
          x[2 * c] = p0 - __uint_as_float(hi[c] << 16);
          x[2 * c + 1] = p1 - __uint_as_float(hi[c] & 0xffff0000u);
        }
      }
      tmem_st32(sb + 32 * wg, hi);
      if (!pref) {
#pragma unroll
        for (int c = 0; c < 32; ++c) hi[c] = pack_bf16x2(x[2 * c], x[2 * c + 1]);
        tmem_st32(sb + 64 + 32 * wg, hi);
      }
      float s0, s1, s2, s3;
      f32x2_split(add_x2(add_x2(ls2[0], ls2[1]), add_x2(ls2[2], ls2[3])), s0, s1);
      l_run += s0 + s1;
      (void)s2;
      (void)s3;
      tmem_wait_st();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) pair2::arrive_cluster(p_full_leader + 8 * b);
    }
    // ---- epilogue: row sum of both warpgroups, then this warpgroup's 64
    // columns of O, normalised (one split) or as a partial
    bool ok = live && __all_sync(0xffffffffu, bounded_wait(&o_done[(n_chunks - 1) % k2Bufs],
                                                           ((n_chunks - 1) / k2Bufs) & 1, P.err,
                                                           abort_flag, 42, wait_ns));
    xch[512 + wg * 128 + row] = l_run;
    named_sync(1, 256);
    tc_fence_after();
    if (ok) {
      const float l_tot = l_run + xch[512 + (1 - wg) * 128 + row];
      const int qi = row_valid ? R / g : 0, hl = row_valid ? R - qi * g : 0;
      const int64_t orow = static_cast<int64_t>(qi) * P.hq + kvh * g + hl;
      const float inv = l_tot > 0.f ? 1.f / l_tot : 0.f;
      const int64_t punit =
          it.part_start + static_cast<int64_t>(kvh * it.tiles + tile) * it.splits + split;
      float* po = P.part_o + (punit * D + 64 * wg) * 128 + row;
#pragma unroll 1
      for (int c = 0; c < 2; ++c) {
        uint32_t r[32];
        tmem_ld32(o_addr + 32 * c, r);
        tmem_wait_ld();
        if (!row_valid) continue;
        if (it.splits == 1) {
          float4* dst = reinterpret_cast<float4*>(it.out + orow * D + 64 * wg + 32 * c);
#pragma unroll
          for (int e = 0; e < 8; ++e)
            dst[e] = make_float4(__uint_as_float(r[4 * e]) * inv, __uint_as_float(r[4 * e + 1]) * inv,
                                 __uint_as_float(r[4 * e + 2]) * inv, __uint_as_float(r[4 * e + 3]) * inv);
        } else {
#pragma unroll
          for (int e = 0; e < 32; ++e) po[(32 * c + e) * 128] = __uint_as_float(r[e]);
        }
      }
      if (row_valid && it.splits > 1 && wg == 0) P.part_ml[punit * 128 + row] = make_float2(m_run, l_tot);
    }
    // ---- split merge (few splits): the CTA whose partial of this (kv head,
    // tile) lands last combines every split's (o, max, sum) for its 128 rows
    // and writes the output; it leaves the arrival counter at zero for the
    // next call.  With many splits, attn_tc_merge_kernel runs instead (one
    // CTA reading many partials back is slower than a grid-wide pass).
    if (P.fuse_merge && it.splits > 1 && tile < it.tiles) {
      int* cnt = P.counters + it.cnt_start + kvh * it.tiles + tile;
      volatile int* last = reinterpret_cast<volatile int*>(xch + 1000);
      __threadfence();
      named_sync(1, 256);
      if (tid == 128) *last = atomicAdd(cnt, 1) == it.splits - 1;
      named_sync(1, 256);
      if (*last) {
        __threadfence();
        const int64_t pu0 = it.part_start + static_cast<int64_t>(kvh * it.tiles + tile) * it.splits;
        if (row_valid) {
          float mt = -INFINITY;
          for (int sp = 0; sp < it.splits; ++sp) mt = fmaxf(mt, __ldcg(P.part_ml + (pu0 + sp) * 128 + row).x);
          float acc[64];
#pragma unroll
          for (int c = 0; c < 64; ++c) acc[c] = 0.f;
          float lt = 0.f;
#pragma unroll 1
          for (int sp = 0; sp < it.splits; ++sp) {
            const float2 ml = __ldcg(P.part_ml + (pu0 + sp) * 128 + row);
            const float w = ml.x == -INFINITY ? 0.f : ex2(ml.x - mt);
            lt = fmaf(w, ml.y, lt);
            const float* po = P.part_o + ((pu0 + sp) * D + 64 * wg) * 128 + row;
#pragma unroll
            for (int c = 0; c < 64; ++c) acc[c] = fmaf(w, __ldcg(po + c * 128), acc[c]);
          }
          const float inv = lt > 0.f ? 1.f / lt : 0.f;
          const int qi = R / g, hl = R - qi * g;
          float4* dst = reinterpret_cast<float4*>(it.out + (static_cast<int64_t>(qi) * P.hq + kvh * g + hl) * D + 64 * wg);
#pragma unroll
          for (int e = 0; e < 16; ++e)
            dst[e] = make_float4(acc[4 * e] * inv, acc[4 * e + 1] * inv, acc[4 * e + 2] * inv, acc[4 * e + 3] * inv);
        }
        if (tid == 128) *cnt = 0;
      }
    }
  }

  // ---- teardown: no MMA of the pair is in flight (the even CTA waited for
  // its drain before reaching the barrier); tensor memory is freed by the
  // warps that allocated it, in both CTAs together
  tc_fence_before();
  pair2::cluster_sync();
  tc_fence_after();
  if (warp == 1) pair2::tmem_dealloc(tmem, k2TmemCols);
}

// Split merge: one block per (kv head, 128-row tile, 32 rows, 32 columns);
// lanes are rows, so every partial load is a coalesced 128-byte line; warp w
// combines columns 4w..4w+3 over the splits; the 32 x 32 result leaves row
// by row through a shared-memory transpose.  kOnce (up to kMergeOnce splits,
// a grid of at most one wave at its occupancy): every partial is loaded at
// once, then the splits' maximum and the weighted sum, so the loads cost one
// round trip, at ~110 registers a thread; otherwise online over the splits
// (running max in log2 units, 32 registers: many blocks per SM for large
// grids).  Partials: o column-major [unit][d][128 rows], (max, sum)
// [unit][128 rows].
struct TcMergeParams {
  TcItem items[kTcMaxItems];
  int block_start[kTcMaxItems + 1];   // first block of each item
  int n_items, hq, hkv, g;
  const float* part_o;
  const float2* part_ml;
};

constexpr int kMergeOnce = 16;

template <int D, bool kOnce>
__global__ void __launch_bounds__(256) attn_tc_merge_kernel(const __grid_constant__ TcMergeParams P) {
  pdl_trigger();   // let a dependent launch of the next kernel start (see pdl_attribute)
  __shared__ float tile[32][33];
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  int item = 0;
  while (item + 1 < P.n_items && static_cast<int>(blockIdx.x) >= P.block_start[item + 1]) ++item;
  const TcItem& it = P.items[item];
  const int S = it.splits;
  int b = blockIdx.x - P.block_start[item];
  const int cb = b % (D / 32);
  b /= D / 32;
  const int rb = b % 4;                          // 4 blocks of 32 rows per tile
  const int pair = b / 4;                        // kv head * tiles + tile
  const int kvh = pair / it.tiles, tp = pair - kvh * it.tiles;
  const int r = rb * 32 + lane;                  // row within the tile
  const int c0 = cb * 32 + 4 * warp;
  const int M = it.m * P.g;
  const int64_t u0 = it.part_start + static_cast<int64_t>(pair) * S;
  float mx = -INFINITY, l = 0.f;
  float acc[4] = {0.f, 0.f, 0.f, 0.f};
  constexpr int kPre = kMergeOnce;
  if (kOnce && 128 * tp + rb * 32 < M) {
    float2 ml[kPre];
    float o[kPre][4];
#pragma unroll
    for (int s = 0; s < kPre; ++s)
      if (s < S) {
        ml[s] = __ldcg(P.part_ml + (u0 + s) * 128 + r);
        const float* po = P.part_o + ((u0 + s) * D + c0) * 128 + r;
#pragma unroll
        for (int e = 0; e < 4; ++e) o[s][e] = __ldcg(po + e * 128);
      }
#pragma unroll
    for (int s = 0; s < kPre; ++s)
      if (s < S) mx = fmaxf(mx, ml[s].x);
#pragma unroll
    for (int s = 0; s < kPre; ++s)
      if (s < S) {
        const float w = ml[s].x == -INFINITY ? 0.f : ex2(ml[s].x - mx);
#pragma unroll
        for (int e = 0; e < 4; ++e) acc[e] = fmaf(w, o[s][e], acc[e]);
        l = fmaf(w, ml[s].y, l);
      }
  } else if (!kOnce && 128 * tp + rb * 32 < M) {
#pragma unroll 4
    for (int s = 0; s < S; ++s) {
      const float2 ml = __ldcg(P.part_ml + (u0 + s) * 128 + r);
      const float* po = P.part_o + ((u0 + s) * D + c0) * 128 + r;
      float o[4];
#pragma unroll
      for (int e = 0; e < 4; ++e) o[e] = __ldcg(po + e * 128);
      const float mn = fmaxf(mx, ml.x);
      const float a = mx == -INFINITY ? 0.f : ex2(mx - mn);
      const float w = ml.x == -INFINITY ? 0.f : ex2(ml.x - mn);
#pragma unroll
      for (int e = 0; e < 4; ++e) acc[e] = acc[e] * a + w * o[e];
      l = l * a + w * ml.y;
      mx = mn;
    }
  }
  const float inv = l > 0.f ? 1.f / l : 0.f;
#pragma unroll
  for (int e = 0; e < 4; ++e) tile[lane][4 * warp + e] = acc[e] * inv;
  __syncthreads();
#pragma unroll
  for (int rr = 0; rr < 4; ++rr) {   // row 4 warp + rr: lanes write 32 consecutive columns
    const int Rg = 128 * tp + rb * 32 + 4 * warp + rr;
    if (Rg < M) {
      const int qi = Rg / P.g, hl = Rg - qi * P.g;
      it.out[(static_cast<int64_t>(qi) * P.hq + kvh * P.g + hl) * D + cb * 32 + lane] =
          tile[4 * warp + rr][lane];
    }
  }
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

// 3-D uint8 tensor map (E4M3 codes) with a (128 x rows_box x 1) box, no swizzle.
static bool encode_3d_u8(CUtensorMap* map, const void* base, uint64_t d0, uint64_t d1,
                         uint64_t d2, uint64_t stride1_bytes, uint64_t stride2_bytes,
                         uint32_t box1) {
  auto fn = encode_fn();
  if (!fn) return false;
  cuuint64_t dims[3] = {d0, d1 ? d1 : 1, d2 ? d2 : 1};
  cuuint64_t strides[2] = {stride1_bytes, stride2_bytes};
  cuuint32_t box[3] = {128, box1, 1};
  cuuint32_t estr[3] = {1, 1, 1};
  return fn(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, const_cast<void*>(base), dims, strides, box,
            estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

bool tc_supported(int head_dim) { return head_dim == 64 || head_dim == 128; }

struct TcPlan {
  int span;
  int splits[kTcMaxItems];
  int tiles[kTcMaxItems];
  int units;            // CTAs (1-SM kernel) or CTA pairs (2-SM kernel)
  int64_t part_units;   // 128-row partial blocks
  int64_t counters;     // split-arrival counters (2-SM kernel)
  int max_splits;
};

// the 2-SM kernel merges splits in the kernel up to this many per tile
constexpr int kFusedMergeMaxSplits = 4;

// Work units per (item, kv head, pair of query tiles).
// two (the 2-SM kernel, a cluster of two CTAs per unit): a split covers
// `span` entries of the item's chunk list (its prefix chunks, then its tree
// chunks).  Otherwise (the 1-SM kernel, one CTA per unit): prefix splits of
// `span` chunks plus one tree split.  The span minimises waves x (span + fixed work
// of a unit, in chunks) plus a small charge per unit for its partials' write
// and read.
static TcPlan plan_tc(const eagle_attn_item* items, int n, int hq, int hkv, int d, int sms,
                      bool two) {
  TcPlan T;
  memset(&T, 0, sizeof(T));
  const int g = hq / hkv;
  int max_span = 1;
  for (int b = 0; b < n; ++b) {
    T.tiles[b] = (items[b].m * g + 127) / 128;
    const int nc = (items[b].prefix_len + kChunk - 1) / kChunk;
    const int nv = nc + (items[b].m + kChunk - 1) / kChunk;
    max_span = std::max(max_span, two ? nv : nc);
  }
  auto splits_of = [&](int b, int span) {
    const int nc = (items[b].prefix_len + kChunk - 1) / kChunk;
    if (two) return (nc + (items[b].m + kChunk - 1) / kChunk + span - 1) / span;
    return (nc + span - 1) / span + 1;
  };
  double best_cost = -1.0;
  for (int span = 1; span <= max_span; ++span) {
    int64_t total = 0;
    for (int b = 0; b < n; ++b)
      total += static_cast<int64_t>(hkv) * ((T.tiles[b] + 1) / 2) * splits_of(b, span);
    const int64_t slots = two ? 2 * total : total;
    const int64_t waves = (slots + sms - 1) / sms;
    const double cost = two ? static_cast<double>(waves * (span + 6)) + 0.02 * static_cast<double>(total)
                            : static_cast<double>(waves * (span + 2)) + 0.04 * static_cast<double>(total);
    if (best_cost < 0.0 || cost <= best_cost) {
      best_cost = cost;
      T.span = span;
    }
  }
  int64_t units = 0, part = 0;
  for (int b = 0; b < n; ++b) {
    T.splits[b] = splits_of(b, T.span);
    units += static_cast<int64_t>(hkv) * ((T.tiles[b] + 1) / 2) * T.splits[b];
    if (T.splits[b] > 1) part += static_cast<int64_t>(hkv) * T.tiles[b] * T.splits[b];
    if (two && T.splits[b] > 1) T.counters += static_cast<int64_t>(hkv) * T.tiles[b];
    T.max_splits = std::max(T.max_splits, T.splits[b]);
  }
  T.units = static_cast<int>(units);
  T.part_units = part;
  return T;
}

static size_t part_bytes(const TcPlan& T, int d) {
  return align_up(sizeof(float) * static_cast<size_t>(T.part_units) * 128 * d, 256) +
         align_up(sizeof(float2) * static_cast<size_t>(T.part_units) * 128, 256) +
         align_up(sizeof(int32_t) * static_cast<size_t>(T.counters), 256);
}

int attn_tc_num_launches(const eagle_attn_item* items, int n, int hq, int hkv, int d, int sms) {
  int count = 0;
  for (int b0 = 0; b0 < n; b0 += kTcMaxItems) {
    const int nb = std::min(kTcMaxItems, n - b0);
    const TcPlan T = plan_tc(items + b0, nb, hq, hkv, d, sms, d == 128);
    count += 1 + (T.part_units > 0 && (d != 128 || T.max_splits > kFusedMergeMaxSplits) ? 1 : 0);
  }
  return count;
}

size_t attn_tc_ws_size(const eagle_attn_item* items, int n, int hq, int hkv, int d, int sms) {
  size_t need = kWsHeader;
  for (int b0 = 0; b0 < n; b0 += kTcMaxItems) {
    const int nb = std::min(kTcMaxItems, n - b0);
    const TcPlan T = plan_tc(items + b0, nb, hq, hkv, d, sms, d == 128);
    need = std::max(need, kWsHeader + part_bytes(T, d));
  }
  return need;
}

// The split merge in its one-round form when every tile's splits fit and the
// grid is one wave at that form's occupancy (two blocks per SM), else online.
template <int D>
static void launch_merge(const TcMergeParams& MP, int blocks, int max_splits, int sms,
                         cudaStream_t stream) {
  if (max_splits <= kMergeOnce && blocks <= 2 * sms)
    attn_tc_merge_kernel<D, true><<<blocks, 256, 0, stream>>>(MP);
  else
    attn_tc_merge_kernel<D, false><<<blocks, 256, 0, stream>>>(MP);
}

// tables / pool_rows: per item, the block table and the pool's rows per head
// of a paged prefix (null arrays: every item contiguous)
template <int D>
static eagle_status launch_d(const eagle_attn_item* items, int n, int hq, int hkv, float scale,
                             void* ws, size_t ws_bytes, cudaStream_t stream, int sms,
                             const int32_t* const* tables = nullptr,
                             const int64_t* pool_rows = nullptr) {
  static_assert(sizeof(TcParams) < 32000, "kernel parameter block too large");
  for (int b0 = 0; b0 < n; b0 += kTcMaxItems) {
    const int nb = std::min(kTcMaxItems, n - b0);
    const eagle_attn_item* its = items + b0;
    const TcPlan T = plan_tc(its, nb, hq, hkv, D, sms, D == 128);
    if (ws_bytes < kWsHeader + part_bytes(T, D)) return EAGLE_ERR_WORKSPACE_TOO_SMALL;
    TcParams P;
    memset(&P, 0, sizeof(P));
    int64_t units = 0, part = 0, cnt = 0;
    for (int b = 0; b < nb; ++b) {
      const eagle_attn_item& x = its[b];
      // rows the prefix maps cover: the prefix, or the whole pool of a paged item
      const bool paged = tables && tables[b0 + b] && x.prefix_len > 0;
      const uint64_t S = paged ? static_cast<uint64_t>(pool_rows[b0 + b])
                               : static_cast<uint64_t>(x.prefix_len);
      const void* kbase = x.prefix_len ? x.k_cache : x.tree_k;
      const void* vbase = x.prefix_len ? x.v_cache : x.tree_v;
      const uint64_t hs = static_cast<uint64_t>(x.cache_head_stride) * 2;
      // boxes: the 2-SM kernel loads half a chunk per CTA (64 keys of K, 64
      // value columns of V), the 1-SM kernel a whole chunk (128 keys)
      const uint32_t kbox = D == 128 ? 64 : kChunk;
      const uint64_t ts = static_cast<uint64_t>(hkv) * D * 2;
      if (!encode_3d(&P.kmap[b], kbase, D, S, hkv, D * 2, x.prefix_len ? hs : D * 2, kbox, 1) ||
          !encode_3d(&P.vmap[b], vbase, D, S, hkv, D * 2, x.prefix_len ? hs : D * 2, kChunk, 1) ||
          !encode_3d(&P.tkmap[b], x.tree_k, D, hkv, x.m, D * 2, ts, 1, kbox) ||
          !encode_3d(&P.tvmap[b], x.tree_v, D, hkv, x.m, D * 2, ts, 1, kChunk))
        return EAGLE_ERR_CUDA;
      TcItem& ti = P.items[b];
      ti.q = static_cast<const __nv_bfloat16*>(x.q);
      ti.table = paged ? tables[b0 + b] : nullptr;
      ti.pool_pages = paged ? static_cast<int>(pool_rows[b0 + b] / kChunk) : 0;
      ti.out = x.out;
      ti.mask = x.mask;
      ti.m = x.m;
      ti.prefix_len = x.prefix_len;
      ti.splits = T.splits[b];
      ti.tiles = T.tiles[b];
      ti.pairs = (T.tiles[b] + 1) / 2;
      ti.unit_start = static_cast<int>(units);
      ti.part_start = part;
      ti.cnt_start = static_cast<int>(cnt);
      if (D == 128 && T.splits[b] > 1) cnt += static_cast<int64_t>(hkv) * T.tiles[b];
      units += static_cast<int64_t>(hkv) * ti.pairs * T.splits[b];
      if (T.splits[b] > 1) part += static_cast<int64_t>(hkv) * T.tiles[b] * T.splits[b];
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
        pbase + align_up(sizeof(float) * static_cast<size_t>(T.part_units) * 128 * D, 256));
    P.fuse_merge = D == 128 && T.max_splits <= kFusedMergeMaxSplits;
    P.counters = reinterpret_cast<int32_t*>(
        pbase + align_up(sizeof(float) * static_cast<size_t>(T.part_units) * 128 * D, 256) +
        align_up(sizeof(float2) * static_cast<size_t>(T.part_units) * 128, 256));
    if constexpr (D == 128) {   // 2-SM kernel: a cluster of two CTAs per unit
      const size_t smem = Sm2::kAlloc;
      EAGLE_CUDA(cudaFuncSetAttribute(attn2_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                      static_cast<int>(smem)));
      attn2_kernel<<<static_cast<unsigned>(2 * units), k2Threads, smem, stream>>>(P);
    } else {
      const size_t smem = TcSmem<D>::kAlloc;
      EAGLE_CUDA(cudaFuncSetAttribute(attn_tc_kernel<D, false>,
                                      cudaFuncAttributeMaxDynamicSharedMemorySize,
                                      static_cast<int>(smem)));
      attn_tc_kernel<D, false><<<static_cast<unsigned>(units), kTcThreads, smem, stream>>>(P);
    }
    eagle_status st = launch_status();
    if (st != EAGLE_OK) return st;
    if (part > 0 && !P.fuse_merge) {
      TcMergeParams MP;
      memset(&MP, 0, sizeof(MP));
      int blocks = 0;
      for (int b = 0; b < nb; ++b) {
        MP.items[b] = P.items[b];
        MP.block_start[b] = blocks;
        if (P.items[b].splits > 1) blocks += hkv * P.items[b].tiles * 4 * (D / 32);
      }
      MP.block_start[nb] = blocks;
      MP.n_items = nb;
      MP.hq = hq;
      MP.hkv = hkv;
      MP.g = hq / hkv;
      MP.part_o = P.part_o;
      MP.part_ml = P.part_ml;
      launch_merge<D>(MP, blocks, T.max_splits, sms, stream);
      if ((st = launch_status()) != EAGLE_OK) return st;
    }
  }
  return EAGLE_OK;
}

eagle_status attn_tc_launch(const eagle_attn_item* items, int n, int hq, int hkv, int d,
                            float scale, void* ws, size_t ws_bytes, cudaStream_t stream, int sms) {
  if (d == 128) return launch_d<128>(items, n, hq, hkv, scale, ws, ws_bytes, stream, sms);
  if (d == 64) return launch_d<64>(items, n, hq, hkv, scale, ws, ws_bytes, stream, sms);
  return EAGLE_ERR_UNSUPPORTED_SHAPE;
}

// ------------------------------------------------------------ E4M3 prefix
// The 1-SM kernel with its prefix chunks staged as E4M3 codes (head_dim 128);
// the tree keys / values are bf16 and go through its tree split as usual.
static eagle_status launch_fp8(const eagle_attn_fp8_item* items, int n, int hq, int hkv,
                               float scale, void* ws, size_t ws_bytes, cudaStream_t stream,
                               int sms) {
  constexpr int D = 128;
  std::vector<eagle_attn_item> flat(n);
  for (int b = 0; b < n; ++b) {
    flat[b].m = items[b].m;
    flat[b].prefix_len = items[b].prefix_len;
  }
  for (int b0 = 0; b0 < n; b0 += kTcMaxItems) {
    const int nb = std::min(kTcMaxItems, n - b0);
    const TcPlan T = plan_tc(flat.data() + b0, nb, hq, hkv, D, sms, false);
    if (ws_bytes < kWsHeader + part_bytes(T, D)) return EAGLE_ERR_WORKSPACE_TOO_SMALL;
    TcParams P;
    memset(&P, 0, sizeof(P));
    int64_t units = 0, part = 0;
    for (int b = 0; b < nb; ++b) {
      const eagle_attn_fp8_item& x = items[b0 + b];
      const uint64_t S = static_cast<uint64_t>(x.prefix_len);
      const uint64_t ts = static_cast<uint64_t>(hkv) * D * 2;
      const void* kb = x.prefix_len ? static_cast<const void*>(x.k_cache) : x.tree_k;
      const void* vb = x.prefix_len ? static_cast<const void*>(x.v_cache) : x.tree_v;
      const uint64_t hs = x.prefix_len ? static_cast<uint64_t>(x.cache_head_stride) : D;
      if (!encode_3d_u8(&P.kmap[b], kb, D, S, hkv, D, hs, kChunk) ||
          !encode_3d_u8(&P.vmap[b], vb, D, S, hkv, D, hs, kChunk) ||
          !encode_3d(&P.tkmap[b], x.tree_k, D, hkv, x.m, D * 2, ts, 1, kChunk) ||
          !encode_3d(&P.tvmap[b], x.tree_v, D, hkv, x.m, D * 2, ts, 1, kChunk))
        return EAGLE_ERR_CUDA;
      TcItem& ti = P.items[b];
      ti.q = static_cast<const __nv_bfloat16*>(x.q);
      ti.out = x.out;
      ti.mask = x.mask;
      ti.m = x.m;
      ti.prefix_len = x.prefix_len;
      ti.splits = T.splits[b];
      ti.tiles = T.tiles[b];
      ti.pairs = (T.tiles[b] + 1) / 2;
      ti.unit_start = static_cast<int>(units);
      ti.part_start = part;
      ti.kscale = x.k_scale;
      ti.vscale = x.v_scale;
      ti.sstride = x.scale_head_stride;
      units += static_cast<int64_t>(hkv) * ti.pairs * T.splits[b];
      if (T.splits[b] > 1) part += static_cast<int64_t>(hkv) * T.tiles[b] * T.splits[b];
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
        pbase + align_up(sizeof(float) * static_cast<size_t>(T.part_units) * 128 * D, 256));
    const size_t smem = TcSmem<D, true>::kAlloc;
    EAGLE_CUDA(cudaFuncSetAttribute(attn_tc_kernel<D, true>,
                                    cudaFuncAttributeMaxDynamicSharedMemorySize,
                                    static_cast<int>(smem)));
    attn_tc_kernel<D, true><<<static_cast<unsigned>(units), kTcThreads, smem, stream>>>(P);
    eagle_status st = launch_status();
    if (st != EAGLE_OK) return st;
    if (part > 0) {
      TcMergeParams MP;
      memset(&MP, 0, sizeof(MP));
      int blocks = 0;
      for (int b = 0; b < nb; ++b) {
        MP.items[b] = P.items[b];
        MP.block_start[b] = blocks;
        if (P.items[b].splits > 1) blocks += hkv * P.items[b].tiles * 4 * (D / 32);
      }
      MP.block_start[nb] = blocks;
      MP.n_items = nb;
      MP.hq = hq;
      MP.hkv = hkv;
      MP.g = hq / hkv;
      MP.part_o = P.part_o;
      MP.part_ml = P.part_ml;
      launch_merge<D>(MP, blocks, T.max_splits, sms, stream);
      if ((st = launch_status()) != EAGLE_OK) return st;
    }
  }
  return EAGLE_OK;
}

static eagle_status fp8_validate(const eagle_attn_fp8_item* items, int n, int hq, int hkv,
                                 int d) {
  EAGLE_CHECK_ARG(items && n >= 1 && n <= (1 << 20) && hq >= 1 && hkv >= 1 && hq % hkv == 0);
  EAGLE_CHECK_SHAPE(d == 128);
  for (int b = 0; b < n; ++b) {
    const eagle_attn_fp8_item& x = items[b];
    EAGLE_CHECK_ARG(x.m >= 1 && x.prefix_len >= 0);
    EAGLE_CHECK_SHAPE(x.m <= EAGLE_MAX_TREE);
    EAGLE_CHECK_ARG(x.q && x.tree_k && x.tree_v && x.mask && x.out);
    EAGLE_CHECK_ARG(aligned16(x.q) && aligned16(x.tree_k) && aligned16(x.tree_v) &&
                    aligned16(x.out));
    if (x.prefix_len > 0) {
      EAGLE_CHECK_ARG(x.k_cache && x.v_cache && x.k_scale && x.v_scale);
      EAGLE_CHECK_ARG(aligned16(x.k_cache) && aligned16(x.v_cache));
      EAGLE_CHECK_ARG(x.cache_head_stride % 16 == 0 &&
                      x.cache_head_stride >= static_cast<int64_t>(x.prefix_len) * d);
      EAGLE_CHECK_ARG(x.scale_head_stride >= (x.prefix_len + kChunk - 1) / kChunk);
    }
  }
  return EAGLE_OK;
}

// ------------------------------------------------------------- paged prefix
static eagle_status paged_items(const eagle_attn_paged_item* items, int n, int hq, int hkv, int d,
                                eagle_attn_item* flat, const int32_t** tables, int64_t* rows) {
  EAGLE_CHECK_ARG(items && n >= 1 && hq >= 1 && hkv >= 1 && hq % hkv == 0);
  EAGLE_CHECK_SHAPE(tc_supported(d));
  static_assert(EAGLE_KV_PAGE_TOKENS == kChunk, "a page is one K/V chunk of the kernel");
  for (int b = 0; b < n; ++b) {
    const eagle_attn_paged_item& x = items[b];
    EAGLE_CHECK_ARG(x.m >= 1 && x.prefix_len >= 0);
    EAGLE_CHECK_SHAPE(x.m <= EAGLE_MAX_TREE);
    EAGLE_CHECK_ARG(x.q && x.tree_k && x.tree_v && x.mask && x.out);
    EAGLE_CHECK_ARG(aligned16(x.q) && aligned16(x.tree_k) && aligned16(x.tree_v) &&
                    aligned16(x.out));
    if (x.prefix_len > 0) {
      EAGLE_CHECK_ARG(x.k_pool && x.v_pool && x.block_table && aligned16(x.k_pool) &&
                      aligned16(x.v_pool));
      EAGLE_CHECK_ARG(x.pool_head_stride % d == 0 && x.pool_head_stride % 8 == 0 &&
                      x.pool_head_stride >= static_cast<int64_t>(kChunk) * d);
    }
    eagle_attn_item& f = flat[b];
    f.q = x.q;
    f.k_cache = x.k_pool;
    f.v_cache = x.v_pool;
    f.tree_k = x.tree_k;
    f.tree_v = x.tree_v;
    f.mask = x.mask;
    f.out = x.out;
    f.cache_head_stride = x.pool_head_stride;
    f.prefix_len = x.prefix_len;
    f.m = x.m;
    tables[b] = x.block_table;
    rows[b] = x.prefix_len > 0 ? x.pool_head_stride / d : 0;
  }
  return EAGLE_OK;
}

}  // namespace eagle

using namespace eagle;

extern "C" size_t eagle_tree_attn_paged_workspace_size(const eagle_attn_paged_item* items,
                                                       int32_t n_items, int32_t n_q_heads,
                                                       int32_t n_kv_heads, int32_t head_dim) {
  if (!items || n_items < 1 || n_items > (1 << 20)) return 0;
  std::vector<eagle_attn_item> flat(n_items);
  std::vector<const int32_t*> tables(n_items);
  std::vector<int64_t> rows(n_items);
  if (paged_items(items, n_items, n_q_heads, n_kv_heads, head_dim, flat.data(), tables.data(),
                  rows.data()) != EAGLE_OK)
    return 0;
  return std::max(attn_tc_ws_size(flat.data(), n_items, n_q_heads, n_kv_heads, head_dim, kPlanSMs),
                  attn_tc_ws_size(flat.data(), n_items, n_q_heads, n_kv_heads, head_dim,
                                  plan_sms()));
}

extern "C" eagle_status eagle_tree_attn_paged_batched(const eagle_attn_paged_item* items,
                                                      int32_t n_items, int32_t n_q_heads,
                                                      int32_t n_kv_heads, int32_t head_dim,
                                                      float scale, void* ws, size_t ws_bytes,
                                                      eagle_stream stream) {
  EAGLE_CHECK_ARG(ws != nullptr && n_items >= 1 && n_items <= (1 << 20));
  std::vector<eagle_attn_item> flat(n_items);
  std::vector<const int32_t*> tables(n_items);
  std::vector<int64_t> rows(n_items);
  eagle_status st = paged_items(items, n_items, n_q_heads, n_kv_heads, head_dim, flat.data(),
                                tables.data(), rows.data());
  if (st != EAGLE_OK) return st;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  const int sms = plan_sms();
  return head_dim == 128
             ? launch_d<128>(flat.data(), n_items, n_q_heads, n_kv_heads, scale, ws, ws_bytes, s,
                             sms, tables.data(), rows.data())
             : launch_d<64>(flat.data(), n_items, n_q_heads, n_kv_heads, scale, ws, ws_bytes, s,
                            sms, tables.data(), rows.data());
}

extern "C" size_t eagle_tree_attn_fp8_workspace_size(const eagle_attn_fp8_item* items,
                                                     int32_t n_items, int32_t n_q_heads,
                                                     int32_t n_kv_heads, int32_t head_dim) {
  if (fp8_validate(items, n_items, n_q_heads, n_kv_heads, head_dim) != EAGLE_OK) return 0;
  std::vector<eagle_attn_item> flat(n_items);
  for (int b = 0; b < n_items; ++b) {
    memset(&flat[b], 0, sizeof(flat[b]));
    flat[b].m = items[b].m;
    flat[b].prefix_len = items[b].prefix_len;
  }
  size_t need = kWsHeader;
  for (const int sms : {kPlanSMs, plan_sms()})
    for (int b0 = 0; b0 < n_items; b0 += kTcMaxItems) {
      const int nb = std::min(kTcMaxItems, n_items - b0);
      const TcPlan T = plan_tc(flat.data() + b0, nb, n_q_heads, n_kv_heads, head_dim, sms, false);
      need = std::max(need, kWsHeader + part_bytes(T, head_dim));
    }
  return need;
}

extern "C" eagle_status eagle_tree_attn_fp8_batched(const eagle_attn_fp8_item* items,
                                                    int32_t n_items, int32_t n_q_heads,
                                                    int32_t n_kv_heads, int32_t head_dim,
                                                    float scale, void* ws, size_t ws_bytes,
                                                    eagle_stream stream) {
  eagle_status st = fp8_validate(items, n_items, n_q_heads, n_kv_heads, head_dim);
  if (st != EAGLE_OK) return st;
  EAGLE_CHECK_ARG(ws != nullptr);
  return launch_fp8(items, n_items, n_q_heads, n_kv_heads, scale, ws, ws_bytes,
                    reinterpret_cast<cudaStream_t>(stream), plan_sms());
}
