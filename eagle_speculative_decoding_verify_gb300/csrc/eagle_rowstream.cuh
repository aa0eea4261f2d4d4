// One HBM pass over rows of fp32 logits, shared by the tree build (draft
// rows) and the verify step (target rows).
//
// Work split: every row is streamed by one thread-block cluster of P CTAs
// (P <= 8, chosen on the host so that one wave fills the GPU).  CTA p of the
// cluster takes the p-th contiguous share of the row's 1024-element tiles
// and streams it through a six-slot shared-memory ring (16 KB slots) filled
// by 1-D bulk (TMA) copies; a slot is released through an mbarrier that each
// warp arrives on once it holds its elements in registers, so no CTA barrier
// is taken per slot.  Per CTA:
//   * max and sum of 2^((x - max) c) per thread (fp32 ex2), combined with
//     fp32 factors and fp64 accumulation;
//   * the exact top-K (value desc, token id asc), K <= 64, in two passes
//     over the CTA's share.  The first (the stream itself) keeps each
//     thread's five best slot maxima (its candidate slots) and each warp's
//     maximum of every slot; at its end the K-th largest of the CTA's 256
//     thread maxima (K distinct elements reach it) becomes the bound.  The
//     second reloads from L2 each thread's candidate slots that reach the
//     bound (about K thread-slots per CTA); a warp with a lane whose fifth
//     candidate slot reaches the bound as well (it may have more) revisits
//     instead every warp-slot whose maximum reaches the bound.  In the
//     verify kernel the next slot's load overlaps the current slot's
//     absorption on both routes.  Each warp keeps the elements at or above
//     the bound in a private buffer: about K per CTA, where a one-pass
//     running bound lets some K ln(n / K) through, nearly one per warp and
//     slot.  A warp whose buffer grows past max(2K, 64) entries cuts it to
//     its best K, which raises its bound to its exact K-th best; that entry
//     is also published as the CTA's running bound (shared-memory atomicMax
//     on the 64-bit key), which every warp reads once per slot;
//   * the argmax (K = 1);
//   * optionally per-tile (max, sum) of every warp for inverse-CDF sampling.
// Row end: every warp ranks its survivors by counting into a sorted list of at
// most K; the CTA merges its 8 lists by counting ranks straight into the
// shared memory of the cluster's rank-0 CTA (distributed shared memory),
// together with its max and sum; after one cluster barrier the rank-0 CTA
// merges the P lists the same way and writes the row record.  The caller then
// runs its per-row step and arrives on the item's counter; the CTA whose row
// arrives last runs the item's final step.  The counter lives in the
// workspace, starts at zero and is reset by its last user; nothing spins on
// it.
#pragma once

#include "eagle_common.cuh"

namespace eagle {

constexpr int kTile = 1024;                   // tokens per tile
constexpr int kSlotTiles = 4;                 // tiles per ring slot
constexpr int kSlotElems = kTile * kSlotTiles;  // 4096 floats = 16 KB
constexpr int kSlots = 6;                     // ring depth
constexpr int kThreads = 256;
constexpr int kWarps = kThreads / 32;
constexpr int kVec = kSlotElems / kThreads / 4;  // float4 per thread per slot (4)
constexpr int kPer = kVec * 4;                // elements per thread per slot (16)
constexpr int kWarpCap = 256;                 // survivors per warp (> K, so cuts progress)
constexpr int kKMax = EAGLE_MAX_TOP_K;
constexpr int kMaxItems = EAGLE_MAX_BATCH;
constexpr int kMaxCluster = 8;                // CTAs per row
constexpr int kTrackSlots = 64;               // slots per CTA with a recorded warp maximum
constexpr int kCand = 5;                      // candidate slots per thread (second pass)
constexpr float kLog2e = 1.4426950408889634f;

enum : int { kWantSum = 1, kWantTileSums = 2 };

struct RowStream {
  const float* base[kMaxItems];  // row 0 of each item
  float exp_scale[kMaxItems];    // factor on (x - max) inside exp: 1/T (1 for draft)
  int16_t topk[kMaxItems];       // K per item (0 = none, 1 = argmax)
  int16_t flags[kMaxItems];      // kWantSum | kWantTileSums
  int64_t row_stride;
  int n_items, rows_per_item, vocab, tiles_per_row, ctas_per_row, rec_k;
  int32_t* err;
  uint32_t* item_cnt;            // [n_items]
  char* rows;                    // [rows] row records
  float2* tile_sums;             // [rows][tiles_per_row][kWarps] or null
};

// Row record:  double sum; float max; int count; float val[rec_k]; int idx[rec_k]
// `sum` is sum_x 2^((x - max) * c) with c = exp_scale * log2(e), i.e. the sum
// of exp((x - max) * exp_scale).
__host__ __device__ constexpr int rec_bytes(int rec_k) {
  return static_cast<int>(align_up(16 + 8 * static_cast<size_t>(rec_k), 16));
}
struct RecHead {
  double sum;
  float max;
  int count;
};
__device__ __forceinline__ float* rec_val(char* rec) { return reinterpret_cast<float*>(rec + 16); }
__device__ __forceinline__ int* rec_idx(char* rec, int rec_k) {
  return reinterpret_cast<int*>(rec + 16 + 4 * rec_k);
}

// (value, token) as one 64-bit key, larger key = earlier in (value desc,
// token asc) order: high word = order-preserving image of the float (-0 taken
// as +0), low word = ~token.  Key 0 marks no element (-inf padding; inputs
// are finite).
using Key = unsigned long long;
constexpr int kNoIndex = 0x7fffffff;
__device__ __forceinline__ uint32_t fkey(float v) {
  uint32_t u = __float_as_uint(v);
  u = (u == 0x80000000u) ? 0u : u;
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}
__device__ __forceinline__ Key mkkey(float v, int i) {
  return v == -INFINITY ? 0ull
                        : (static_cast<Key>(fkey(v)) << 32) | static_cast<uint32_t>(~i);
}
__device__ __forceinline__ float key_v(Key k) {
  const uint32_t h = static_cast<uint32_t>(k >> 32);
  return k ? __uint_as_float((h & 0x80000000u) ? (h & 0x7fffffffu) : ~h) : -INFINITY;
}
__device__ __forceinline__ float fkey_value(uint32_t h) {   // inverse of fkey
  return __uint_as_float((h & 0x80000000u) ? (h & 0x7fffffffu) : ~h);
}
__device__ __forceinline__ int key_i(Key k) {
  return k ? static_cast<int>(~static_cast<uint32_t>(k)) : kNoIndex;
}
__device__ __forceinline__ Key warp_max_key(Key k) {
#pragma unroll
  for (int o = 16; o; o >>= 1) {
    const Key y = __shfl_xor_sync(0xffffffffu, k, o);
    k = y > k ? y : k;
  }
  return k;
}

static_assert(kWarps * kKMax >= kThreads, "the warp lists hold one key per thread (first-slot bound)");

struct StreamSmem {
  // 96 KB: the stream's ring; then (second pass) the warp survivor buffers,
  // kWarpCap keys per warp at its start; then the callers' final steps
  float ring[kSlots][kSlotElems];
  Key wlist[kWarps * kKMax];           // warp lists, stride K
  Key clist[kMaxCluster * kKMax];      // rank-0 CTA: the cluster's CTA lists, stride max(K, 1)
  Key rlist[kKMax];                    // rank-0 CTA: the row's list (best first)
  double csum[kMaxCluster];
  float cmax[kMaxCluster];
  int ccnt[kMaxCluster];
  double red_d[kWarps];
  float red_f[kWarps];
  int lcnt[kWarps];
  Key red_best[kWarps];
  double rsum;                         // rank-0 CTA: row sum, max, count
  float rmax;
  int rcount;
  int flag;
  int ncand;                           // second-pass bound: candidate thread maxima
  uint32_t wbound[kWarps];             // second-pass bound: per-warp bounds (value keys)
  uint32_t tkey;                       // second-pass bound (value key; 0: none)
  float wsmax[kWarps][kTrackSlots];    // first pass: every warp's maximum of every slot
  Key cta_bound;                       // running bound: K-th best of the CTA so far
  int aux[2 * EAGLE_MAX_TREE];         // callers' own data (never touched by the stream)
  unsigned long long aux_key;          // (callers' own)
  double aux_d;                        // (callers' own)
  uint64_t full[kSlots];
  uint64_t empty[kSlots];
};
// bytes of the region (the ring) the final steps reuse
constexpr size_t kScratchBytes = sizeof(float) * kSlots * kSlotElems;
static_assert(sizeof(Key) * kWarps * kWarpCap <= kScratchBytes, "warp buffers live in the ring");
// two CTAs per SM: 228 KB of shared memory per SM, 1 KB of it reserved per CTA
static_assert(2 * (sizeof(StreamSmem) + 1024) <= 228 * 1024, "two stream CTAs per SM");

// ------------------------------------------------------------ cluster helpers
__device__ __forceinline__ uint32_t map_rank0(const void* p) {
  uint32_t a;
  asm volatile("mapa.shared::cluster.u32 %0, %1, 0;" : "=r"(a) : "r"(smem_addr(p)));
  return a;
}
// address of p in the shared memory of CTA r of the cluster
__device__ __forceinline__ uint32_t map_rank(const void* p, uint32_t r) {
  uint32_t a;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(a) : "r"(smem_addr(p)), "r"(r));
  return a;
}
__device__ __forceinline__ unsigned long long ld_cluster_u64(uint32_t a) {
  unsigned long long v;
  asm volatile("ld.shared::cluster.u64 %0, [%1];" : "=l"(v) : "r"(a) : "memory");
  return v;
}
__device__ __forceinline__ uint32_t ld_cluster_u32(uint32_t a) {
  uint32_t v;
  asm volatile("ld.shared::cluster.u32 %0, [%1];" : "=r"(v) : "r"(a) : "memory");
  return v;
}
__device__ __forceinline__ uint32_t atom_add_cluster_u32(uint32_t a, uint32_t v) {
  uint32_t old;
  asm volatile("atom.shared::cluster.add.u32 %0, [%1], %2;" : "=r"(old) : "r"(a), "r"(v) : "memory");
  return old;
}
__device__ __forceinline__ void st_cluster(uint32_t a, Key v) {
  asm volatile("st.shared::cluster.u64 [%0], %1;" ::"r"(a), "l"(v) : "memory");
}
__device__ __forceinline__ void st_cluster(uint32_t a, float v) {
  asm volatile("st.shared::cluster.f32 [%0], %1;" ::"r"(a), "f"(v) : "memory");
}
__device__ __forceinline__ void st_cluster(uint32_t a, double v) {
  asm volatile("st.shared::cluster.f64 [%0], %1;" ::"r"(a), "d"(v) : "memory");
}
__device__ __forceinline__ void st_cluster(uint32_t a, int v) {
  asm volatile("st.shared::cluster.s32 [%0], %1;" ::"r"(a), "r"(v) : "memory");
}
__device__ __forceinline__ void cluster_arrive_relaxed() {
  asm volatile("barrier.cluster.arrive.relaxed.aligned;" ::: "memory");
}
__device__ __forceinline__ void cluster_arrive_release() {
  asm volatile("barrier.cluster.arrive.release.aligned;" ::: "memory");
}
__device__ __forceinline__ void cluster_wait() {
  asm volatile("barrier.cluster.wait.acquire.aligned;" ::: "memory");
}

// ------------------------------------------------------------ selections
// Ranks by counting: every lane holds E entries (positions lane + 32 r) of
// buf[0, n); rank = entries before it.  Writes the entries of rank < K to
// dst[rank] (dst may alias buf: all reads finish before the first write).
template <int E>
__device__ __forceinline__ void rank_count(const Key* buf, int n, int K, Key* dst) {
  const int lane = threadIdx.x & 31;
  Key mine[E];
  int rk[E];
#pragma unroll
  for (int r = 0; r < E; ++r) {
    const int a = lane + 32 * r;
    mine[r] = a < n ? buf[a] : 0ull;
    rk[r] = 0;
  }
#pragma unroll 4
  for (int b = 0; b < n; ++b) {
    const Key o = buf[b];
#pragma unroll
    for (int r = 0; r < E; ++r) rk[r] += o > mine[r] ? 1 : 0;
  }
  __syncwarp();
#pragma unroll
  for (int r = 0; r < E; ++r) {
    const int a = lane + 32 * r;
    if (a < n && rk[r] < K) dst[rk[r]] = mine[r];
  }
  __syncwarp();
}

// Best min(n, K) of the n <= kWarpCap entries of buf, best first into dst;
// one warp.  Returns min(n, K).
static __device__ __noinline__ int warp_select(const Key* buf, int n, int K, Key* dst) {
  if (n <= 32) rank_count<1>(buf, n, K, dst);
  else if (n <= 64) rank_count<2>(buf, n, K, dst);
  else if (n <= 128) rank_count<4>(buf, n, K, dst);
  else rank_count<8>(buf, n, K, dst);
  return n < K ? n : K;
}

// Rank of entry c of list p in the union of nl lists at stride `stride`
// (each sorted best first, counts cnt, keys distinct): c plus, for every
// other list, the number of its entries before it -- counted over the whole
// list with independent loads (a dependent binary-search probe costs ~90
// cycles on this part, so a search over lists of up to 127 entries is slower
// than the count).
__device__ __forceinline__ int union_rank(const Key* L, const int* cnt, int nl, int stride, int p,
                                          int c) {
  const Key e = L[p * stride + c];
  int r = c;
  for (int q = 0; q < nl; ++q) {
    if (q == p) continue;
    const Key* lq = L + q * stride;
    const int n = cnt[q];
    int before = 0;
#pragma unroll 8
    for (int i = 0; i < n; ++i) before += lq[i] > e ? 1 : 0;
    r += before;
  }
  return r;
}

// Before a merge (one warp, nl <= 32 sorted lists at `stride`): a bound with
// K entries of the union at or before it, below which nothing can be among
// the union's best K -- the best of the lists' K-th entries (K entries in
// that list), and, when every list has q = ceil(K / nl) entries, the worst of
// the lists' q-th entries (nl q >= K entries).  Cuts every list's count to
// its entries at or before the better bound.
__device__ __forceinline__ void prune_lists(const Key* L, int* cnt, int nl, int K, int stride) {
  const int lane = threadIdx.x & 31;
  const int q = (K + nl - 1) / nl;
  const int n = lane < nl ? cnt[lane] : 0;
  const bool full = n == K;
  Key tau = warp_max_key(full ? L[lane * stride + K - 1] : 0ull);
  if (__all_sync(0xffffffffu, lane >= nl || n >= q)) {
    Key t2 = lane < nl ? L[lane * stride + q - 1] : ~0ull;
#pragma unroll
    for (int o = 16; o; o >>= 1) {
      const Key y = __shfl_xor_sync(0xffffffffu, t2, o);
      t2 = y < t2 ? y : t2;
    }
    tau = t2 > tau ? t2 : tau;
  }
  if (tau == 0ull) return;
  if (lane < nl) {
    const Key* lq = L + lane * stride;
    const int n = cnt[lane];   // entries at or before tau form a prefix: count them
    int keep = 0;
#pragma unroll 8
    for (int i = 0; i < n; ++i) keep += lq[i] >= tau ? 1 : 0;
    cnt[lane] = keep;
  }
  __syncwarp();
}

// ------------------------------------------------------------ the stream
struct RowCtx {
  int64_t row;      // global row (item * rows_per_item + row of the item)
  int item;
  bool leader;      // rank 0 of the row's cluster: holds the row result
};

// One cluster's row: where it is, what to compute, where the result goes.
struct RowJob {
  const float* src;   // the row's logits
  char* rec;          // the row record
  float2* tsums;      // the row's per-(tile, warp) sums (kWantTileSums)
  int32_t* err;       // error word
  int64_t row;        // global row (item * rows_per_item + row of the item)
  int item, vocab, TR, PC, rank, K, flags, rec_k;
  float c2;           // exp scale * log2(e)
};

// The job of CTA `rank` of the cluster that streams global row `row`.
static __device__ __forceinline__ RowJob row_job(const RowStream& P, int64_t row, int rank) {
  RowJob J;
  J.row = row;
  J.item = static_cast<int>(row / P.rows_per_item);
  const int lrow = static_cast<int>(row - static_cast<int64_t>(J.item) * P.rows_per_item);
  J.src = P.base[J.item] + lrow * P.row_stride;
  J.rec = P.rows + row * rec_bytes(P.rec_k);
  J.tsums = P.tile_sums ? P.tile_sums + row * P.tiles_per_row * kWarps : nullptr;
  J.err = P.err;
  J.vocab = P.vocab;
  J.TR = P.tiles_per_row;
  J.PC = P.ctas_per_row;
  J.rank = rank;
  J.K = P.topk[J.item];
  J.flags = P.flags[J.item];
  J.rec_k = P.rec_k;
  J.c2 = P.exp_scale[J.item] * kLog2e;
  return J;
}

// Code warm-up.  The code that runs once per row at its end (the CTA and row
// merges, the callers' per-row and final steps) is not in L2 when the row's
// data has just been flushed through it, and fetching it from HBM by the
// leaders of every row at once costs several microseconds.  One extra
// cluster streams a short row of its own through the same code (same call
// sites) at launch, so that the code is in L2 when the real rows reach it.
// Only worth it when the rows are long enough for the warm-up to run ahead of
// them (stream_warm_up); on short rows it would only lengthen the launch.
//
// The warm-up reads and writes only library-owned static memory, never the
// caller's buffers, so that it may run before the launch's dependency on
// the previous kernel is resolved (pdl_wait): its row is one tile per CTA of
// g_warm_row, written by that CTA (a descending ramp); its record, tile sums
// and error word go to g_warm_out.  Launches that overlap write the same
// values or outputs nothing reads.
constexpr int kWarmMinTilesPerCta = 16;
__host__ __device__ constexpr bool stream_warm_up(int tiles_per_row, int ctas_per_row) {
  return tiles_per_row >= kWarmMinTilesPerCta * ctas_per_row;
}
static __device__ __align__(16) float g_warm_row[kMaxCluster * kTile];
static __device__ __align__(16) char g_warm_out[32 + rec_bytes(kKMax) + sizeof(float2) * kMaxCluster * kWarps];

// CTA `rank` of the warm-up cluster: writes its tile of the warm-up row, and
// returns its job (item 0's statistics, the cluster's PC tiles).
static __device__ __forceinline__ RowJob warm_row_job(const RowStream& P, int rank) {
  RowJob J = row_job(P, 0, rank);
  for (int i = threadIdx.x; i < kTile; i += kThreads)
    g_warm_row[rank * kTile + i] = -static_cast<float>(rank * kTile + i) * (1.0f / 1024.0f);
  fence_proxy_async_global();   // generic writes, then bulk-copy reads of them
  __syncthreads();
  J.src = g_warm_row;
  J.vocab = P.ctas_per_row * kTile;
  J.TR = P.ctas_per_row;
  J.err = reinterpret_cast<int32_t*>(g_warm_out);
  J.rec = g_warm_out + 32;
  J.tsums = J.tsums ? reinterpret_cast<float2*>(g_warm_out + 32 + rec_bytes(kKMax)) : nullptr;
  return J;
}

// Streams this CTA's share of its row; on return the leader has written the
// row record and holds it in S.rlist / rmax / rsum / rcount.  Every CTA of
// the grid calls it exactly once (it contains cluster barriers).
// kOverlapReload: in the second pass, a thread's next candidate slot is
// loaded before the current one is absorbed (two slot buffers: it pays where
// the kernel's registers allow it; measured: the verify kernel 1.5 us faster,
// the build kernel, which then spilled, 4.5 us slower).
template <bool kOverlapReload = false>
static __device__ __forceinline__ RowCtx stream_row(const RowJob& Jb, StreamSmem& S) {
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int PC = Jb.PC;
  RowCtx cx;
  cx.row = Jb.row;
  const int rank = Jb.rank;
  cx.leader = rank == 0;
  cx.item = Jb.item;
  const float* src = Jb.src;
  const int TR = Jb.TR;
  const int tile0 = rank * TR / PC;
  const int e_begin = tile0 * kTile;
  const int e_end = min(Jb.vocab, ((rank + 1) * TR / PC) * kTile);
  const int n_el = e_end > e_begin ? e_end - e_begin : 0;
  const int n_slots = (n_el + kSlotElems - 1) / kSlotElems;
  const int K = Jb.K;
  const int flags = Jb.flags;
  const float c2 = Jb.c2;

  auto issue = [&](int j) {  // thread 0: bulk copy of slot j
    const int off = j * kSlotElems;
    int nel = n_el - off;
    if (nel > kSlotElems) nel = kSlotElems;
    const uint32_t bytes = static_cast<uint32_t>(nel & ~3) * 4u;
    uint64_t* bar = &S.full[j % kSlots];
    mbar_arrive_expect_tx(bar, bytes);
    if (bytes) bulk_copy_g2s(S.ring[j % kSlots], src + e_begin + off, bytes, bar);
  };

  if (tid == 0) {
    for (int s = 0; s < kSlots; ++s) {
      mbar_init(&S.full[s], 1);
      mbar_init(&S.empty[s], kWarps);
    }
    fence_barrier_init();
    S.ncand = 0;
    S.tkey = 0u;
    S.cta_bound = 0ull;
  }
  __syncthreads();
  if (tid == 0)
    for (int j = 0; j < kSlots && j < n_slots; ++j) issue(j);
  __syncwarp();
  cluster_arrive_relaxed();   // every CTA of the cluster has started (waited on at row end)

  float m_run = -INFINITY, s_run = 0.f;       // per-thread running max / sum
  // K >= 2: this thread's kCand best slot maxima (cv, best first) and their
  // slots (cs); a slot enters only with a larger maximum, so of equal maxima
  // the earlier slot stays
  float cv[kCand];
  int cs[kCand];
#pragma unroll
  for (int r = 0; r < kCand; ++r) {
    cv[r] = -INFINITY;
    cs[r] = 0;
  }
  float best_v = -INFINITY;                    // per-thread argmax (K == 1)
  int best_i = kNoIndex;
  float thr_v = INFINITY;                      // warp survivor bound (K >= 2): elements
  int thr_i = kNoIndex;                        // at or before (thr_v, thr_i)
  int wn = 0;                                  // entries in this warp's buffer
  // the warp's survivor buffer, in the ring: written only in the second pass,
  // after the first pass's last CTA barrier (every thread has then read its
  // last slot and no bulk copy is in flight)
  Key* wb = reinterpret_cast<Key*>(S.ring) + warp * kWarpCap;

  for (int j = 0; j < n_slots; ++j) {
    const int b = j % kSlots;
    const uint32_t par = (j / kSlots) & 1;
    if (!mbar_wait(&S.full[b], par)) {
      record_error(Jb.err, kDevTimeout, 1);
      mbar_wait(&S.full[b], par);  // give an in-flight copy a last chance to land
    }
    const int off = j * kSlotElems;
    int nel = n_el - off;
    if (nel > kSlotElems) nel = kSlotElems;
    const int n4 = nel & ~3;  // elements delivered by the bulk copy
    float x[kPer];
#pragma unroll
    for (int q = 0; q < kVec; ++q) {
      const int e = (q * kThreads + tid) * 4;
      float4 f = make_float4(-INFINITY, -INFINITY, -INFINITY, -INFINITY);
      if (e + 4 <= n4) {
        f = *reinterpret_cast<const float4*>(&S.ring[b][e]);
      } else if (e < nel) {  // ragged row tail (vocab % 4 != 0): read it directly
        const float* g = src + e_begin + off + e;
        const int avail = nel - e;
        f.x = __ldg(g);
        if (avail > 1) f.y = __ldg(g + 1);
        if (avail > 2) f.z = __ldg(g + 2);
      }
      x[4 * q + 0] = f.x;
      x[4 * q + 1] = f.y;
      x[4 * q + 2] = f.z;
      x[4 * q + 3] = f.w;
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(&S.empty[b]);   // one arrival per warp
    if (tid == 0 && j + kSlots < n_slots) {    // refill once every warp has read the slot
      if (!mbar_wait(&S.empty[b], par)) record_error(Jb.err, kDevTimeout, 2);
      fence_proxy_async_smem();
      issue(j + kSlots);
    }

    const int tbase = e_begin + off + tid * 4;  // token of element (q, c) = tbase + q * 1024 + c

    float lm;
    {
      float m4[4];
#pragma unroll
      for (int a = 0; a < 4; ++a) m4[a] = fmaxf(fmaxf(x[a], x[4 + a]), fmaxf(x[8 + a], x[12 + a]));
      lm = fmaxf(fmaxf(m4[0], m4[1]), fmaxf(m4[2], m4[3]));
    }

    // ---- sum of exp (invalid elements are -inf and contribute 0)
    if (flags & kWantSum) {
      const float mn = fmaxf(m_run, lm);
      if (mn != -INFINITY) {
        s_run *= ex2((m_run - mn) * c2);
        const float offc = mn * c2;
        float acc[4];
#pragma unroll
        for (int a = 0; a < 4; ++a) acc[a] = ex2(fmaf(x[a], c2, -offc));
#pragma unroll
        for (int e = 4; e < kPer; ++e) acc[e & 3] += ex2(fmaf(x[e], c2, -offc));
        s_run += (acc[0] + acc[1]) + (acc[2] + acc[3]);
        m_run = mn;
      }
    }

    // ---- per-tile (max, sum) of this warp's 128 elements of every tile
    if (flags & kWantTileSums) {
      float tm[kVec], ts[kVec];
#pragma unroll
      for (int q = 0; q < kVec; ++q)
        tm[q] = fmaxf(fmaxf(x[4 * q], x[4 * q + 1]), fmaxf(x[4 * q + 2], x[4 * q + 3]));
#pragma unroll
      for (int o = 16; o; o >>= 1)
#pragma unroll
        for (int q = 0; q < kVec; ++q) tm[q] = fmaxf(tm[q], __shfl_xor_sync(0xffffffffu, tm[q], o));
#pragma unroll
      for (int q = 0; q < kVec; ++q) {
        ts[q] = 0.f;
        if (tm[q] != -INFINITY) {
#pragma unroll
          for (int c = 0; c < 4; ++c) ts[q] += ex2((x[4 * q + c] - tm[q]) * c2);
        }
      }
#pragma unroll
      for (int o = 16; o; o >>= 1)
#pragma unroll
        for (int q = 0; q < kVec; ++q) ts[q] += __shfl_xor_sync(0xffffffffu, ts[q], o);
      if (lane == 0) {
#pragma unroll
        for (int q = 0; q < kVec; ++q)
          if (q * kTile < nel)
            Jb.tsums[(tile0 + j * kSlotTiles + q) * kWarps + warp] =
                make_float2(tm[q], ts[q]);
      }
    }

    // ---- argmax (each thread sees its tokens in increasing order)
    if (K == 1) {
#pragma unroll
      for (int q = 0; q < kVec; ++q)
#pragma unroll
        for (int c = 0; c < 4; ++c) {
          const bool t = x[4 * q + c] > best_v;
          best_v = t ? x[4 * q + c] : best_v;
          best_i = t ? tbase + q * kTile + c : best_i;
        }
    }

    // ---- end of the first pass (K >= 2): the second pass's bound.  The
    // K-th largest of the CTA's thread maxima has K distinct elements at or
    // above it, so the CTA's best K are all at or above it as well.  First a
    // per-warp bound, the largest lane maximum that q = ceil(K / 8) lanes
    // reach; the smallest of the eight is reached by 8 q >= K lanes (0: fewer
    // valid lanes, no bound).  Then the exact K-th largest among the lane
    // maxima at or above it, by counting.  Values only: an element equal to
    // the bound survives whatever its token, which keeps a superset.
    if (K >= 2) {
      {   // insert (lm, j): entry r takes entry r-1 if lm beats that, else lm if it beats r
        bool g[kCand];
#pragma unroll
        for (int r = 0; r < kCand; ++r) g[r] = lm > cv[r];
#pragma unroll
        for (int r = kCand - 1; r > 0; --r) {
          cv[r] = g[r - 1] ? cv[r - 1] : (g[r] ? lm : cv[r]);
          cs[r] = g[r - 1] ? cs[r - 1] : (g[r] ? j : cs[r]);
        }
        cv[0] = g[0] ? lm : cv[0];
        cs[0] = g[0] ? j : cs[0];
      }
      const float wm = warp_max(lm);
      if (lane == 0 && j < kTrackSlots) S.wsmax[warp][j] = wm;
      if (j == n_slots - 1) {
        const float tmax = cv[0];   // this thread's maximum
        const uint32_t c0 = tmax == -INFINITY ? 0u : fkey(tmax);
        const int q = (K + kWarps - 1) / kWarps;
        int ge = 0;
#pragma unroll 8
        for (int s = 0; s < 32; ++s) ge += __shfl_sync(0xffffffffu, c0, s) >= c0 ? 1 : 0;
        const uint32_t wq = __reduce_max_sync(0xffffffffu, (ge >= q && c0 != 0u) ? c0 : 0u);
        if (lane == 0) S.wbound[warp] = wq;
        __syncthreads();
        uint32_t cb = S.wbound[0];
#pragma unroll
        for (int w = 1; w < kWarps; ++w) cb = S.wbound[w] < cb ? S.wbound[w] : cb;
        if (cb != 0u) {   // the same in every thread
          const bool cand = c0 >= cb;
          const unsigned bm = __ballot_sync(0xffffffffu, cand);
          int o = 0;
          if (lane == 0 && bm) o = atomicAdd(&S.ncand, __popc(bm));
          o = __shfl_sync(0xffffffffu, o, 0);
          uint32_t* ck = reinterpret_cast<uint32_t*>(S.wlist);  // filled only after the stream
          if (cand) ck[o + __popc(bm & ((1u << lane) - 1u))] = c0;
          __syncthreads();
          if (cand) {
            const int n = S.ncand;
            int g = 0;   // thread maxima at or above this one, itself included
            for (int i = 0; i < n; ++i) g += ck[i] >= c0 ? 1 : 0;
            if (g >= K) atomicMax(&S.tkey, c0);
          }
          __syncthreads();
        }
        const uint32_t t = S.tkey;
        thr_v = t ? fkey_value(t) : -INFINITY;   // -inf: every valid element survives
        thr_i = kNoIndex;
      }
    }
  }

  // ---- second pass (K >= 2): reload, now from L2, only what can hold
  // survivors (elements at or before the bound).  Every survivor lies in a
  // thread-slot (one thread's 16 elements of one slot) whose maximum reaches
  // the bound, and a thread's kCand best slot maxima cover all its such slots
  // unless the last of them reaches the bound as well.  So a warp none of whose
  // threads is in that case reloads only its threads' qualifying candidate
  // slots (about K thread-slots per CTA); otherwise it revisits every
  // warp-slot whose recorded maximum reaches the bound, 512 elements each
  // (slots past kTrackSlots have no recorded maximum and are always
  // reloaded).
  if (K >= 2) {
    // this lane's 16 elements of slot j, in the ring's layout
    auto load_slot = [&](int j, float (&x)[kPer]) {
      const int off = j * kSlotElems;
      int nel = n_el - off;
      if (nel > kSlotElems) nel = kSlotElems;
      const float* g0 = src + e_begin + off;
#pragma unroll
      for (int q = 0; q < kVec; ++q) {
        const int e = (q * kThreads + tid) * 4;
        float4 f = make_float4(-INFINITY, -INFINITY, -INFINITY, -INFINITY);
        if (e + 4 <= nel) {
          f = __ldcg(reinterpret_cast<const float4*>(g0 + e));
        } else if (e < nel) {
          const int avail = nel - e;
          f.x = __ldcg(g0 + e);
          if (avail > 1) f.y = __ldcg(g0 + e + 1);
          if (avail > 2) f.z = __ldcg(g0 + e + 2);
        }
        x[4 * q + 0] = f.x;
        x[4 * q + 1] = f.y;
        x[4 * q + 2] = f.z;
        x[4 * q + 3] = f.w;
      }
    };
    // add this lane's survivors among x (tokens from tbase) to the warp buffer
    auto absorb = [&](float (&x)[kPer], int tbase) {
      float lm;
      {
        float m4[4];
#pragma unroll
        for (int a = 0; a < 4; ++a) m4[a] = fmaxf(fmaxf(x[a], x[4 + a]), fmaxf(x[8 + a], x[12 + a]));
        lm = fmaxf(fmaxf(m4[0], m4[1]), fmaxf(m4[2], m4[3]));
      }
      if (__any_sync(0xffffffffu, lm >= thr_v)) {
        auto survives = [&](int e) {
          const float xv = x[e];
          const int xi = tbase + (e >> 2) * kTile + (e & 3);
          return (xv != -INFINITY) & ((xv > thr_v) | ((xv == thr_v) & (xi <= thr_i)));
        };
        uint32_t pm = 0;
        if (lm >= thr_v) {
#pragma unroll
          for (int e = 0; e < kPer; ++e) pm |= survives(e) ? (1u << e) : 0u;
        }
        // common case: no lane holds more than one survivor.  A lone survivor
        // has the lane maximum's value (any survivor of a lane whose maximum
        // is above the bound is that maximum; at the bound all share its
        // value); its token follows from its bit; positions from a ballot.
        const unsigned one = __ballot_sync(0xffffffffu, pm != 0u);
        if (__all_sync(0xffffffffu, (pm & (pm - 1u)) == 0u) && wn + __popc(one) <= kWarpCap) {
          if (pm) {
            const int e = __ffs(pm) - 1;
            wb[wn + __popc(one & ((1u << lane) - 1u))] = mkkey(lm, tbase + (e >> 2) * kTile + (e & 3));
          }
          wn += __popc(one);
          __syncwarp();
          pm = 0u;
        }
        while (__any_sync(0xffffffffu, pm != 0u)) {
          const int cntp = __popc(pm);
          int incl = cntp;
#pragma unroll
          for (int o = 1; o < 32; o <<= 1) {
            const int y = __shfl_up_sync(0xffffffffu, incl, o);
            if (lane >= o) incl += y;
          }
          const int total = __shfl_sync(0xffffffffu, incl, 31);
          const bool fits = wn + total <= kWarpCap;
          // append (all, or the first kWarpCap - wn in lane order)
          int take = cntp;
          if (!fits) take = max(0, min(cntp, kWarpCap - wn - (incl - cntp)));
          int pos = wn + incl - cntp;
          if (take) {
            int taken = 0;
#pragma unroll
            for (int e = 0; e < kPer; ++e)   // static indices keep x in registers
              if (((pm >> e) & 1u) && taken < take) {
                wb[pos++] = mkkey(x[e], tbase + (e >> 2) * kTile + (e & 3));
                pm &= ~(1u << e);
                ++taken;
              }
          }
          __syncwarp();
          if (fits) {
            wn += total;
            break;
          }
          // buffer full: keep the best K, raise this warp's bound, drop what no
          // longer survives, and go on with the rest of this slot
          wn = warp_select(wb, kWarpCap, K, wb);
          if (wn >= K && before(key_v(wb[K - 1]), key_i(wb[K - 1]), thr_v, thr_i)) {
            thr_v = key_v(wb[K - 1]);
            thr_i = key_i(wb[K - 1]);
            if (lane == 0) atomicMax(&S.cta_bound, wb[K - 1]);
          }
          uint32_t keep = 0;
#pragma unroll
          for (int e = 0; e < kPer; ++e) keep |= survives(e) ? (1u << e) : 0u;
          pm &= keep;
          if (!__any_sync(0xffffffffu, pm != 0u)) break;
        }
      }
      // keep the buffer short: past max(2K, 64) entries cut it to the best K,
      // which raises this warp's bound and, through the shared running bound,
      // every other warp's
      if (wn > (2 * K > 64 ? 2 * K : 64)) {
        wn = warp_select(wb, wn, K, wb);
        if (before(key_v(wb[K - 1]), key_i(wb[K - 1]), thr_v, thr_i)) {
          thr_v = key_v(wb[K - 1]);
          thr_i = key_i(wb[K - 1]);
          if (lane == 0) atomicMax(&S.cta_bound, wb[K - 1]);
        }
      }
    };
    const bool over = cv[kCand - 1] != -INFINITY && cv[kCand - 1] >= thr_v;
    if (!__any_sync(0xffffffffu, over)) {
      auto load_cand = [&](int r, float (&x)[kPer]) {
        if (cv[r] != -INFINITY && cv[r] >= thr_v) {
          load_slot(cs[r], x);
        } else {
#pragma unroll
          for (int e = 0; e < kPer; ++e) x[e] = -INFINITY;
        }
      };
      if constexpr (kOverlapReload) {
        // candidate slot r + 1 is loaded before slot r is absorbed, so that
        // the L2 round trips overlap (two buffers, static indices)
        float xa[kPer], xb[kPer];
        load_cand(0, xa);
#pragma unroll
        for (int r = 0; r < kCand; ++r) {
          const bool q = cv[r] != -INFINITY && cv[r] >= thr_v;
          if (!__any_sync(0xffffffffu, q)) break;
          if (r + 1 < kCand) load_cand(r + 1, (r & 1) ? xa : xb);
          absorb((r & 1) ? xb : xa, e_begin + cs[r] * kSlotElems + tid * 4);
        }
      } else {
#pragma unroll
        for (int r = 0; r < kCand; ++r) {
          const bool q = cv[r] != -INFINITY && cv[r] >= thr_v;
          if (!__any_sync(0xffffffffu, q)) break;
          float x[kPer];
          load_cand(r, x);
          absorb(x, e_begin + cs[r] * kSlotElems + tid * 4);
        }
      }
    } else {
      // the running bound: the best K-th entry any warp has cut to so far
      auto refresh = [&]() {
        const Key cb = *reinterpret_cast<volatile Key*>(&S.cta_bound);
        if (cb != 0ull && before(key_v(cb), key_i(cb), thr_v, thr_i)) {
          thr_v = key_v(cb);
          thr_i = key_i(cb);
        }
      };
      if constexpr (kOverlapReload) {
        // the next warp-slot at or after j whose recorded maximum reaches
        // the bound (n_slots: none), the same in every lane of the warp.  It
        // is loaded before the current slot is absorbed, so the L2 round
        // trips overlap; the bound it was chosen with may since have risen,
        // which only loads a slot whose elements then all fail the bound.
        auto next_slot = [&](int j) {
          refresh();
          for (; j < n_slots; ++j)
            if ((j < kTrackSlots ? S.wsmax[warp][j] : INFINITY) >= thr_v) break;
          return j;
        };
        float xa[kPer], xb[kPer];
        int j = next_slot(0);
        if (j < n_slots) load_slot(j, xa);
        while (j < n_slots) {
          const int j1 = next_slot(j + 1);
          if (j1 < n_slots) load_slot(j1, xb);
          absorb(xa, e_begin + j * kSlotElems + tid * 4);
          if (j1 >= n_slots) break;
          j = next_slot(j1 + 1);
          if (j < n_slots) load_slot(j, xa);
          absorb(xb, e_begin + j1 * kSlotElems + tid * 4);
        }
      } else {
        for (int j = 0; j < n_slots; ++j) {
          refresh();
          const float wmax = j < kTrackSlots ? S.wsmax[warp][j] : INFINITY;
          if (!(wmax >= thr_v)) continue;   // the same in every lane of the warp
          float x[kPer];
          load_slot(j, x);
          absorb(x, e_begin + j * kSlotElems + tid * 4);
        }
      }
    }
  }

  // ================================================================ CTA result
  if (flags & kWantSum) {
    const float wm = warp_max(m_run);
    double sd = (s_run > 0.f)
                    ? static_cast<double>(s_run) * static_cast<double>(ex2((m_run - wm) * c2))
                    : 0.0;
    sd = warp_sum_d(sd);
    if (lane == 0) {
      S.red_f[warp] = wm;
      S.red_d[warp] = sd;
    }
  }
  if (K == 1) {
    const Key b = warp_max_key(mkkey(best_v, best_i));
    if (lane == 0) S.red_best[warp] = b;
  }
  if (K >= 2) {
    const int kept = warp_select(wb, wn, K, S.wlist + warp * K);
    if (lane == 0) S.lcnt[warp] = kept;
  }
  __syncthreads();
  if (K >= 2) {
    if (warp == 0) prune_lists(S.wlist, S.lcnt, kWarps, K, K);
    __syncthreads();
  }
  cluster_wait();   // (relaxed arrival above) every CTA of the cluster runs
  const int KL = K > 1 ? K : 1;   // list stride
  if (K >= 2) {
    const uint32_t dst = map_rank0(S.clist + rank * KL);
    for (int e = tid; e < kWarps * K; e += kThreads) {
      const int w = e / K, c = e - w * K;
      if (c >= S.lcnt[w]) continue;
      const Key ent = S.wlist[e];
      const int r = union_rank(S.wlist, S.lcnt, kWarps, K, w, c);
      if (r < K) st_cluster(dst + 8u * static_cast<uint32_t>(r), ent);
    }
  }
  if (tid < 32) {
    float M = -INFINITY;
    double Ssum = 0.0;
    if (flags & kWantSum) {
      const float fm = lane < kWarps ? S.red_f[lane] : -INFINITY;
      M = warp_max(fm);
      double d = 0.0;
      if (lane < kWarps && S.red_d[lane] > 0.0)
        d = S.red_d[lane] * static_cast<double>(ex2((S.red_f[lane] - M) * c2));
      Ssum = warp_sum_d(d);
    }
    int cnt = 0;
    if (K == 1) {
      const Key b = warp_max_key(lane < kWarps ? S.red_best[lane] : 0ull);
      if (lane == 0) st_cluster(map_rank0(S.clist + rank), b);
      cnt = 1;
    } else if (K >= 2) {
      int t = lane < kWarps ? S.lcnt[lane] : 0;
      t = warp_sum_i(t);
      cnt = t < K ? t : K;
    }
    if (lane == 0) {
      st_cluster(map_rank0(&S.cmax[rank]), M);
      st_cluster(map_rank0(&S.csum[rank]), Ssum);
      st_cluster(map_rank0(&S.ccnt[rank]), cnt);
    }
  }
  __syncwarp();
  cluster_arrive_release();
  cluster_wait();   // the CTA lists have landed in the rank-0 CTA
  if (!cx.leader) return cx;

  // ================================================================ row result (rank 0)
  char* rec = Jb.rec;
  if (K >= 2) {
    if (warp == 0) prune_lists(S.clist, S.ccnt, PC, K, K);
    __syncthreads();
    for (int e = tid; e < PC * K; e += kThreads) {
      const int p = e / K, c = e - p * K;
      if (c >= S.ccnt[p]) continue;
      const Key ent = S.clist[e];
      const int r = union_rank(S.clist, S.ccnt, PC, K, p, c);
      if (r < K) {
        S.rlist[r] = ent;
        rec_val(rec)[r] = key_v(ent);
        rec_idx(rec, Jb.rec_k)[r] = key_i(ent);
      }
    }
  }
  if (tid < 32) {
    float M = -INFINITY;
    double Ssum = 0.0;
    int cnt = 0;
    if (flags & kWantSum) {
      const float fm = lane < PC ? S.cmax[lane] : -INFINITY;
      M = warp_max(fm);
      double d = 0.0;
      if (lane < PC && S.csum[lane] > 0.0)
        d = S.csum[lane] * static_cast<double>(ex2((S.cmax[lane] - M) * c2));
      Ssum = warp_sum_d(d);
    }
    if (K == 1) {
      const Key b = warp_max_key(lane < PC ? S.clist[lane] : 0ull);
      if (!(flags & kWantSum)) M = key_v(b);
      if (lane == 0) {
        S.rlist[0] = b;
        rec_val(rec)[0] = key_v(b);
        rec_idx(rec, Jb.rec_k)[0] = key_i(b);
      }
      cnt = 1;
    } else if (K >= 2) {
      int t = lane < PC ? S.ccnt[lane] : 0;
      t = warp_sum_i(t);
      cnt = t < K ? t : K;
      if (!(flags & kWantSum))   // row max = best of the CTA heads
        M = key_v(warp_max_key((lane < PC && S.ccnt[lane] > 0) ? S.clist[lane * K] : 0ull));
    }
    if (lane == 0) {
      RecHead h;
      h.sum = Ssum;
      h.max = M;
      h.count = cnt;
      *reinterpret_cast<RecHead*>(rec) = h;
      S.rsum = Ssum;
      S.rmax = M;
      S.rcount = cnt;
    }
  }
  __syncthreads();
  return cx;
}

// The row's leader arrives on its item's counter after the caller's per-row
// step; true for the one CTA whose row arrives last (it then runs the item's
// final step and may read every row result of the item).  One
// acquire-release atomic at GPU scope orders both ways: the CTA barrier before
// it puts every thread's row writes before the release (cumulative), and the
// barrier after it puts the acquire before every thread's later reads.
static __device__ __forceinline__ bool item_arrive(const RowStream& P, StreamSmem& S, int item) {
  __syncthreads();
  if (threadIdx.x == 0) {
    uint32_t old;
    asm volatile("atom.acq_rel.gpu.global.add.u32 %0, [%1], 1;"
                 : "=r"(old)
                 : "l"(P.item_cnt + item)
                 : "memory");
    const bool last = old == static_cast<uint32_t>(P.rows_per_item - 1);
    if (last) P.item_cnt[item] = 0u;
    S.flag = last ? 1 : 0;
  }
  __syncthreads();
  return S.flag != 0;
}

}  // namespace eagle
