// One HBM pass over rows of fp32 logits, shared by the tree build (draft
// rows) and the verify walk (target rows).
//
// Work split: the rows of all items are cut into 1024-element tiles and the
// grid (a whole number of CTAs per SM) takes equal contiguous tile ranges.
// A CTA streams its range through a two-slot shared-memory ring filled by
// 1-D bulk (TMA) copies; a slot is released through an mbarrier that every
// thread arrives on once it holds its 32 elements in registers, so no CTA
// barrier is taken per slot.  Per row segment the CTA computes:
//   * max and sum of 2^((x - max) * c) per thread (fp32 ex2), combined per
//     segment with fp32 factors and fp64 accumulation,
//   * the exact top-K (value desc, token id asc), K <= 64: the survivor
//     threshold is the K-th best of the top-2 of every thread in the
//     segment's first slot (distinct elements, so a lower bound of the K-th
//     value of the segment); each warp keeps the elements >= threshold in a
//     private buffer (sorted and cut to its best K when full, which raises
//     its threshold); at the end of the segment every warp sorts its buffer
//     and the CTA merges the eight sorted lists by binary-search ranks,
//   * optionally per-tile (max, sum) of every warp for inverse-CDF sampling.
// Each segment is written as a piece record.  The CTA whose piece arrives
// last for a row merges the row's pieces into a row record; the CTA whose
// row arrives last for an item runs the item's final step (tree assembly or
// acceptance walk).  Arrival counters live in the workspace, start at zero
// and are reset by their last user; nothing ever spins on them.
#pragma once

#include "eagle_common.cuh"

namespace eagle {

constexpr int kTile = 1024;                 // tokens per tile
constexpr int kSubTiles = 8;                // tiles per ring slot
constexpr int kSub = kTile * kSubTiles;     // 8192 floats = 32 KB per slot
constexpr int kThreads = 256;
constexpr int kWarps = kThreads / 32;
constexpr int kVec = kSub / kThreads / 4;   // float4 per thread per slot (8)
constexpr int kWarpCap = 128;               // survivors per warp (> K, so merges progress)
constexpr int kKMax = EAGLE_MAX_TOP_K;
constexpr int kMaxItems = EAGLE_MAX_BATCH;
constexpr int kMaxPieces = 16;              // CTAs sharing one row (host keeps it)
constexpr float kLog2e = 1.4426950408889634f;

enum : int { kWantSum = 1, kWantTileSums = 2 };

struct RowStream {
  const float* base[kMaxItems];  // row 0 of each item
  float exp_scale[kMaxItems];    // factor on (x - max) inside exp: 1/T (1 for draft)
  int16_t topk[kMaxItems];       // K per item (0 = none, 1 = argmax)
  int16_t flags[kMaxItems];      // kWantSum | kWantTileSums
  int64_t row_stride;
  int64_t total_tiles;
  int n_items, rows_per_item, vocab, tiles_per_row;
  int grid, max_pieces, rec_k;
  int32_t* err;
  uint32_t* row_cnt;             // [n_items * rows_per_item]
  uint32_t* item_cnt;            // [n_items]
  char* pieces;                  // [rows][max_pieces] piece records
  char* rows;                    // [rows] row records
  float2* tile_sums;             // [rows][tiles_per_row][kWarps] or null
};

// Piece record (one row segment of one CTA) and row record share a layout:
//   double sum; float max; int count; float val[rec_k]; int idx[rec_k]
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

struct StreamSmem {
  int n_done_items;                   // items whose final step this CTA runs
  int done_items[kMaxItems + 31];     // (padded so that the ring starts 16-byte aligned)
  float buf[2][kSub];                 // ring; from here on reused by the item final step
  float wv[kWarps][kWarpCap];         // warp survivor buffers
  int wi[kWarps][kWarpCap];
  float mv[kMaxPieces * kKMax];       // merge staging (piece lists / warp lists)
  int mi[kMaxPieces * kKMax];
  int lcnt[kWarps];                   // entries of each warp's sorted list
  float thr;                          // CTA survivor threshold of the segment
  float list_v[kKMax];
  int list_i[kKMax];
  float red_f[kWarps];
  double red_d[kWarps];
  int wcnt[kWarps];
  uint64_t full[2];
  uint64_t empty[2];
  int is_last;
  int cnt[kMaxPieces];
  float pmax[kMaxPieces];
  double psum[kMaxPieces];
};


__device__ __forceinline__ int64_t tile_owner(int64_t t, int64_t T, int G) {
  return ((t + 1) * G - 1) / T;
}

__device__ __forceinline__ int64_t next_slot(int64_t t, int64_t t_end, int TR) {
  const int64_t row_end = (t / TR + 1) * TR;
  int64_t n = row_end - t;
  if (n > kSubTiles) n = kSubTiles;
  const int64_t e = t + n;
  return e < t_end ? e : t_end;
}

// Issue the bulk copy of the slot starting at tile t into ring buffer b.
__device__ __forceinline__ void issue_slot(const RowStream& P, StreamSmem& S, int64_t t,
                                           int64_t t_end, int b) {
  const int64_t row = t / P.tiles_per_row;
  const int tir = static_cast<int>(t - row * P.tiles_per_row);
  const int ntiles = static_cast<int>(next_slot(t, t_end, P.tiles_per_row) - t);
  int nel = ntiles * kTile;
  const int rem = P.vocab - tir * kTile;
  if (nel > rem) nel = rem;
  const uint32_t bytes = static_cast<uint32_t>(nel & ~3) * 4u;
  const int item = static_cast<int>(row / P.rows_per_item);
  const int lrow = static_cast<int>(row - static_cast<int64_t>(item) * P.rows_per_item);
  const float* src = P.base[item] + lrow * P.row_stride + static_cast<int64_t>(tir) * kTile;
  mbar_arrive_expect_tx(&S.full[b], bytes);
  if (bytes) bulk_copy_g2s(S.buf[b], src, bytes, &S.full[b]);
}

// best k of n (v, i) entries (distinct i) from smem, sorted into out; all threads.
__device__ __forceinline__ void rank_select(const float* v, const int* id, int n, int k,
                                            float* out_v, int* out_i) {
  for (int a = threadIdx.x; a < n; a += blockDim.x) {
    const float va = v[a];
    const int ia = id[a];
    int rank = 0;
    for (int b = 0; b < n; ++b) rank += before(v[b], id[b], va, ia) ? 1 : 0;
    if (rank < k) {
      out_v[rank] = va;
      out_i[rank] = ia;
    }
  }
}

// Warp bitonic sort of 32E (v, i) pairs held E per lane (position p = lane
// + 32 r) into (value desc, index asc) order: position 0 holds the best.
template <int E>
__device__ __forceinline__ void warp_sort(float (&v)[E], int (&id)[E]) {
  const int lane = threadIdx.x & 31;
#pragma unroll 1
  for (int k = 2; k <= 32 * E; k <<= 1) {
#pragma unroll 1
    for (int j = k >> 1; j > 0; j >>= 1) {
      if (j >= 32) {  // partner is another register of the same lane
        auto cx = [&](float& va, int& ia, float& vb, int& ib, int p) {   // (a lower, b upper)
          const bool best_first = (p & k) == 0;
          const bool b_first = before(vb, ib, va, ia);
          const bool swap = best_first == b_first;
          const float tv = swap ? vb : va, tw = swap ? va : vb;
          const int ti = swap ? ib : ia, tj = swap ? ia : ib;
          va = tv; vb = tw; ia = ti; ib = tj;
        };
        if constexpr (E == 2) {
          cx(v[0], id[0], v[1], id[1], lane);
        } else if constexpr (E == 4) {
          if (j == 64) {
            cx(v[0], id[0], v[2], id[2], lane);
            cx(v[1], id[1], v[3], id[3], lane + 32);
          } else {
            cx(v[0], id[0], v[1], id[1], lane);
            cx(v[2], id[2], v[3], id[3], lane + 64);
          }
        }
      } else {
#pragma unroll
        for (int r = 0; r < E; ++r) {
          const int p = lane + 32 * r;
          const float ov = __shfl_xor_sync(0xffffffffu, v[r], j);
          const int oi = __shfl_xor_sync(0xffffffffu, id[r], j);
          const bool lower = (p & j) == 0;
          const bool best_first = (p & k) == 0;   // direction of this block
          const bool other_first = before(ov, oi, v[r], id[r]);
          // keep the better one at (lower == best_first), the worse one otherwise
          const bool take = (lower == best_first) == other_first;
          v[r] = take ? ov : v[r];
          id[r] = take ? oi : id[r];
        }
      }
    }
  }
}

__device__ __forceinline__ void warp_sort64(float (&v)[2], int (&id)[2]) { warp_sort<2>(v, id); }

// Sort a warp's buffer (n <= kWarpCap entries) best first, in place; returns n.
static __device__ __noinline__ int warp_sort_buffer(float* bv, int* bi, int n) {
  const int lane = threadIdx.x & 31;
  constexpr int E = kWarpCap / 32;
  float v[E];
  int id[E];
#pragma unroll
  for (int r = 0; r < E; ++r) {
    const int a = lane + 32 * r;
    v[r] = a < n ? bv[a] : -INFINITY;
    id[r] = a < n ? bi[a] : 0x7fffffff;
  }
  warp_sort<E>(v, id);
  __syncwarp();
#pragma unroll
  for (int r = 0; r < E; ++r) {
    const int a = lane + 32 * r;
    if (a < n) {
      bv[a] = v[r];
      bi[a] = id[r];
    }
  }
  __syncwarp();
  return n;
}

// Rank of entry (v, id) of sorted list `self` among the union of `nl` sorted
// lists stored at stride `stride` (counts in `cnt`): its position plus the
// number of entries of every other list that come before it.
static __device__ __noinline__ int merged_rank(const float* lv, const int* li, const int* cnt, int nl,
                                               int stride, int self, int pos, float v, int id) {
  int rank = pos;
  for (int q = 0; q < nl; ++q) {
    // entries of list q before (v, id): fixed 7 halving steps (lists <= 64)
    int lo = 0, hi = cnt[q];
#pragma unroll
    for (int step = 0; step < 7; ++step) {
      const int mid = (lo + hi) >> 1;
      const bool go = (lo < hi) & before(lv[q * stride + mid], li[q * stride + mid], v, id);
      const bool stay = (lo < hi) & !go;
      lo = go ? mid + 1 : lo;
      hi = stay ? mid : hi;
    }
    rank += (q == self) ? 0 : lo;
  }
  return rank;
}

// K-th best of every thread's top-2 (sv, si) over the CTA: each warp sorts
// its 64 samples, the CTA ranks the warps' best K by binary search.  Every
// thread of the CTA calls this (two CTA barriers).
static __device__ __noinline__ float cta_threshold(StreamSmem& S, float (&sv)[2], int (&si)[2],
                                                   int K) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  warp_sort64(sv, si);
  const int keep = K < 64 ? K : 64;
#pragma unroll
  for (int r = 0; r < 2; ++r) {
    const int a = lane + 32 * r;
    if (a < keep) {
      S.mv[warp * kKMax + a] = sv[r];
      S.mi[warp * kKMax + a] = si[r];
    }
  }
  if (lane == 0) {
    S.lcnt[warp] = keep;
    S.wcnt[warp] = 0;
  }
  __syncthreads();
  for (int e = threadIdx.x; e < kWarps * keep; e += kThreads) {
    const int w = e / keep, c = e - w * keep;
    const float v = S.mv[w * kKMax + c];
    if (merged_rank(S.mv, S.mi, S.lcnt, kWarps, kKMax, w, c, v, S.mi[w * kKMax + c]) == K - 1)
      S.thr = v;   // -inf when the slot holds fewer than K elements
  }
  __syncthreads();
  return S.thr;
}

// ------------------------------------------------------------ row finalize
// Merge the pieces of `row` into its row record.  Piece lists are sorted, so
// an entry's rank is its position plus, for every other piece, the number of
// that piece's entries that come before it (binary search).
static __device__ __noinline__ void finalize_row(const RowStream& P, StreamSmem& S, int64_t row) {
  const int TR = P.tiles_per_row;
  const int64_t T = P.total_tiles;
  const int item = static_cast<int>(row / P.rows_per_item);
  const int K = P.topk[item];
  const int64_t p0 = tile_owner(row * TR, T, P.grid);
  const int np = static_cast<int>(tile_owner(row * TR + TR - 1, T, P.grid) - p0 + 1);
  const int rb = rec_bytes(P.rec_k);
  char* prow = P.pieces + (row * P.max_pieces) * rb;
  for (int p = threadIdx.x; p < np; p += blockDim.x) {
    const volatile RecHead* h = reinterpret_cast<volatile RecHead*>(prow + p * rb);
    S.cnt[p] = h->count;
    S.pmax[p] = h->max;
    S.psum[p] = h->sum;
  }
  __syncthreads();
  for (int e = threadIdx.x; e < np * K; e += blockDim.x) {
    const int p = e / K, c = e - p * K;
    char* rec = prow + p * rb;
    if (c < S.cnt[p]) {
      S.mv[e] = __ldcg(rec_val(rec) + c);
      S.mi[e] = __ldcg(rec_idx(rec, P.rec_k) + c);
    }
  }
  __syncthreads();
  char* out = P.rows + row * rb;
  for (int e = threadIdx.x; e < np * K; e += blockDim.x) {
    const int p = e / K, c = e - p * K;
    if (c >= S.cnt[p]) continue;
    const int rank = merged_rank(S.mv, S.mi, S.cnt, np, K, p, c, S.mv[e], S.mi[e]);
    if (rank < K) {
      rec_val(out)[rank] = S.mv[e];
      rec_idx(out, P.rec_k)[rank] = S.mi[e];
    }
  }
  if (threadIdx.x < 32) {
    const float c2 = P.exp_scale[item] * kLog2e;
    float m = -INFINITY;
    int total = 0;
    for (int p = threadIdx.x; p < np; p += 32) {
      m = fmaxf(m, S.pmax[p]);
      total += S.cnt[p];
    }
    m = warp_max(m);
    total = warp_sum_i(total);
    double s = 0.0;
    for (int p = threadIdx.x; p < np; p += 32)
      if (S.psum[p] > 0.0) s += S.psum[p] * static_cast<double>(ex2((S.pmax[p] - m) * c2));
    s = warp_sum_d(s);
    if (threadIdx.x == 0) {
      RecHead h;
      h.sum = s;
      h.max = m;
      h.count = total < K ? total : K;
      *reinterpret_cast<RecHead*>(out) = h;
    }
  }
  __syncthreads();
}

// ------------------------------------------------------------ the stream
// Processes this CTA's tile range; returns with S.done_items listing the
// items whose last row this CTA finalized (their final step is the caller's).
static __device__ void run_stream(const RowStream& P, StreamSmem& S) {
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int TR = P.tiles_per_row;
  const int64_t T = P.total_tiles;
  const int64_t t_begin = static_cast<int64_t>(blockIdx.x) * T / P.grid;
  const int64_t t_end = static_cast<int64_t>(blockIdx.x + 1) * T / P.grid;

  if (tid == 0) {
    for (int b = 0; b < 2; ++b) {
      mbar_init(&S.full[b], 1);
      mbar_init(&S.empty[b], kWarps);
    }
    fence_barrier_init();
    S.n_done_items = 0;
  }
  if (lane == 0) S.wcnt[warp] = 0;
  __syncthreads();

  int64_t pf = t_begin;  // producer cursor (thread 0)
  if (tid == 0) {
    for (int b = 0; b < 2 && pf < t_end; ++b) {
      issue_slot(P, S, pf, t_end, b);
      pf = next_slot(pf, t_end, TR);
    }
  }

  float m_run = -INFINITY, s_run = 0.f;       // per-thread running max / sum
  float best_v = -INFINITY;                    // per-thread argmax (K == 1)
  int best_i = 0x7fffffff;
  float thr_v = INFINITY;                      // warp survivor threshold (K >= 2):
  int thr_i = 0x7fffffff;                      // survivors come at or before (thr_v, thr_i)
  int64_t cur = t_begin;
  for (int j = 0; cur < t_end; ++j) {
    const int b = j & 1;
    const int64_t nxt = next_slot(cur, t_end, TR);
    const int64_t row = cur / TR;
    const int tir = static_cast<int>(cur - row * TR);
    int nel = static_cast<int>(nxt - cur) * kTile;
    const int rem = P.vocab - tir * kTile;
    if (nel > rem) nel = rem;
    const int item = static_cast<int>(row / P.rows_per_item);
    const int K = P.topk[item];
    const int flags = P.flags[item];
    const float c2 = P.exp_scale[item] * kLog2e;

    if (!mbar_wait(&S.full[b], (j >> 1) & 1)) {
      record_error(P.err, kDevTimeout, 1);
      mbar_wait(&S.full[b], (j >> 1) & 1);  // give an in-flight copy a last chance to land
    }
    float x[kVec * 4];
    const int tok0 = tir * kTile;
    const int n4 = nel & ~3;  // elements delivered by the bulk copy
#pragma unroll
    for (int q = 0; q < kVec; ++q) {
      const int e = (q * kThreads + tid) * 4;
      float4 f = make_float4(-INFINITY, -INFINITY, -INFINITY, -INFINITY);
      if (e + 4 <= n4) {
        f = *reinterpret_cast<const float4*>(&S.buf[b][e]);
      } else if (e < nel) {  // ragged row tail (vocab % 4 != 0): read it directly
        const int lrow = static_cast<int>(row - static_cast<int64_t>(item) * P.rows_per_item);
        const float* g = P.base[item] + lrow * P.row_stride + tok0 + e;
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
    if (tid == 0 && pf < t_end) {  // refill this slot once every warp has read it
      if (!mbar_wait(&S.empty[b], (j >> 1) & 1)) record_error(P.err, kDevTimeout, 2);
      fence_proxy_async_smem();
      issue_slot(P, S, pf, t_end, b);
      pf = next_slot(pf, t_end, TR);
    }

    const bool seg_first = (cur == t_begin) || (tir == 0);
    const bool seg_last = (nxt == t_end) || (nxt % TR == 0);
    const int tbase = tok0 + tid * 4;   // token of element (q, c) = tbase + q * 1024 + c

    float lm;
    {
      float m4[4];
#pragma unroll
      for (int a = 0; a < 4; ++a) m4[a] = fmaxf(fmaxf(x[a], x[4 + a]), fmaxf(x[8 + a], x[12 + a]));
#pragma unroll
      for (int a = 0; a < 4; ++a)
        m4[a] = fmaxf(m4[a], fmaxf(fmaxf(x[16 + a], x[20 + a]), fmaxf(x[24 + a], x[28 + a])));
      lm = fmaxf(fmaxf(m4[0], m4[1]), fmaxf(m4[2], m4[3]));
    }

    // ---- sum of exp (invalid elements are -inf and contribute 0)
    if (flags & kWantSum) {
      const float mn = fmaxf(m_run, lm);
      if (mn != -INFINITY) {
        s_run *= ex2((m_run - mn) * c2);
        const float off = mn * c2;
        float acc[8];
#pragma unroll
        for (int a = 0; a < 8; ++a) acc[a] = ex2(fmaf(x[a], c2, -off));
#pragma unroll
        for (int e = 8; e < kVec * 4; ++e) acc[e & 7] += ex2(fmaf(x[e], c2, -off));
        s_run += ((acc[0] + acc[1]) + (acc[2] + acc[3])) + ((acc[4] + acc[5]) + (acc[6] + acc[7]));
        m_run = mn;
      }
    }

    // ---- per-tile (max, sum) of this warp's 128 elements of every tile
    if (flags & kWantTileSums) {
      const int ntl = static_cast<int>(nxt - cur);
#pragma unroll
      for (int q = 0; q < kVec; ++q) {
        float tm = fmaxf(fmaxf(x[4 * q], x[4 * q + 1]), fmaxf(x[4 * q + 2], x[4 * q + 3]));
        tm = warp_max(tm);
        float ts = 0.f;
        if (tm != -INFINITY) {
#pragma unroll
          for (int c = 0; c < 4; ++c) ts += ex2((x[4 * q + c] - tm) * c2);
        }
#pragma unroll
        for (int o = 16; o; o >>= 1) ts += __shfl_xor_sync(0xffffffffu, ts, o);
        if (lane == 0 && q < ntl)
          P.tile_sums[(row * TR + tir + q) * kWarps + warp] = make_float2(tm, ts);
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

    // ---- top-K survivors, K >= 2
    if (K >= 2) {
      float* bv = S.wv[warp];
      int* bi = S.wi[warp];
      if (seg_first) {
        // threshold: K-th best of the threads' top-2 over the whole CTA
        float sv[2] = {-INFINITY, -INFINITY};
        int si[2] = {0x7fffffff, 0x7fffffff};
#pragma unroll
        for (int q = 0; q < kVec; ++q)
#pragma unroll
          for (int c = 0; c < 4; ++c) {
            const float xv = x[4 * q + c];
            const int xi = tbase + q * kTile + c;
            const bool gt1 = xv > sv[1], gt0 = xv > sv[0];
            sv[1] = gt0 ? sv[0] : (gt1 ? xv : sv[1]);
            si[1] = gt0 ? si[0] : (gt1 ? xi : si[1]);
            sv[0] = gt0 ? xv : sv[0];
            si[0] = gt0 ? xi : si[0];
          }
        thr_v = cta_threshold(S, sv, si, K);
        thr_i = 0x7fffffff;
      }
      if (__any_sync(0xffffffffu, lm >= thr_v)) {
        auto survives = [&](int e) {
          const float xv = x[e];
          const int xi = tbase + (e >> 2) * kTile + (e & 3);
          return (xv != -INFINITY) & ((xv > thr_v) | ((xv == thr_v) & (xi <= thr_i)));
        };
        uint32_t pm = 0;
#pragma unroll
        for (int e = 0; e < kVec * 4; ++e) pm |= survives(e) ? (1u << e) : 0u;
        for (;;) {
          const int cntp = __popc(pm);
          int incl = cntp;
#pragma unroll
          for (int o = 1; o < 32; o <<= 1) {
            const int y = __shfl_up_sync(0xffffffffu, incl, o);
            if (lane >= o) incl += y;
          }
          const int total = __shfl_sync(0xffffffffu, incl, 31);
          const int n = S.wcnt[warp];
          const bool fits = n + total <= kWarpCap;
          // append (all, or the first kWarpCap - n in lane order)
          int take = cntp;
          if (!fits) take = max(0, min(cntp, kWarpCap - n - (incl - cntp)));
          int pos = n + incl - cntp;
          if (take) {
            int taken = 0;
#pragma unroll
            for (int e = 0; e < kVec * 4; ++e)   // static indices keep x in registers
              if (((pm >> e) & 1u) && taken < take) {
                bv[pos++] = x[e];
                bi[pos - 1] = tbase + (e >> 2) * kTile + (e & 3);
                pm &= ~(1u << e);
                ++taken;
              }
          }
          __syncwarp();
          if (fits) {
            if (lane == 0) S.wcnt[warp] = n + total;
            __syncwarp();
            break;
          }
          // buffer full: keep the best K, raise this warp's bar, drop what no
          // longer survives, and go on with the rest of this slot
          const int kept = min(warp_sort_buffer(bv, bi, kWarpCap), K);
          if (kept >= K && before(bv[K - 1], bi[K - 1], thr_v, thr_i)) {
            thr_v = bv[K - 1];
            thr_i = bi[K - 1];
          }
          uint32_t keep = 0;
#pragma unroll
          for (int e = 0; e < kVec * 4; ++e) keep |= survives(e) ? (1u << e) : 0u;
          pm &= keep;
          if (lane == 0) S.wcnt[warp] = kept;
          __syncwarp();
          if (!__any_sync(0xffffffffu, pm != 0u)) break;
        }
      }
    }

    // ---- end of a row segment: piece record, arrival counters, finalize
    if (seg_last) {
      float M = -INFINITY;
      double Ssum = 0.0;
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
        float v = best_v;
        int i = best_i;
        warp_best(v, i);
        if (lane == 0) {
          S.list_v[warp] = v;   // staged per warp
          S.list_i[warp] = i;
        }
      }
      __syncthreads();
      if (tid < 32) {
        if (flags & kWantSum) {
          const float fm = lane < kWarps ? S.red_f[lane] : -INFINITY;
          M = warp_max(fm);
          double d = 0.0;
          if (lane < kWarps && S.red_d[lane] > 0.0)
            d = S.red_d[lane] * static_cast<double>(ex2((S.red_f[lane] - M) * c2));
          Ssum = warp_sum_d(d);
        }
        if (K == 1) {
          float v = lane < kWarps ? S.list_v[lane] : -INFINITY;
          int i = lane < kWarps ? S.list_i[lane] : 0x7fffffff;
          warp_best(v, i);
          if (!(flags & kWantSum)) M = v;
          if (lane == 0) {
            S.mv[0] = v;
            S.mi[0] = i;
          }
        }
      }
      int nl = 0;
      if (K >= 2) {
        // every warp sorts its survivors; the CTA merges the sorted lists
        {
          float* bv = S.wv[warp];
          int* bi = S.wi[warp];
          const int n = warp_sort_buffer(bv, bi, S.wcnt[warp]);
          const int keep = n < K ? n : K;
          for (int a = lane; a < keep; a += 32) {
            S.mv[warp * kKMax + a] = bv[a];
            S.mi[warp * kKMax + a] = bi[a];
          }
          if (lane == 0) S.lcnt[warp] = keep;
        }
        __syncthreads();
        int total = 0;
        for (int w = 0; w < kWarps; ++w) total += S.lcnt[w];
        for (int e = tid; e < kWarps * kKMax; e += kThreads) {
          const int w = e / kKMax, c = e - w * kKMax;
          if (c >= S.lcnt[w]) continue;
          const float v = S.mv[e];
          const int id = S.mi[e];
          const int rank = merged_rank(S.mv, S.mi, S.lcnt, kWarps, kKMax, w, c, v, id);
          if (rank < K) {
            S.list_v[rank] = v;
            S.list_i[rank] = id;
          }
        }
        nl = total < K ? total : K;
        __syncthreads();
        for (int a = tid; a < nl; a += kThreads) {
          S.mv[a] = S.list_v[a];
          S.mi[a] = S.list_i[a];
        }
        if (!(flags & kWantSum) && tid == 0) M = S.list_v[0];
      } else if (K == 1) {
        nl = 1;
      }
      __syncthreads();
      const int64_t piece = static_cast<int64_t>(blockIdx.x) - tile_owner(row * TR, T, P.grid);
      const int rb = rec_bytes(P.rec_k);
      char* rec = P.pieces + (row * P.max_pieces + piece) * rb;
      for (int a = tid; a < nl; a += kThreads) {
        rec_val(rec)[a] = S.mv[a];
        rec_idx(rec, P.rec_k)[a] = S.mi[a];
      }
      if (tid == 0) {
        RecHead h;
        h.sum = Ssum;
        h.max = M;
        h.count = nl;
        *reinterpret_cast<RecHead*>(rec) = h;
      }
      // reset per-segment state
      m_run = -INFINITY;
      s_run = 0.f;
      best_v = -INFINITY;
      best_i = 0x7fffffff;
      thr_v = INFINITY;
      thr_i = 0x7fffffff;
      if (lane == 0) S.wcnt[warp] = 0;
      __threadfence();
      __syncthreads();
      if (tid == 0) {
        const int np = static_cast<int>(tile_owner(row * TR + TR - 1, T, P.grid) -
                                        tile_owner(row * TR, T, P.grid) + 1);
        const uint32_t old = atomicAdd(&P.row_cnt[row], 1u);
        S.is_last = (old == static_cast<uint32_t>(np - 1));
      }
      __syncthreads();
      if (S.is_last) {
        __threadfence();
        finalize_row(P, S, row);
        __threadfence();
        __syncthreads();
        if (tid == 0) {
          P.row_cnt[row] = 0u;
          const uint32_t old = atomicAdd(&P.item_cnt[item], 1u);
          if (old == static_cast<uint32_t>(P.rows_per_item - 1)) {
            P.item_cnt[item] = 0u;
            S.done_items[S.n_done_items++] = item;
          }
        }
        __syncthreads();
      }
    }
    cur = nxt;
  }
  // every issued copy has been consumed above; the ring is free again
  __syncthreads();
  if (S.n_done_items) __threadfence();
}

}  // namespace eagle
