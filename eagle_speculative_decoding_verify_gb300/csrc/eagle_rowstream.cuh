// One HBM pass over rows of fp32 logits, shared by the tree build (draft
// rows) and the verify walk (target rows).
//
// Work split: the rows of all items are cut into 1024-element tiles; the
// grid (a whole number of CTAs per SM) takes equal contiguous tile ranges.
// A CTA streams its range through a two-deep shared-memory ring filled by
// 1-D bulk (TMA) copies and computes, per row segment it owns:
//   * max and sum of exp((x - max) * scale) (fp32 exps, fp64 combine),
//   * the exact top-K (value desc, token id asc), K <= 64, by filtering
//     against a lower bound of the K-th value (the K-th best of a sample of
//     per-lane maxima, then the running list) and ranking the few survivors,
//   * optionally (max, sum) per 1024-token tile for inverse-CDF sampling.
// Each segment is written as a "piece" record.  The CTA whose piece arrives
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
constexpr int kCandCap = 1024;              // survivor buffer (entries)
constexpr int kKMax = EAGLE_MAX_TOP_K;
constexpr int kMaxItems = EAGLE_MAX_BATCH;
constexpr int kMaxPieces = 16;              // CTAs sharing one row (host keeps it)

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
  float2* tile_sums;             // [rows][tiles_per_row] or null
};

// Piece record (one row segment of one CTA) and row record share a layout:
//   double sum; float max; int count; float val[rec_k]; int idx[rec_k]
// For row records of the draft rows `sum` holds the logsumexp instead.
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
  float buf[2][kSub];                 // ring (also reused by the item final step)
  float cand_v[kCandCap];
  int cand_i[kCandCap];
  float list_v[kKMax];
  int list_i[kKMax];
  float tmp_v[kKMax];
  int tmp_i[kKMax];
  float red_f[kWarps][kSubTiles];
  float red_g[kWarps][kSubTiles];
  double red_d[kWarps];
  int red_i[kWarps];
  uint64_t bar[2];
  int cand_n;
  int list_n;
  int overflow;
  int is_last;
  float thr_v;
  int thr_i;
  int n_done_items;
  int done_items[kMaxItems];
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

// Issue the bulk copy of slot starting at tile t into ring buffer b.
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
  mbar_arrive_expect_tx(&S.bar[b], bytes);
  if (bytes) bulk_copy_g2s(S.buf[b], src, bytes, &S.bar[b]);
}

// best k of n (v, i) entries (all distinct i), sorted into out; all threads.
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

// ------------------------------------------------------------ row finalize
// Merge the pieces of `row` into its row record.  Piece lists are sorted, so
// an entry's rank is its position plus, for every other piece, the number of
// that piece's entries that come before it (binary search).
static __device__ void finalize_row(const RowStream& P, StreamSmem& S, int64_t row) {
  const int TR = P.tiles_per_row;
  const int64_t T = P.total_tiles;
  const int item = static_cast<int>(row / P.rows_per_item);
  const int K = P.topk[item];
  const int64_t p0 = tile_owner(row * TR, T, P.grid);
  const int np = static_cast<int>(tile_owner(row * TR + TR - 1, T, P.grid) - p0 + 1);
  const int rb = rec_bytes(P.rec_k);
  char* prow = P.pieces + (row * P.max_pieces) * rb;
  // stage piece lists in the survivor buffer: piece p at offset p * K
  float* pv = S.cand_v;
  int* pi = S.cand_i;
  __shared__ int cnt[kMaxPieces];
  __shared__ float pmax[kMaxPieces];
  __shared__ double psum[kMaxPieces];
  for (int p = threadIdx.x; p < np; p += blockDim.x) {
    char* rec = prow + p * rb;
    const volatile RecHead* h = reinterpret_cast<volatile RecHead*>(rec);
    cnt[p] = h->count;
    pmax[p] = h->max;
    psum[p] = h->sum;
  }
  __syncthreads();
  for (int e = threadIdx.x; e < np * K; e += blockDim.x) {
    const int p = e / K, c = e - p * K;
    char* rec = prow + p * rb;
    if (c < cnt[p]) {
      pv[e] = __ldcg(rec_val(rec) + c);
      pi[e] = __ldcg(rec_idx(rec, P.rec_k) + c);
    }
  }
  __syncthreads();
  char* out = P.rows + row * rb;
  for (int e = threadIdx.x; e < np * K; e += blockDim.x) {
    const int p = e / K, c = e - p * K;
    if (c >= cnt[p]) continue;
    const float v = pv[e];
    const int id = pi[e];
    int rank = c;
    for (int q = 0; q < np; ++q) {
      if (q == p) continue;
      int lo = 0, hi = cnt[q];          // count entries of piece q before (v, id)
      while (lo < hi) {
        const int mid = (lo + hi) >> 1;
        if (before(pv[q * K + mid], pi[q * K + mid], v, id)) lo = mid + 1; else hi = mid;
      }
      rank += lo;
    }
    if (rank < K) {
      rec_val(out)[rank] = v;
      rec_idx(out, P.rec_k)[rank] = id;
    }
  }
  if (threadIdx.x == 0) {
    float m = -INFINITY;
    int total = 0;
    for (int p = 0; p < np; ++p) {
      m = fmaxf(m, pmax[p]);
      total += cnt[p];
    }
    double s = 0.0;
    const double sc = static_cast<double>(P.exp_scale[item]);
    for (int p = 0; p < np; ++p)
      if (psum[p] > 0.0) s += psum[p] * exp((static_cast<double>(pmax[p]) - m) * sc);
    RecHead h;
    h.sum = s;
    h.max = m;
    h.count = total < K ? total : K;
    *reinterpret_cast<RecHead*>(out) = h;
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
    mbar_init(&S.bar[0], 1);
    mbar_init(&S.bar[1], 1);
    fence_barrier_init();
    S.n_done_items = 0;
    S.list_n = 0;
  }
  __syncthreads();

  int64_t pf = t_begin;  // producer cursor (thread 0 only)
  if (tid == 0) {
    for (int b = 0; b < 2 && pf < t_end; ++b) {
      issue_slot(P, S, pf, t_end, b);
      pf = next_slot(pf, t_end, TR);
    }
  }

  float m_run = -INFINITY, s_run = 0.f;       // per-thread running max / sum
  float best_v = -INFINITY;                    // per-thread argmax (K == 1)
  int best_i = 0x7fffffff;
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
    const float c2 = P.exp_scale[item] * 1.4426950408889634f;  // scale * log2(e)

    if (!mbar_wait(&S.bar[b], (j >> 1) & 1)) {
      record_error(P.err, kDevTimeout, 1);
      mbar_wait(&S.bar[b], (j >> 1) & 1);  // give an in-flight copy a last chance to land
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
    __syncthreads();  // ring slot b fully read
    if (tid == 0 && pf < t_end) {
      fence_proxy_async_smem();
      issue_slot(P, S, pf, t_end, b);
      pf = next_slot(pf, t_end, TR);
    }

    const bool seg_first = (cur == t_begin) || (tir == 0);
    const bool seg_last = (nxt == t_end) || (nxt % TR == 0);
    auto valid = [&](int q, int c) { return (q * kThreads + tid) * 4 + c < nel; };
    auto token = [&](int q, int c) { return tok0 + (q * kThreads + tid) * 4 + c; };

    // ---- max / sum of exp
    if (flags & kWantSum) {
      float lm = -INFINITY;
#pragma unroll
      for (int e = 0; e < kVec * 4; ++e) lm = fmaxf(lm, x[e]);
      if (lm > m_run) {
        s_run *= exp2f((m_run - lm) * c2);
        m_run = lm;
      }
      const float off = m_run * c2;
#pragma unroll
      for (int q = 0; q < kVec; ++q)
#pragma unroll
        for (int c = 0; c < 4; ++c)
          if (valid(q, c)) s_run += exp2f(fmaf(x[4 * q + c], c2, -off));
    }

    // ---- per-tile (max, sum) for inverse-CDF sampling
    if (flags & kWantTileSums) {
#pragma unroll
      for (int q = 0; q < kVec; ++q) {
        float tm = -INFINITY, ts = 0.f;
#pragma unroll
        for (int c = 0; c < 4; ++c) tm = fmaxf(tm, x[4 * q + c]);
#pragma unroll
        for (int c = 0; c < 4; ++c)
          if (valid(q, c)) ts += exp2f((x[4 * q + c] - tm) * c2);
#pragma unroll
        for (int o = 16; o; o >>= 1) {
          const float om = __shfl_xor_sync(0xffffffffu, tm, o);
          const float os = __shfl_xor_sync(0xffffffffu, ts, o);
          const float nm = fmaxf(tm, om);
          ts = (nm == -INFINITY) ? 0.f
                                 : ts * exp2f((tm - nm) * c2) + os * exp2f((om - nm) * c2);
          tm = nm;
        }
        if (lane == 0) {
          S.red_f[warp][q] = tm;
          S.red_g[warp][q] = ts;
        }
      }
      __syncthreads();
      const int ntl = static_cast<int>(nxt - cur);
      if (tid < ntl) {
        float tm = -INFINITY;
        for (int w = 0; w < kWarps; ++w) tm = fmaxf(tm, S.red_f[w][tid]);
        float ts = 0.f;
        for (int w = 0; w < kWarps; ++w)
          if (S.red_g[w][tid] > 0.f) ts += S.red_g[w][tid] * exp2f((S.red_f[w][tid] - tm) * c2);
        P.tile_sums[row * TR + tir + tid] = make_float2(tm, ts);
      }
    }

    // ---- argmax
    if (K == 1) {
#pragma unroll
      for (int q = 0; q < kVec; ++q)
#pragma unroll
        for (int c = 0; c < 4; ++c)
          if (valid(q, c) && before(x[4 * q + c], token(q, c), best_v, best_i)) {
            best_v = x[4 * q + c];
            best_i = token(q, c);
          }
    }

    // ---- exact top-K, K >= 2
    if (K >= 2) {
      if (seg_first) {
        // lower bound of the K-th value: K-th best of the per-warp top-qn
        // lane maxima (distinct elements of this row)
        float lv = -INFINITY;
        int li = 0x7fffffff;
#pragma unroll
        for (int q = 0; q < kVec; ++q)
#pragma unroll
          for (int c = 0; c < 4; ++c)
            if (valid(q, c) && before(x[4 * q + c], token(q, c), lv, li)) {
              lv = x[4 * q + c];
              li = token(q, c);
            }
        const int qn = (K + kWarps - 1) / kWarps;
        for (int r = 0; r < qn; ++r) {
          float wv = lv;
          int wi = li;
          warp_best(wv, wi);
          if (lane == 0) {
            S.tmp_v[warp * qn + r] = wv;
            S.tmp_i[warp * qn + r] = wi;
          }
          if (tid == 0 && r == 0) {
            S.thr_v = -INFINITY;  // default: every valid element survives
            S.thr_i = 0x7fffffff;
          }
          if (li == wi) {
            lv = -INFINITY;
            li = 0x7fffffff;
          }
        }
        __syncthreads();
        const int ns = qn * kWarps;
        if (tid < ns) {
          const float va = S.tmp_v[tid];
          const int ia = S.tmp_i[tid];
          int rank = 0;
          for (int b2 = 0; b2 < ns; ++b2) rank += before(S.tmp_v[b2], S.tmp_i[b2], va, ia) ? 1 : 0;
          if (rank == K - 1) {
            S.thr_v = va;
            S.thr_i = ia;
          }
        }
        if (tid == 0) S.list_n = 0;
        __syncthreads();
      } else if (tid == 0) {
        if (S.list_n >= K) {
          S.thr_v = S.list_v[K - 1];
          S.thr_i = S.list_i[K - 1];
        } else {
          S.thr_v = -INFINITY;
          S.thr_i = 0x7fffffff;
        }
      }
      for (int round = 0;; ++round) {
        if (tid == 0) {
          S.cand_n = 0;
          S.overflow = 0;
        }
        __syncthreads();
        const float tv = S.thr_v;
        const int ti = S.thr_i;
        int npass = 0;
#pragma unroll
        for (int q = 0; q < kVec; ++q)
#pragma unroll
          for (int c = 0; c < 4; ++c) {
            const float xv = x[4 * q + c];
            const int xi = token(q, c);
            npass += (valid(q, c) && (before(xv, xi, tv, ti) || (xv == tv && xi == ti))) ? 1 : 0;
          }
        if (__any_sync(0xffffffffu, npass > 0)) {
          int incl = npass;
#pragma unroll
          for (int o = 1; o < 32; o <<= 1) {
            const int y = __shfl_up_sync(0xffffffffu, incl, o);
            if (lane >= o) incl += y;
          }
          const int total = __shfl_sync(0xffffffffu, incl, 31);
          int base = 0;
          if (lane == 31) base = atomicAdd(&S.cand_n, total);
          base = __shfl_sync(0xffffffffu, base, 31);
          int pos = base + incl - npass;
#pragma unroll
          for (int q = 0; q < kVec; ++q)
#pragma unroll
            for (int c = 0; c < 4; ++c) {
              const float xv = x[4 * q + c];
              const int xi = token(q, c);
              if (valid(q, c) && (before(xv, xi, tv, ti) || (xv == tv && xi == ti))) {
                if (pos < kCandCap) {
                  S.cand_v[pos] = xv;
                  S.cand_i[pos] = xi;
                } else {
                  S.overflow = 1;
                }
                ++pos;
              }
            }
        }
        __syncthreads();
        // merge running list + survivors -> best K
        const int nc = S.cand_n < kCandCap ? S.cand_n : kCandCap;
        const int nl = S.list_n;
        // append list entries behind the survivors (room kept by the cap check)
        for (int a = tid; a < nl; a += kThreads) {
          if (nc + a < kCandCap) {
            S.cand_v[nc + a] = S.list_v[a];
            S.cand_i[nc + a] = S.list_i[a];
          }
        }
        __syncthreads();
        const int ntot = (nc + nl) < kCandCap ? (nc + nl) : kCandCap;
        const bool ovf = S.overflow || (nc + nl) > kCandCap;
        rank_select(S.cand_v, S.cand_i, ntot, K, S.tmp_v, S.tmp_i);
        __syncthreads();
        const int kept = ntot < K ? ntot : K;
        if (!ovf) {
          for (int a = tid; a < kept; a += kThreads) {
            S.list_v[a] = S.tmp_v[a];
            S.list_i[a] = S.tmp_i[a];
          }
          if (tid == 0) S.list_n = kept;
          __syncthreads();
          break;
        }
        // too many survivors: raise the bound to the K-th of what was seen and
        // collect this slot again (the running list is unchanged)
        if (tid == 0) {
          S.thr_v = S.tmp_v[K - 1];
          S.thr_i = S.tmp_i[K - 1];
        }
        __syncthreads();
        if (round > 64) {
          record_error(P.err, kDevAssert, 2);
          break;
        }
      }
    }

    // ---- end of a row segment: write this CTA's piece record
    if (seg_last) {
      float M = -INFINITY;
      double Ssum = 0.0;
      if (flags & kWantSum) {
        const float wm = warp_max(m_run);
        double sd = (s_run > 0.f) ? static_cast<double>(s_run) * exp2((static_cast<double>(m_run) - wm) * c2) : 0.0;
        sd = warp_sum_d(sd);
        if (lane == 0) {
          S.red_f[warp][0] = wm;
          S.red_d[warp] = sd;
        }
        __syncthreads();
        if (tid == 0) {
          for (int w = 0; w < kWarps; ++w) M = fmaxf(M, S.red_f[w][0]);
          for (int w = 0; w < kWarps; ++w)
            if (S.red_d[w] > 0.0)
              Ssum += S.red_d[w] * exp2((static_cast<double>(S.red_f[w][0]) - M) * c2);
        }
      }
      if (K == 1) {
        float v = best_v;
        int i = best_i;
        warp_best(v, i);
        if (lane == 0) {
          S.red_g[warp][0] = v;
          S.red_i[warp] = i;
        }
        __syncthreads();
        if (tid == 0) {
          float bv = -INFINITY;
          int bi = 0x7fffffff;
          for (int w = 0; w < kWarps; ++w)
            if (before(S.red_g[w][0], S.red_i[w], bv, bi)) {
              bv = S.red_g[w][0];
              bi = S.red_i[w];
            }
          S.list_v[0] = bv;
          S.list_i[0] = bi;
          S.list_n = 1;
          if (!(flags & kWantSum)) M = bv;
        }
        __syncthreads();
      }
      const int64_t piece = static_cast<int64_t>(blockIdx.x) - tile_owner(row * TR, T, P.grid);
      const int rb = rec_bytes(P.rec_k);
      char* rec = P.pieces + (row * P.max_pieces + piece) * rb;
      const int nl = (K >= 1) ? S.list_n : 0;
      for (int a = tid; a < nl; a += kThreads) {
        rec_val(rec)[a] = S.list_v[a];
        rec_idx(rec, P.rec_k)[a] = S.list_i[a];
      }
      if (tid == 0) {
        RecHead h;
        h.sum = Ssum;
        h.max = (K >= 2 && !(flags & kWantSum)) ? S.list_v[0] : M;
        h.count = nl;
        *reinterpret_cast<RecHead*>(rec) = h;
      }
      // reset per-segment state
      m_run = -INFINITY;
      s_run = 0.f;
      best_v = -INFINITY;
      best_i = 0x7fffffff;
      __threadfence();
      __syncthreads();
      if (tid == 0) {
        const int np = static_cast<int>(tile_owner(row * TR + TR - 1, T, P.grid) -
                                        tile_owner(row * TR, T, P.grid) + 1);
        const uint32_t old = atomicAdd(&P.row_cnt[row], 1u);
        S.is_last = (old == static_cast<uint32_t>(np - 1));
        S.list_n = 0;
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
  __syncthreads();
  if (S.n_done_items) __threadfence();
}

}  // namespace eagle
