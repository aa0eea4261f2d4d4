// eagle_tree_verify: target logits + draft tree -> accepted path and bonus
// token, one fused launch.
//
// Sources: "EAGLE-2: Feature-Level Speculative Decoding Guide", "Single-Pass
// Tree Verification" (the target scores every node at once; the verifier
// walks from the root accepting matching tokens until the first discrepancy;
// the output equals vanilla decoding) and "True Lossless Acceleration";
// "Support Eagle-3 Speculative Decoding in llama.cpp", proposal (acceptance /
// rejection strategy = speculative sampling); "EAGLE-2 Speculative Decoding
// Support for llama.cpp - Phase 1", "Performance Notes" (temperature + top_k
// + top_p).
//
// Phase 1 (one cluster per row, eagle_rowstream.cuh): one HBM pass over the
// m target rows of every item -> per row the argmax (greedy), the top_k
// logits (sampling with top_k) or the max, sum of exp((x-max)/T) and
// per-tile sums (sampling over the full vocabulary).
// Phase 2 (the row's leader CTA, one warp): the walk's decision at that
// node -- the accepted child, or the bonus token if the walk stops there.
// Phase 3 (the CTA whose row of an item arrives last): follow the decisions
// from the root.
// Sampling follows recursive speculative sampling with one-hot draft
// distributions (tree children are deterministic top-k picks): accept child j
// iff u_j (1 - rho) < p(token_j), else rho += p(token_j); on rejection of all
// children (or at a leaf) draw the bonus token by inverse CDF over token ids
// ascending with the rejected tokens removed.  Probabilities of individual
// tokens and all decisions are fp64.
#include "eagle_philox.cuh"
#include "eagle_stream_host.h"

namespace eagle {

enum : int { kModeGreedy = 0, kModeTopK = 1, kModeFull = 2, kModeNucleus = 3 };

struct VerifyArgs {
  RowStream rs;
  int m;
  int mode[kMaxItems];
  double inv_temperature[kMaxItems];   // 1 / T
  float top_p[kMaxItems];
  int top_k[kMaxItems];
  const int32_t* parents[kMaxItems];
  const int32_t* tokens[kMaxItems];
  int32_t* accepted[kMaxItems];
  uint64_t seed[kMaxItems];
  uint64_t step;
  int32_t* n_accepted;
  int32_t* bonus;
  int2* dec;                      // [rows] per-node decision: (accepted child or -1, bonus)
  int n_warm;                     // code warm-up clusters after the rows' (0 or 2)
};

__device__ __forceinline__ double warp_incl_scan_d(double v) {
  const int lane = threadIdx.x & 31;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const double y = __shfl_up_sync(0xffffffffu, v, o);
    if (lane >= o) v += y;
  }
  return v;
}

// ------------------------------------------------ nucleus over the vocabulary
// (top_p < 1 without top_k).  The kept set is the shortest prefix of the
// row in (probability desc, token asc) order -- the order of the 64-bit keys
// mkkey(logit, token), larger first -- whose mass reaches top_p of the total,
// the crossing token included.  Masses are exp((x - max) / T) as fixed-point
// integers, units of 2^-31 of the max's, summed exactly in 64 bits, so sums
// do not depend on their order.  The crossing token is found by bins of u = log2 of
// the max's mass over the token's, (max - x) c2 >= 0, which is monotone in
// the logit: 32 bins per unit of u, then 1024 sub-bins of the crossing bin,
// then the crossing sub-bin's tokens (few unless many share a logit) ranked
// by their keys; more than kNucCap of them are resolved by a radix select on
// the key, 8 bits per pass.  All warps of the row's leader CTA, over the row
// in L2 (the stream has just read it); the ring is their scratch.  Results:
// S.aux_key = the crossing key (kept iff key >= it), S.aux_d = the kept mass
// in units of the max's; per-tile kept masses at ring byte offset kNucTiles
// (read by the residual draw).
constexpr size_t kNucTiles = 65536;                  // u64 [tiles], after the histograms
constexpr size_t kNucScratch = kScratchBytes - 512;  // the searches' scratch, at the ring's end
constexpr int kNucMaxTiles = static_cast<int>((kNucScratch - kNucTiles) / 8);
constexpr int kNucBins = 1024;                       // per warp, per level
constexpr int kNucCap = 1024;                        // tokens ranked exactly
constexpr float kQUnit = 2147483648.0f;              // 2^31: a token's mass fits 32 bits

// Bin b of H[0..nb) (nb = kThreads * per, all threads) with above(b) < t <=
// above(b) + H[b], above(b) = sum of H over the bins before b (bin 0 first);
// scratch[kWarps] = b, scratch[kWarps + 1] = above(b), scratch[kWarps + 2] =
// sum of H.
static __device__ __forceinline__ void find_cut_bin(const unsigned long long* H, int nb, double t,
                                                    unsigned long long* scratch) {
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int per = nb / kThreads;
  const int lo = tid * per;   // this thread's bins [lo, lo + per)
  unsigned long long cs = 0;
  for (int b = lo; b < lo + per; ++b) cs += H[b];
  unsigned long long incl = cs;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const unsigned long long y = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += y;
  }
  if (lane == 31) scratch[warp] = incl;
  if (tid == 0) {
    scratch[kWarps] = static_cast<unsigned long long>(nb - 1);
    scratch[kWarps + 1] = 0;
  }
  __syncthreads();
  unsigned long long wbase = 0, total = 0;
  for (int w = 0; w < kWarps; ++w) {
    if (w < warp) wbase += scratch[w];
    total += scratch[w];
  }
  const unsigned long long above = wbase + incl - cs;
  if (cs > 0 && static_cast<double>(above) < t && t <= static_cast<double>(above + cs)) {
    unsigned long long acc = above;
    for (int b = lo; b < lo + per; ++b) {
      if (H[b] > 0 && static_cast<double>(acc + H[b]) >= t) {
        scratch[kWarps] = static_cast<unsigned long long>(b);
        scratch[kWarps + 1] = acc;
        break;
      }
      acc += H[b];
    }
  }
  if (tid == 0) scratch[kWarps + 2] = total;
  __syncthreads();
}

// Block sums (all threads) of three u64 and one int; every thread gets them.
static __device__ __forceinline__ void block_sum4(unsigned long long& a, unsigned long long& b,
                                                  unsigned long long& c, int& n,
                                                  unsigned long long* scratch) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
#pragma unroll
  for (int o = 16; o; o >>= 1) {
    a += __shfl_xor_sync(0xffffffffu, a, o);
    b += __shfl_xor_sync(0xffffffffu, b, o);
    c += __shfl_xor_sync(0xffffffffu, c, o);
    n += __shfl_xor_sync(0xffffffffu, n, o);
  }
  if (lane == 0) {
    scratch[4 * warp] = a;
    scratch[4 * warp + 1] = b;
    scratch[4 * warp + 2] = c;
    scratch[4 * warp + 3] = static_cast<unsigned long long>(n);
  }
  __syncthreads();
  a = b = c = 0;
  n = 0;
  for (int w = 0; w < kWarps; ++w) {
    a += scratch[4 * w];
    b += scratch[4 * w + 1];
    c += scratch[4 * w + 2];
    n += static_cast<int>(scratch[4 * w + 3]);
  }
  __syncthreads();
}

// The nucleus cut, by every CTA of the row's cluster over its own share of
// the row (the tiles it streamed), the shares combined in the leader's
// shared memory (distributed shared memory) between cluster barriers:
//   1. approximate masses of the bins of u (32-bit sums of each token's mass
//      relative to its bin's top, 2^-12 units) -> the leader's approximate
//      crossing bin;
//   2. exact fixed-point sums above / in the bin and the total -> the leader
//      confirms the bin (or moves to a neighbour and the pass repeats);
//   3. the bin's tokens appended to the leader's list, and every tile's mass
//      above the bin written to the leader's tile array;
// then the leader alone ranks the list (or, past kNucCap tokens, runs the
// radix select on the key over the whole row) and completes the tiles.
// Called by every CTA of the cluster after stream_row, the leader's row max
// in place.
struct NucShare {
  uint32_t bin;          // leader: the bin under test / confirmed
  uint32_t done;         // leader: 1 when confirmed
  unsigned long long above, t_bits;   // leader: mass above the bin; t as double bits
  unsigned long long part[4];         // every CTA: above, in, total, count of its share
  uint32_t cnt;          // leader: tokens of the bin collected
};

static __device__ __noinline__ void nucleus_cut(const float* row, int V, int rank, int PC,
                                                float c2, double top_p, StreamSmem& S) {
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const bool leader = rank == 0;
  char* ring = reinterpret_cast<char*>(S.ring);
  uint32_t* ch = reinterpret_cast<uint32_t*>(ring);                       // [kWarps][kNucBins]
  float* fh = reinterpret_cast<float*>(ring + kWarps * kNucBins * 4);     // leader: [kNucBins]
  unsigned long long* wh = reinterpret_cast<unsigned long long*>(ring);   // (fallback) [kWarps][256]
  unsigned long long* tiles = reinterpret_cast<unsigned long long*>(ring + kNucTiles);
  unsigned long long* scr = reinterpret_cast<unsigned long long*>(ring + kNucScratch);  // [16]
  NucShare* sh = reinterpret_cast<NucShare*>(ring + kNucScratch + 128);
  unsigned long long* red = reinterpret_cast<unsigned long long*>(ring + kNucScratch + 256);  // [4 kWarps]
  unsigned long long* lkey = reinterpret_cast<unsigned long long*>(ring + 36864);  // [kNucCap]
  unsigned long long* lq = lkey + kNucCap;        // [kNucCap] their masses
  unsigned long long* sq = lq + kNucCap;          // [kNucCap] masses in key order
  int* ord = reinterpret_cast<int*>(sq + kNucCap);   // [kNucCap] entry of each rank
  const uint32_t lead_sh = map_rank(sh, 0);
  auto lead = [&](const void* p) { return lead_sh + static_cast<uint32_t>(reinterpret_cast<const char*>(p) - reinterpret_cast<const char*>(sh)); };
  const float M = __uint_as_float(ld_cluster_u32(map_rank(&S.rmax, 0)));
  const int TR = (V + kTile - 1) / kTile;
  const int tile0 = rank * TR / PC, tile1 = (rank + 1) * TR / PC;   // this CTA's share
  // the tokens of a range of tiles: f(x, token, u); x = -inf past the row's
  // end.  A round loads kNucUnroll 16-byte pieces per thread before using
  // any; every lane of a warp runs the same rounds.
  constexpr int kNucUnroll = 8;
  auto load4 = [&](int i, float (&xs)[4]) {
    if (i + 4 <= V) {
      const float4 v = __ldcg(reinterpret_cast<const float4*>(row + i));
      xs[0] = v.x, xs[1] = v.y, xs[2] = v.z, xs[3] = v.w;
    } else {
#pragma unroll
      for (int c = 0; c < 4; ++c) xs[c] = i + c < V ? __ldcg(row + i + c) : -INFINITY;
    }
  };
  auto for_tiles = [&](int t0, int t1, auto f) {
    const int b0 = t0 * kTile, b1 = t1 * kTile;
    for (int i0 = b0 + tid * 4; i0 < b1; i0 += kThreads * 4 * kNucUnroll) {
      float xs[kNucUnroll][4];
#pragma unroll
      for (int j = 0; j < kNucUnroll; ++j) {
        const int i = i0 + j * kThreads * 4;
        if (i < b1) load4(i, xs[j]);
        else xs[j][0] = xs[j][1] = xs[j][2] = xs[j][3] = -INFINITY;
      }
#pragma unroll
      for (int j = 0; j < kNucUnroll; ++j)
#pragma unroll
        for (int c = 0; c < 4; ++c) f(xs[j][c], i0 + j * kThreads * 4 + c, (M - xs[j][c]) * c2);
    }
  };
  auto qof = [&](float u) {   // (a 32-bit conversion: the 64-bit one is slow here)
    return static_cast<unsigned long long>(__float2uint_rn(ex2(-u) * kQUnit));
  };
  auto bin1 = [&](float u) { return min(kNucBins - 1, __float2int_rz(u * 32.f)); };

  // ---- 1. approximate bin masses over the share: a token of bin b adds
  // 2^(b/32 - u) in (2^-1/32, 1] in units of 2^-12 (a warp's bin would wrap
  // past 2^20 tokens)
  for (int b = tid; b < kWarps * kNucBins; b += kThreads) ch[b] = 0u;
  for (int b = tile0 + tid; b < tile1; b += kThreads) tiles[b] = 0ull;
  if (leader && tid == 0) {
    sh->cnt = 0u;
    sh->done = 0u;
  }
  __syncthreads();
  for_tiles(tile0, tile1, [&](float x, int, float u) {
    if (x == -INFINITY) return;
    const int b = bin1(u);
    atomicAdd(&ch[warp * kNucBins + b],
              __float2uint_rn(ex2(static_cast<float>(b) * (1.0f / 32.0f) - u) * 4096.0f));
  });
  __syncthreads();
  unsigned long long* ch64 = reinterpret_cast<unsigned long long*>(ring);   // [kNucBins] the CTA's sums
  {
    unsigned long long cs[kNucBins / kThreads];
#pragma unroll
    for (int k = 0; k < kNucBins / kThreads; ++k) {
      cs[k] = 0;
      for (int w = 0; w < kWarps; ++w) cs[k] += ch[w * kNucBins + tid + k * kThreads];
    }
    __syncthreads();
#pragma unroll
    for (int k = 0; k < kNucBins / kThreads; ++k) ch64[tid + k * kThreads] = cs[k];
  }
  __syncwarp();
  cluster_arrive_release();
  cluster_wait();
  if (leader) {
    for (int b = tid; b < kNucBins; b += kThreads) {
      unsigned long long c = 0;
      for (int r = 0; r < PC; ++r) c += ld_cluster_u64(map_rank(ch64 + b, static_cast<uint32_t>(r)));
      fh[b] = static_cast<float>(c) * (1.0f / 4096.0f) * ex2(-static_cast<float>(b) * (1.0f / 32.0f));
    }
    __syncthreads();
    if (warp == 0) {
      double tot = 0.0;
      for (int b = lane; b < kNucBins; b += 32) tot += fh[b];
      tot = warp_sum_d(tot);
      const double ta = top_p * tot;
      double cum = 0.0;
      int pick = kNucBins - 1;
      for (int base = 0; base < kNucBins; base += 32) {
        const double m = fh[base + lane];
        const double incl = warp_incl_scan_d(m) + cum;
        const unsigned bal = __ballot_sync(0xffffffffu, m > 0.0 && incl >= ta);
        if (bal) {
          pick = base + __ffs(bal) - 1;
          break;
        }
        cum = __shfl_sync(0xffffffffu, incl, 31);
      }
      if (lane == 0) sh->bin = static_cast<uint32_t>(pick);
    }
  }
  __syncwarp();
  cluster_arrive_release();
  cluster_wait();
  // ---- 2. exact sums for the bin under test; the leader confirms or moves it
  int b1 = 0;
  unsigned long long above = 0;
  double t = 0.0;
  for (int guard = 0; guard < kNucBins; ++guard) {
    b1 = static_cast<int>(ld_cluster_u32(lead(&sh->bin)));
    unsigned long long ab = 0, in = 0, Z = 0;
    int n_in = 0;
    for_tiles(tile0, tile1, [&](float x, int, float u) {
      if (x == -INFINITY) return;
      const unsigned long long q = qof(u);
      const int b = bin1(u);
      Z += q;
      if (b < b1) ab += q;
      else if (b == b1) in += q, ++n_in;
    });
    block_sum4(ab, in, Z, n_in, red);
    if (tid == 0) {
      sh->part[0] = ab;
      sh->part[1] = in;
      sh->part[2] = Z;
      sh->part[3] = static_cast<unsigned long long>(n_in);
    }
    __syncwarp();
    cluster_arrive_release();
    cluster_wait();
    if (leader && tid == 0) {
      unsigned long long A = 0, I = 0, T = 0;
      for (int r = 0; r < PC; ++r) {
        A += ld_cluster_u64(map_rank(&sh->part[0], static_cast<uint32_t>(r)));
        I += ld_cluster_u64(map_rank(&sh->part[1], static_cast<uint32_t>(r)));
        T += ld_cluster_u64(map_rank(&sh->part[2], static_cast<uint32_t>(r)));
      }
      const double tt = top_p * static_cast<double>(T);
      sh->above = A;
      sh->t_bits = static_cast<unsigned long long>(__double_as_longlong(tt));
      if (static_cast<double>(A) >= tt && b1 > 0) sh->bin = static_cast<uint32_t>(b1 - 1);
      else if (static_cast<double>(A + I) < tt && b1 < kNucBins - 1) sh->bin = static_cast<uint32_t>(b1 + 1);
      else sh->done = 1u;
    }
    __syncwarp();
    cluster_arrive_release();
    cluster_wait();
    if (ld_cluster_u32(lead(&sh->done))) {
      above = ld_cluster_u64(lead(&sh->above));
      t = __longlong_as_double(static_cast<long long>(ld_cluster_u64(lead(&sh->t_bits))));
      break;
    }
  }
  // ---- 3. the bin's tokens to the leader's list; each tile's mass above the
  // bin (a warp's 128 tokens of a piece lie in one tile: one add per warp and
  // piece) into this CTA's own tile array, then copied to the leader's
  for (int i0 = tile0 * kTile + tid * 4; i0 < tile1 * kTile; i0 += kThreads * 4 * kNucUnroll) {
    float xs[kNucUnroll][4];
#pragma unroll
    for (int j = 0; j < kNucUnroll; ++j) {
      const int i = i0 + j * kThreads * 4;
      if (i < tile1 * kTile) load4(i, xs[j]);
      else xs[j][0] = xs[j][1] = xs[j][2] = xs[j][3] = -INFINITY;
    }
#pragma unroll
    for (int j = 0; j < kNucUnroll; ++j) {
      const int i = i0 + j * kThreads * 4;
      unsigned long long q = 0;
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        const float x = xs[j][c];
        if (x == -INFINITY) continue;
        const float u = (M - x) * c2;
        const int b = bin1(u);
        if (b < b1) {
          q += qof(u);
        } else if (b == b1) {
          const uint32_t e = atom_add_cluster_u32(lead(&sh->cnt), 1u);
          if (e < static_cast<uint32_t>(kNucCap)) {
            st_cluster(map_rank(lkey + e, 0), mkkey(x, i + c));
            st_cluster(map_rank(lq + e, 0), static_cast<Key>(qof(u)));
          }
        }
      }
#pragma unroll
      for (int o = 16; o; o >>= 1) q += __shfl_xor_sync(0xffffffffu, q, o);
      if (lane == 0 && q && i < tile1 * kTile) atomicAdd(&tiles[i / kTile], q);
    }
  }
  __syncthreads();
  if (!leader)
    for (int b = tile0 + tid; b < tile1; b += kThreads)
      st_cluster(map_rank(tiles + b, 0), static_cast<Key>(tiles[b]));
  __syncwarp();
  cluster_arrive_release();
  cluster_wait();
  if (!leader) return;
  const int n = static_cast<int>(sh->cnt);
  unsigned long long kb = 0, keep = 0;
  if (n <= kNucCap) {
    // rank by counting (keys distinct), masses in key order, first prefix
    // reaching t
    for (int e = tid; e < n; e += kThreads) {
      const unsigned long long k = lkey[e];
      int r = 0;
      for (int f = 0; f < n; ++f) r += lkey[f] > k ? 1 : 0;
      sq[r] = lq[e];
      ord[r] = e;
    }
    __syncthreads();
    if (warp == 0) {
      unsigned long long cum = above;
      int pick = n - 1;
      bool found = false;
      for (int base = 0; base < n && !found; base += 32) {
        const unsigned long long q = base + lane < n ? sq[base + lane] : 0ull;
        unsigned long long incl = q;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
          const unsigned long long y = __shfl_up_sync(0xffffffffu, incl, o);
          if (lane >= o) incl += y;
        }
        const unsigned bal =
            __ballot_sync(0xffffffffu, base + lane < n && static_cast<double>(cum + incl) >= t);
        const int l = bal ? __ffs(bal) - 1 : 31;
        if (bal) {
          pick = base + l;
          found = true;
        }
        cum += __shfl_sync(0xffffffffu, incl, l);
      }
      if (lane == 0) {
        scr[kWarps + 1] = cum;
        scr[kWarps + 3] = static_cast<unsigned long long>(pick);
      }
    }
    __syncthreads();
    keep = scr[kWarps + 1];
    kb = lkey[ord[static_cast<int>(scr[kWarps + 3])]];
    // the bin's kept tokens complete their tiles
    for (int e = tid; e < n; e += kThreads)
      if (lkey[e] >= kb) atomicAdd(&tiles[static_cast<int>(~static_cast<uint32_t>(lkey[e])) / kTile], lq[e]);
  } else {
    // many tokens share the crossing bin: radix select on the 64-bit key
    // among them over the whole row, 8 bits per pass from the top (exact
    // 64-bit sums), by the leader alone
    unsigned long long prefix = 0, pmask = 0;
    for (int shf = 56; shf >= 0; shf -= 8) {
      for (int b = tid; b < kWarps * 256; b += kThreads) wh[b] = 0ull;
      __syncthreads();
      for_tiles(0, TR, [&](float x, int id, float u) {
        if (x == -INFINITY || bin1(u) != b1) return;
        const unsigned long long k = mkkey(x, id);
        if ((k & pmask) == prefix) atomicAdd(&wh[warp * 256 + static_cast<int>((k >> shf) & 255u)], qof(u));
      });
      __syncthreads();
      unsigned long long* rev = wh + kWarps * 256;   // bins in key order, largest first
      for (int b = tid; b < 256; b += kThreads) {
        unsigned long long sum = 0;
        for (int w = 0; w < kWarps; ++w) sum += wh[w * 256 + 255 - b];
        rev[b] = sum;
      }
      __syncthreads();
      find_cut_bin(rev, 256, t - static_cast<double>(above), scr);
      const int b = 255 - static_cast<int>(scr[kWarps]);
      above += scr[kWarps + 1];
      prefix |= static_cast<unsigned long long>(b) << shf;
      pmask |= 255ull << shf;
      __syncthreads();
    }
    kb = prefix;   // one token (keys are distinct); its own mass completes the sum
    for_tiles(0, TR, [&](float x, int id, float u) {
      if (x != -INFINITY && mkkey(x, id) == kb) scr[kWarps + 1] = qof(u);
    });
    __syncthreads();
    keep = above + scr[kWarps + 1];
    // the bin's kept tokens complete their tiles
    for (int i0 = tid * 4; i0 < TR * kTile; i0 += kThreads * 4) {
      float xs[4];
      load4(i0, xs);
      unsigned long long q = 0;
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        const float u = (M - xs[c]) * c2;
        if (xs[c] != -INFINITY && bin1(u) == b1 && mkkey(xs[c], i0 + c) >= kb) q += qof(u);
      }
#pragma unroll
      for (int o = 16; o; o >>= 1) q += __shfl_xor_sync(0xffffffffu, q, o);
      if (lane == 0 && q) atomicAdd(&tiles[i0 / kTile], q);
    }
  }
  if (tid == 0) {
    S.aux_key = kb;
    S.aux_d = static_cast<double>(keep) / static_cast<double>(kQUnit);
  }
  __syncthreads();
}

// One node's decision: its row, its place in the tree, the sampling
// parameters of its item, and where the decision goes.
struct NodeJob {
  const float* lrow;     // the node's target row
  const float2* tsums;   // the row's per-(tile, warp) sums (full vocabulary)
  const unsigned long long* ntiles;   // per-tile kept masses (nucleus; see nucleus_cut)
  int2* dec;             // out: (accepted child or -1, bonus)
  double invT, top_p;
  uint64_t seed, step;
  float c2;              // 1/T * log2(e), the tile sums' exponent scale
  int node, m, mode, K, TR, vocab;
};

// Decision of the walk at one node (warp 0 of the node's row leader): the
// child accepted there (-1 if none) and the token emitted when the walk stops
// there.  It depends only on the node's own row, its children and the
// uniforms keyed by (seed, step, node, j), so every node decides on its own,
// in parallel, and the item's final step follows the decisions from the root.
// The tree (parents, tokens) is in S.aux.
static __device__ __noinline__ void node_decision(const NodeJob& J, StreamSmem& S) {
  const int lane = threadIdx.x & 31;
  const int m = J.m;
  const int node = J.node;
  const int mode = J.mode;
  const double invT = J.invT;
  const double top_p = J.top_p;
  const int K = J.K;
  const uint64_t seed = J.seed;
  const int* parents = S.aux;                   // prefetched at kernel start
  const int* tokens = S.aux + EAGLE_MAX_TREE;
  const int TR = J.TR;

  int* kn = reinterpret_cast<int*>(S.ring[0]);          // children (node ids), node order
  int* kt = kn + EAGLE_MAX_TREE;                         // their tokens
  double* kp = reinterpret_cast<double*>(S.ring[1]);     // kept probabilities, by rank
  int* kid = reinterpret_cast<int*>(kp + kKMax);         // kept ids, by rank
  double* sp = reinterpret_cast<double*>(kid + kKMax);   // kept probabilities sorted by id
  int* sid = reinterpret_cast<int*>(sp + kKMax);
  double* pc = reinterpret_cast<double*>(S.ring[2]);     // children probabilities (top-k mode)
  int* krej = reinterpret_cast<int*>(pc + EAGLE_MAX_TREE);  // kept entry is a child's token

  // ---- the children of this node, in node order
  int nk = 0;
  {
    int pv[EAGLE_MAX_TREE / 32];
#pragma unroll
    for (int r = 0; r < EAGLE_MAX_TREE / 32; ++r) {
      const int i = lane + 32 * r;
      pv[r] = (i > node && i < m) ? parents[i] : -2;
    }
#pragma unroll
    for (int r = 0; r < EAGLE_MAX_TREE / 32; ++r) {
      const int i = lane + 32 * r;
      const bool is = pv[r] == node;
      const unsigned bal = __ballot_sync(0xffffffffu, is);
      if (is) {
        const int pos = nk + __popc(bal & ((1u << lane) - 1u));
        kn[pos] = i;
        kt[pos] = tokens[i];
      }
      nk += __popc(bal);
    }
  }
  __syncwarp();

  int child = -1, bonus = -1;
  if (mode == kModeGreedy) {
    const int a = key_i(S.rlist[0]);   // argmax
    for (int b = 0; b < nk && child < 0; b += 32) {
      const bool hit = b + lane < nk && kt[b + lane] == a;
      const unsigned bal = __ballot_sync(0xffffffffu, hit);
      if (bal) child = kn[b + __ffs(bal) - 1];
    }
    bonus = a;
  } else {
    // ---- the warped target distribution at this node
    const float* lrow = J.lrow;
    double rowmax = 0.0, zsum = 1.0, izsum = 1.0;
    int nkeep = 0;
    if (mode == kModeTopK) {
      // lane l holds the entries of rank 2l and 2l + 1: one scan of the pair
      // sums gives every prefix mass and the total
      int cnt = S.rcount;
      if (cnt > K) cnt = K;
      const int ea = 2 * lane, eb = ea + 1;
      const double z0 = static_cast<double>(key_v(S.rlist[0])) * invT;
      double pa = 0.0, pb = 0.0;   // exp((z - z0)), unnormalised
      int ia = kNoIndex, ib = kNoIndex;
      if (ea < cnt) {
        pa = exp_d(static_cast<double>(key_v(S.rlist[ea])) * invT - z0);
        ia = key_i(S.rlist[ea]);
      }
      if (eb < cnt) {
        pb = exp_d(static_cast<double>(key_v(S.rlist[eb])) * invT - z0);
        ib = key_i(S.rlist[eb]);
      }
      const double incl = warp_incl_scan_d(pa + pb);
      double kept = __shfl_sync(0xffffffffu, incl, 31);
      nkeep = cnt;
      if (top_p < 1.0) {
        // entries are in probability order; keep the shortest prefix whose
        // normalised cumulative mass reaches top_p (the crossing entry included)
        const double lim = top_p * kept;
        const unsigned ba = __ballot_sync(0xffffffffu, ea < cnt && incl - pb >= lim);
        const unsigned bb = __ballot_sync(0xffffffffu, eb < cnt && incl >= lim);
        const int fa = ba ? 2 * (__ffs(ba) - 1) : cnt;
        const int fb = bb ? 2 * (__ffs(bb) - 1) + 1 : cnt;
        const int last = (fa < fb ? fa : fb) < cnt ? (fa < fb ? fa : fb) : cnt - 1;
        nkeep = last + 1;
        const double at = __shfl_sync(0xffffffffu, (last & 1) ? incl : incl - pb, last >> 1);
        kept = at;
      }
      const double ik = 1.0 / kept;
      const bool ka = ea < nkeep, kb = eb < nkeep;
      kp[ea] = ka ? pa * ik : 0.0;
      kid[ea] = ka ? ia : kNoIndex;
      kp[eb] = kb ? pb * ik : 0.0;
      kid[eb] = kb ? ib : kNoIndex;
      // children probabilities: every kept entry looks for its token among
      // the children (a child whose token is not kept has probability 0)
      for (int j = lane; j < nk; j += 32) pc[j] = 0.0;
      __syncwarp();
      int ra = 0, rb = 0;
      for (int r = 0; r < nk; ++r) {
        const int t = kt[r];
        if (ka && t == ia) {
          pc[r] = pa * ik;
          ra = 1;
        }
        if (kb && t == ib) {
          pc[r] = pb * ik;
          rb = 1;
        }
      }
      krej[ea] = ra;
      krej[eb] = rb;
      __syncwarp();
    } else {  // full vocabulary, or its nucleus (kept mass and set from nucleus_cut)
      rowmax = static_cast<double>(S.rmax);
      zsum = mode == kModeNucleus ? S.aux_d : S.rsum;
      izsum = 1.0 / zsum;
    }
    const unsigned long long kcut = mode == kModeNucleus ? S.aux_key : 0ull;
    auto prob_tok = [&](int t) -> double {  // token t, full vocabulary or nucleus (lane-local)
      const float x = __ldg(lrow + t);
      if (mkkey(x, t) < kcut) return 0.0;   // outside the nucleus
      return exp_d((static_cast<double>(x) - rowmax) * invT) * izsum;
    };
    auto prob_of = [&](int j) -> double {  // child j (lane-local)
      if (mode == kModeTopK) return pc[j];
      return prob_tok(kt[j]);
    };

    // ---- children in node order, 32 at a time: child j is accepted iff
    // u_j (1 - rho_j) < p(token_j), rho_j = mass of the children before it
    // (all of them rejected when j is reached)
    double rho_all = 0.0;
    for (int b = 0; b < nk && child < 0; b += 32) {
      const int j = b + lane;
      const bool valid = j < nk;
      const double pt = valid ? prob_of(j) : 0.0;
      const double incl = warp_incl_scan_d(pt);
      const double rho = rho_all + (incl - pt);
      const double u = valid ? philox_uniform(seed, J.step, static_cast<uint32_t>(node),
                                              static_cast<uint32_t>(j))
                             : 1.0;
      const unsigned bal = __ballot_sync(0xffffffffu, valid && (u * (1.0 - rho) < pt));
      if (bal) child = kn[b + __ffs(bal) - 1];
      rho_all += __shfl_sync(0xffffffffu, incl, 31);
    }

    if (child < 0) {
      // ---- every child rejected (or a leaf): residual draw by inverse CDF
      // over ids ascending, the children's tokens removed
      const double thr =
          philox_uniform(seed, J.step, static_cast<uint32_t>(node), kResidualChild) *
          (1.0 - rho_all);
      auto is_rejected = [&](int t) {
        for (int r = 0; r < nk; ++r)
          if (kt[r] == t) return true;
        return false;
      };
      if (mode == kModeTopK) {
        // kept entries sorted by token id (rank by counting); the children's
        // tokens (all rejected here) carry no mass
#pragma unroll
        for (int hh = 0; hh < 2; ++hh) {
          const int e = 2 * lane + hh;
          if (e < nkeep) {
            const int me = kid[e];
            int r = 0;
            for (int f = 0; f < nkeep; ++f) r += kid[f] < me ? 1 : 0;
            sid[r] = me;
            sp[r] = krej[e] ? 0.0 : kp[e];
          }
        }
        __syncwarp();
        // lane l holds sorted entries 2l and 2l + 1
        const int ea = 2 * lane, eb = ea + 1;
        const double ma = ea < nkeep ? sp[ea] : 0.0, mb = eb < nkeep ? sp[eb] : 0.0;
        const double incl = warp_incl_scan_d(ma + mb);
        const unsigned ba = __ballot_sync(0xffffffffu, ea < nkeep && incl - mb > thr);
        const unsigned bb = __ballot_sync(0xffffffffu, eb < nkeep && incl > thr);
        const int fa = ba ? 2 * (__ffs(ba) - 1) : kKMax;
        const int fb = bb ? 2 * (__ffs(bb) - 1) + 1 : kKMax;
        int pick = fa < fb ? fa : fb;
        if (pick >= kKMax) {   // rounding: the last entry with mass
          const unsigned nza = __ballot_sync(0xffffffffu, ea < nkeep && ma > 0.0);
          const unsigned nzb = __ballot_sync(0xffffffffu, eb < nkeep && mb > 0.0);
          const int la = nza ? 2 * (31 - __clz(nza)) : -1;
          const int lb = nzb ? 2 * (31 - __clz(nzb)) + 1 : -1;
          pick = la > lb ? la : lb;
          if (pick < 0) pick = nkeep - 1;
        }
        bonus = sid[pick];
      } else {
        // tile masses (tile sums were taken relative to each tile's max)
        const float2* ts = J.tsums;
        const double c2 = static_cast<double>(J.c2);
        double cum = 0.0;
        int tile = -1;
        double before_tile = 0.0;
        for (int base = 0; base < TR && tile < 0; base += 32) {
          const int t = base + lane;
          double mass = 0.0;
          if (t < TR && mode == kModeNucleus) {
            mass = static_cast<double>(J.ntiles[t]) * (1.0 / static_cast<double>(kQUnit)) * izsum;
          } else if (t < TR) {
            // combine the per-warp partials of tile t (max, sum of 2^((x - max) c2))
            const float2* tw = ts + static_cast<int64_t>(t) * kWarps;
            for (int w = 0; w < kWarps; ++w) {
              const float2 v = __ldcg(tw + w);
              if (v.y > 0.f)
                mass += static_cast<double>(v.y) *
                        static_cast<double>(ex2((v.x - static_cast<float>(rowmax)) * static_cast<float>(c2)));
            }
            mass *= izsum;
          }
          if (t < TR) {
            for (int r = 0; r < nk; ++r) {   // rejected tokens of this tile, each once
              const int rt = kt[r];
              if (rt / kTile != t) continue;
              bool first = true;
              for (int r2 = 0; r2 < r; ++r2) first &= kt[r2] != rt;
              if (first) mass -= prob_tok(rt);
            }
            if (mass < 0.0) mass = 0.0;
          }
          const double incl = warp_incl_scan_d(mass) + cum;
          const unsigned bal = __ballot_sync(0xffffffffu, t < TR && incl > thr);
          if (bal) {
            const int l = __ffs(bal) - 1;
            tile = base + l;
            before_tile = __shfl_sync(0xffffffffu, incl - mass, l);
          }
          cum = __shfl_sync(0xffffffffu, incl, 31);
        }
        if (tile < 0) tile = TR - 1, before_tile = cum;  // rounding: take the last tile
        // scan inside the tile: lane owns 32 consecutive tokens
        const int v0 = tile * kTile + lane * 32;
        double lm[32];
        double lsum = 0.0;
#pragma unroll
        for (int q = 0; q < 32; ++q) {
          const int t = v0 + q;
          double mass = 0.0;
          if (t < J.vocab && !is_rejected(t)) {
            const float x = __ldg(lrow + t);
            if (mkkey(x, t) >= kcut)
              mass = static_cast<double>(exp2f((x - static_cast<float>(rowmax)) * static_cast<float>(c2))) * izsum;
          }
          lm[q] = mass;
          lsum += mass;
        }
        const double incl = warp_incl_scan_d(lsum) + before_tile;
        const unsigned bal = __ballot_sync(0xffffffffu, incl > thr);
        int pick = -1;
        if (bal) {
          const int l = __ffs(bal) - 1;
          if (lane == l) {
            double c = incl - lsum;
            for (int q = 0; q < 32; ++q) {
              c += lm[q];
              if (lm[q] > 0.0 && c > thr) {
                pick = v0 + q;
                break;
              }
            }
            if (pick < 0) pick = v0 + 31;
          }
          pick = __shfl_sync(0xffffffffu, pick, l);
        } else {  // rounding: last token of the tile with mass
          int last = -1;
          for (int q = 31; q >= 0; --q)
            if (lm[q] > 0.0) {
              last = v0 + q;
              break;
            }
          const unsigned b2 = __ballot_sync(0xffffffffu, last >= 0);
          const int l = b2 ? 31 - __clz(b2) : 0;
          pick = __shfl_sync(0xffffffffu, last, l);
          if (pick < 0) pick = tile * kTile;
        }
        bonus = pick;
      }
    }
  }
  if (lane == 0) *J.dec = make_int2(child, bonus);
  __syncwarp();
}

// Warp 0 of a row leader, after its decision (written by lane 0): arrive on
// the item's counter; true in the warp whose row arrives last.  Lane 0 wrote
// the decision and performs the arrival itself, so the atomic's release
// orders that write and its acquire (in the last arrival) makes every row's
// decision visible to lane 0, and through the warp barrier to the warp.  The
// last arrival resets the counter for the next launch.
static __device__ __forceinline__ bool warp_item_arrive(const VerifyArgs& A, int item) {
  const int lane = threadIdx.x & 31;
  int last = 0;
  if (lane == 0) {
    uint32_t old;
    asm volatile("atom.acq_rel.gpu.global.add.u32 %0, [%1], 1;"
                 : "=r"(old)
                 : "l"(A.rs.item_cnt + item)
                 : "memory");
    last = old == static_cast<uint32_t>(A.rs.rows_per_item - 1);
    if (last) A.rs.item_cnt[item] = 0u;
  }
  last = __shfl_sync(0xffffffffu, last, 0);
  __syncwarp();
  return last != 0;
}

// The item's final step (warp 0 of the CTA whose row arrived last): follow
// the m decisions at `src` from the root into acc / n_acc / bonus.
static __device__ __noinline__ void follow_path(const int2* src, int m, int32_t* acc,
                                                int32_t* n_acc, int32_t* bonus, StreamSmem& S) {
  const int lane = threadIdx.x & 31;
  int2* dec = reinterpret_cast<int2*>(S.ring[0]);
  for (int i = lane; i < m; i += 32) dec[i] = __ldcg(src + i);
  __syncwarp();
  if (lane == 0) {
    int node = 0, n = 0;
    acc[0] = 0;
    for (int guard = 0; guard < m; ++guard) {
      const int c = dec[node].x;
      if (c <= node || c >= m) break;   // -1: the walk stops here
      node = c;
      acc[++n] = node;
    }
    *n_acc = n;
    *bonus = dec[node].y;
  }
  __syncwarp();
}

// The decision code warm-up's scratch (library-owned, see warm_row_job):
// decision, tile sums of one tile, path outputs of a two-node tree.
constexpr size_t kDecisionWarmBytes = 16 + sizeof(float2) * kWarps + 16;
static __device__ __align__(16) char g_warm_decision[kDecisionWarmBytes];

// The decision code warm-up (warp 0 of one CTA, at launch): node_decision
// and follow_path on made-up inputs of item 0's mode -- the root of a
// two-node tree, a row list of K entries with distinct tokens, the first tile
// of the stream warm-up's row (g_warm_row) for the full-vocabulary path,
// zero tile sums -- with every output in g_warm_decision, so that their code
// is in L2 before the first real row reaches it (the L2 holds other data when
// a verify step starts, and fetching the code from HBM after the row's
// stream costs several microseconds).  It touches no caller memory.
static __device__ __noinline__ void warm_decision(const VerifyArgs& A, StreamSmem& S) {
  const int lane = threadIdx.x & 31;
  char* w = g_warm_decision;
  int2* dec = reinterpret_cast<int2*>(w);
  float2* ts = reinterpret_cast<float2*>(w + 16);
  int32_t* outs = reinterpret_cast<int32_t*>(w + 16 + sizeof(float2) * kWarps);
  const int vocab = kTile;
  const int K = A.top_k[0];
  if (lane < kWarps) ts[lane] = make_float2(0.f, 0.f);
  unsigned long long* ntiles = reinterpret_cast<unsigned long long*>(reinterpret_cast<char*>(S.ring) + kNucTiles);
  if (lane == 0) {
    ntiles[0] = 0ull;
    S.aux_key = 0ull;   // nucleus: every token kept, mass 1
    S.aux_d = 1.0;
  }
  for (int e = lane; e < kKMax; e += 32)
    S.rlist[e] = e < K ? mkkey(-0.5f * static_cast<float>(e), (e * 7) % vocab) : 0ull;
  if (lane == 0) {
    S.aux[0] = -1;
    S.aux[1] = 0;
    S.aux[EAGLE_MAX_TREE] = 0;
    S.aux[EAGLE_MAX_TREE + 1] = vocab - 1;
    S.rcount = K > 1 ? K : 1;
    S.rmax = 0.f;
    S.rsum = 1.0;
  }
  __syncwarp();
  NodeJob J;
  J.lrow = g_warm_row;
  J.tsums = ts;
  J.ntiles = ntiles;
  J.dec = dec;
  J.node = 0;
  J.m = 2;
  J.mode = A.mode[0];
  J.K = K;
  J.invT = A.inv_temperature[0];
  J.top_p = static_cast<double>(A.top_p[0]);
  J.seed = A.seed[0];
  J.step = A.step;
  J.c2 = A.rs.exp_scale[0] * kLog2e;
  J.TR = 1;
  J.vocab = vocab;
  node_decision(J, S);
  follow_path(dec, 1, outs, outs + 2, outs + 3, S);
}

// Grid: one cluster per row, then (long rows: stream_warm_up) two clusters
// for the code warm-ups: the first streams the short warm-up row (see
// warm_row_job) and decides node 0 of a two-node tree of its own on it,
// stopping before the arrival; warp 0 of the first CTA of the second runs
// warm_decision at launch.
__global__ void __launch_bounds__(kThreads, 2) verify_kernel(const __grid_constant__ VerifyArgs A) {
  extern __shared__ __align__(128) char smem_raw[];
  StreamSmem& S = *reinterpret_cast<StreamSmem*>(smem_raw);
  const int PC = A.rs.ctas_per_row;
  const int64_t cl = blockIdx.x / PC;
  const int rank = static_cast<int>(blockIdx.x - cl * PC);
  const int64_t rows = static_cast<int64_t>(A.rs.n_items) * A.m;
  pdl_trigger();
  if (cl > rows) {
    if (rank == 0 && threadIdx.x < 32) warm_decision(A, S);
    return;
  }
  const bool warm = cl == rows;
  if (!warm) pdl_wait();          // the warm-ups touch no caller memory
  const RowJob R = warm ? warm_row_job(A.rs, rank) : row_job(A.rs, cl, rank);
  // the row leader's warp 0 prefetches its item's tree (parents, tokens)
  // while the stream runs; the warm-up's tree is root -> one child
  if (rank == 0 && threadIdx.x < 32) {
    if (warm) {
      if (threadIdx.x == 0) {
        S.aux[0] = -1;
        S.aux[1] = 0;
        S.aux[EAGLE_MAX_TREE] = 0;
        S.aux[EAGLE_MAX_TREE + 1] = R.vocab - 1;
      }
    } else {
      for (int i = threadIdx.x; i < A.m; i += 32) {
        cp_async4(S.aux + i, A.parents[R.item] + i);
        cp_async4(S.aux + EAGLE_MAX_TREE + i, A.tokens[R.item] + i);
      }
    }
    cp_async_commit();
  }
  const RowCtx cx = stream_row<true>(R, S);
  if (A.mode[cx.item] == kModeNucleus) {   // every CTA of the cluster, once the row max is in place
    __syncwarp();
    cluster_arrive_release();
    cluster_wait();
    nucleus_cut(R.src, R.vocab, rank, R.PC, R.c2, static_cast<double>(A.top_p[cx.item]), S);
  }
  if (!cx.leader) return;
  if (threadIdx.x >= 32) return;         // warp 0 of the leader from here on
  cp_async_wait_all();
  __syncwarp();
  NodeJob J;
  const int item = cx.item;
  J.lrow = R.src;
  J.tsums = R.tsums;
  J.ntiles = reinterpret_cast<const unsigned long long*>(reinterpret_cast<char*>(S.ring) + kNucTiles);
  J.node = warm ? 0 : static_cast<int>(cx.row - static_cast<int64_t>(item) * A.m);
  J.m = warm ? 2 : A.m;
  J.dec = warm ? reinterpret_cast<int2*>(g_warm_decision) : A.dec + cx.row;
  J.mode = A.mode[item];
  J.K = A.top_k[item];
  J.invT = A.inv_temperature[item];
  J.top_p = static_cast<double>(A.top_p[item]);
  J.seed = A.seed[item];
  J.step = A.step;
  J.c2 = R.c2;
  J.TR = R.TR;
  J.vocab = R.vocab;
  node_decision(J, S);
  if (warm) return;
  if (warp_item_arrive(A, item))
    follow_path(A.dec + static_cast<int64_t>(item) * A.m, A.m, A.accepted[item],
                A.n_accepted + item, A.bonus + item, S);
}

static eagle_status verify_impl(int32_t n_items, const float* const* logits, int64_t row_stride,
                                int32_t vocab, const eagle_tree* trees,
                                const eagle_sampling* params, const uint64_t* seeds,
                                uint64_t step, int32_t* const* accepted, int32_t* n_accepted,
                                int32_t* bonus, void* ws, size_t ws_bytes,
                                cudaStream_t stream) {
  EAGLE_CHECK_ARG(logits && trees && params && seeds && accepted && n_accepted && bonus && ws);
  EAGLE_CHECK_ARG(n_items >= 1 && vocab >= 1);
  EAGLE_CHECK_SHAPE(n_items <= kMaxItems);
  EAGLE_CHECK_ARG(row_stride >= vocab && row_stride % 4 == 0);
  const int m = trees[0].m;
  EAGLE_CHECK_ARG(m >= 1);
  EAGLE_CHECK_SHAPE(m <= EAGLE_MAX_TREE);
  VerifyArgs A;
  memset(&A, 0, sizeof(A));
  int rec_k = 1;
  for (int i = 0; i < n_items; ++i) {
    EAGLE_CHECK_ARG(logits[i] && aligned16(logits[i]) && accepted[i]);
    EAGLE_CHECK_ARG(trees[i].parents && trees[i].tokens && trees[i].m == m);
    const eagle_sampling& p = params[i];
    int mode, k = 0;
    if (p.greedy) {
      mode = kModeGreedy;
      k = 1;
    } else {
      EAGLE_CHECK_ARG(p.temperature > 0.f && p.top_p > 0.f && p.top_p <= 1.f && p.top_k >= 0);
      k = p.top_k >= vocab ? (vocab <= kKMax ? vocab : 0) : p.top_k;
      EAGLE_CHECK_SHAPE(k <= kKMax);
      mode = k > 0 ? kModeTopK : (p.top_p < 1.f ? kModeNucleus : kModeFull);
      EAGLE_CHECK_SHAPE(mode != kModeNucleus || (vocab + kTile - 1) / kTile <= kNucMaxTiles);
    }
    A.mode[i] = mode;
    A.top_k[i] = k;
    A.inv_temperature[i] = p.greedy ? 1.0 : 1.0 / static_cast<double>(p.temperature);
    A.top_p[i] = p.greedy ? 1.f : p.top_p;
    A.parents[i] = trees[i].parents;
    A.tokens[i] = trees[i].tokens;
    A.accepted[i] = accepted[i];
    A.seed[i] = seeds[i];
    A.rs.base[i] = logits[i];
    A.rs.exp_scale[i] = p.greedy ? 1.f : 1.f / p.temperature;
    A.rs.topk[i] = static_cast<int16_t>(mode == kModeTopK || mode == kModeGreedy ? k : 0);
    A.rs.flags[i] = mode == kModeFull ? (kWantSum | kWantTileSums) : mode == kModeNucleus ? kWantSum : 0;
    if (k > rec_k) rec_k = k;
  }
  const StreamLayout L = stream_layout(n_items, m, vocab, kKMax, true, true);
  if (ws_bytes < L.total) return EAGLE_ERR_WORKSPACE_TOO_SMALL;
  const int occ = stream_ctas_per_sm(verify_kernel);
  if (occ <= 0) return EAGLE_ERR_CUDA;
  const int ctas = stream_ctas_per_row(verify_kernel, L, occ, 2);
  if (ctas <= 0) return EAGLE_ERR_CUDA;
  fill_stream(A.rs, L, static_cast<char*>(ws), n_items, m, vocab, row_stride, ctas, true);
  A.m = m;
  A.step = step;
  A.n_accepted = n_accepted;
  A.bonus = bonus;
  A.dec = reinterpret_cast<int2*>(static_cast<char*>(ws) + L.off_dec);
  A.n_warm = stream_warm_up(L.tiles_per_row, ctas) ? 2 : 0;
  return launch_stream(verify_kernel, A, L.n_rows + A.n_warm, ctas, stream);
}

}  // namespace eagle

using namespace eagle;

extern "C" size_t eagle_tree_verify_workspace_size(int32_t n_items, int32_t m, int32_t vocab) {
  if (n_items < 1 || m < 1 || vocab < 1) return 0;
  return stream_layout(n_items, m, vocab, kKMax, true, true).total;
}

extern "C" eagle_status eagle_tree_verify(const float* target_logits, int64_t row_stride,
                                          int32_t vocab, eagle_tree tree,
                                          const eagle_sampling* params, uint64_t seed,
                                          uint64_t step, int32_t* accepted,
                                          int32_t* n_accepted, int32_t* bonus_token, void* ws,
                                          size_t ws_bytes, eagle_stream stream) {
  return verify_impl(1, &target_logits, row_stride, vocab, &tree, params, &seed, step,
                     &accepted, n_accepted, bonus_token, ws, ws_bytes,
                     reinterpret_cast<cudaStream_t>(stream));
}

extern "C" eagle_status eagle_tree_verify_batched(int32_t n_items,
                                                  const float* const* target_logits,
                                                  int64_t row_stride, int32_t vocab,
                                                  const eagle_tree* trees,
                                                  const eagle_sampling* params,
                                                  const uint64_t* seeds, uint64_t step,
                                                  int32_t* const* accepted,
                                                  int32_t* n_accepted, int32_t* bonus_tokens,
                                                  void* ws, size_t ws_bytes,
                                                  eagle_stream stream) {
  return verify_impl(n_items, target_logits, row_stride, vocab, trees, params, seeds, step,
                     accepted, n_accepted, bonus_tokens, ws, ws_bytes,
                     reinterpret_cast<cudaStream_t>(stream));
}
