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

enum : int { kModeGreedy = 0, kModeTopK = 1, kModeFull = 2 };

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

// p(t) under the full-vocabulary target distribution (lane-local).
__device__ __forceinline__ double full_prob(const float* lrow, int t, double rowmax, double invT,
                                            double inv_zsum) {
  return exp_d((static_cast<double>(__ldg(lrow + t)) - rowmax) * invT) * inv_zsum;
}

// Decision of the walk at one node (warp 0 of the node's row leader): the
// child accepted there (-1 if none) and the token emitted when the walk stops
// there.  It depends only on the node's own row, its children and the
// uniforms keyed by (seed, step, node, j), so every node decides on its own,
// in parallel, and the item's final step follows the decisions from the root.
static __device__ __noinline__ void node_decision(const VerifyArgs& A, int64_t row, int item,
                                                  StreamSmem& S) {
  const int lane = threadIdx.x & 31;
  const int m = A.m;
  const int node = static_cast<int>(row - static_cast<int64_t>(item) * m);
  const int mode = A.mode[item];
  const double invT = A.inv_temperature[item];
  const double top_p = static_cast<double>(A.top_p[item]);
  const int K = A.top_k[item];
  const uint64_t seed = A.seed[item];
  const int* parents = S.aux;                   // prefetched at kernel start
  const int* tokens = S.aux + EAGLE_MAX_TREE;
  const int TR = A.rs.tiles_per_row;

  int* kn = reinterpret_cast<int*>(S.ring[0]);          // children (node ids), node order
  int* kt = kn + EAGLE_MAX_TREE;                         // their tokens
  double* kp = reinterpret_cast<double*>(S.ring[1]);     // kept probabilities, by rank
  int* kid = reinterpret_cast<int*>(kp + kKMax);         // kept ids, by rank
  double* sp = reinterpret_cast<double*>(kid + kKMax);   // kept probabilities sorted by id
  int* sid = reinterpret_cast<int*>(sp + kKMax);

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
    const float* lrow = A.rs.base[item] + static_cast<int64_t>(node) * A.rs.row_stride;
    double rowmax = 0.0, zsum = 1.0, izsum = 1.0;
    int nkeep = 0;
    if (mode == kModeTopK) {
      int cnt = S.rcount;
      if (cnt > K) cnt = K;
      double z[2], pr[2];
      int id[2];
      const double z0 = static_cast<double>(key_v(S.rlist[0])) * invT;
#pragma unroll
      for (int hh = 0; hh < 2; ++hh) {
        const int e = lane + 32 * hh;
        if (e < cnt) {
          z[hh] = static_cast<double>(key_v(S.rlist[e])) * invT;
          id[hh] = key_i(S.rlist[e]);
          pr[hh] = exp_d(z[hh] - z0);
        } else {
          pr[hh] = 0.0;
          id[hh] = kNoIndex;
        }
      }
      const double itot = 1.0 / warp_sum_d(pr[0] + pr[1]);
      pr[0] *= itot;
      pr[1] *= itot;
      nkeep = cnt;
      if (top_p < 1.0) {
        // entries are in probability order; keep the shortest prefix whose
        // cumulative mass reaches top_p (the crossing entry included)
        const double c0 = warp_incl_scan_d(pr[0]);
        const double t0 = __shfl_sync(0xffffffffu, c0, 31);
        const double c1 = warp_incl_scan_d(pr[1]) + t0;
        const unsigned b0 = __ballot_sync(0xffffffffu, lane < cnt && c0 >= top_p);
        const unsigned b1 = __ballot_sync(0xffffffffu, lane + 32 < cnt && c1 >= top_p);
        int last = cnt - 1;
        if (b0) last = __ffs(b0) - 1;
        else if (b1) last = 32 + __ffs(b1) - 1;
        nkeep = last + 1;
        if (lane > last) pr[0] = 0.0;
        if (lane + 32 > last) pr[1] = 0.0;
        const double itot2 = 1.0 / warp_sum_d(pr[0] + pr[1]);
        pr[0] *= itot2;
        pr[1] *= itot2;
      }
      kp[lane] = pr[0];
      kid[lane] = lane < nkeep ? id[0] : kNoIndex;
      kp[lane + 32] = pr[1];
      kid[lane + 32] = lane + 32 < nkeep ? id[1] : kNoIndex;
      __syncwarp();
    } else {  // full vocabulary
      rowmax = static_cast<double>(S.rmax);
      zsum = S.rsum;
      izsum = 1.0 / zsum;
    }
    auto prob_of = [&](int t) -> double {  // lane-local
      if (mode == kModeTopK) {
        double v = 0.0;
        for (int e = 0; e < nkeep; ++e)
          if (kid[e] == t) v = kp[e];
        return v;
      }
      return full_prob(lrow, t, rowmax, invT, izsum);
    };

    // ---- children in node order, 32 at a time: child j is accepted iff
    // u_j (1 - rho_j) < p(token_j), rho_j = mass of the children before it
    // (all of them rejected when j is reached)
    double rho_all = 0.0;
    for (int b = 0; b < nk && child < 0; b += 32) {
      const int j = b + lane;
      const bool valid = j < nk;
      const double pt = valid ? prob_of(kt[j]) : 0.0;
      const double incl = warp_incl_scan_d(pt);
      const double rho = rho_all + (incl - pt);
      const double u = valid ? philox_uniform(seed, A.step, static_cast<uint32_t>(node),
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
          philox_uniform(seed, A.step, static_cast<uint32_t>(node), kResidualChild) *
          (1.0 - rho_all);
      auto is_rejected = [&](int t) {
        for (int r = 0; r < nk; ++r)
          if (kt[r] == t) return true;
        return false;
      };
      if (mode == kModeTopK) {
        // kept entries sorted by token id (rank by counting)
#pragma unroll
        for (int hh = 0; hh < 2; ++hh) {
          const int e = lane + 32 * hh;
          if (e < nkeep) {
            int r = 0;
            for (int f = 0; f < nkeep; ++f) r += kid[f] < kid[e] ? 1 : 0;
            sid[r] = kid[e];
            sp[r] = is_rejected(kid[e]) ? 0.0 : kp[e];
          }
        }
        __syncwarp();
        int pick = -1, last = -1;
        double cum = 0.0;
        for (int hh = 0; hh < 2 && pick < 0; ++hh) {
          const int r = lane + 32 * hh;
          const double mass = r < nkeep ? sp[r] : 0.0;
          const double incl = warp_incl_scan_d(mass) + cum;
          const unsigned bal = __ballot_sync(0xffffffffu, r < nkeep && incl > thr);
          if (bal) pick = 32 * hh + __ffs(bal) - 1;
          const unsigned nz = __ballot_sync(0xffffffffu, r < nkeep && mass > 0.0);
          if (nz) last = 32 * hh + 31 - __clz(nz);
          cum = __shfl_sync(0xffffffffu, incl, 31);
        }
        if (pick < 0) pick = last >= 0 ? last : nkeep - 1;
        bonus = sid[pick];
      } else {
        // tile masses (tile sums were taken relative to each tile's max)
        const float2* ts = A.rs.tile_sums + row * TR * kWarps;
        const double c2 = static_cast<double>(A.rs.exp_scale[item]) * 1.4426950408889634;
        double cum = 0.0;
        int tile = -1;
        double before_tile = 0.0;
        for (int base = 0; base < TR && tile < 0; base += 32) {
          const int t = base + lane;
          double mass = 0.0;
          if (t < TR) {
            // combine the per-warp partials of tile t (max, sum of 2^((x - max) c2))
            const float2* tw = ts + static_cast<int64_t>(t) * kWarps;
            for (int w = 0; w < kWarps; ++w) {
              const float2 v = __ldcg(tw + w);
              if (v.y > 0.f)
                mass += static_cast<double>(v.y) *
                        static_cast<double>(ex2((v.x - static_cast<float>(rowmax)) * static_cast<float>(c2)));
            }
            mass *= izsum;
            for (int r = 0; r < nk; ++r) {   // rejected tokens of this tile, each once
              const int rt = kt[r];
              if (rt / kTile != t) continue;
              bool first = true;
              for (int r2 = 0; r2 < r; ++r2) first &= kt[r2] != rt;
              if (first) mass -= full_prob(lrow, rt, rowmax, invT, izsum);
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
          if (t < A.rs.vocab && !is_rejected(t)) {
            const float x = __ldg(lrow + t);
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
  if (lane == 0) A.dec[row] = make_int2(child, bonus);
  __syncwarp();
}

// The item's final step (warp 0 of the CTA whose row arrived last): follow
// the decisions from the root.
static __device__ __noinline__ void follow_path(const VerifyArgs& A, int item, StreamSmem& S) {
  const int lane = threadIdx.x & 31;
  const int m = A.m;
  int2* dec = reinterpret_cast<int2*>(S.ring[0]);
  const int2* src = A.dec + static_cast<int64_t>(item) * m;
  for (int i = lane; i < m; i += 32) dec[i] = __ldcg(src + i);
  __syncwarp();
  if (lane == 0) {
    int32_t* acc = A.accepted[item];
    int node = 0, n = 0;
    acc[0] = 0;
    for (int guard = 0; guard < m; ++guard) {
      const int c = dec[node].x;
      if (c <= node || c >= m) break;   // -1: the walk stops here
      node = c;
      acc[++n] = node;
    }
    A.n_accepted[item] = n;
    A.bonus[item] = dec[node].y;
  }
  __syncwarp();
}

__global__ void __launch_bounds__(kThreads, 2) verify_kernel(const __grid_constant__ VerifyArgs A) {
  extern __shared__ __align__(128) char smem_raw[];
  StreamSmem& S = *reinterpret_cast<StreamSmem*>(smem_raw);
  // the row leader's warp 0 prefetches its item's tree (parents, tokens)
  // while the stream runs
  const int PC = A.rs.ctas_per_row;
  if (blockIdx.x % PC == 0 && threadIdx.x < 32) {
    const int item = static_cast<int>((blockIdx.x / PC) / A.m);
    for (int i = threadIdx.x; i < A.m; i += 32) {
      cp_async4(S.aux + i, A.parents[item] + i);
      cp_async4(S.aux + EAGLE_MAX_TREE + i, A.tokens[item] + i);
    }
    cp_async_commit();
  }
  const RowCtx cx = stream_row(A.rs, S);
  if (!cx.leader) return;
  if (threadIdx.x < 32) {
    cp_async_wait_all();
    __syncwarp();
    node_decision(A, cx.row, cx.item, S);
  }
  if (item_arrive(A.rs, S, cx.item) && threadIdx.x < 32) follow_path(A, cx.item, S);
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
  bool any_full = false;
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
      EAGLE_CHECK_SHAPE(k > 0 || p.top_p >= 1.f);  // nucleus needs a top_k bound
      mode = k > 0 ? kModeTopK : kModeFull;
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
    A.rs.topk[i] = static_cast<int16_t>(mode == kModeFull ? 0 : k);
    A.rs.flags[i] = mode == kModeFull ? (kWantSum | kWantTileSums) : 0;
    if (k > rec_k) rec_k = k;
    any_full |= mode == kModeFull;
  }
  (void)any_full;
  const StreamLayout L = stream_layout(n_items, m, vocab, kKMax, true, true);
  if (ws_bytes < L.total) return EAGLE_ERR_WORKSPACE_TOO_SMALL;
  const int occ = stream_ctas_per_sm(verify_kernel);
  if (occ <= 0) return EAGLE_ERR_CUDA;
  const int ctas = stream_ctas_per_row(verify_kernel, L, occ);
  if (ctas <= 0) return EAGLE_ERR_CUDA;
  fill_stream(A.rs, L, static_cast<char*>(ws), n_items, m, vocab, row_stride, ctas, true);
  A.m = m;
  A.step = step;
  A.n_accepted = n_accepted;
  A.bonus = bonus;
  A.dec = reinterpret_cast<int2*>(static_cast<char*>(ws) + L.off_dec);
  return launch_stream(verify_kernel, A, L.n_rows, ctas, stream);
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
