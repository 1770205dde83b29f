// One token's routing, split over four threads that each own a quarter of its logits (whole
// 32-expert chunks): scoring, the group limit, Top-k with renormalisation and the token's
// load-balance contributions ["MoE 路由数学" §2.1 and §3.2; "Systems for Mixture-of-Experts
// Models" §5.3 router walk-through].
//
// The four threads of a token are lanes of four warps with the same TMEM lane quarter, so in
// the router GEMM's epilogue each reads its chunks straight from the accumulator; the same
// phases run from global memory in route_rows_stats_kernel, so the GEMM epilogue and the
// separate statistics kernel compute the same bits.  Phases (shared memory between them):
//   A  per thread: max logit, sum of exp(g - max) (kept online across its chunks), sum of
//      sigmoids, and each chunk's two largest selection keys;
//   B  per thread: the token's max, exp-sum and sigmoid-sum (its four parts combined in thread
//      order), the group limit, the top-k of its kept chunks, and its P contributions;
//   C  one thread per token: the k best of the four lists, and the weights.
// The arithmetic matches the warp-per-token kernels where it decides: sigmoid as
// 1 / (1 + expf(-g)), selection keys s + b (sigmoid) or g (softmax), a group's score = its two
// largest keys added in float32, the (key descending, index ascending) order everywhere, and
// weights exp(g_j - g_top) / sum or s_j / sum times the route scale.
#pragma once

#include "common.cuh"

namespace moe {

constexpr int kRouteMaxChunks = 8;   // E <= 256
constexpr int kRouteMaxK = 8;
constexpr int kRouteSubs = 4;        // threads per token
constexpr int kRouteTile = 128;      // tokens per tile

struct RouteThreadCfg {
  int nc;             // E / 32
  int k;
  int score;          // MOE_SCORE_*
  int cpg;            // 32-expert chunks per group (group limit on), else 0
  int topk_groups;
  int renorm;
  float scale;
  int select;         // 1: choose experts and weights; 0: statistics only (given selection)
};

// Shared memory of the phases for one tile of 128 tokens.  The token slot is the innermost
// index everywhere, so the 32 lanes of a warp (32 consecutive slots) touch 32 consecutive words.
struct RouteSmem {
  float bias[256];
  float stat[kRouteSubs][3][kRouteTile];          // per thread part: max, exp-sum, sigmoid-sum
  float ctop[kRouteMaxChunks][2][kRouteTile];     // per chunk: two largest keys
  float ckey[kRouteSubs][kRouteMaxK][kRouteTile]; // per thread part: its top-k list
  int cidx[kRouteSubs][kRouteMaxK][kRouteTile];
  float cval[kRouteSubs][kRouteMaxK][kRouteTile];
  float P[4][256];                                // per TMEM lane quarter: column sums
  int cnt[256];
  float Z[4];
};

// 1 / (1 + e^-g); __frcp_rn is the correctly rounded reciprocal, the same bits as the
// division 1.0f / x, without its general-divisor path
__device__ __forceinline__ float sigm(float g) { return __frcp_rn(1.0f + expf(-g)); }

__device__ __forceinline__ void route_chunk_range(const RouteThreadCfg& rc, int sub, int& c0,
                                                  int& c1) {
  c0 = sub * rc.nc / kRouteSubs;
  c1 = (sub + 1) * rc.nc / kRouteSubs;
}

// Insertion of (key, e, val) into the descending list (bk, bi, bv) of kRouteMaxK entries, from
// the bottom up; equal keys keep the lower index first.
__device__ __forceinline__ void topk_insert(float key, int e, float val, float (&bk)[kRouteMaxK],
                                            int (&bi)[kRouteMaxK], float (&bv)[kRouteMaxK]) {
#pragma unroll
  for (int j = kRouteMaxK - 1; j >= 0; --j) {
    const bool here = ranks_before(key, e, bk[j], bi[j]);
    const bool above = j == 0 ? true : ranks_before(key, e, bk[j - 1], bi[j - 1]);
    if (here) {
      if (above && j > 0) {
        bk[j] = bk[j - 1];
        bi[j] = bi[j - 1];
        bv[j] = bv[j - 1];
      } else {
        bk[j] = key;
        bi[j] = e;
        bv[j] = val;
      }
    }
  }
}

// Column sums of a warp's 32 x 32 block (lane = token, register = expert of the chunk):
// afterwards lane l holds the sum over the 32 lanes of column l, added in a fixed butterfly
// order (deterministic).
__device__ __forceinline__ float warp_column_sum(float (&v)[32]) {
  const int lane = threadIdx.x & 31;
#pragma unroll
  for (int off = 16; off >= 1; off >>= 1) {
    const bool upper = (lane & off) != 0;
#pragma unroll
    for (int i = 0; i < off; ++i) {
      const float send = upper ? v[i] : v[i + off];
      const float keep = upper ? v[i + off] : v[i];
      v[i] = keep + __shfl_xor_sync(0xffffffffu, send, off);
    }
  }
  return v[0];
}

// Phase A for this thread's chunks of token slot r.  Loader: void(int chunk, float (&v)[32]).
// Also hands each chunk to `each(c, v)` (the epilogue writes the logits from there).
template <typename Loader, typename Each>
__device__ __forceinline__ void route_phase_a(const RouteThreadCfg& rc, RouteSmem& sm, int r,
                                              int sub, Loader load, Each each) {
  const bool sig = rc.score == MOE_SCORE_SIGMOID;
  const bool limit = sig && rc.cpg > 0 && rc.select;
  int c0, c1;
  route_chunk_range(rc, sub, c0, c1);
  float m = -INFINITY, se = 0.f, ss = 0.f;
#pragma unroll 1
  for (int c = c0; c < c1; ++c) {
    float v[32];
    load(c, v);
    each(c, v);
    float cm = v[0];
#pragma unroll
    for (int i = 1; i < 32; ++i) cm = fmaxf(cm, v[i]);
    if (cm > m) {                      // online exp-sum: rescale to the new maximum
      se = (m == -INFINITY) ? 0.f : se * expf(m - cm);
      m = cm;
    }
    float a = -INFINITY, b = -INFINITY;
#pragma unroll
    for (int i = 0; i < 32; ++i) {
      se += expf(v[i] - m);
      if (sig) {
        const float s = sigm(v[i]);
        ss += s;
        if (limit) {
          const float key = s + sm.bias[c * 32 + i];
          if (key > a) {
            b = a;
            a = key;
          } else if (key > b) {
            b = key;
          }
        }
      }
    }
    sm.ctop[c][0][r] = a;
    sm.ctop[c][1][r] = b;
  }
  sm.stat[sub][0][r] = m;
  sm.stat[sub][1][r] = se;
  sm.stat[sub][2][r] = ss;
}

// The token's max, exp-sum and sigmoid-sum from the four parts, in thread order.
struct RouteTotals {
  float m, se, ss;
};
__device__ __forceinline__ RouteTotals route_totals(const RouteSmem& sm, int r) {
  RouteTotals t{-INFINITY, 0.f, 0.f};
#pragma unroll
  for (int s = 0; s < kRouteSubs; ++s) t.m = fmaxf(t.m, sm.stat[s][0][r]);
#pragma unroll
  for (int s = 0; s < kRouteSubs; ++s) {
    const float ms = sm.stat[s][0][r];
    if (ms != -INFINITY) t.se += sm.stat[s][1][r] * expf(ms - t.m);
    t.ss += sm.stat[s][2][r];
  }
  return t;
}

// Phase B: the group limit (kept chunks), this thread's P contributions (column sums of the
// warp's 32 tokens into sm.P[q]) over its own chunks, and the top-k of its share of the
// token's kept chunks into the candidate lists.  The kept chunks are dealt out in chunk order
// (the j-th to thread part j mod 4), so every part of a token gets the same count whichever
// groups the token keeps, and a warp's threads insert in step; load_row(c, v) reads chunk c of
// the thread's own token row (any chunk, per thread).  live: the slot holds a token.
template <typename Loader, typename RowLoader>
__device__ __forceinline__ void route_phase_b(const RouteThreadCfg& rc, RouteSmem& sm, int r,
                                              int sub, int q, bool live, Loader load,
                                              RowLoader load_row) {
  const bool sig = rc.score == MOE_SCORE_SIGMOID;
  const bool limit = sig && rc.cpg > 0 && rc.select;
  const RouteTotals tot = route_totals(sm, r);
  uint32_t kept = 0xffffffffu;
  if (limit) {
    float gsc[kRouteMaxChunks];
    const int ng = rc.nc / rc.cpg;
#pragma unroll 1
    for (int g = 0; g < ng; ++g) {
      float a = -INFINITY, b = -INFINITY;        // two largest over the group's chunks
      for (int c = g * rc.cpg; c < (g + 1) * rc.cpg; ++c) {
        const float x1 = sm.ctop[c][0][r], x2 = sm.ctop[c][1][r];
        if (x1 > a) {
          b = fmaxf(a, x2);
          a = x1;
        } else if (x1 > b) {
          b = x1;
        }
      }
      gsc[g] = a + b;
    }
    kept = 0u;
#pragma unroll 1
    for (int g = 0; g < ng; ++g) {
      int rank = 0;
      for (int g2 = 0; g2 < ng; ++g2) rank += ranks_before(gsc[g2], g2, gsc[g], g) ? 1 : 0;
      if (rank < rc.topk_groups)
        for (int c = g * rc.cpg; c < (g + 1) * rc.cpg; ++c) kept |= 1u << c;
    }
  }
  int c0, c1;
  route_chunk_range(rc, sub, c0, c1);
  float bk[kRouteMaxK], bv[kRouteMaxK];
  int bi[kRouteMaxK];
#pragma unroll
  for (int j = 0; j < kRouteMaxK; ++j) {
    bk[j] = -INFINITY;
    bv[j] = 0.f;
    bi[j] = 0x7fffffff;
  }
  const float inv_ss = 1.0f / tot.ss, inv_se = 1.0f / tot.se;
#pragma unroll 1
  for (int c = c0; c < c1; ++c) {
    float v[32], pr[32];
    load(c, v);
#pragma unroll
    for (int i = 0; i < 32; ++i) {
      const float s = sig ? sigm(v[i]) : 0.f;
      pr[i] = live ? (sig ? s * inv_ss : expf(v[i] - tot.m) * inv_se) : 0.f;
    }
    sm.P[q][c * 32 + (threadIdx.x & 31)] = warp_column_sum(pr);
  }
  if (rc.select) {
    // this part's share of the kept chunks: every kRouteSubs-th set bit, from bit `sub`
    uint32_t mine = 0u;
    {
      uint32_t rest = live ? kept & ((rc.nc >= 32) ? 0xffffffffu : ((1u << rc.nc) - 1u)) : 0u;
      for (int j = 0; rest; ++j) {
        const uint32_t low = rest & (0u - rest);
        if ((j % kRouteSubs) == sub) mine |= low;
        rest ^= low;
      }
    }
#pragma unroll 1
    while (__any_sync(0xffffffffu, mine != 0u)) {
      if (mine) {
        const int c = __ffs(mine) - 1;
        mine &= mine - 1u;
        float v[32];
        load_row(c, v);
#pragma unroll
        for (int i = 0; i < 32; ++i) {
          const int e = c * 32 + i;
          const float s = sig ? sigm(v[i]) : 0.f;
          const float key = sig ? s + sm.bias[e] : v[i];
          const float val = sig ? s : v[i];
          if (ranks_before(key, e, bk[kRouteMaxK - 1], bi[kRouteMaxK - 1]))
            topk_insert(key, e, val, bk, bi, bv);
        }
      }
    }
  }
#pragma unroll
  for (int j = 0; j < kRouteMaxK; ++j) {
    sm.ckey[sub][j][r] = bk[j];
    sm.cidx[sub][j][r] = bi[j];
    sm.cval[sub][j][r] = bv[j];
  }
}

// Phase C (one thread per token): the k best of the four candidate lists, in rank order, and
// the weights.  Returns the token's lse for the z-loss.
__device__ __forceinline__ float route_phase_c(const RouteThreadCfg& rc, const RouteSmem& sm,
                                               int r, int (&idx)[kRouteMaxK],
                                               float (&w)[kRouteMaxK]) {
  const bool sig = rc.score == MOE_SCORE_SIGMOID;
  const RouteTotals tot = route_totals(sm, r);
  float bk[kRouteMaxK], bv[kRouteMaxK];
  int bi[kRouteMaxK];
#pragma unroll
  for (int j = 0; j < kRouteMaxK; ++j) {
    bk[j] = sm.ckey[0][j][r];
    bi[j] = sm.cidx[0][j][r];
    bv[j] = sm.cval[0][j][r];
  }
#pragma unroll 1
  for (int s = 1; s < kRouteSubs; ++s) {
    for (int j = 0; j < kRouteMaxK; ++j) {      // each list is sorted: stop at its first miss
      const float key = sm.ckey[s][j][r];
      const int e = sm.cidx[s][j][r];
      if (!ranks_before(key, e, bk[kRouteMaxK - 1], bi[kRouteMaxK - 1])) break;
      topk_insert(key, e, sm.cval[s][j][r], bk, bi, bv);
    }
  }
  float num[kRouteMaxK], den = 0.f;
#pragma unroll
  for (int j = 0; j < kRouteMaxK; ++j) {
    num[j] = 0.f;
    if (j >= rc.k) continue;
    num[j] = sig ? bv[j] : expf(bv[j] - bv[0]);
    den += num[j];
  }
  if (!rc.renorm) den = sig ? 1.f : tot.se * expf(tot.m - bv[0]);
#pragma unroll
  for (int j = 0; j < kRouteMaxK; ++j) {
    idx[j] = bi[j];
    w[j] = (num[j] / den) * rc.scale;
  }
  return tot.m + logf(tot.se);
}

}  // namespace moe
