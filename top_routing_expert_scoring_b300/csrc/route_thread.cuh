// One token's routing, done by one thread over its row of logits read 32 experts at a time:
// scoring, the group limit, Top-k with renormalisation and the token's load-balance
// contributions ["MoE 路由数学" §2.1 and §3.2; "Systems for Mixture-of-Experts Models" §5.3
// router walk-through].  The row comes from a loader (a TMEM chunk in the router GEMM's
// epilogue, or global memory in route_rows_kernel), so the GEMM epilogue and the separate
// kernels compute the same bits.
//
// The arithmetic matches the warp-per-token kernels: sigmoid as 1 / (1 + expf(-g)), selection
// keys s + b (sigmoid) or g (softmax), a group's score = its two largest keys added in float32,
// the (key descending, index ascending) order everywhere, weights exp(g_j - g_top) / sum or
// s_j / sum times the route scale.  Experts are read in index order, so equal keys keep the
// lower index first.
#pragma once

#include "common.cuh"

namespace moe {

constexpr int kRouteMaxChunks = 8;   // E <= 256
constexpr int kRouteMaxK = 8;

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

// Result of one token's routing: the k selected experts in rank order with their weights, and
// the token's statistics terms (its z term; P contributions are produced chunk by chunk by the
// caller through token_probs).
struct RouteThreadOut {
  int idx[kRouteMaxK];
  float w[kRouteMaxK];
  float m;            // max logit
  float se;           // sum_e exp(g_e - m)
  float ss;           // sum_e sigmoid(g_e) (sigmoid scoring)
};

__device__ __forceinline__ float sigm(float g) { return 1.0f / (1.0f + expf(-g)); }

// Passes 1 and 2 over the row.  Loader: void(int chunk, float (&v)[32]) returning experts
// 32*chunk .. 32*chunk+31.  bias: shared-memory copy of the selection bias (sigmoid) or nullptr.
template <typename Loader>
__device__ __forceinline__ void route_thread(const RouteThreadCfg& rc, const float* bias,
                                             Loader load, RouteThreadOut& o) {
  const bool sig = rc.score == MOE_SCORE_SIGMOID;
  // ---- pass 1: max logit, sum of sigmoids, per-chunk two largest keys ------------------
  float m = -INFINITY, ss = 0.f;
  float ct1[kRouteMaxChunks], ct2[kRouteMaxChunks];
#pragma unroll
  for (int c = 0; c < kRouteMaxChunks; ++c) {
    ct1[c] = -INFINITY;
    ct2[c] = -INFINITY;
    if (c >= rc.nc) continue;
    float v[32];
    load(c, v);
#pragma unroll
    for (int i = 0; i < 32; ++i) {
      m = fmaxf(m, v[i]);
      if (sig) {
        const float s = sigm(v[i]);
        ss += s;
        if (rc.cpg > 0) {
          const float key = s + bias[c * 32 + i];
          if (key > ct1[c]) {
            ct2[c] = ct1[c];
            ct1[c] = key;
          } else if (key > ct2[c]) {
            ct2[c] = key;
          }
        }
      }
    }
  }
  // group limit: a group's score is the sum of its two largest keys; a group is kept when
  // fewer than topk_groups groups rank before it (ties: lower group)
  uint32_t kept = 0xffffffffu;
  if (sig && rc.cpg > 0 && rc.select) {
    float gsc[kRouteMaxChunks];
#pragma unroll
    for (int c = 0; c < kRouteMaxChunks; ++c) {
      float a = -INFINITY, b = -INFINITY;       // two largest over the chunks of c's group
#pragma unroll
      for (int c2 = 0; c2 < kRouteMaxChunks; ++c2) {
        if (c2 < rc.nc && c < rc.nc && c2 / rc.cpg == c / rc.cpg) {
          const float x1 = ct1[c2], x2 = ct2[c2];
          if (x1 > a) {
            b = fmaxf(a, x2);
            a = x1;
          } else if (x1 > b) {
            b = x1;
          }
        }
      }
      gsc[c] = a + b;
    }
    kept = 0u;
#pragma unroll
    for (int c = 0; c < kRouteMaxChunks; ++c) {
      if (c >= rc.nc) continue;
      const int q = c / rc.cpg;
      int rank = 0;
#pragma unroll
      for (int c2 = 0; c2 < kRouteMaxChunks; ++c2)
        if (c2 < rc.nc && c2 % rc.cpg == 0 && ranks_before(gsc[c2], c2 / rc.cpg, gsc[c], q))
          ++rank;
      if (rank < rc.topk_groups) kept |= 1u << c;
    }
  }
  // ---- pass 2: sum of exp(g - m); Top-k over the kept experts -------------------------
  float se = 0.f;
  float bk[kRouteMaxK], bv[kRouteMaxK];
  int bi[kRouteMaxK];
#pragma unroll
  for (int j = 0; j < kRouteMaxK; ++j) {
    bk[j] = -INFINITY;
    bv[j] = 0.f;
    bi[j] = 0x7fffffff;
  }
#pragma unroll
  for (int c = 0; c < kRouteMaxChunks; ++c) {
    if (c >= rc.nc) continue;
    float v[32];
    load(c, v);
    const bool live = (kept >> c) & 1u;
#pragma unroll
    for (int i = 0; i < 32; ++i) {
      se += expf(v[i] - m);
      if (!rc.select || !live) continue;
      const int e = c * 32 + i;
      float key, val;
      if (sig) {
        val = sigm(v[i]);
        key = val + bias[e];
      } else {
        val = v[i];
        key = v[i];
      }
      if (ranks_before(key, e, bk[kRouteMaxK - 1], bi[kRouteMaxK - 1])) {
        // insertion into the sorted list, from the bottom up
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
    }
  }
  o.m = m;
  o.se = se;
  o.ss = ss;
  if (!rc.select) return;
  // weights of the k selected experts, in rank order
  float num[kRouteMaxK], den = 0.f;
#pragma unroll
  for (int j = 0; j < kRouteMaxK; ++j) {
    num[j] = 0.f;
    if (j >= rc.k) continue;
    num[j] = sig ? bv[j] : expf(bv[j] - bv[0]);
    den += num[j];
  }
  if (!rc.renorm) den = sig ? 1.f : se * expf(m - bv[0]);
#pragma unroll
  for (int j = 0; j < kRouteMaxK; ++j) {
    o.idx[j] = bi[j];
    o.w[j] = (num[j] / den) * rc.scale;
  }
}

// Pass 3: the token's P contributions for one 32-expert chunk (softmax(g)_e, or s_e / sum s).
__device__ __forceinline__ void token_probs(const RouteThreadCfg& rc, const RouteThreadOut& o,
                                            const float (&v)[32], float (&p)[32]) {
#pragma unroll
  for (int i = 0; i < 32; ++i)
    p[i] = rc.score == MOE_SCORE_SIGMOID ? sigm(v[i]) / o.ss : expf(v[i] - o.m) / o.se;
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

}  // namespace moe
