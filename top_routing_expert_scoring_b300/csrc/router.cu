// Router kernels: logits, scoring + Top-k + weights, and the load-balance statistics.
//
//   g = x W_gate                                   ["MoE 路由数学" §2.1]
//   softmax:  p = softmax(g), S = TopK(g, k), w = p_S / sum_S p     (same section)
//   sigmoid:  s = sigmoid(g), selection on s + b, groups limited by the sum of each group's
//             two best biased scores, w = route_scale * s_S / sum_S s
//                                                  ["Systems for Mixture-of-Experts Models"
//                                                   §5.3 router walk-through]
//   stats:    f_i, P_i, L = E sum f_i P_i, z = mean (logsumexp g)^2
//                                                  ["MoE 路由数学" §3.2; "Mixture of Experts 架构"
//                                                   load_balancing_loss / router_z_loss blocks]
#include <cuda_bf16.h>

#include <cstdlib>
#include <cstring>

#include "common.cuh"
#include "kernels.h"
#include "route_thread.cuh"

namespace moe {

// ------------------------------------------------------------------------------------------
// Logits on CUDA cores, general case (float32 path, or shapes the other two kernels do not
// take): one CTA computes a 32-token x 64-expert tile, K in chunks of 32.
// ------------------------------------------------------------------------------------------
template <typename T>
__global__ void __launch_bounds__(256) router_logits_simt(const T* __restrict__ x,
                                                         const T* __restrict__ w,
                                                         float* __restrict__ g, int Tn, int d,
                                                         int E) {
  pdl_prologue();
  constexpr int TT = 32, TE = 64, TK = 32;
  __shared__ float xs[TK][TT + 1];
  __shared__ float wsm[TK][TE + 1];
  const int t0 = blockIdx.x * TT, e0 = blockIdx.y * TE;
  const int tid = threadIdx.x;
  const int tx = tid % 16, ty = tid / 16;      // ty: token pair, tx: 4 experts
  float acc[2][4] = {};
  for (int k0 = 0; k0 < d; k0 += TK) {
    for (int i = tid; i < TT * TK; i += 256) {
      int r = i / TK, kk = i % TK;
      int t = t0 + r, c = k0 + kk;
      xs[kk][r] = (t < Tn && c < d) ? to_f32(x[(size_t)t * d + c]) : 0.f;
    }
    for (int i = tid; i < TE * TK; i += 256) {
      int r = i / TK, kk = i % TK;
      int e = e0 + r, c = k0 + kk;
      wsm[kk][r] = (e < E && c < d) ? to_f32(w[(size_t)e * d + c]) : 0.f;
    }
    __syncthreads();
#pragma unroll 8
    for (int kk = 0; kk < TK; ++kk) {
      float a0 = xs[kk][ty * 2], a1 = xs[kk][ty * 2 + 1];
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        float b = wsm[kk][tx * 4 + j];
        acc[0][j] = fmaf(a0, b, acc[0][j]);
        acc[1][j] = fmaf(a1, b, acc[1][j]);
      }
    }
    __syncthreads();
  }
#pragma unroll
  for (int r = 0; r < 2; ++r) {
    int t = t0 + ty * 2 + r;
    if (t >= Tn) continue;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      int e = e0 + tx * 4 + j;
      if (e < E) g[(size_t)t * E + e] = acc[r][j];
    }
  }
}

// ------------------------------------------------------------------------------------------
// Logits for a small expert count (E <= 32, bf16): the router weights stay in shared memory
// and each warp streams TPW token rows at once with 16-byte loads (two for E <= 8: each weight
// vector read from shared memory then serves both; one for more experts, to stay within the
// registers), keeping E partial dot products per token and lane; a butterfly reduction (fixed
// order) finishes them.  HBM-bound on reading x.
// ------------------------------------------------------------------------------------------
template <int EP>
__global__ void __launch_bounds__(512, 1) router_logits_stream(const uint4* __restrict__ x,
                                                           const uint4* __restrict__ w,
                                                           float* __restrict__ g, int Tn,
                                                           int d8, int E) {
  constexpr int TPW = EP <= 8 ? 2 : 1;
  pdl_prologue();
  extern __shared__ uint4 wsm[];                  // [EP][d8]: 8 bf16 per uint4
  for (int i = threadIdx.x; i < EP * d8; i += blockDim.x) {
    const int e = i / d8;
    wsm[i] = e < E ? w[i] : make_uint4(0u, 0u, 0u, 0u);
  }
  __syncthreads();
  const int lane = threadIdx.x & 31;
  const int warps = (gridDim.x * blockDim.x) >> 5;
  const int groups = (Tn + TPW - 1) / TPW;
  for (int tg = (blockIdx.x * blockDim.x + threadIdx.x) >> 5; tg < groups; tg += warps) {
    const int t0 = TPW * tg;
    const int nt = min(TPW, Tn - t0);
    float acc[TPW][EP];
#pragma unroll
    for (int q = 0; q < TPW; ++q)
#pragma unroll
      for (int e = 0; e < EP; ++e) acc[q][e] = 0.f;
    const uint4* xr[TPW];
#pragma unroll
    for (int q = 0; q < TPW; ++q) xr[q] = x + (size_t)(t0 + (q < nt ? q : 0)) * d8;
    // per token four independent 16-byte loads in flight per lane, then their products in order
    for (int c0 = lane; c0 < d8; c0 += 128) {
      uint4 xv[TPW][4];
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        const bool in = c0 + 32 * u < d8;
#pragma unroll
        for (int q = 0; q < TPW; ++q)
          xv[q][u] = in ? __ldg(xr[q] + c0 + 32 * u) : make_uint4(0u, 0u, 0u, 0u);
      }
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        const int c = c0 + 32 * u;
        if (c >= d8) break;
        float xf[TPW][8];
#pragma unroll
        for (int q = 0; q < TPW; ++q) {
          const __nv_bfloat162* xh = reinterpret_cast<const __nv_bfloat162*>(&xv[q][u]);
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            const float2 f = __bfloat1622float2(xh[i]);
            xf[q][2 * i] = f.x;
            xf[q][2 * i + 1] = f.y;
          }
        }
#pragma unroll
        for (int e = 0; e < EP; ++e) {
          const uint4 wv = wsm[e * d8 + c];
          const __nv_bfloat162* wh = reinterpret_cast<const __nv_bfloat162*>(&wv);
#pragma unroll
          for (int q = 0; q < TPW; ++q) {
            float a = acc[q][e];
#pragma unroll
            for (int i = 0; i < 4; ++i) {
              const float2 f = __bfloat1622float2(wh[i]);
              a = fmaf(xf[q][2 * i], f.x, a);
              a = fmaf(xf[q][2 * i + 1], f.y, a);
            }
            acc[q][e] = a;
          }
        }
      }
    }
#pragma unroll
    for (int q = 0; q < TPW; ++q) {
      if (q >= nt) break;
#pragma unroll
      for (int e = 0; e < EP; ++e) acc[q][e] = warp_sum(acc[q][e]);
#pragma unroll
      for (int e = 0; e < EP; ++e)
        if (lane == e && e < E) g[(size_t)(t0 + q) * E + e] = acc[q][e];
    }
  }
}

template <int EP>
static cudaError_t launch_stream(const moe_config& c, const void* x, const void* w_gate,
                                 float* logits, cudaStream_t s) {
  const int d8 = c.d_model / 8;
  const size_t smem = (size_t)EP * d8 * sizeof(uint4);
  cudaError_t e = smem_attr_once(reinterpret_cast<const void*>(router_logits_stream<EP>),
                                 200 * 1024);
  if (e != cudaSuccess) return e;
  // one CTA of 16 warps per SM: the router weights are staged once per SM, and each warp
  // then streams its share of the token rows
  int blocks = ceil_div(c.T, 16);
  if (blocks > num_sms()) blocks = num_sms();
  launch_pdl(router_logits_stream<EP>, blocks, 512, smem, s, (const uint4*)x, (const uint4*)w_gate, logits,
                                                     c.T, d8, c.E);
  return cudaGetLastError();
}

// ------------------------------------------------------------------------------------------
// Logits for decode-sized batches (bf16): one CTA per (expert, group of TP tokens) streams
// that expert's router row (16-byte loads; its 8 warps take one eighth of d each) and forms
// the group's dot products against the token rows, which stay in L1/L2; the 8 partial sums are
// added in a fixed order.  Spreads the work over many SMs instead of one tile; the router row
// is re-read from L2 once per token group and x once per expert, so this is for small E or
// very small T.
// ------------------------------------------------------------------------------------------
template <int TP>
__global__ void __launch_bounds__(256) router_logits_few(const uint4* __restrict__ x,
                                                        const uint4* __restrict__ w,
                                                        float* __restrict__ g, int Tn, int d8,
                                                        int E) {
  pdl_prologue();
  __shared__ float part[8][TP];
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int e = blockIdx.x;
  const int t_base = blockIdx.y * TP;
  x += (size_t)t_base * d8;
  Tn -= t_base;
  float acc[TP];
#pragma unroll
  for (int t = 0; t < TP; ++t) acc[t] = 0.f;
  const uint4* wr = w + (size_t)e * d8;
  const int per = ceil_div(d8, 8);
  const int c0 = warp * per, c1 = min(d8, c0 + per);
  for (int c = c0 + lane; c < c1; c += 32) {
    const uint4 wv = __ldg(wr + c);
    const __nv_bfloat162* wh = reinterpret_cast<const __nv_bfloat162*>(&wv);
    float wf[8];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const float2 f2 = __bfloat1622float2(wh[i]);
      wf[2 * i] = f2.x;
      wf[2 * i + 1] = f2.y;
    }
#pragma unroll
    for (int t = 0; t < TP; ++t) {
      if (t < Tn) {
        const uint4 xv = __ldg(x + (size_t)t * d8 + c);
        const __nv_bfloat162* xh = reinterpret_cast<const __nv_bfloat162*>(&xv);
        float a = acc[t];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const float2 f2 = __bfloat1622float2(xh[i]);
          a = fmaf(wf[2 * i], f2.x, a);
          a = fmaf(wf[2 * i + 1], f2.y, a);
        }
        acc[t] = a;
      }
    }
  }
#pragma unroll
  for (int t = 0; t < TP; ++t) {
    const float v = warp_sum(acc[t]);
    if (lane == 0) part[warp][t] = v;
  }
  __syncthreads();
  if (threadIdx.x < TP && threadIdx.x < Tn) {
    float v = 0.f;
#pragma unroll
    for (int q = 0; q < 8; ++q) v += part[q][threadIdx.x];
    g[(size_t)(t_base + threadIdx.x) * E + e] = v;
  }
}

cudaError_t launch_router_logits(const moe_config& c, const void* x, const void* w_gate,
                                 float* logits, cudaStream_t s, float* part, DevStatus* st) {
  if (part && router_split(c) > 0) return launch_router_split(c, x, w_gate, part, logits, st, s);
  if (c.dtype == MOE_DTYPE_BF16 && (c.T <= 16 || (c.E <= 32 && c.T <= 512))) {
    // four tokens per CTA: a lane keeps the four token loads of a step in flight together
    launch_pdl(router_logits_few<4>, dim3(c.E, ceil_div(c.T, 4)), 256, 0, s,
               (const uint4*)x, (const uint4*)w_gate, logits, c.T, c.d_model / 8, c.E);
    return cudaGetLastError();
  }
  if (c.dtype == MOE_DTYPE_BF16) {
    if (c.E >= 32 && c.E % 32 == 0) return launch_router_tc(c, x, w_gate, logits, s);
    const size_t row_bytes = (size_t)c.d_model * 2;
    if (c.E <= 8 && 8 * row_bytes <= 200 * 1024) return launch_stream<8>(c, x, w_gate, logits, s);
    if (c.E <= 16 && 16 * row_bytes <= 200 * 1024)
      return launch_stream<16>(c, x, w_gate, logits, s);
    if (c.E <= 32 && 32 * row_bytes <= 200 * 1024)
      return launch_stream<32>(c, x, w_gate, logits, s);
  }
  dim3 grid(ceil_div(c.T, 32), ceil_div(c.E, 64));
  if (c.dtype == MOE_DTYPE_F32)
    launch_pdl(router_logits_simt<float>, grid, 256, 0, s, (const float*)x, (const float*)w_gate, logits,
                                                   c.T, c.d_model, c.E);
  else
    launch_pdl(router_logits_simt<__nv_bfloat16>, grid, 256, 0, s, (const __nv_bfloat16*)x,
                                                           (const __nv_bfloat16*)w_gate, logits,
                                                           c.T, c.d_model, c.E);
  return cudaGetLastError();
}

// ------------------------------------------------------------------------------------------
// Scoring, group limit, Top-k and weights: one warp per token.  Lane l holds experts
// l*V .. l*V+V-1 (V = ceil(E/32)); the selection is k rounds of a warp-wide (key, index)
// maximum, which ranks equal keys by the lower expert index.
// ------------------------------------------------------------------------------------------
struct RouteArgs {
  const float* g;
  const float* bias;
  int T, E, k, score, n_groups, topk_groups, renorm;
  float scale;
  int32_t* idx;
  float* w;
  float* part_P;            // optional load-balance partials (see aux_partial_kernel)
  int32_t* part_cnt;
  float* part_z;
};

constexpr int kAuxWarps = 8;

// One token's contribution to the load-balance statistics, identical in every kernel that
// takes it: P_i gets softmax(g)_i (sigmoid scoring: s_i / sum_j s_j), z gets lse(g)^2.
template <int V>
__device__ __forceinline__ void token_stats(const float (&gv)[V], int lane, int E, int score,
                                            float (&accP)[V], float& zacc) {
  float m = -INFINITY;
#pragma unroll
  for (int i = 0; i < V; ++i) m = fmaxf(m, gv[i]);
  m = warp_max(m);
  float ex[V], se = 0.f;
#pragma unroll
  for (int i = 0; i < V; ++i) {
    ex[i] = (lane * V + i) < E ? expf(gv[i] - m) : 0.f;
    se += ex[i];
  }
  se = warp_sum(se);
  const float lse = m + logf(se);
  if (score == MOE_SCORE_SOFTMAX) {
#pragma unroll
    for (int i = 0; i < V; ++i) accP[i] += ex[i] / se;
  } else {
    float sv[V], ss = 0.f;
#pragma unroll
    for (int i = 0; i < V; ++i) {
      sv[i] = (lane * V + i) < E ? 1.0f / (1.0f + expf(-gv[i])) : 0.f;
      ss += sv[i];
    }
    ss = warp_sum(ss);
#pragma unroll
    for (int i = 0; i < V; ++i) accP[i] += sv[i] / ss;
  }
  if (lane == 0) zacc += lse * lse;
}

// The CTA's warps add their partials in a fixed order and write one row per CTA.
template <int V>
__device__ __forceinline__ void write_block_stats(const float (&accP)[V], const int (&cnt)[V],
                                                  float zacc, int E, float* part_P,
                                                  int32_t* part_cnt, float* part_z,
                                                  unsigned char* smem) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  float* sP = reinterpret_cast<float*>(smem);                       // [warps][E]
  int* sC = reinterpret_cast<int*>(sP + kAuxWarps * E);              // [warps][E]
  float* sZ = reinterpret_cast<float*>(sC + kAuxWarps * E);
  __syncthreads();
#pragma unroll
  for (int i = 0; i < V; ++i) {
    const int e = lane * V + i;
    if (e < E) {
      sP[warp * E + e] = accP[i];
      sC[warp * E + e] = cnt[i];
    }
  }
  if (lane == 0) sZ[warp] = zacc;
  __syncthreads();
  for (int e = threadIdx.x; e < E; e += blockDim.x) {
    float pv = 0.f;
    int c = 0;
    for (int w = 0; w < kAuxWarps; ++w) { pv += sP[w * E + e]; c += sC[w * E + e]; }
    part_P[(size_t)blockIdx.x * E + e] = pv;
    part_cnt[(size_t)blockIdx.x * E + e] = c;
  }
  if (threadIdx.x == 0) {
    float z = 0.f;
    for (int w = 0; w < kAuxWarps; ++w) z += sZ[w];
    part_z[blockIdx.x] = z;
  }
}

template <int V>
__global__ void __launch_bounds__(256) route_topk_kernel(RouteArgs a) {
  pdl_prologue();
  extern __shared__ float route_smem[];
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, wpb = blockDim.x >> 5;
  const int E = a.E, k = a.k;
  const bool grouped = a.score == MOE_SCORE_SIGMOID && a.n_groups > 1 && a.topk_groups < a.n_groups;
  float* row = route_smem + warp * (E + 32);
  float* gsc = row + E;
  const bool stats = a.part_P != nullptr;
  float accP[V];
  int cnt[V];
#pragma unroll
  for (int i = 0; i < V; ++i) { accP[i] = 0.f; cnt[i] = 0; }
  float zacc = 0.f;
  for (int t = blockIdx.x * wpb + warp; t < a.T; t += gridDim.x * wpb) {
    float key[V], val[V], graw[V];
#pragma unroll
    for (int i = 0; i < V; ++i) {
      const int e = lane * V + i;
      const float gv = e < E ? a.g[(size_t)t * E + e] : -INFINITY;
      graw[i] = gv;
      if (a.score == MOE_SCORE_SOFTMAX) {
        key[i] = gv;
        val[i] = gv;
      } else {
        const float sv = e < E ? 1.0f / (1.0f + expf(-gv)) : 0.f;
        const float b = (e < E && a.bias) ? a.bias[e] : 0.f;
        val[i] = sv;
        key[i] = e < E ? sv + b : -INFINITY;
      }
    }
    if (stats) token_stats<V>(graw, lane, E, a.score, accP, zacc);
    if (grouped) {
      const int per = E / a.n_groups;
#pragma unroll
      for (int i = 0; i < V; ++i) {
        const int e = lane * V + i;
        if (e < E) row[e] = key[i];
      }
      __syncwarp();
      if (lane < a.n_groups) {
        float b1 = -INFINITY, b2 = -INFINITY;      // two largest of the group
        for (int q = 0; q < per; ++q) {
          const float v = row[lane * per + q];
          if (v > b1) { b2 = b1; b1 = v; } else if (v > b2) { b2 = v; }
        }
        gsc[lane] = b1 + b2;
      }
      __syncwarp();
      float gk = lane < a.n_groups ? gsc[lane] : -INFINITY;
      bool gtaken = lane >= a.n_groups;
      uint32_t keep = 0;
      for (int r = 0; r < a.topk_groups; ++r) {
        float bk = gtaken ? -INFINITY : gk;
        int bi = gtaken ? 0x7fffffff : lane;
        warp_best(bk, bi);
        keep |= 1u << bi;
        if (lane == bi) gtaken = true;
      }
#pragma unroll
      for (int i = 0; i < V; ++i) {
        const int e = lane * V + i;
        if (e < E && !((keep >> (e / per)) & 1u)) key[i] = -INFINITY;
      }
      __syncwarp();
    }
    // k rounds of the warp-wide best remaining (key, index)
    uint32_t taken = 0;
    int my_sel = -1;
    float my_val = 0.f;
    float first_val = 0.f;
    for (int j = 0; j < k; ++j) {
      float bk = -INFINITY;
      int bi = 0x7fffffff;
      float bv = 0.f;
#pragma unroll
      for (int i = 0; i < V; ++i) {
        const int e = lane * V + i;
        if (!((taken >> i) & 1u) && e < E && ranks_before(key[i], e, bk, bi)) {
          bk = key[i];
          bi = e;
          bv = val[i];
        }
      }
      const int mine = bi;
      warp_best(bk, bi);
      const int owner = bi / V;
      if (lane == owner) {
#pragma unroll
        for (int i = 0; i < V; ++i)
          if (lane * V + i == bi) {
            taken |= 1u << i;
            cnt[i] += 1;
          }
      }
      const float v = __shfl_sync(0xffffffffu, bv, owner);
      (void)mine;
      if (j == 0) first_val = v;
      if (lane == j) { my_sel = bi; my_val = v; }
    }
    // weights of the k selected experts (lanes 0..k-1 hold one each)
    float num = 0.f;
    if (a.score == MOE_SCORE_SOFTMAX) {
      // p_j = exp(g_j - m) / sum_all exp(g - m) with m = the largest logit (= first selected)
      num = lane < k ? expf(my_val - first_val) : 0.f;
    } else {
      num = lane < k ? my_val : 0.f;
    }
    float den;
    if (a.renorm) {
      den = warp_sum(num);
    } else if (a.score == MOE_SCORE_SOFTMAX) {
      float part = 0.f;
#pragma unroll
      for (int i = 0; i < V; ++i) {
        const int e = lane * V + i;
        if (e < E) part += expf(val[i] - first_val);
      }
      den = warp_sum(part);
    } else {
      den = 1.f;
    }
    if (lane < k) {
      a.idx[(size_t)t * k + lane] = my_sel;
      a.w[(size_t)t * k + lane] = (num / den) * a.scale;
    }
  }
  if (stats)
    write_block_stats<V>(accP, cnt, zacc, E, a.part_P, a.part_cnt, a.part_z,
                         reinterpret_cast<unsigned char*>(route_smem));
}

// ------------------------------------------------------------------------------------------
// Decode batches with E > 32: one CTA per token, thread e <-> expert e (E <= 256).  The warp
// kernel above gives each lane E/32 experts and then walks k rounds of a warp-wide arg-max,
// a long serial chain when a step has only a few tokens.  Here every step is a parallel count:
//   1. each expert's rank within its segment (its group under a group limit, else its warp's
//      32 experts) = the number of segment members that rank before it;
//   2. group limit: a group's score is its rank-0 plus rank-1 key (its two largest), a group is
//      kept when fewer than topk_groups groups rank before it (ties: lower group);
//   3. candidates = kept experts of segment rank < k (the k best of the kept experts are among
//      them); a candidate's rank among the candidates is its rank among all kept experts, and
//      ranks 0..k-1 are the selection in rank order.
// The order is the same strict (key descending, index ascending) order as everywhere, so the
// selection is the same set in the same order; renormalised weights are formed as in the warp
// kernel (lanes 0..k-1 of warp 0 in rank order).  With the statistics, each token writes its
// own partial row (p_t, the selection indicator and lse_t^2); aux_token_kernel writes the same
// rows for the separate statistics call, so both reduce to the same bits.
// ------------------------------------------------------------------------------------------
constexpr int kRouteCtaMaxT = 64;

bool route_cta(const moe_config& c) {
  return c.routing == MOE_ROUTE_TOKEN_CHOICE && c.E > 32 && c.T <= kRouteCtaMaxT;
}

// Prefill batches of a bf16 router with E a multiple of 32 (<= 256, by default >= 128) and
// groups of whole 32-expert chunks: the router GEMM's epilogue does the scoring, the Top-k and
// the statistics terms (launch_router_fused), one partial row per 128-token tile.
constexpr int kRouterFusedMinE = 128;

bool router_fused(const moe_config& c) {
  if (c.dtype != MOE_DTYPE_BF16 || c.routing != MOE_ROUTE_TOKEN_CHOICE) return false;
  if (c.E < 32 || c.E > 256 || c.E % 32 || c.k > 8 || c.T <= kRouterSplitMaxT) return false;
  const bool limit = c.score == MOE_SCORE_SIGMOID && c.n_groups > 1 &&
                     c.topk_groups < c.n_groups;
  if (limit && (c.E / c.n_groups) % 32) return false;
  // Measured: at E = 256 (the DeepSeek-V3 router) the fused path matches the separate logits
  // GEMM + Top-k pass; at E = 64 (DeepSeekMoE-16B) its four threads per token share two
  // 32-expert chunks, and the separate pass is 25 us per step faster.  MOE_B300_ROUTER=fused
  // takes the fused path for every eligible router, =separate for none.
  const char* env = getenv("MOE_B300_ROUTER");
  if (env && strcmp(env, "separate") == 0) return false;
  if (env && strcmp(env, "fused") == 0) return true;
  return c.E >= kRouterFusedMinE;
}

int aux_rows(const moe_config& c) {
  if (router_fused(c)) return ceil_div(c.T, 128);
  return route_cta(c) ? c.T : aux_blocks(c);
}

// The fused router's statistics rows for a given selection (moe_aux_stats), from logits in
// global memory: the same 128-token tiles, the same four threads per token (thread group w =
// warp + 2 takes TMEM lane quarter w % 4 and chunk quarter w / 4, as in the epilogue), the
// same token-to-slot mapping (a last tile of <= 64 rows puts rows 16q..16q+15 on lanes 0..15
// of quarter q, as the M = 64 accumulator does) and the same phases, so both give the same
// bits.
__global__ void __launch_bounds__(512) route_rows_stats_kernel(const float* __restrict__ g,
                                                               const int32_t* __restrict__ idx,
                                                               int T, RouteThreadCfg rc,
                                                               float* part_P, int32_t* part_cnt,
                                                               float* part_z) {
  pdl_prologue();
  extern __shared__ unsigned char route_rows_smem[];
  RouteSmem& sm = *reinterpret_cast<RouteSmem*>(route_rows_smem);
  const int E = rc.nc * 32;
  const int tile = blockIdx.x;
  const int row0 = tile * kRouteTile;
  const int rows = min(kRouteTile, T - row0);
  const int w = (threadIdx.x >> 5) + 2, lane = threadIdx.x & 31;
  const int q = w & 3, sub = (w - 2) >> 2;
  const int r = q * 32 + lane;
  const bool half = rows <= 64;
  const int row = half ? q * 16 + lane : r;
  const bool live = half ? (lane < 16 && row < rows) : (r < rows);
  const size_t t = static_cast<size_t>(row0 + (live ? row : 0));
  for (int e = threadIdx.x; e < 256; e += 512) {
    sm.bias[e] = 0.f;
    sm.cnt[e] = 0;
  }
  __syncthreads();
  auto load = [&](int c, float (&v)[32]) {
    const float4* src = reinterpret_cast<const float4*>(g + t * E + c * 32);
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const float4 f = live ? src[i] : make_float4(0.f, 0.f, 0.f, 0.f);
      v[4 * i] = f.x;
      v[4 * i + 1] = f.y;
      v[4 * i + 2] = f.z;
      v[4 * i + 3] = f.w;
    }
  };
  route_phase_a(rc, sm, r, sub, load, [](int, const float (&)[32]) {});
  __syncthreads();
  route_phase_b(rc, sm, r, sub, q, live, load, load);
  __syncthreads();
  if (sub == 0) {
    const RouteTotals tot = route_totals(sm, r);
    const float lse = tot.m + logf(tot.se);
    if (live)
      for (int j = 0; j < rc.k; ++j) {
        const int e = idx[t * rc.k + j];
        if (e >= 0 && e < E) atomicAdd(&sm.cnt[e], 1);    // caller's indices: range-checked
      }
    const float zt = warp_sum(live ? lse * lse : 0.f);
    if (lane == 0) sm.Z[q] = zt;
  }
  __syncthreads();
  for (int e = threadIdx.x; e < E; e += 512) {
    part_P[static_cast<size_t>(tile) * E + e] =
        ((sm.P[0][e] + sm.P[1][e]) + sm.P[2][e]) + sm.P[3][e];
    part_cnt[static_cast<size_t>(tile) * E + e] = sm.cnt[e];
  }
  if (threadIdx.x == 0) part_z[tile] = ((sm.Z[0] + sm.Z[1]) + sm.Z[2]) + sm.Z[3];
}

// Block-wide reductions over blockDim/32 warps (every thread gets the result); red holds one
// value per warp and is free again on return.
__device__ __forceinline__ float block_max(float v, float* red) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nw = blockDim.x >> 5;
  v = warp_max(v);
  if (lane == 0) red[warp] = v;
  __syncthreads();
  float m = red[0];
  for (int w = 1; w < nw; ++w) m = fmaxf(m, red[w]);
  __syncthreads();
  return m;
}

__device__ __forceinline__ float block_sum(float v, float* red) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nw = blockDim.x >> 5;
  v = warp_sum(v);
  if (lane == 0) red[warp] = v;
  __syncthreads();
  float t = red[0];
  for (int w = 1; w < nw; ++w) t += red[w];
  __syncthreads();
  return t;
}

// One token's statistics in the CTA layout (thread e holds g_e; invalid threads hold nothing):
// P contribution softmax(g)_e (sigmoid scoring: s_e / sum_j s_j) and lse(g).
__device__ __forceinline__ void token_stats_cta(float gv, bool valid, int score, float* red,
                                                float& pc, float& lse) {
  const float m = block_max(valid ? gv : -INFINITY, red);
  const float ex = valid ? expf(gv - m) : 0.f;
  const float se = block_sum(ex, red);
  lse = m + logf(se);
  if (score == MOE_SCORE_SOFTMAX) {
    pc = ex / se;
  } else {
    const float sv = valid ? 1.0f / (1.0f + expf(-gv)) : 0.f;
    const float ss = block_sum(sv, red);
    pc = sv / ss;
  }
}

__global__ void __launch_bounds__(256) route_topk_cta_kernel(RouteArgs a) {
  pdl_prologue();
  __shared__ float skey[256];
  __shared__ float sval[256];
  __shared__ float slot_key[256];
  __shared__ int slot_idx[256];
  __shared__ float gtop[2][32];
  __shared__ int sel_idx[8];
  __shared__ float sel_val[8];
  __shared__ float red[8];
  const int t = blockIdx.x, e = threadIdx.x, lane = e & 31, warp = e >> 5;
  const int E = a.E, k = a.k;
  const bool valid = e < E;
  const float gv = valid ? a.g[(size_t)t * E + e] : -INFINITY;
  float key, val;
  if (a.score == MOE_SCORE_SOFTMAX) {
    key = gv;
    val = gv;
  } else {
    const float sv = valid ? 1.0f / (1.0f + expf(-gv)) : 0.f;
    const float b = (valid && a.bias) ? a.bias[e] : 0.f;
    val = sv;
    key = valid ? sv + b : -INFINITY;
  }
  skey[e] = key;
  sval[e] = val;
  slot_idx[e] = -1;
  float pc = 0.f, lse = 0.f;
  const bool stats = a.part_P != nullptr;
  if (stats) token_stats_cta(gv, valid, a.score, red, pc, lse);
  __syncthreads();
  const bool grouped =
      a.score == MOE_SCORE_SIGMOID && a.n_groups > 1 && a.topk_groups < a.n_groups;
  const int seg_len = grouped ? E / a.n_groups : 32;
  const int seg = e / seg_len;
  const int s0 = seg * seg_len, s1 = min(E, s0 + seg_len);
  int r_seg = 0;
  if (valid)
    for (int q = s0; q < s1; ++q) r_seg += ranks_before(skey[q], q, key, e) ? 1 : 0;
  bool kept = true;
  if (grouped) {
    if (valid && r_seg < 2) gtop[r_seg][seg] = key;
    __syncthreads();
    if (valid) {
      const float gs = gtop[0][seg] + gtop[1][seg];
      int grank = 0;
      for (int q = 0; q < a.n_groups; ++q)
        grank += ranks_before(gtop[0][q] + gtop[1][q], q, gs, seg) ? 1 : 0;
      kept = grank < a.topk_groups;
    }
  }
  const int kk = min(seg_len, k);
  const bool cand = valid && kept && r_seg < kk;
  if (cand) {
    slot_key[seg * kk + r_seg] = key;
    slot_idx[seg * kk + r_seg] = e;
  }
  __syncthreads();
  const int nslots = ceil_div(E, seg_len) * kk;
  bool selected = false;
  if (cand) {
    int rank = 0;
    for (int q = 0; q < nslots; ++q) {
      const int qi = slot_idx[q];
      if (qi >= 0 && ranks_before(slot_key[q], qi, key, e)) ++rank;
    }
    if (rank < k) {
      sel_idx[rank] = e;
      sel_val[rank] = val;
      selected = true;
    }
  }
  __syncthreads();
  if (warp == 0) {
    const int my_sel = lane < k ? sel_idx[lane] : -1;
    const float my_val = lane < k ? sel_val[lane] : 0.f;
    const float first_val = sel_val[0];
    float num;
    if (a.score == MOE_SCORE_SOFTMAX) num = lane < k ? expf(my_val - first_val) : 0.f;
    else num = lane < k ? my_val : 0.f;
    float den;
    if (a.renorm) {
      den = warp_sum(num);
    } else if (a.score == MOE_SCORE_SOFTMAX) {
      float part = 0.f;
      for (int q = lane; q < E; q += 32) part += expf(sval[q] - first_val);
      den = warp_sum(part);
    } else {
      den = 1.f;
    }
    if (lane < k) {
      a.idx[(size_t)t * k + lane] = my_sel;
      a.w[(size_t)t * k + lane] = (num / den) * a.scale;
    }
  }
  if (stats && valid) {
    a.part_P[(size_t)t * E + e] = pc;
    a.part_cnt[(size_t)t * E + e] = selected ? 1 : 0;
    if (e == 0) a.part_z[t] = lse * lse;
  }
}

// The statistics rows of route_topk_cta_kernel for a given selection (moe_aux_stats).
__global__ void __launch_bounds__(256) aux_token_kernel(const float* __restrict__ g,
                                                       const int32_t* __restrict__ idx, int E,
                                                       int k, int score, float* part_P,
                                                       int32_t* part_cnt, float* part_z) {
  pdl_prologue();
  __shared__ float red[8];
  const int t = blockIdx.x, e = threadIdx.x;
  const bool valid = e < E;
  const float gv = valid ? g[(size_t)t * E + e] : -INFINITY;
  float pc, lse;
  token_stats_cta(gv, valid, score, red, pc, lse);
  if (!valid) return;
  int c = 0;
  for (int j = 0; j < k; ++j) c |= idx[(size_t)t * k + j] == e ? 1 : 0;
  part_P[(size_t)t * E + e] = pc;
  part_cnt[(size_t)t * E + e] = c;
  if (e == 0) part_z[t] = lse * lse;
}

cudaError_t launch_route_topk(const moe_config& c, const float* logits, const float* bias,
                              int32_t* idx, float* w, DevStatus* st, cudaStream_t s,
                              float* part_P, int32_t* part_cnt, float* part_z) {
  (void)st;
  RouteArgs a{logits, bias, c.T, c.E, c.k, c.score, c.n_groups, c.topk_groups, c.renormalize,
              c.route_scale, idx, w, part_P, part_cnt, part_z};
  if (route_cta(c)) {
    launch_pdl(route_topk_cta_kernel, c.T, 32 * ceil_div(c.E, 32), 0, s, a);
    return cudaGetLastError();
  }
  const int wpb = kAuxWarps;
  // with the statistics, the grid is the statistics' fixed block count (fixed token sets)
  const int blocks = part_P ? aux_blocks(c) : ceil_div(c.T, wpb);
  const size_t route_bytes = (size_t)wpb * (c.E + 32) * sizeof(float);
  const size_t stats_bytes = (size_t)kAuxWarps * c.E * 8 + kAuxWarps * 4 + 16;
  const size_t smem = route_bytes > stats_bytes ? route_bytes : stats_bytes;
  if (c.E <= 32) launch_pdl(route_topk_kernel<1>, blocks, wpb * 32, smem, s, a);
  else if (c.E <= 64) launch_pdl(route_topk_kernel<2>, blocks, wpb * 32, smem, s, a);
  else if (c.E <= 128) launch_pdl(route_topk_kernel<4>, blocks, wpb * 32, smem, s, a);
  else launch_pdl(route_topk_kernel<8>, blocks, wpb * 32, smem, s, a);
  return cudaGetLastError();
}

// ------------------------------------------------------------------------------------------
// Statistics.  Each CTA owns a fixed set of tokens (warp w of CTA b takes tokens
// b*8 + w + i*gridDim*8), accumulates per-expert sums in registers, reduces its warps in a
// fixed order and writes one partial row; a single CTA then sums the rows in float32 in a
// fixed order.  No floating-point atomics, so the results are reproducible bit for bit.
// ------------------------------------------------------------------------------------------
struct AuxArgs {
  const float* g;
  const int32_t* idx;       // [T,k] or NULL when ec_C > 0
  int T, E, k, score;
  int ec_C;                 // expert choice: every expert holds ec_C tokens
  float* part_P;            // [nblk][E]
  int32_t* part_cnt;        // [nblk][E]
  float* part_z;            // [nblk]
};

template <int V>
__global__ void __launch_bounds__(kAuxWarps * 32) aux_partial_kernel(AuxArgs a) {
  pdl_prologue();
  extern __shared__ unsigned char aux_smem[];
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int E = a.E;
  float accP[V];
  int cnt[V];
#pragma unroll
  for (int i = 0; i < V; ++i) { accP[i] = 0.f; cnt[i] = 0; }
  float zacc = 0.f;
  for (int t = blockIdx.x * kAuxWarps + warp; t < a.T; t += gridDim.x * kAuxWarps) {
    float gv[V];
#pragma unroll
    for (int i = 0; i < V; ++i) {
      const int e = lane * V + i;
      gv[i] = e < E ? a.g[(size_t)t * E + e] : -INFINITY;
    }
    token_stats<V>(gv, lane, E, a.score, accP, zacc);
    if (a.ec_C <= 0) {
      for (int j = 0; j < a.k; ++j) {
        const int e = a.idx[(size_t)t * a.k + j];
        if (e >= 0 && e < E && e / V == lane) {
#pragma unroll
          for (int i = 0; i < V; ++i)
            if (lane * V + i == e) cnt[i] += 1;
        }
      }
    }
  }
  write_block_stats<V>(accP, cnt, zacc, E, a.part_P, a.part_cnt, a.part_z, aux_smem);
}

// Lanes own consecutive experts (coalesced reads of a partial row); the 32 warps split into
// G = 32-expert groups x W = 32/G block strides.  Each thread sums blocks sub, sub+W, ... of its
// expert (float32 for P, integers for counts), then thread (sub 0) adds the W sums in order;
// warp 0 also sums the z partials.  Deterministic for a given block count.  (No float64: its
// throughput on this part is a tiny fraction.)
__global__ void __launch_bounds__(1024) aux_final_kernel(const float* part_P,
                                                        const int32_t* part_cnt,
                                                        const float* part_z, int nblk, int T,
                                                        int E, int ec_C, float* f, float* P,
                                                        float* l_balance, float* z_loss) {
  pdl_prologue();
  __shared__ float sp[1024];
  __shared__ int sc[1024];
  __shared__ float prod[256];
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  int G = 1;
  while (G * 32 < E) G <<= 1;                  // expert groups of 32 (E <= 256: G <= 8)
  const int W = 32 / G;                        // warps per group = block stride
  const int g = warp % G, sub = warp / G;
  const int e = g * 32 + lane;
  float p = 0.f;
  int c = 0;
  if (e < E) {
    // eight rows' loads in flight, then added in row order
    for (int b0 = sub; b0 < nblk; b0 += 8 * W) {
      float qp[8];
      int qc[8];
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        const int b = b0 + i * W;
        if (b < nblk) {
          qp[i] = part_P[(size_t)b * E + e];
          qc[i] = part_cnt[(size_t)b * E + e];
        }
      }
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        if (b0 + i * W >= nblk) break;
        p += qp[i];
        c += qc[i];
      }
    }
  }
  sp[sub * 32 * G + e] = p;
  sc[sub * 32 * G + e] = c;
  __syncthreads();
  const float invT = 1.0f / (float)T;
  if (sub == 0 && e < E) {
    float ps = 0.f;
    int cs = 0;
    for (int w = 0; w < W; ++w) {
      ps += sp[w * 32 * G + e];
      cs += sc[w * 32 * G + e];
    }
    if (ec_C > 0) cs = ec_C;
    const float fe = (float)cs * invT, Pe = ps * invT;
    if (f) f[e] = fe;
    if (P) P[e] = Pe;
    prod[e] = fe * Pe;
  }
  __syncthreads();
  if (warp == 0) {
    float acc = 0.f;
    for (int x = lane; x < E; x += 32) acc += prod[x];
    acc = warp_sum(acc);
    float z = 0.f;
    for (int b = lane; b < nblk; b += 32) z += part_z[b];
    z = warp_sum(z);
    if (lane == 0) {
      if (l_balance) *l_balance = (float)E * acc;
      if (z_loss) *z_loss = z * invT;
    }
  }
}

int aux_blocks(const moe_config& c) {
  int b = ceil_div(c.T, kAuxWarps * 2);
  return b < 1 ? 1 : (b > 512 ? 512 : b);
}

cudaError_t launch_aux_stats(const moe_config& c, const float* logits, const int32_t* idx,
                             const int32_t* /*ec_counts*/, float* part_P, int32_t* part_cnt,
                             float* part_z, int nblocks, float* f, float* P, float* l_balance,
                             float* z_loss, DevStatus* st, cudaStream_t s) {
  (void)st;
  if (router_fused(c)) {              // the fused router's 128-token rows
    const bool limit = c.score == MOE_SCORE_SIGMOID && c.n_groups > 1 &&
                       c.topk_groups < c.n_groups;
    RouteThreadCfg rc{c.E / 32, c.k, c.score, limit ? (c.E / c.n_groups) / 32 : 0,
                      c.topk_groups, c.renormalize, c.route_scale, 0};
    const int tiles = ceil_div(c.T, kRouteTile);
    cudaError_t ea = smem_attr_once(reinterpret_cast<const void*>(route_rows_stats_kernel),
                                    static_cast<int>(sizeof(RouteSmem)));
    if (ea != cudaSuccess) return ea;
    launch_pdl(route_rows_stats_kernel, tiles, 512, sizeof(RouteSmem), s, logits, idx, c.T, rc,
               part_P, part_cnt, part_z);
    cudaError_t err = cudaGetLastError();
    if (err != cudaSuccess) return err;
    return launch_aux_final(c, part_P, part_cnt, part_z, tiles, f, P, l_balance, z_loss, s);
  }
  if (route_cta(c)) {                 // per-token rows, as the fused Top-k pass writes them
    launch_pdl(aux_token_kernel, c.T, 32 * ceil_div(c.E, 32), 0, s, logits, idx, c.E, c.k,
               c.score, part_P, part_cnt, part_z);
    cudaError_t err = cudaGetLastError();
    if (err != cudaSuccess) return err;
    return launch_aux_final(c, part_P, part_cnt, part_z, c.T, f, P, l_balance, z_loss, s);
  }
  const int ecC = c.routing == MOE_ROUTE_EXPERT_CHOICE ? (int)((long long)c.T * c.k / c.E) : 0;
  AuxArgs a{logits, idx, c.T, c.E, c.k, c.score, ecC, part_P, part_cnt, part_z};
  const size_t smem = (size_t)kAuxWarps * c.E * 8 + kAuxWarps * 4 + 16;
  if (c.E <= 32) launch_pdl(aux_partial_kernel<1>, nblocks, kAuxWarps * 32, smem, s, a);
  else if (c.E <= 64) launch_pdl(aux_partial_kernel<2>, nblocks, kAuxWarps * 32, smem, s, a);
  else if (c.E <= 128) launch_pdl(aux_partial_kernel<4>, nblocks, kAuxWarps * 32, smem, s, a);
  else launch_pdl(aux_partial_kernel<8>, nblocks, kAuxWarps * 32, smem, s, a);
  cudaError_t err = cudaGetLastError();
  if (err != cudaSuccess) return err;
  return launch_aux_final(c, part_P, part_cnt, part_z, nblocks, f, P, l_balance, z_loss, s);
}

cudaError_t launch_aux_final(const moe_config& c, const float* part_P, const int32_t* part_cnt,
                             const float* part_z, int nblocks, float* f, float* P,
                             float* l_balance, float* z_loss, cudaStream_t s) {
  const int ecC = c.routing == MOE_ROUTE_EXPERT_CHOICE ? (int)((long long)c.T * c.k / c.E) : 0;
  launch_pdl(aux_final_kernel, 1, 1024, 0, s, part_P, part_cnt, part_z, nblocks, c.T, c.E, ecC, f, P,
                                      l_balance, z_loss);
  return cudaGetLastError();
}

}  // namespace moe
