// Router-side backward and the selection-bias update (sm_103a).
//
// The loss differentiated here is  alpha * L_balance + beta * z + <d_w, w>:
//   * L_balance = E * sum_i f_i P_i with f a count, so only P_i carries a gradient
//     ("MoE 路由数学" §3.4; "Systems for Mixture-of-Experts Models" §3.2);
//   * z = mean over tokens of logsumexp(g)^2 (router_z_loss code block of the "Mixture of
//     Experts 架构" page);
//   * w = the routing weights, d_w their upstream gradient (nullable); the selection is a
//     discrete choice and the sigmoid route's bias only enters the selection (§3.4 of the
//     lecture), so neither has a gradient.
// The steps on the device:
//   1. router_bw_scores_kernel: one warp per token recomputes p (and s), lse and the chain rule
//      of the scoring function in fp32; writes dL/dg as fp32 and, for the tensor-core GEMMs,
//      as bf16 in both [T, E64] and [E64, T] layouts (E64 = E rounded up to 64, zero padded).
//   2. One router_grad_gemm_kernel launch for both gradient products, its tiles taken from a
//      counter (dW's first):
//      dW_gate = dg^T x with M = d (x read MN-major: T is the reduction axis and x's row
//      index), N = E64 (dg^T K-major), K = T, split along K into fixed slices;
//      dx = dg W_gate with M = T (dg K-major), N = 256 columns of d (W_gate read MN-major),
//      K = E64.
//   3. splitk_reduce_kernel sums dW's float32 slices in slice order (deterministic).
// The float32 configuration runs the two products as plain SIMT loops.
//
// The bias update ("Systems for Mixture-of-Experts Models" §3.4; update_bias code block of the
// "Mixture of Experts 架构" page): b_i -= gamma when expert i's load exceeds the mean load
// T*k/E, b_i += gamma when it is below, unchanged when equal; loads are recovered exactly from
// the frequencies f_i = load_i / T.
#include <cuda.h>
#include <cuda_bf16.h>

#include <cmath>

#include "common.cuh"
#include "kernels.h"
#include "tc_ptx.cuh"

namespace moe {
namespace {

constexpr int kBwTokens = 16;     // tokens per CTA of the scores kernel (one per warp)
constexpr int kBwWarps = 16;
// shared row of the transposed tile: 18 bf16 = 9 words, odd, so the 32 lanes writing 32
// experts of one token hit 32 different banks
constexpr int kTPad = kBwTokens + 2;

int e64_of(int E) { return (E + 63) / 64 * 64; }
long long t64_of(int T) { return ((long long)T + 63) / 64 * 64; }   // >= every CTA's tokens

struct ScoresArgs {
  int T, E, E64, k, score, renorm;
  long long T64;
  float route_scale, alpha, beta;
  const float* logits;
  const int32_t* idx;
  const float* d_w;       // nullable
  const float* f;         // nullable
  float* d_logits;        // nullable
  __nv_bfloat16* dg16;    // nullable: [T, E64]
  __nv_bfloat16* dgT;     // nullable: [E64, T64]
  int* tile_counter;      // nullable: zeroed here for the gradient GEMM launch that follows
  DevStatus* st;
};

template <int V>
__global__ void __launch_bounds__(kBwWarps * 32, 2) router_bw_scores_kernel(const ScoresArgs a) {
  pdl_prologue();
  if (a.tile_counter && blockIdx.x == 0 && threadIdx.x == 0) *a.tile_counter = 0;
  __shared__ __nv_bfloat16 sT[256][kTPad];
  __shared__ int sSel[kBwWarps][256];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int t_base = blockIdx.x * kBwTokens;
  const float inv_T = 1.0f / static_cast<float>(a.T);
  const float bal = a.alpha * static_cast<float>(a.E) * inv_T;     // dL/dprob = bal * f_i
  const float zc = 2.0f * a.beta * inv_T;

  float c[V];
#pragma unroll
  for (int i = 0; i < V; ++i) {
    const int e = lane + 32 * i;
    c[i] = (a.f && e < a.E) ? bal * a.f[e] : 0.0f;
  }

  for (int j8 = 0; j8 < kBwTokens / kBwWarps; ++j8) {
    const int tl = warp * (kBwTokens / kBwWarps) + j8;
    const int t = t_base + tl;
    float dg[V];
    if (t < a.T) {
      const float* gr = a.logits + static_cast<size_t>(t) * a.E;
      // every load of the token is issued here, before any arithmetic: lane j holds choice j
      // (k <= 8), broadcast below
      int e_l = 0;
      float dw_l = 0.0f;
      if (a.d_w && lane < a.k) {
        e_l = a.idx[static_cast<size_t>(t) * a.k + lane];
        dw_l = a.d_w[static_cast<size_t>(t) * a.k + lane];
      }
      float g[V];
      float m = -INFINITY;
#pragma unroll
      for (int i = 0; i < V; ++i) {
        const int e = lane + 32 * i;
        g[i] = e < a.E ? gr[e] : -INFINITY;
        m = fmaxf(m, g[i]);
      }
      m = warp_max(m);
      float p[V], zsum = 0.0f;
#pragma unroll
      for (int i = 0; i < V; ++i) {
        p[i] = (lane + 32 * i) < a.E ? expf(g[i] - m) : 0.0f;
        zsum += p[i];
      }
      zsum = warp_sum(zsum);
      const float inv_z = 1.0f / zsum;
#pragma unroll
      for (int i = 0; i < V; ++i) p[i] *= inv_z;
      const float lse = m + logf(zsum);

      // scores v the weights are built from: p (softmax) or s = sigmoid(g)
      float v[V];
      if (a.score == MOE_SCORE_SOFTMAX) {
#pragma unroll
        for (int i = 0; i < V; ++i) v[i] = p[i];
      } else {
#pragma unroll
        for (int i = 0; i < V; ++i)
          v[i] = (lane + 32 * i) < a.E ? __frcp_rn(1.0f + expf(-g[i])) : 0.0f;
      }

      // gate-weight term: dL/dv on the selected experts
      float dv[V];
#pragma unroll
      for (int i = 0; i < V; ++i) dv[i] = 0.0f;
      if (a.d_w) {
        float dwv[V];
        float sum_s = 0.0f, sum_dws = 0.0f;
#pragma unroll
        for (int i = 0; i < V; ++i) dwv[i] = 0.0f;
        // choice j of the token marks expert e_j in the warp's row of slots (j + 1; the
        // last choice naming an expert wins), then each lane reads its own experts' slots
        int* slot = sSel[warp];
#pragma unroll
        for (int i = 0; i < V; ++i) slot[lane + 32 * i] = 0;
        __syncwarp();
        if (lane < a.k) {
          if (e_l < 0 || e_l >= a.E) record_error(a.st, MOE_ERR_ARG, t);
          else atomicMax(&slot[e_l], lane + 1);
        }
        __syncwarp();
        bool sel[V];
#pragma unroll
        for (int i = 0; i < V; ++i) {
          const int j1 = slot[lane + 32 * i];
          const float dwj = __shfl_sync(0xffffffffu, dw_l, j1 > 0 ? j1 - 1 : 0);
          sel[i] = j1 > 0;
          dwv[i] = sel[i] ? dwj : 0.0f;
        }
#pragma unroll
        for (int i = 0; i < V; ++i)
          if (sel[i]) { sum_s += v[i]; sum_dws += dwv[i] * v[i]; }
        sum_s = warp_sum(sum_s);
        sum_dws = warp_sum(sum_dws);
        // w_j = scale * v_j / sum_S v: dL/dv_j = scale * (d_w_j - sum_S d_w v / sum_S v) / sum_S v
        const float inv_ss = 1.0f / sum_s;
        const float mean_dw = sum_dws * inv_ss;
#pragma unroll
        for (int i = 0; i < V; ++i)
          if (sel[i])
            dv[i] = a.renorm ? a.route_scale * (dwv[i] - mean_dw) * inv_ss
                             : a.route_scale * dwv[i];
      }

      if (a.score == MOE_SCORE_SOFTMAX) {
        float gp = 0.0f;
#pragma unroll
        for (int i = 0; i < V; ++i) gp += (dv[i] + c[i]) * p[i];
        gp = warp_sum(gp);
#pragma unroll
        for (int i = 0; i < V; ++i) dg[i] = p[i] * (dv[i] + c[i] - gp);
      } else {
        float ssum = 0.0f;
#pragma unroll
        for (int i = 0; i < V; ++i) ssum += v[i];
        ssum = warp_sum(ssum);
        const float inv_s = 1.0f / ssum;
        float cq = 0.0f;
#pragma unroll
        for (int i = 0; i < V; ++i) cq += c[i] * v[i];
        cq = warp_sum(cq) * inv_s;                       // <c, q>, q = s / sum s
#pragma unroll
        for (int i = 0; i < V; ++i) {
          const float ds = dv[i] + (c[i] - cq) * inv_s;
          dg[i] = ds * v[i] * (1.0f - v[i]);
        }
      }
#pragma unroll
      for (int i = 0; i < V; ++i) dg[i] += zc * lse * p[i];

      if (a.d_logits) {
        float* out = a.d_logits + static_cast<size_t>(t) * a.E;
#pragma unroll
        for (int i = 0; i < V; ++i)
          if (lane + 32 * i < a.E) out[lane + 32 * i] = dg[i];
      }
      if (a.dg16) {
        __nv_bfloat16* out = a.dg16 + static_cast<size_t>(t) * a.E64;
#pragma unroll
        for (int i = 0; i < V; ++i)
          if (lane + 32 * i < a.E) out[lane + 32 * i] = __float2bfloat16_rn(dg[i]);
        for (int e = a.E + lane; e < a.E64; e += 32) out[e] = __float2bfloat16_rn(0.0f);
      }
    } else {
#pragma unroll
      for (int i = 0; i < V; ++i) dg[i] = 0.0f;
    }
    if (a.dgT) {
#pragma unroll
      for (int i = 0; i < V; ++i)
        if (lane + 32 * i < a.E) sT[lane + 32 * i][tl] = __float2bfloat16_rn(dg[i]);
      for (int e = a.E + lane; e < a.E64; e += 32) sT[e][tl] = __float2bfloat16_rn(0.0f);
    }
  }
  if (a.dgT) {
    __syncthreads();
    // row e of the transposed block: 16 tokens = 8 words = one 32-byte sector; a warp writes
    // 4 rows per instruction, 8 lanes per row
    const int sub = lane >> 3, wd = lane & 7;
    for (int e = warp * 4 + sub; e < a.E64; e += kBwWarps * 4) {
      const uint32_t wv = *reinterpret_cast<const uint32_t*>(&sT[e][2 * wd]);
      *reinterpret_cast<uint32_t*>(a.dgT + static_cast<size_t>(e) * a.T64 + t_base + 2 * wd) =
          wv;
    }
  }
}

// ---------------------------------------------------------------------------------------------
// tcgen05 GEMM D[M, N] = sum_k A(m, k) B(n, k), either operand K-major ([rows, K], K
// contiguous) or MN-major ([K, rows], rows contiguous), float32 accumulate, split along K.
// ---------------------------------------------------------------------------------------------
namespace rg {

using namespace tc;

constexpr int BM = 128;
constexpr int BK = 64;
constexpr int STAGES = 4;
constexpr int A_STAGE = BM * BK * 2;          // 16 KB
constexpr int B_STAGE = 256 * BK * 2;         // up to 32 KB
constexpr int MN_ATOM = 64 * BK * 2;          // one 64-column MN-major box: 8 KB
constexpr int TMEM_COLS = 512;
constexpr int EPI_WARPS = 8;                  // two per TMEM lane quarter, one column half each
constexpr int THREADS = 64 + 32 * EPI_WARPS;
constexpr int NQ = 4;                         // tile ids queued from the producer
// full, empty, tmem full x2, tmem empty x2, drain, tile queue full x NQ, empty x NQ
constexpr int NBARS = 2 * STAGES + 5 + 2 * NQ;
constexpr int STAGE_OUT = 32 * 32 * 4;       // one 32-row x 32-column fp32 chunk, 4 KB
// ring | per epilogue warp one chunk buffer (1024-byte aligned, 128-byte swizzle) | barriers
constexpr size_t SMEM_BYTES =
    1024 + (size_t)STAGES * (A_STAGE + B_STAGE) + EPI_WARPS * STAGE_OUT + 256;
static_assert(SMEM_BYTES <= 232448, "shared memory of one CTA");

struct Params {
  int M, N, KB;           // rows of D, MMA N, K blocks of 64
  int a_mn, b_mn;
  int m_tiles, n_tiles, splits;
  float* out;
  int out_mode;           // 0: out[m * ldo + n]; 1: out[(split * n_valid + n) * ldo + m]
  int ldo, n_valid;
  DevStatus* st;
};

// One launch runs up to two GEMMs (the dW and dx products of one backward call): tile ids
// [0, ntiles[0]) belong to job 0, the next ntiles[1] to job 1.  CTAs take tile ids from a
// global counter (zeroed by the kernel before), so the long dW tiles, handed out first, and
// the short dx tiles spread over the GPU together: dW's reads of x overlap dx's writes.
struct Jobs {
  Params p[2];
  int ntiles[2];
  int njobs;
  int* counter;
};

// Descriptor of an MN-major operand with the 128-byte swizzle: 64-element (128-byte) rows
// along MN, 8 K-rows per 1024-byte atom (stride byte offset), 64-column atoms lbo bytes apart
// along MN (leading byte offset).  Advancing K by 16 adds two atoms: 2048 bytes.
__device__ __forceinline__ uint64_t mn_desc(uint32_t saddr, uint32_t lbo) {
  uint64_t d = 0;
  d |= static_cast<uint64_t>((saddr & 0x3FFFFu) >> 4);
  d |= static_cast<uint64_t>((lbo >> 4) & 0x3FFFu) << 16;
  d |= static_cast<uint64_t>(1024 >> 4) << 32;
  d |= static_cast<uint64_t>(1) << 46;
  d |= static_cast<uint64_t>(2) << 61;
  return d;
}

struct Tile {
  int mt, nt, s, kb0, kb1;
};
__device__ __forceinline__ Tile tile_of(int tile, const Params& p) {
  Tile t;
  t.mt = tile % p.m_tiles;
  const int r = tile / p.m_tiles;
  t.nt = r % p.n_tiles;
  t.s = r / p.n_tiles;
  t.kb0 = static_cast<int>((long long)t.s * p.KB / p.splits);
  t.kb1 = static_cast<int>((long long)(t.s + 1) * p.KB / p.splits);
  return t;
}

__global__ void __launch_bounds__(THREADS, 1)
    router_grad_gemm_kernel(const __grid_constant__ CUtensorMap tmA0,
                            const __grid_constant__ CUtensorMap tmB0,
                            const __grid_constant__ CUtensorMap tmO0,
                            const __grid_constant__ CUtensorMap tmA1,
                            const __grid_constant__ CUtensorMap tmB1,
                            const __grid_constant__ CUtensorMap tmO1, const Jobs J) {
  pdl_prologue();
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  uint8_t* sA = smem;
  uint8_t* sB = smem + STAGES * A_STAGE;
  uint8_t* sOut = sB + STAGES * B_STAGE;
  uint64_t* bars = reinterpret_cast<uint64_t*>(sOut + EPI_WARPS * STAGE_OUT);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + NBARS);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  volatile int* queue = reinterpret_cast<volatile int*>(tmem_slot + 2);   // [NQ] tile ids

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t full0 = smem_u32(bars);
  const uint32_t empty0 = full0 + 8 * STAGES;
  const uint32_t tfull0 = empty0 + 8 * STAGES;
  const uint32_t tempty0 = tfull0 + 16;
  const uint32_t drain = tempty0 + 16;
  const uint32_t qfull0 = drain + 8;
  const uint32_t qempty0 = qfull0 + 8 * NQ;
  const Params* P = J.p;
  const int total = J.ntiles[0] + (J.njobs > 1 ? J.ntiles[1] : 0);

  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(full0 + 8 * s, 1);
      mbar_init(empty0 + 8 * s, 1);
    }
    for (int a = 0; a < 2; ++a) {
      mbar_init(tfull0 + 8 * a, 1);
      mbar_init(tempty0 + 8 * a, EPI_WARPS);
    }
    mbar_init(drain, 1);
    for (int q = 0; q < NQ; ++q) {
      mbar_init(qfull0 + 8 * q, 1);        // the producer publishes a tile id
      mbar_init(qempty0 + 8 * q, 1 + EPI_WARPS);   // the MMA issuer and every epilogue warp took it
    }
    *abort_flag = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  if (warp == 1) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                     smem_u32(tmem_slot)),
                 "r"(TMEM_COLS)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;

  // the i-th tile id this CTA works on (consumers): -1 ends the sequence
  auto next_tile = [&](int i, DevStatus* st, int where) -> int {
    const int q = i % NQ;
    if (!wait_bounded(qfull0 + 8 * q, static_cast<uint32_t>((i / NQ) & 1), abort_flag, st,
                      where, true))
      return -2;
    const int t = queue[q];
    return t;
  };

  if (warp == 0 && lane == 0) {
    // ------------------------------- TMA producer -------------------------------------------
    int stage = 0;
    uint32_t ph = 0;
    uint32_t issued = 0, last_par = 0;
    bool ok = true;
    for (int i = 0; ok; ++i) {
      int tile = atomicAdd(J.counter, 1);
      if (tile >= total) tile = -1;
      const int q = i % NQ;
      if (!wait_bounded(qempty0 + 8 * q, static_cast<uint32_t>(((i / NQ) & 1) ^ 1), abort_flag,
                        P[0].st, 27, true)) {
        ok = false;
        break;
      }
      queue[q] = tile;
      mbar_arrive(qfull0 + 8 * q);
      if (tile < 0) break;
      const int job = tile < J.ntiles[0] ? 0 : 1;
      const Params& p = P[job];
      const CUtensorMap* tmA = job ? &tmA1 : &tmA0;
      const CUtensorMap* tmB = job ? &tmB1 : &tmB0;
      const Tile ti = tile_of(tile - (job ? J.ntiles[0] : 0), p);
      const uint32_t bytes = A_STAGE + p.N * BK * 2;
      const int m0 = ti.mt * BM, n0 = ti.nt * p.N;
      for (int kb = ti.kb0; kb < ti.kb1; ++kb) {
        if (!wait_bounded(empty0 + 8 * stage, ph ^ 1u, abort_flag, p.st, 21, true)) {
          ok = false;
          break;
        }
        const uint32_t fb = full0 + 8 * stage;
        mbar_expect_tx(fb, bytes);
        const uint32_t a_dst = smem_u32(sA + stage * A_STAGE);
        const uint32_t b_dst = smem_u32(sB + stage * B_STAGE);
        if (p.a_mn) {
          tma_load_2d(a_dst, tmA, fb, m0, kb * BK);
          tma_load_2d(a_dst + MN_ATOM, tmA, fb, m0 + 64, kb * BK);
        } else {
          tma_load_2d(a_dst, tmA, fb, kb * BK, m0);
        }
        if (p.b_mn) {
          for (int i2 = 0; i2 < p.N / 64; ++i2)
            tma_load_2d(b_dst + i2 * MN_ATOM, tmB, fb, n0 + 64 * i2, kb * BK);
        } else {
          tma_load_2d(b_dst, tmB, fb, kb * BK, n0);
        }
        issued |= 1u << stage;
        last_par = (last_par & ~(1u << stage)) | (ph << stage);
        if (++stage == STAGES) {
          stage = 0;
          ph ^= 1u;
        }
      }
    }
    if (!ok) {
      for (int s = 0; s < STAGES; ++s)
        if ((issued >> s) & 1u)
          wait_bounded(full0 + 8 * s, (last_par >> s) & 1u, abort_flag, P[0].st, 25, false);
    }
  } else if (warp == 1 && lane == 0) {
    // ------------------------------- MMA issuer ---------------------------------------------
    const uint32_t a_lbo = MN_ATOM, b_lbo = MN_ATOM;
    int stage = 0, acc = 0;
    uint32_t ph = 0, aph = 0;
    bool ok = true;
    for (int i = 0; ok; ++i) {
      const int tile = next_tile(i, P[0].st, 28);
      mbar_arrive(qempty0 + 8 * (i % NQ));
      if (tile < 0) break;
      const int job = tile < J.ntiles[0] ? 0 : 1;
      const Params& p = P[job];
      const Tile ti = tile_of(tile - (job ? J.ntiles[0] : 0), p);
      const uint32_t idesc = idesc_bf16_f32(BM, p.N) | (static_cast<uint32_t>(p.a_mn) << 15) |
                             (static_cast<uint32_t>(p.b_mn) << 16);
      if (!wait_bounded(tempty0 + 8 * acc, aph ^ 1u, abort_flag, p.st, 22, true)) {
        ok = false;
        break;
      }
      tc_fence_after();
      const uint32_t dt = tmem_base + static_cast<uint32_t>(acc * 256);
      for (int kb = ti.kb0; kb < ti.kb1; ++kb) {
        if (!wait_bounded(full0 + 8 * stage, ph, abort_flag, p.st, 23, true)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t a0 = smem_u32(sA + stage * A_STAGE);
        const uint32_t b0 = smem_u32(sB + stage * B_STAGE);
#pragma unroll
        for (int kk = 0; kk < BK / 16; ++kk) {
          const uint64_t ad = p.a_mn ? mn_desc(a0 + kk * 2048, a_lbo) : sw128_desc(a0 + kk * 32);
          const uint64_t bd = p.b_mn ? mn_desc(b0 + kk * 2048, b_lbo) : sw128_desc(b0 + kk * 32);
          tc_mma(dt, ad, bd, idesc, (kb > ti.kb0 || kk != 0) ? 1u : 0u);
        }
        tc_commit(empty0 + 8 * stage);
        if (++stage == STAGES) {
          stage = 0;
          ph ^= 1u;
        }
      }
      if (!ok) break;
      tc_commit(tfull0 + 8 * acc);
      acc ^= 1;
      if (acc == 0) aph ^= 1u;
    }
    tc_commit(drain);
    wait_bounded(drain, 0u, abort_flag, P[0].st, 26, false);
  } else if (warp >= 2) {
    // ------------------------------- epilogue -----------------------------------------------
    const int q = warp & 3;                     // TMEM lane quarter this warp may read
    const int h = (warp - 2) >> 2;              // column half
    const int r = q * 32 + lane;
    const uint32_t buf = smem_u32(sOut) + (warp - 2) * STAGE_OUT;
    int acc = 0;
    uint32_t aph = 0;
    for (int i = 0;; ++i) {
      int tile = 0;
      if (lane == 0) {
        tile = next_tile(i, P[0].st, 29);
        mbar_arrive(qempty0 + 8 * (i % NQ));
      }
      tile = __shfl_sync(0xffffffffu, tile, 0);
      if (tile < 0) break;
      const int job = tile < J.ntiles[0] ? 0 : 1;
      const Params& p = P[job];
      const CUtensorMap* tmO = job ? &tmO1 : &tmO0;
      const Tile ti = tile_of(tile - (job ? J.ntiles[0] : 0), p);
      int ok = 1;
      if (lane == 0) ok = wait_bounded(tfull0 + 8 * acc, aph, abort_flag, p.st, 24, true) ? 1 : 0;
      ok = __shfl_sync(0xffffffffu, ok, 0);
      if (!ok) break;
      tc_fence_after();
      const uint32_t tb = tmem_base + static_cast<uint32_t>(acc * 256) +
                          (static_cast<uint32_t>(q * 32) << 16);
      const int m = ti.mt * BM + r;
      const bool live = m < p.M;
      const int n0 = ti.nt * p.N;
#pragma unroll 1
      for (int c = h * (p.N / 64); c < (h + 1) * (p.N / 64); ++c) {
        uint32_t vr[32];
        tmem_ld32(tb + c * 32, vr);
        if (p.out_mode == 0) {
          // The warp's 32 rows x 32 columns go to its shared buffer in the
          // 128-byte-swizzled layout (16-byte chunk j of row i at chunk j ^ (i & 7):
          // conflict-free), then leave as one TMA store; rows past M are clipped by the TMA.
          if (lane == 0) bulk_wait_read<0>();     // the previous store has read the buffer
          __syncwarp();
#pragma unroll
          for (int j = 0; j < 8; ++j)
            asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(
                             buf + lane * 128 + ((j ^ (lane & 7)) << 4)),
                         "r"(vr[4 * j]), "r"(vr[4 * j + 1]), "r"(vr[4 * j + 2]),
                         "r"(vr[4 * j + 3])
                         : "memory");
          fence_async_smem();
          __syncwarp();
          if (lane == 0) {
            tma_store_2d(tmO, buf, n0 + c * 32, ti.mt * BM + q * 32);
            bulk_commit();
          }
        } else if (live) {
          // column n of this row goes to row n of the transposed partial: lanes hold
          // consecutive m, so each store instruction writes 128 contiguous bytes
#pragma unroll
          for (int i2 = 0; i2 < 32; ++i2) {
            const int n = n0 + c * 32 + i2;
            if (n < p.n_valid)
              p.out[(static_cast<size_t>(ti.s) * p.n_valid + n) * p.ldo + m] =
                  __uint_as_float(vr[i2]);
          }
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(tempty0 + 8 * acc);
      acc ^= 1;
      if (acc == 0) aph ^= 1u;
    }
    if (lane == 0) bulk_wait_all();              // this warp's TMA stores are complete
  }

  __syncthreads();
  if (warp == 1) {
    __syncwarp();
    tc_fence_after();
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem_base),
                 "r"(TMEM_COLS)
                 : "memory");
  }
}

// One launch of up to two GEMMs (jobs); counter: a workspace int zeroed by the kernel before.
cudaError_t launch(const CUtensorMap* a, const CUtensorMap* b, const CUtensorMap* o,
                   const Params* p, int njobs, int* counter, cudaStream_t s) {
  cudaError_t e = smem_attr_once(reinterpret_cast<const void*>(router_grad_gemm_kernel),
                                 static_cast<int>(SMEM_BYTES));
  if (e != cudaSuccess) return e;
  Jobs J{};
  int total = 0;
  for (int j = 0; j < njobs; ++j) {
    J.p[j] = p[j];
    J.ntiles[j] = p[j].m_tiles * p[j].n_tiles * p[j].splits;
    total += J.ntiles[j];
  }
  J.njobs = njobs;
  J.counter = counter;
  const int k1 = njobs > 1 ? 1 : 0;
  int grid = num_sms();
  if (total < grid) grid = total;
  launch_pdl(router_grad_gemm_kernel, grid, THREADS, SMEM_BYTES, s, a[0], b[0], o[0], a[k1], b[k1],
             o[k1], J);
  return cudaGetLastError();
}

}  // namespace rg

// dW[e, c] = sum over slices s (in order) of part[s, e, c]
__global__ void splitk_reduce_kernel(const float4* __restrict__ part, float4* __restrict__ out,
                                     long long n4, int splits) {
  pdl_prologue();
  for (long long i = blockIdx.x * (long long)blockDim.x + threadIdx.x; i < n4;
       i += (long long)gridDim.x * blockDim.x) {
    float4 a = part[i];
    for (int s = 1; s < splits; ++s) {
      const float4 b = part[(long long)s * n4 + i];
      a.x += b.x; a.y += b.y; a.z += b.z; a.w += b.w;
    }
    out[i] = a;
  }
}

// float32 configuration: dW[e, c] = sum_t dg[t, e] x[t, c]; dx[t, c] = sum_e dg[t, e] W[e, c]
__global__ void dw_simt_kernel(const float* __restrict__ dg, const float* __restrict__ x,
                               float* __restrict__ dw, int T, int E, int d) {
  pdl_prologue();
  const long long n = (long long)E * d;
  for (long long i = blockIdx.x * (long long)blockDim.x + threadIdx.x; i < n;
       i += (long long)gridDim.x * blockDim.x) {
    const int e = static_cast<int>(i / d), cc = static_cast<int>(i % d);
    float acc = 0.0f;
    for (int t = 0; t < T; ++t) acc = fmaf(dg[(size_t)t * E + e], x[(size_t)t * d + cc], acc);
    dw[i] = acc;
  }
}
__global__ void dx_simt_kernel(const float* __restrict__ dg, const float* __restrict__ w,
                               float* __restrict__ dx, int T, int E, int d) {
  pdl_prologue();
  const long long n = (long long)T * d;
  for (long long i = blockIdx.x * (long long)blockDim.x + threadIdx.x; i < n;
       i += (long long)gridDim.x * blockDim.x) {
    const int t = static_cast<int>(i / d), cc = static_cast<int>(i % d);
    float acc = 0.0f;
    for (int e = 0; e < E; ++e) acc = fmaf(dg[(size_t)t * E + e], w[(size_t)e * d + cc], acc);
    dx[i] = acc;
  }
}

__global__ void bias_update_kernel(const float* __restrict__ f, float* __restrict__ bias, int T,
                                   int k, int E, float gamma) {
  pdl_prologue();
  const int e = blockIdx.x * blockDim.x + threadIdx.x;
  if (e >= E) return;
  // f = load / T rounded once to float32; load < 2^23, so rint(f * T) is the load exactly
  const long long load = llrint(static_cast<double>(f[e]) * static_cast<double>(T));
  const long long lhs = load * E, rhs = (long long)T * k;
  const float b = bias[e];
  if (lhs > rhs) bias[e] = b - gamma;
  else if (lhs < rhs) bias[e] = b + gamma;
}

// ---------------------------------------------------------------------------------------------
// Host side
// ---------------------------------------------------------------------------------------------
struct BwLayout {
  size_t status, counter, dg16, dgT, part, dg32, total;
  int splits;         // K slices of dW when the launch also runs dx
  int splits_alone;   // K slices of dW when it runs alone (no dx requested)
};

constexpr size_t kAlignBw = 256;
size_t align_bw(size_t v) { return (v + kAlignBw - 1) & ~(kAlignBw - 1); }

// K slices of the dW GEMM when it runs alone.  Cost in units of one K block of one tile:
// waves x (blocks per slice + 4 for the pipeline fill), plus the partials' write and read
// expressed in the same unit (one wave-wide K block moves num_sms x 16 KB of x).
int dw_splits_alone(const moe_config& c) {
  const int m_tiles = c.d_model / rg::BM;
  const int KB = ceil_div(c.T, rg::BK);
  const int sms = num_sms();
  const double unit_bytes = (double)sms * rg::A_STAGE;
  int best = 1;
  double best_cost = 1e300;
  for (int s = 1; s <= 32 && s <= KB; ++s) {
    const int waves = ceil_div(m_tiles * s, sms);
    double cost = waves * (double)(ceil_div(KB, s) + 4);
    if (s > 1) cost += (double)s * c.E * c.d_model * 8.0 / unit_bytes;
    if (cost < best_cost - 1e-9) {
      best_cost = cost;
      best = s;
    }
  }
  return best;
}

// K slices of the dW GEMM sharing its launch with dx, whose tiles fill the SMs around the dW
// tiles: the fewest slices whose tile (K blocks per slice) is no longer than the launch's
// balanced length, all dW and dx work over the SMs, with a dx tile (its 128 KB float32
// epilogue) counted as 7 K blocks of dW (measured rates).  Fewer slices write and reduce fewer
// partials: measured, V3 1 slice 107 us against 111 with 2, Mixtral 2 slices 33.5 us against
// 34.9 with 4, DeepSeekMoE 4 slices equal to 9.
int dw_splits_merged(const moe_config& c) {
  const int m_tiles = c.d_model / rg::BM;
  const int KB = ceil_div(c.T, rg::BK);
  const int bn = c.d_model % 256 == 0 ? 256 : 128;
  const double dx_units = (double)ceil_div(c.T, rg::BM) * (c.d_model / bn) * (bn == 256 ? 7.0 : 3.5);
  const double balanced = ((double)m_tiles * KB + dx_units) / num_sms();
  for (int s = 1; s <= 32 && s <= KB; ++s)
    if (ceil_div(KB, s) <= balanced) return s;
  return KB < 32 ? KB : 32;
}

BwLayout bw_layout(const moe_config& c) {
  BwLayout L{};
  size_t o = 0;
  auto take = [&](size_t bytes) {
    size_t at = o;
    o = align_bw(o + (bytes ? bytes : 1));
    return at;
  };
  const size_t T = c.T, E = c.E, d = c.d_model, E64 = e64_of(c.E), T64 = t64_of(c.T);
  L.status = take(sizeof(DevStatus));
  L.counter = take(sizeof(int));
  if (c.dtype == MOE_DTYPE_BF16) {
    L.splits = dw_splits_merged(c);
    L.splits_alone = dw_splits_alone(c);
    L.dg16 = take(T * E64 * 2);
    L.dgT = take(E64 * T64 * 2);
    const int smax = L.splits > L.splits_alone ? L.splits : L.splits_alone;
    L.part = take(smax > 1 ? (size_t)smax * E * d * 4 : 0);
  } else {
    L.splits = 1;
    L.splits_alone = 1;
    L.dg32 = take(T * E * 4);
  }
  L.total = o;
  return L;
}

template <typename P>
P* at_bw(void* ws, size_t off) {
  return reinterpret_cast<P*>(static_cast<unsigned char*>(ws) + off);
}

cudaError_t launch_scores(const ScoresArgs& a, cudaStream_t s) {
  const int grid = ceil_div(a.T, kBwTokens);
  const int V = ceil_div(a.E, 32);
  switch (V) {
#define MOE_BW_CASE(n) \
  case n: launch_pdl(router_bw_scores_kernel<n>, grid, kBwWarps * 32, 0, s, a); break;
    MOE_BW_CASE(1) MOE_BW_CASE(2) MOE_BW_CASE(3) MOE_BW_CASE(4)
    MOE_BW_CASE(5) MOE_BW_CASE(6) MOE_BW_CASE(7) MOE_BW_CASE(8)
#undef MOE_BW_CASE
    default: return cudaErrorInvalidValue;
  }
  return cudaGetLastError();
}

}  // namespace
}  // namespace moe

using namespace moe;

extern "C" {

int moe_router_backward_workspace_size(const moe_config* c, size_t* bytes) {
  int st = moe_check_config(c);
  if (st) return st;
  if (!bytes) return MOE_ERR_ARG;
  *bytes = bw_layout(*c).total;
  return MOE_OK;
}

int moe_router_backward(const moe_config* c, const void* x, const void* w_gate,
                        const float* logits, const int32_t* topk_idx, const float* d_topk_w,
                        const float* f, float alpha, float beta, float* d_logits,
                        float* d_w_gate, float* d_x, void* ws, void* stream) {
  int st = moe_check_config(c);
  if (st) return st;
  if (c->routing != MOE_ROUTE_TOKEN_CHOICE) return MOE_ERR_UNSUPPORTED;
  if (!x || !w_gate || !logits || !d_w_gate) return MOE_ERR_ARG;
  if (d_topk_w && !topk_idx) return MOE_ERR_ARG;
  if (alpha != 0.0f && !f) return MOE_ERR_ARG;
  if (!std::isfinite(alpha) || !std::isfinite(beta)) return MOE_ERR_ARG;
  if (!ws || reinterpret_cast<uintptr_t>(ws) % kAlignBw) return MOE_ERR_WORKSPACE;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const BwLayout L = bw_layout(*c);
  DevStatus* dst = at_bw<DevStatus>(ws, L.status);
  const bool tc = c->dtype == MOE_DTYPE_BF16;
  const int E64 = e64_of(c->E);
  const long long T64 = t64_of(c->T);

  ScoresArgs a{};
  a.T = c->T;
  a.E = c->E;
  a.E64 = E64;
  a.k = c->k;
  a.score = c->score;
  a.renorm = c->renormalize;
  a.T64 = T64;
  a.route_scale = c->route_scale;
  a.alpha = alpha;
  a.beta = beta;
  a.logits = logits;
  a.idx = topk_idx;
  a.d_w = d_topk_w;
  a.f = alpha != 0.0f ? f : nullptr;
  a.st = dst;
  float* dg32 = nullptr;
  if (tc) {
    a.d_logits = d_logits;
    a.dg16 = d_x ? at_bw<__nv_bfloat16>(ws, L.dg16) : nullptr;
    a.dgT = at_bw<__nv_bfloat16>(ws, L.dgT);
    a.tile_counter = at_bw<int>(ws, L.counter);
  } else {
    dg32 = d_logits ? d_logits : at_bw<float>(ws, L.dg32);
    a.d_logits = dg32;
  }
  cudaError_t e = launch_scores(a, s);
  if (e != cudaSuccess) return MOE_ERR_CUDA;

  const int T = c->T, E = c->E, d = c->d_model;
  if (!tc) {
    launch_pdl(dw_simt_kernel, num_sms() * 4, 256, 0, s, dg32, static_cast<const float*>(x), d_w_gate,
                                                 T, E, d);
    if (d_x)
      launch_pdl(dx_simt_kernel, num_sms() * 4, 256, 0, s, dg32, static_cast<const float*>(w_gate), d_x,
                                                   T, E, d);
    return cudaGetLastError() == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
  }

  // One launch for both gradient GEMMs (tiles handed out by a counter, dW's first):
  //   dW_gate = dg^T x: M = d (x MN-major), N = E64 (dg^T K-major), K = T, split along K
  //   dx = dg W_gate:   M = T (dg K-major), N = 256 (or 128) columns of d (W_gate MN-major),
  //                     K = E64
  CUtensorMap ma[2], mb[2], mo[2];
  rg::Params p[2] = {};
  if (!tc::make_map_box(&ma[0], x, (uint64_t)T, (uint64_t)d, 64) ||
      !tc::make_map_strided(&mb[0], a.dgT, (uint64_t)E64, (uint64_t)T, (uint64_t)T64, E64))
    return MOE_ERR_CUDA;
  mo[0] = mb[0];                      // transposed-partial mode: no store map
  p[0].M = d;
  p[0].N = E64;
  p[0].KB = ceil_div(T, rg::BK);
  p[0].a_mn = 1;
  p[0].b_mn = 0;
  p[0].m_tiles = d / rg::BM;
  p[0].n_tiles = 1;
  const int splits = d_x ? L.splits : L.splits_alone;
  p[0].splits = splits;
  p[0].out_mode = 1;
  p[0].ldo = d;
  p[0].n_valid = E;
  p[0].st = dst;
  p[0].out = splits > 1 ? at_bw<float>(ws, L.part) : d_w_gate;
  int njobs = 1;
  if (d_x) {
    const int bn = d % 256 == 0 ? 256 : 128;
    if (!tc::make_map_box(&ma[1], a.dg16, (uint64_t)T, (uint64_t)E64, 128) ||
        !tc::make_map_box(&mb[1], w_gate, (uint64_t)E, (uint64_t)d, 64) ||
        !tc::make_map_f32_store(&mo[1], d_x, (uint64_t)T, (uint64_t)d))
      return MOE_ERR_CUDA;
    p[1].M = T;
    p[1].N = bn;
    p[1].KB = E64 / rg::BK;
    p[1].a_mn = 0;
    p[1].b_mn = 1;
    p[1].m_tiles = ceil_div(T, rg::BM);
    p[1].n_tiles = d / bn;
    p[1].splits = 1;
    p[1].out = d_x;
    p[1].out_mode = 0;
    p[1].ldo = d;
    p[1].n_valid = d;
    p[1].st = dst;
    njobs = 2;
  }
  e = rg::launch(ma, mb, mo, p, njobs, at_bw<int>(ws, L.counter), s);
  if (e == cudaSuccess && splits > 1) {
    const long long n4 = (long long)E * d / 4;
    launch_pdl(splitk_reduce_kernel, num_sms() * 4, 256, 0, s, at_bw<const float4>(ws, L.part),
                                                        reinterpret_cast<float4*>(d_w_gate), n4,
                                                        splits);
    e = cudaGetLastError();
  }
  if (e != cudaSuccess) return MOE_ERR_CUDA;
  return MOE_OK;
}

int moe_bias_update(const moe_config* c, const float* f, float* bias, float gamma, void* stream) {
  int st = moe_check_config(c);
  if (st) return st;
  if (!f || !bias) return MOE_ERR_ARG;
  if (!std::isfinite(gamma)) return MOE_ERR_ARG;
  if ((long long)c->T * c->k >= (1ll << 23)) return MOE_ERR_SHAPE;
  launch_pdl(bias_update_kernel, ceil_div(c->E, 256), 256, 0, static_cast<cudaStream_t>(stream),
      
      f, bias, c->T, c->k, c->E, gamma);
  return cudaGetLastError() == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
}

}  // extern "C"
