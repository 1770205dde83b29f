// Expert GEMMs for decode-sized batches (few tokens per expert), tcgen05, sm_103a.
//
// Same SwiGLU products as the prefill kernels ["Systems for Mixture-of-Experts Models" §5.2],
// computed transposed so that the weights fill the MMA's M = 128 rows and the few tokens of an
// expert fill N (16..128):
//   GEMM 1:  G^T = W1_e X^T and U^T = W3_e X^T  ->  h[t, f] = SiLU(G[f,t]) * U[f,t]
//   GEMM 2:  Y^T = W2_e H^T (two 128-row halves of a 256-row W2 block)
// At decode sizes the layer is bound by reading the touched experts' weights once
// ("Systems for MoE Models" §1.4: a batch touches about E(1-(1-k/E)^B) experts), so each tile
// streams 256 weight rows through a 4-stage TMA ring while the token rows stay small.  The
// shared experts are one more entry of the same tile list (their token rows are appended to the
// expert-ordered rows), so every SM streams weights even for a single token.
//
// Tile list: entry j in [0, E) is routed expert j, entry E the shared expert (if any); entry j
// has n_j rows, cut into chunks of NP rows; its tiles are (weight block, chunk) with the chunk
// fastest so the CTAs reading one weight block run together.  Every wait is bounded as in the
// prefill kernels.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp8.h>

#include "common.cuh"
#include "kernels.h"
#include "tc_ptx.cuh"

namespace moe {
namespace dec {

using namespace tc;

constexpr int BK = 64;
constexpr int MAX_STAGES = 8;
constexpr int A_BOX = 128 * BK * 2;           // 16 KB: 128 weight rows
constexpr int A_STAGE = 2 * A_BOX;            // two 128-row weight blocks
constexpr int NP_MAX = 128;                   // token rows per chunk (B box height)
constexpr int TMEM_COLS = 512;                // 2 buffers x (2 x 128 columns)
constexpr int THREADS = 192;
constexpr int MAX_J = 257;
constexpr int NBARS = 2 * MAX_STAGES + 5;
constexpr size_t CTRL_BYTES = 8 * NBARS + 16 + (MAX_J + 1) * 4;
constexpr size_t SMEM_LIMIT = 227 * 1024;
// The ring's stage holds 256 weight rows and the largest token chunk (np_max rows) of one
// 64-wide K slice; as many stages as fit (up to 8): 6 for 16-row chunks, 4 for 128-row chunks.
inline int stage_bytes(int np_max) { return A_STAGE + ((np_max * BK * 2 + 1023) / 1024) * 1024; }
inline int num_stages(int np_max) {
  const int n = static_cast<int>((SMEM_LIMIT - 1024 - CTRL_BYTES) / stage_bytes(np_max));
  return n < MAX_STAGES ? n : MAX_STAGES;
}

struct Params {
  const int32_t* offsets;   // [E+1] routed row offsets
  int E;
  int has_shared;
  int T;                    // tokens (rows of the shared entry, appended after offsets[E])
  int NP;                   // routed chunk rows = routed B box height (16, 32, 64 or 128)
  int NPs;                  // shared chunk rows = shared B box height
  int gemm;                 // 1 = gate/up + SwiGLU, 2 = down
  int K_routed, K_shared;   // reduction lengths (GEMM 1: d, d; GEMM 2: F, Fs)
  int wb_routed, wb_shared; // weight blocks per entry (GEMM 1: F/128, Fs/128; GEMM 2: d/256)
  int a_rows_routed;        // rows of A per routed expert (GEMM 1: 2F; GEMM 2: d)
  int up_routed, up_shared; // GEMM 1: offset of the up rows (F, Fs)
  void* out;                // GEMM 1: h bf16 [rows, ldo]; GEMM 2: y f32 [rows, ldo]
  float* out_shared;        // GEMM 2: shared output f32 [T, ldo]
  int ldo;
  int ksplit;               // K is cut into ksplit slices, each a tile of its own
  float* gu;                // GEMM 1 with ksplit > 1: fp32 gate | up partials [ksplit][rows][2 ldo]
  size_t part_stride;       // elements between consecutive K-slice partials of the outputs
  size_t shared_stride;     // GEMM 2: elements between K-slice partials of out_shared
  int stages;               // ring depth
  int stage;                // bytes per ring stage
  int fp8;                  // operands are E4M3 codes (kind::f8f6f4) instead of bf16
  int bk;                   // K elements per ring stage: 64 (bf16) or 128 (E4M3), 128 bytes
  const float* sa;          // E4M3: scale of each routed weight row (row index of A)
  const float* sa_shared;   // E4M3: scale of each shared weight row
  const float* sb;          // E4M3: scale of each token row (row index of B)
  float* hf;                // GEMM 1, E4M3, one K slice: h = SiLU(g) * u in float32 [rows, ldo]
  DevStatus* st;
};

struct DTile {
  int j, wb, ks, row0, n;   // entry, weight block, K slice, first row of the chunk, valid rows
};

__device__ __forceinline__ int entry_rows(const Params& p, int j) {
  return j < p.E ? p.offsets[j + 1] - p.offsets[j] : p.T;
}
// First row of an entry; with no routed entries (E = 0, the router logits) the shared entry's
// rows start at 0 and offsets may be null.
__device__ __forceinline__ int shared_row0(const Params& p) {
  return p.E > 0 ? p.offsets[p.E] : 0;
}
__device__ __forceinline__ int entry_row0(const Params& p, int j) {
  return j < p.E ? p.offsets[j] : shared_row0(p);
}

__device__ __forceinline__ int entry_np(const Params& p, int j) {
  return j < p.E ? p.NP : p.NPs;
}

__device__ __forceinline__ DTile decode_dtile(int tile, const Params& p, const int* prefix,
                                              int J) {
  int lo = 0, hi = J;
  while (hi - lo > 1) {
    const int mid = (lo + hi) >> 1;
    if (prefix[mid] <= tile) lo = mid; else hi = mid;
  }
  DTile t;
  t.j = lo;
  const int n_j = entry_rows(p, lo);
  const int np = entry_np(p, lo);
  const int chunks = ceil_div(n_j, np);
  int tt = tile - prefix[lo];
  const int c = tt % chunks;          // chunk fastest: CTAs on one weight slice run together
  tt /= chunks;
  t.ks = tt % p.ksplit;
  t.wb = tt / p.ksplit;
  t.row0 = entry_row0(p, lo) + c * np;
  t.n = min(np, n_j - c * np);
  return t;
}

__global__ void __launch_bounds__(THREADS, 1)
    decode_gemm_kernel(const __grid_constant__ CUtensorMap tmA,
                       const __grid_constant__ CUtensorMap tmAs,
                       const __grid_constant__ CUtensorMap tmB,
                       const __grid_constant__ CUtensorMap tmBs, const Params p) {
  pdl_prologue();
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  const int STAGES = p.stages;
  const int STAGE = p.stage;
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + STAGES * STAGE);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + NBARS);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  int* prefix = reinterpret_cast<int*>(tmem_slot + 4);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t full0 = smem_u32(bars);
  const uint32_t empty0 = full0 + 8 * STAGES;
  const uint32_t tfull0 = empty0 + 8 * STAGES;
  const uint32_t tempty0 = tfull0 + 16;
  const uint32_t drain = tempty0 + 16;
  const int J = p.E + (p.has_shared ? 1 : 0);

  for (int j = threadIdx.x; j < J; j += blockDim.x)
    prefix[j + 1] = ceil_div(entry_rows(p, j), entry_np(p, j)) *
                    (j < p.E ? p.wb_routed : p.wb_shared) * p.ksplit;
  __syncthreads();
  if (threadIdx.x == 0) {
    prefix[0] = 0;
    for (int j = 1; j <= J; ++j) prefix[j] += prefix[j - 1];
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(full0 + 8 * s, 1);
      mbar_init(empty0 + 8 * s, 1);
    }
    for (int a = 0; a < 2; ++a) {
      mbar_init(tfull0 + 8 * a, 1);
      mbar_init(tempty0 + 8 * a, 4);
    }
    mbar_init(drain, 1);
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
  const int total = prefix[J];

  if (warp == 0 && lane == 0) {
    // ------------------------------- TMA producer -------------------------------------------
    int stage = 0;
    uint32_t ph = 0, issued = 0, last_par = 0;
    bool ok = true;
    for (int tile = blockIdx.x; ok && tile < total; tile += gridDim.x) {
      const DTile t = decode_dtile(tile, p, prefix, J);
      const bool sh = t.j >= p.E;
      const CUtensorMap* am = sh ? &tmAs : &tmA;
      const CUtensorMap* bm = sh ? &tmBs : &tmB;
      const uint32_t b_bytes = static_cast<uint32_t>(entry_np(p, t.j)) * BK * 2;
      int a0, a1;
      if (p.gemm == 1) {
        const int base = sh ? 0 : t.j * p.a_rows_routed;
        a0 = base + t.wb * 128;
        a1 = a0 + (sh ? p.up_shared : p.up_routed);
      } else {
        a0 = (sh ? 0 : t.j * p.a_rows_routed) + t.wb * 256;
        a1 = a0 + 128;
      }
      const int KB = (sh ? p.K_shared : p.K_routed) / p.bk;
      const int kb0 = t.ks * KB / p.ksplit, kb1 = (t.ks + 1) * KB / p.ksplit;
      for (int kb = kb0; kb < kb1; ++kb) {
        if (!wait_bounded(empty0 + 8 * stage, ph ^ 1u, abort_flag, p.st, 21, true)) {
          ok = false;
          break;
        }
        const uint32_t fb = full0 + 8 * stage;
        const uint32_t sa = smem_u32(smem + stage * STAGE);
        mbar_expect_tx(fb, A_STAGE + b_bytes);
        tma_load_2d(sa, am, fb, kb * p.bk, a0);
        tma_load_2d(sa + A_BOX, am, fb, kb * p.bk, a1);
        tma_load_2d(sa + A_STAGE, bm, fb, kb * p.bk, t.row0);
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
          wait_bounded(full0 + 8 * s, (last_par >> s) & 1u, abort_flag, p.st, 25, false);
    }
  } else if (warp == 1 && lane == 0) {
    // ------------------------------- MMA issuer ---------------------------------------------
    int stage = 0, acc = 0;
    uint32_t ph = 0, aph = 0;
    bool ok = true;
    for (int tile = blockIdx.x; ok && tile < total; tile += gridDim.x) {
      const DTile t = decode_dtile(tile, p, prefix, J);
      const int n16 = (t.n + 15) & ~15;
      const uint32_t idesc = p.fp8 ? idesc_e4m3_f32(128, n16) : idesc_bf16_f32(128, n16);
      const int KB = (t.j >= p.E ? p.K_shared : p.K_routed) / p.bk;
      const int kb0 = t.ks * KB / p.ksplit, kb1 = (t.ks + 1) * KB / p.ksplit;
      if (!wait_bounded(tempty0 + 8 * acc, aph ^ 1u, abort_flag, p.st, 22, true)) {
        ok = false;
        break;
      }
      tc_fence_after();
      const uint32_t d0 = tmem_base + static_cast<uint32_t>(acc * 256);
      for (int kb = kb0; kb < kb1; ++kb) {
        if (!wait_bounded(full0 + 8 * stage, ph, abort_flag, p.st, 23, true)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t sa = smem_u32(smem + stage * STAGE);
        const uint32_t sb = sa + A_STAGE;
        // four MMAs per 128-byte stage row: K = 16 bf16 or K = 32 E4M3 each, 32 bytes apart
        if (p.fp8) {
#pragma unroll
          for (int kk = 0; kk < 4; ++kk) {
            const uint64_t bdesc = sw128_desc(sb + kk * 32);
            const uint32_t accum = (kb != kb0 || kk != 0) ? 1u : 0u;
            tc_mma_f8(d0, sw128_desc(sa + kk * 32), bdesc, idesc, accum);
            tc_mma_f8(d0 + 128, sw128_desc(sa + A_BOX + kk * 32), bdesc, idesc, accum);
          }
        } else {
#pragma unroll
          for (int kk = 0; kk < 4; ++kk) {
            const uint64_t bdesc = sw128_desc(sb + kk * 32);
            const uint32_t accum = (kb != kb0 || kk != 0) ? 1u : 0u;
            tc_mma(d0, sw128_desc(sa + kk * 32), bdesc, idesc, accum);
            tc_mma(d0 + 128, sw128_desc(sa + A_BOX + kk * 32), bdesc, idesc, accum);
          }
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
    wait_bounded(drain, 0u, abort_flag, p.st, 26, false);
  } else if (warp >= 2) {
    // ------------------------------- epilogue -----------------------------------------------
    // Thread = one weight row f (TMEM lane); columns = tokens.  For each token the warp's 32
    // lanes write 32 consecutive outputs.
    const int q = warp & 3;
    const int f = q * 32 + lane;
    int acc = 0;
    uint32_t aph = 0;
    for (int tile = blockIdx.x; tile < total; tile += gridDim.x) {
      const DTile t = decode_dtile(tile, p, prefix, J);
      int ok = 1;
      if (lane == 0) ok = wait_bounded(tfull0 + 8 * acc, aph, abort_flag, p.st, 24, true) ? 1 : 0;
      ok = __shfl_sync(0xffffffffu, ok, 0);
      if (!ok) break;
      tc_fence_after();
      const uint32_t tb = tmem_base + static_cast<uint32_t>(acc * 256) +
                          (static_cast<uint32_t>(q * 32) << 16);
      const bool sh = t.j >= p.E;
      // E4M3: this thread's two weight rows carry scales s_lo, s_hi; token rows carry sb[row]
      float s_lo = 1.0f, s_hi = 1.0f;
      if (p.fp8) {
        const float* sa = sh ? p.sa_shared : p.sa;
        int a0;
        if (p.gemm == 1) {
          a0 = (sh ? 0 : t.j * p.a_rows_routed) + t.wb * 128 + f;
          s_lo = sa[a0];
          s_hi = sa[a0 + (sh ? p.up_shared : p.up_routed)];
        } else {
          a0 = (sh ? 0 : t.j * p.a_rows_routed) + t.wb * 256 + f;
          s_lo = sa[a0];
          s_hi = sa[a0 + 128];
        }
      }
#pragma unroll 1
      for (int c0 = 0; c0 < t.n; c0 += 32) {
        uint32_t lo[32], hi[32];
        tmem_ld32(tb + c0, lo);
        tmem_ld32(tb + 128 + c0, hi);
        const int m = min(32, t.n - c0);
        if (p.fp8) {
#pragma unroll
          for (int i = 0; i < 32; ++i) {
            if (i < m) {
              const float sr = p.sb[t.row0 + c0 + i];
              lo[i] = __float_as_uint(__uint_as_float(lo[i]) * s_lo * sr);
              hi[i] = __float_as_uint(__uint_as_float(hi[i]) * s_hi * sr);
            }
          }
        }
        if (p.gemm == 1 && p.hf) {
          // one K slice: h in float32, formed as the quantising pass would form it
#pragma unroll
          for (int i = 0; i < 32; ++i) {
            if (i < m) {
              const float g = __uint_as_float(lo[i]), u = __uint_as_float(hi[i]);
              p.hf[static_cast<size_t>(t.row0 + c0 + i) * p.ldo + t.wb * 128 + f] =
                  (g / (1.0f + expf(-g))) * u;
            }
          }
        } else if (p.gemm == 1 && p.gu == nullptr) {
          __nv_bfloat16* out = static_cast<__nv_bfloat16*>(p.out);
#pragma unroll
          for (int i = 0; i < 32; ++i) {
            if (i < m) {
              const float g = __uint_as_float(lo[i]), u = __uint_as_float(hi[i]);
              const float hv = (g / (1.0f + expf(-g))) * u;
              out[static_cast<size_t>(t.row0 + c0 + i) * p.ldo + t.wb * 128 + f] =
                  __float2bfloat16_rn(hv);
            }
          }
        } else if (p.gemm == 1) {
          // raw gate | up partial sums of this K slice; a finalize pass forms SiLU(g) * u
          float* gu = p.gu + static_cast<size_t>(t.ks) * p.part_stride;
#pragma unroll
          for (int i = 0; i < 32; ++i) {
            if (i < m) {
              float* o = gu + static_cast<size_t>(t.row0 + c0 + i) * (2 * p.ldo) + t.wb * 128 + f;
              o[0] = __uint_as_float(lo[i]);
              o[p.ldo] = __uint_as_float(hi[i]);
            }
          }
        } else {
          float* out = sh ? p.out_shared + static_cast<size_t>(t.ks) * p.shared_stride
                          : static_cast<float*>(p.out) + static_cast<size_t>(t.ks) * p.part_stride;
          const int rbase = sh ? t.row0 - shared_row0(p) : t.row0;
#pragma unroll
          for (int i = 0; i < 32; ++i) {
            if (i < m) {
              float* o = out + static_cast<size_t>(rbase + c0 + i) * p.ldo + t.wb * 256 + f;
              o[0] = __uint_as_float(lo[i]);
              o[128] = __uint_as_float(hi[i]);
            }
          }
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(tempty0 + 8 * acc);
      acc ^= 1;
      if (acc == 0) aph ^= 1u;
    }
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

// h[r][f] = SiLU(sum_s gate_s[r][f]) * sum_s up_s[r][f], slices summed in order s = 0.. ;
// routed rows r < offsets[E] have F columns, the appended shared rows F_shared.
__global__ void __launch_bounds__(256) swiglu_finalize_kernel(const float* __restrict__ gu,
                                                             size_t part_stride, int S,
                                                             const int32_t* __restrict__ offsets,
                                                             int E, int T, int F, int Fs, int ldo,
                                                             __nv_bfloat16* __restrict__ h) {
  pdl_prologue();
  const int nk = offsets[E];
  const int rows = nk + T;
  const size_t total = static_cast<size_t>(rows) * ldo;
  for (size_t i = blockIdx.x * (size_t)blockDim.x + threadIdx.x; i < total;
       i += (size_t)gridDim.x * blockDim.x) {
    const int r = static_cast<int>(i / ldo), f = static_cast<int>(i - (size_t)r * ldo);
    if (f >= (r < nk ? F : Fs)) continue;
    float g = 0.f, u = 0.f;
    const float* src = gu + static_cast<size_t>(r) * (2 * ldo) + f;
    for (int s0 = 0; s0 < S; s0 += 8) {            // eight slices' loads in flight, then adds
      float qg[8], qu[8];
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        if (s0 + i < S) {
          qg[i] = src[(s0 + i) * part_stride];
          qu[i] = src[(s0 + i) * part_stride + ldo];
        }
      }
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        if (s0 + i >= S) break;
        g += qg[i];
        u += qu[i];
      }
    }
    h[i] = __float2bfloat16_rn((g / (1.0f + expf(-g))) * u);
  }
}

// Gate and up sums over S K slices (part_stride apart), in slice order, of two groups of four
// consecutive columns (pa, and pb when two): the loads of two slices of both groups are in
// flight together.
__device__ __forceinline__ void add4(float4& a, const float4& b) {
  a.x += b.x; a.y += b.y; a.z += b.z; a.w += b.w;
}
__device__ __forceinline__ void sum_slices4x2(const float4* pa, const float4* pb, bool two,
                                              size_t ps4, size_t up4, int S, float4 (&g)[2],
                                              float4 (&u)[2]) {
  g[0] = pa[0];
  u[0] = pa[up4];
  if (two) {
    g[1] = pb[0];
    u[1] = pb[up4];
  }
  for (int sl = 1; sl < S; sl += 2) {
    const bool more = sl + 1 < S;
    const float4 ga = pa[sl * ps4], ua = pa[sl * ps4 + up4];
    float4 gb = ga, ub = ua, gc = ga, uc = ua, gd = ga, ud = ua;
    if (more) { gb = pa[(sl + 1) * ps4]; ub = pa[(sl + 1) * ps4 + up4]; }
    if (two) {
      gc = pb[sl * ps4];
      uc = pb[sl * ps4 + up4];
      if (more) { gd = pb[(sl + 1) * ps4]; ud = pb[(sl + 1) * ps4 + up4]; }
    }
    add4(g[0], ga); add4(u[0], ua);
    if (more) { add4(g[0], gb); add4(u[0], ub); }
    if (two) {
      add4(g[1], gc); add4(u[1], uc);
      if (more) { add4(g[1], gd); add4(u[1], ud); }
    }
  }
}

__device__ __forceinline__ uint32_t cluster_ctarank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}
__device__ __forceinline__ uint32_t cluster_nctarank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_nctarank;" : "=r"(r));
  return r;
}
__device__ __forceinline__ float ld_cluster_f32(const float* local, uint32_t rank) {
  uint32_t remote;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;"
               : "=r"(remote)
               : "r"(static_cast<uint32_t>(__cvta_generic_to_shared(local))), "r"(rank));
  float v;
  asm volatile("ld.shared::cluster.f32 %0, [%1];" : "=f"(v) : "r"(remote) : "memory");
  return v;
}

// E4M3 path: h[r][:] = SiLU(sum_s gate_s[r][:]) * sum_s up_s[r][:] (slices in order), then the
// row is quantised as every E4M3 operand: amax = max |h|, inv = 448 / amax, code = e4m3(h * inv)
// (round to nearest even, saturating), scale = amax / 448; a zero row gets codes 0, scale 0.
// With one K slice the gate/up GEMM has formed h itself (h_ready: gu is one float32 plane).
// Row r is split over the CTAs of a cluster (a cluster of one CTA when rows are many), one
// column range each; h stays in shared memory between the two passes, and the row's amax is
// the maximum of the CTAs' maxima, read through distributed shared memory.  A maximum does not
// depend on how the row is split, so the bytes do not either.
__global__ void __launch_bounds__(1024, 1) swiglu_quant_kernel(const float* __restrict__ gu,
                                                           size_t part_stride, int S,
                                                           const int32_t* __restrict__ offsets,
                                                           int E, int n_shared_rows, int F,
                                                           int Fs, int ldo, int h_ready,
                                                           uint8_t* __restrict__ h8,
                                                           float* __restrict__ hs) {
  pdl_prologue();
  extern __shared__ float4 hrow4[];
  __shared__ float red[32];
  __shared__ float cta_amax, row_amax;
  const uint32_t crank = cluster_ctarank(), csize = cluster_nctarank();
  const int nk = offsets[E];
  const int r = blockIdx.x / csize;
  if (r >= nk + n_shared_rows) return;        // the whole cluster shares r
  const int F4 = (r < nk ? F : Fs) / 4;
  const int chunk = ceil_div(F4, static_cast<int>(csize));
  const int f0 = static_cast<int>(crank) * chunk;
  const int f1 = min(F4, f0 + chunk);
  // h_ready: gu holds h itself, one float32 plane [rows, ldo] written by the gate/up GEMM
  const float4* src =
      reinterpret_cast<const float4*>(gu + static_cast<size_t>(r) * (h_ready ? ldo : 2 * ldo));
  const size_t ps4 = part_stride / 4, up4 = static_cast<size_t>(ldo) / 4;
  float amax = 0.f;
  for (int f = f0 + threadIdx.x; f < f1; f += 2 * blockDim.x) {
    const int fb = f + blockDim.x;
    const bool two = fb < f1;
    float4 hh[2];
    if (h_ready) {
      hh[0] = src[f];
      if (two) hh[1] = src[fb];
    } else {
      float4 g[2], u[2];
      sum_slices4x2(src + f, src + (two ? fb : f), two, ps4, up4, S, g, u);
#pragma unroll
      for (int c = 0; c < 2; ++c) {
        hh[c].x = (g[c].x / (1.0f + expf(-g[c].x))) * u[c].x;
        hh[c].y = (g[c].y / (1.0f + expf(-g[c].y))) * u[c].y;
        hh[c].z = (g[c].z / (1.0f + expf(-g[c].z))) * u[c].z;
        hh[c].w = (g[c].w / (1.0f + expf(-g[c].w))) * u[c].w;
      }
    }
#pragma unroll
    for (int c = 0; c < 2; ++c) {
      if (c == 1 && !two) break;
      const float4 hv = hh[c];
      hrow4[(c ? fb : f) - f0] = hv;
      amax = fmaxf(amax,
                   fmaxf(fmaxf(fabsf(hv.x), fabsf(hv.y)), fmaxf(fabsf(hv.z), fabsf(hv.w))));
    }
  }
  amax = warp_max(amax);
  const int nw = blockDim.x >> 5;
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = amax;
  __syncthreads();
  if (threadIdx.x == 0) {
    float m = red[0];
    for (int w = 1; w < nw; ++w) m = fmaxf(m, red[w]);
    cta_amax = m;
  }
  // every CTA's maximum is visible cluster-wide after this barrier
  asm volatile("barrier.cluster.arrive.release.aligned;\n"
               "barrier.cluster.wait.acquire.aligned;" ::: "memory");
  if (threadIdx.x < 32) {                     // lane q reads CTA q's maximum (csize <= 8)
    float m = threadIdx.x < csize ? ld_cluster_f32(&cta_amax, threadIdx.x) : 0.f;
    m = warp_max(m);
    if (threadIdx.x == 0) row_amax = m;
  }
  __syncthreads();
  // done reading the other CTAs' shared memory; no CTA leaves before all have arrived here
  asm volatile("barrier.cluster.arrive.release.aligned;" ::: "memory");
  amax = row_amax;
  const float inv = amax > 0.f ? 448.0f / amax : 0.f;
  uint32_t* dst = reinterpret_cast<uint32_t*>(h8 + static_cast<size_t>(r) * ldo);
  for (int f = f0 + threadIdx.x; f < f1; f += blockDim.x) {
    const float4 hv = hrow4[f - f0];
    const uint32_t q0 = __nv_cvt_float2_to_fp8x2(make_float2(hv.x * inv, hv.y * inv),
                                                 __NV_SATFINITE, __NV_E4M3);
    const uint32_t q1 = __nv_cvt_float2_to_fp8x2(make_float2(hv.z * inv, hv.w * inv),
                                                 __NV_SATFINITE, __NV_E4M3);
    dst[f] = (q0 & 0xFFFFu) | (q1 << 16);
  }
  if (crank == 0 && threadIdx.x == 0) hs[r] = amax > 0.f ? amax / 448.0f : 0.f;
  asm volatile("barrier.cluster.wait.acquire.aligned;" ::: "memory");
}

// Cluster size for the quantising finalize: split each row over up to 8 CTAs while the rows
// alone give fewer than two CTAs per SM and every CTA keeps at least 32 four-column groups.
static int swiglu_quant_cluster(int rows, int F4) {
  int cn = 1;
  while (cn < 8 && static_cast<long long>(rows) * cn < 2ll * num_sms() && F4 / (2 * cn) >= 32)
    cn *= 2;
  return cn;
}

static cudaError_t launch(const CUtensorMap& a, const CUtensorMap& as, const CUtensorMap& b,
                          const CUtensorMap& bs, Params p, int upper_tiles, cudaStream_t s) {
  cudaError_t e = smem_attr_once(reinterpret_cast<const void*>(decode_gemm_kernel),
                                 static_cast<int>(SMEM_LIMIT));
  if (e != cudaSuccess) return e;
  const int np_max = p.NP > p.NPs ? p.NP : p.NPs;
  p.stage = stage_bytes(np_max);
  p.stages = num_stages(np_max);
  const size_t smem = 1024 + static_cast<size_t>(p.stages) * p.stage + CTRL_BYTES;
  int grid = num_sms();
  if (upper_tiles < grid) grid = upper_tiles;
  if (grid < 1) grid = 1;
  launch_pdl(decode_gemm_kernel, grid, THREADS, smem, s, a, as, b, bs, p);
  return cudaGetLastError();
}

// logits[t][e] = sum over K slices of part[s][t][e] in a fixed order: the slices are cut into
// 8 consecutive groups, each group summed in slice order by its own thread (its loads in flight
// together), then the group sums added in group order.  A CTA covers 32 four-column outputs.
constexpr int kReduceGroups = 8;
__global__ void __launch_bounds__(256) router_slices_reduce_kernel(const float4* __restrict__ part,
                                                                  int S, size_t stride4,
                                                                  size_t n4,
                                                                  float4* __restrict__ logits) {
  pdl_prologue();
  __shared__ float4 gsum[kReduceGroups][32];
  const int o = threadIdx.x & 31, grp = threadIdx.x >> 5;
  const size_t i = blockIdx.x * (size_t)32 + o;
  const int per = (S + kReduceGroups - 1) / kReduceGroups;
  const int s0 = grp * per, s1 = min(S, s0 + per);
  if (i < n4 && s0 < s1) {
    float4 q[8];
#pragma unroll
    for (int j = 0; j < 8; ++j)
      if (s0 + j < s1) q[j] = part[(s0 + j) * stride4 + i];
    float4 v = q[0];
#pragma unroll
    for (int j = 1; j < 8; ++j)
      if (s0 + j < s1) add4(v, q[j]);
    for (int s = s0 + 8; s < s1; ++s) add4(v, part[s * stride4 + i]);
    gsum[grp][o] = v;
  }
  __syncthreads();
  if (grp != 0 || i >= n4) return;
  float4 v = gsum[0][o];
  for (int g = 1; g < kReduceGroups && g * per < S; ++g) add4(v, gsum[g][o]);
  logits[i] = v;
}

}  // namespace dec

// Router logits of a decode-sized batch with E a multiple of 256: g^T = W_gate x^T on the
// decode kernel (W_gate's rows fill the MMA's M as one shared entry of E / 256 weight blocks,
// the tokens fill N), with K = d cut into slices so that W_gate's stream spreads over many
// SMs; a second pass sums the slices in order.
int router_split(const moe_config& c) {
  if (c.dtype != MOE_DTYPE_BF16 || c.E % 256 != 0 || c.d_model % 256 != 0) return 0;
  if (c.T <= 16 || c.T > kRouterSplitMaxT) return 0;
  const int chunks = ceil_div(c.T, 128);
  const int kb = c.d_model / dec::BK;
  int S = num_sms() / (chunks * (c.E / 256));
  if (S > kb / 4) S = kb / 4;                       // at least four K blocks per slice
  return S < 1 ? 1 : S;
}

size_t router_split_bytes(const moe_config& c) {
  const int S = router_split(c);
  return S ? (size_t)S * c.T * c.E * 4 : 0;
}

cudaError_t launch_router_split(const moe_config& c, const void* x, const void* w_gate,
                                float* part, float* logits, DevStatus* st, cudaStream_t s) {
  using namespace dec;
  const int S = router_split(c);
  if (S < 1 || !part) return cudaErrorInvalidValue;
  int np = 16;
  while (np < c.T && np < NP_MAX) np <<= 1;
  CUtensorMap mw, mx;
  if (!tc::make_map_box(&mw, w_gate, (uint64_t)c.E, (uint64_t)c.d_model, 128) ||
      !tc::make_map_box(&mx, x, (uint64_t)c.T, (uint64_t)c.d_model, np))
    return cudaErrorInvalidValue;
  Params p{};
  p.offsets = nullptr;
  p.E = 0;
  p.has_shared = 1;
  p.T = c.T;
  p.NP = np;
  p.NPs = np;
  p.gemm = 2;
  p.K_routed = c.d_model;
  p.K_shared = c.d_model;
  p.wb_routed = 0;
  p.wb_shared = c.E / 256;
  p.a_rows_routed = 0;
  p.out = nullptr;
  p.out_shared = part;
  p.ldo = c.E;
  p.ksplit = S;
  p.gu = nullptr;
  p.part_stride = 0;
  p.shared_stride = (size_t)c.T * c.E;
  p.fp8 = 0;
  p.bk = BK;
  p.st = st;
  cudaError_t e = launch(mw, mw, mx, mx, p, ceil_div(c.T, np) * p.wb_shared * S, s);
  if (e != cudaSuccess) return e;
  const size_t n4 = (size_t)c.T * c.E / 4;
  launch_pdl(router_slices_reduce_kernel, static_cast<int>((n4 + 31) / 32), 256, 0, s,
             reinterpret_cast<const float4*>(part), S, (size_t)c.T * c.E / 4, n4,
             reinterpret_cast<float4*>(logits));
  return cudaGetLastError();
}

cudaError_t launch_ffn_decode(const DecodeFFN& g, DevStatus* st, cudaStream_t s) {
  using namespace dec;
  if (g.np > NP_MAX || g.np_shared > NP_MAX) return cudaErrorInvalidValue;
  const bool sh = g.F_shared > 0;
  const int Fmax = g.F > g.F_shared ? g.F : g.F_shared;
  // bf16: boxes of 64 elements; E4M3: boxes of 128 one-byte codes (the same 128-byte rows)
  auto map = [&](CUtensorMap* m, const void* base, uint64_t rows, uint64_t cols, uint32_t box) {
    return g.fp8 ? tc::make_map_u8(m, base, rows, cols, box)
                 : tc::make_map_box(m, base, rows, cols, box);
  };
  CUtensorMap ma1, mas1, mb1, mbs1, ma2, mas2, mb2, mbs2;
  if (!map(&ma1, g.w13, (uint64_t)g.E * 2 * g.F, (uint64_t)g.d, 128) ||
      !map(&ma2, g.w2, (uint64_t)g.E * g.d, (uint64_t)g.F, 128) ||
      !map(&mb1, g.x, (uint64_t)g.max_rows, (uint64_t)g.d, g.np) ||
      !map(&mb2, g.h, (uint64_t)g.max_rows, (uint64_t)Fmax, g.np) ||
      !map(&mbs1, g.x, (uint64_t)g.max_rows, (uint64_t)g.d, g.np_shared) ||
      !map(&mbs2, g.h, (uint64_t)g.max_rows, (uint64_t)Fmax, g.np_shared))
    return cudaErrorInvalidValue;
  if (sh) {
    if (!map(&mas1, g.ws13, (uint64_t)2 * g.F_shared, (uint64_t)g.d, 128) ||
        !map(&mas2, g.ws2, (uint64_t)g.d, (uint64_t)g.F_shared, 128))
      return cudaErrorInvalidValue;
  } else {
    mas1 = ma1;
    mas2 = ma2;
  }
  Params p1{};
  p1.offsets = g.offsets;
  p1.E = g.E;
  p1.has_shared = sh ? 1 : 0;
  p1.T = g.T;
  p1.NP = g.np;
  p1.NPs = g.np_shared;
  p1.gemm = 1;
  p1.K_routed = g.d;
  p1.K_shared = g.d;
  p1.wb_routed = g.F / 128;
  p1.wb_shared = sh ? g.F_shared / 128 : 0;
  p1.a_rows_routed = 2 * g.F;
  p1.up_routed = g.F;
  p1.up_shared = g.F_shared;
  p1.out = g.h;
  p1.out_shared = nullptr;
  p1.ldo = Fmax;
  p1.ksplit = g.ksplit1;
  p1.gu = g.gu;
  p1.part_stride = static_cast<size_t>(g.max_rows) * 2 * Fmax;
  p1.shared_stride = 0;
  p1.fp8 = g.fp8;
  p1.bk = g.fp8 ? 128 : 64;
  p1.sa = g.s13;
  p1.sa_shared = g.ss13;
  p1.sb = g.sx;
  // E4M3 with one K slice: the gate/up GEMM writes h itself (half the bytes of gate | up)
  const bool h_ready = g.fp8 && g.ksplit1 == 1;
  if (h_ready) {
    p1.hf = g.gu;
    p1.gu = nullptr;
  }
  p1.st = st;
  // upper bound of the tile count: every routed row in its own chunk is impossible to exceed
  const int chunks_upper = ceil_div(g.max_rows, g.np) + g.E + ceil_div(g.T, g.np_shared) + 1;
  const int wbmax1 = p1.wb_routed > p1.wb_shared ? p1.wb_routed : p1.wb_shared;
  cudaError_t err = launch(ma1, mas1, mb1, mbs1, p1, chunks_upper * wbmax1 * g.ksplit1, s);
  if (err != cudaSuccess) return err;
  if (g.fp8) {
    err = smem_attr_once(reinterpret_cast<const void*>(swiglu_quant_kernel), 200 * 1024);
    if (err != cudaSuccess) return err;
    const int cn = swiglu_quant_cluster(g.max_rows, Fmax / 4);
    const int chunk = ceil_div(Fmax / 4, cn);
    int threads = ((chunk + 1) / 2 + 31) / 32 * 32;     // two column groups per thread
    if (threads > 1024) threads = 1024;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(g.max_rows * cn);
    cfg.blockDim = dim3(threads);
    cfg.dynamicSmemBytes = static_cast<size_t>(chunk) * 16;
    cfg.stream = s;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = cn;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;   // see pdl_prologue
    attr[1].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 2;
    err = cudaLaunchKernelEx(&cfg, swiglu_quant_kernel, static_cast<const float*>(g.gu),
                             p1.part_stride, g.ksplit1, g.offsets, g.E, sh ? g.T : 0, g.F,
                             sh ? g.F_shared : 0, Fmax, h_ready ? 1 : 0,
                             static_cast<uint8_t*>(g.h), g.hs);
    if (err != cudaSuccess) return err;
  } else if (g.ksplit1 > 1) {
    const long long work = static_cast<long long>(g.max_rows) * Fmax;
    int blocks = static_cast<int>((work + 255) / 256);
    if (blocks > num_sms() * 8) blocks = num_sms() * 8;
    launch_pdl(swiglu_finalize_kernel, blocks, 256, 0, s, g.gu, p1.part_stride, g.ksplit1, g.offsets, g.E,
                                                  g.T, g.F, sh ? g.F_shared : 0, Fmax,
                                                  static_cast<__nv_bfloat16*>(g.h));
    if ((err = cudaGetLastError()) != cudaSuccess) return err;
  }
  Params p2 = p1;
  p2.gemm = 2;
  p2.K_routed = g.F;
  p2.K_shared = g.F_shared;
  p2.wb_routed = g.d / 256;
  p2.wb_shared = sh ? g.d / 256 : 0;
  p2.a_rows_routed = g.d;
  p2.up_routed = 0;
  p2.up_shared = 0;
  p2.out = g.y;
  p2.out_shared = g.shared_out;
  p2.ldo = g.d;
  p2.ksplit = g.ksplit2;
  p2.gu = nullptr;
  p2.part_stride = g.y_part_stride;
  p2.shared_stride = g.shared_part_stride;
  p2.sa = g.s2;
  p2.sa_shared = g.ss2;
  p2.sb = g.hs;
  return launch(ma2, mas2, mb2, mbs2, p2, chunks_upper * p2.wb_routed * g.ksplit2, s);
}

}  // namespace moe
