// Gate/up grouped GEMM with two M blocks per tile (tcgen05, single CTA, sm_103a).
//
//   h = SiLU(X W1_e^T) * (X W3_e^T)     ["Systems for Mixture-of-Experts Models" §5.2 SwiGLU]
//
// over expert-ordered rows, like the gate/up launch of grouped_gemm_tc.cu, but a tile is 256
// rows of one expert (two M blocks of 128) against one N = 256 weight tile (128 gate rows and
// the matching 128 up rows).  Each K step loads both blocks' A rows and the weight tile once
// and issues two M = 128 MMAs on the same B stage, one per accumulator (TMEM columns 0..255 and
// 256..511).  Per unit of tensor work the ring moves 32 KB instead of 48 KB, so its 3 stages x
// 64 KB cover half as much again of the load latency as the 4 x 48 KB ring of one-block tiles,
// and L2 serves a third fewer bytes.  Unlike a CTA pair (cta_group::2), the two blocks live in
// one CTA, so an expert's last tile may hold a single block, and a block of <= 64 rows runs as
// an M = 64 MMA: the padding stays that of 128-row tiles with M = 64 tails.
//
// The price is the accumulators: both fill TMEM, so a tile's epilogue (SiLU * up, bf16 rows)
// is not overlapped with the next tile's MMAs; the ring keeps loading meanwhile.
//
// Roles: warp 0 lane 0 TMA producer, warp 1 lane 0 MMA issuer (and TMEM owner), warps 2-5
// epilogue.  Every mbarrier wait is bounded (about 2 s); on expiry the CTA records
// MOE_ERR_TIMEOUT, stops its loops, waits (bounded) for its own copies and MMAs, frees TMEM and
// returns.
#include <cuda.h>
#include <cuda_bf16.h>

#include "common.cuh"
#include "kernels.h"
#include "tc_ptx.cuh"

namespace moe {
namespace dm {

using namespace tc;

constexpr int BM = 128;                      // rows per block
constexpr int TR = 2 * BM;                   // rows per tile
constexpr int BK = 64;
constexpr int STAGES = 3;
constexpr int A_BLOCK = BM * BK * 2;         // 16 KB
constexpr int A_STAGE = 2 * A_BLOCK;         // 32 KB
constexpr int B_BOX = 128 * BK * 2;          // 16 KB
constexpr int B_STAGE = 2 * B_BOX;           // 32 KB (gate box, up box)
constexpr int STAGE = A_STAGE + B_STAGE;     // 64 KB
constexpr int TMEM_COLS = 512;               // block 0 at column 0, block 1 at column 256
constexpr int THREADS = 192;
constexpr int NBARS = 2 * STAGES + 3;        // full, empty, tmem full, tmem empty, drain
constexpr int SCHED_BYTES = (257 + 256) * 4;
constexpr size_t SMEM_BYTES = 1024 + (size_t)STAGES * STAGE + 256 + SCHED_BYTES;

struct Params {
  const int32_t* offsets;   // [E+1]
  int E;
  int uniform_rows;         // >= 0: one group of this many rows
  int K;                    // d (multiple of 64)
  int n_tiles;              // F / 128
  int b_rows;               // 2F
  int up_off;               // F
  __nv_bfloat16* out;       // h [rows, F]
  int ldo;                  // F
  int order;                // 1: experts interleaved by row count
  DevStatus* st;
};

struct Tile {
  int e, row0, r0, r1, nt;  // rows of block 0 and block 1 (r1 may be 0)
};

// Tile list: per expert ceil(rows / 256) tiles per N tile, M fastest; experts in schedule
// order (position j holds expert ord[j], mtp[j] tiles precede it).
__device__ __forceinline__ Tile decode(int tile, const Params& p, const int32_t* mtp,
                                       const int32_t* ord) {
  Tile t;
  int base, mt_e, row_base, row_end;
  if (p.uniform_rows >= 0) {
    t.e = 0;
    base = 0;
    mt_e = ceil_div(p.uniform_rows, TR);
    row_base = 0;
    row_end = p.uniform_rows;
  } else {
    int lo = 0, hi = p.E;
    while (hi - lo > 1) {
      const int mid = (lo + hi) >> 1;
      if (mtp[mid] * p.n_tiles <= tile) lo = mid; else hi = mid;
    }
    t.e = ord ? ord[lo] : lo;
    base = mtp[lo];
    mt_e = mtp[lo + 1] - base;
    row_base = p.offsets[t.e];
    row_end = p.offsets[t.e + 1];
  }
  const int tt = tile - base * p.n_tiles;
  t.nt = tt / mt_e;
  const int mt = tt - t.nt * mt_e;
  t.row0 = row_base + mt * TR;
  const int rows = min(TR, row_end - t.row0);
  t.r0 = min(BM, rows);
  t.r1 = rows - t.r0;
  return t;
}

// Schedule of 256-row tiles: index order, or interleaved by row count (largest, smallest,
// second largest, ...) so that weight-streaming and compute-heavy experts run side by side.
__device__ void build_schedule(const Params& p, int32_t* s_mtp, int32_t* s_ord) {
  const int E = p.E;
  for (int e = threadIdx.x; e < E; e += blockDim.x) {
    const int ce = p.offsets[e + 1] - p.offsets[e];
    int pos = e;
    if (p.order == 1) {
      int rank = 0;
      for (int f = 0; f < E; ++f) {
        const int cf = p.offsets[f + 1] - p.offsets[f];
        rank += (cf > ce || (cf == ce && f < e)) ? 1 : 0;
      }
      const int half = (E + 1) >> 1;
      pos = rank < half ? 2 * rank : 2 * (E - 1 - rank) + 1;
    }
    s_ord[pos] = e;
    s_mtp[pos + 1] = ceil_div(ce, TR);
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    s_mtp[0] = 0;
    for (int j = 0; j < E; ++j) s_mtp[j + 1] += s_mtp[j];
  }
  __syncthreads();
}

__global__ void __launch_bounds__(THREADS, 1)
    grouped_gemm_dm_kernel(const __grid_constant__ CUtensorMap tmA,
                           const __grid_constant__ CUtensorMap tmB, const Params p) {
  pdl_prologue();
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + STAGES * STAGE);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + NBARS);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  int32_t* s_mtp = reinterpret_cast<int32_t*>(smem + STAGES * STAGE + 256);
  int32_t* s_ord = s_mtp + 257;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t full0 = smem_u32(bars);
  const uint32_t empty0 = full0 + 8 * STAGES;
  const uint32_t tfull = empty0 + 8 * STAGES;
  const uint32_t tempty = tfull + 8;
  const uint32_t drain = tempty + 8;

  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(full0 + 8 * s, 1);
      mbar_init(empty0 + 8 * s, 1);
    }
    mbar_init(tfull, 1);
    mbar_init(tempty, 4);
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
  const int32_t* mtp = s_mtp;
  const int32_t* ord = s_ord;
  if (p.uniform_rows < 0) build_schedule(p, s_mtp, s_ord);
  const int ntiles =
      (p.uniform_rows >= 0 ? ceil_div(p.uniform_rows, TR) : s_mtp[p.E]) * p.n_tiles;
  const int KB = p.K / BK;

  if (warp == 0 && lane == 0) {
    // ------------------------------- TMA producer -------------------------------------------
    int stage = 0;
    uint32_t ph = 0;
    uint32_t issued = 0, last_par = 0;
    bool ok = true;
    for (int tile = blockIdx.x; ok && tile < ntiles; tile += gridDim.x) {
      const Tile ti = decode(tile, p, mtp, ord);
      const int b0 = ti.e * p.b_rows + ti.nt * 128;
      const int b1 = b0 + p.up_off;
      const uint32_t bytes = (ti.r1 > 0 ? 2 : 1) * A_BLOCK + B_STAGE;
      for (int kb = 0; kb < KB; ++kb) {
        if (!wait_bounded(empty0 + 8 * stage, ph ^ 1u, abort_flag, p.st, 21, true)) {
          ok = false;
          break;
        }
        const uint32_t fb = full0 + 8 * stage;
        const uint32_t st_a = smem_u32(smem + stage * STAGE);
        const uint32_t st_b = st_a + A_STAGE;
        mbar_expect_tx(fb, bytes);
        tma_load_2d(st_a, &tmA, fb, kb * BK, ti.row0);
        if (ti.r1 > 0) tma_load_2d(st_a + A_BLOCK, &tmA, fb, kb * BK, ti.row0 + BM);
        tma_load_2d(st_b, &tmB, fb, kb * BK, b0);
        tma_load_2d(st_b + B_BOX, &tmB, fb, kb * BK, b1);
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
    int stage = 0;
    uint32_t ph = 0, tph = 0;
    bool ok = true;
    for (int tile = blockIdx.x; ok && tile < ntiles; tile += gridDim.x) {
      const Tile tm = decode(tile, p, mtp, ord);
      // a block of <= 64 rows runs as an M = 64 MMA
      const uint32_t id0 = idesc_bf16_f32(tm.r0 <= 64 ? 64 : BM, 256);
      const uint32_t id1 = idesc_bf16_f32(tm.r1 <= 64 ? 64 : BM, 256);
      if (!wait_bounded(tempty, tph ^ 1u, abort_flag, p.st, 22, true)) {
        ok = false;
        break;
      }
      tc_fence_after();
      for (int kb = 0; kb < KB; ++kb) {
        if (!wait_bounded(full0 + 8 * stage, ph, abort_flag, p.st, 23, true)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t a0 = smem_u32(smem + stage * STAGE);
        const uint32_t b0 = a0 + A_STAGE;
#pragma unroll
        for (int kk = 0; kk < BK / 16; ++kk) {
          const uint32_t acc = (kb | kk) != 0 ? 1u : 0u;
          tc_mma(tmem_base, sw128_desc(a0 + kk * 32), sw128_desc(b0 + kk * 32), id0, acc);
          if (tm.r1 > 0)
            tc_mma(tmem_base + 256u, sw128_desc(a0 + A_BLOCK + kk * 32),
                   sw128_desc(b0 + kk * 32), id1, acc);
        }
        tc_commit(empty0 + 8 * stage);
        if (++stage == STAGES) {
          stage = 0;
          ph ^= 1u;
        }
      }
      if (!ok) break;
      tc_commit(tfull);
      tph ^= 1u;
    }
    tc_commit(drain);
    wait_bounded(drain, 0u, abort_flag, p.st, 26, false);
  } else if (warp >= 2) {
    // ------------------------------- epilogue -----------------------------------------------
    const int q = warp & 3;                 // TMEM lanes 32q .. 32q+31 belong to this warp
    uint32_t tph = 0;
    for (int tile = blockIdx.x; tile < ntiles; tile += gridDim.x) {
      const Tile ti = decode(tile, p, mtp, ord);
      int ok = 1;
      if (lane == 0) ok = wait_bounded(tfull, tph, abort_flag, p.st, 24, true) ? 1 : 0;
      ok = __shfl_sync(0xffffffffu, ok, 0);
      if (!ok) break;
      tc_fence_after();
#pragma unroll 1
      for (int b = 0; b < 2; ++b) {
        const int rows = b ? ti.r1 : ti.r0;
        if (rows == 0) continue;
        const uint32_t tb = tmem_base + static_cast<uint32_t>(b * 256) +
                            (static_cast<uint32_t>(q * 32) << 16);
        // M = 128: row 32q + lane in TMEM lane 32q + lane.  M = 64: rows 16q .. 16q+15 in the
        // first 16 lanes of the warp's quarter.
        const bool half = rows <= 64;
        const int row = half ? q * 16 + lane : q * 32 + lane;
        const bool live = half ? (lane < 16 && row < rows) : (row < rows);
        __nv_bfloat16* orow = p.out + static_cast<size_t>(ti.row0 + b * BM + row) * p.ldo +
                              ti.nt * 128;
#pragma unroll 1
        for (int c = 0; c < 4; ++c) {
          uint32_t gr[32], ur[32];
          tmem_ld32(tb + c * 32, gr);
          tmem_ld32(tb + 128 + c * 32, ur);
          uint32_t packed[16];
#pragma unroll
          for (int i = 0; i < 16; ++i) {
            const float g0 = __uint_as_float(gr[2 * i]), g1 = __uint_as_float(gr[2 * i + 1]);
            const float u0 = __uint_as_float(ur[2 * i]), u1 = __uint_as_float(ur[2 * i + 1]);
            const float h0 = (g0 / (1.0f + expf(-g0))) * u0;
            const float h1 = (g1 / (1.0f + expf(-g1))) * u1;
            __nv_bfloat162 hv = __floats2bfloat162_rn(h0, h1);
            packed[i] = *reinterpret_cast<uint32_t*>(&hv);
          }
          if (live) {
            uint4* dst = reinterpret_cast<uint4*>(orow + c * 32);
#pragma unroll
            for (int v = 0; v < 4; ++v)
              dst[v] = make_uint4(packed[4 * v], packed[4 * v + 1], packed[4 * v + 2],
                                  packed[4 * v + 3]);
          }
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(tempty);
      tph ^= 1u;
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

}  // namespace dm

// The gate/up GEMM of a grouped SwiGLU on two-block tiles (see above).
cudaError_t launch_gateup_dm(const GroupedFFN& g, int order, DevStatus* st, cudaStream_t s) {
  using namespace dm;
  CUtensorMap mx, mw13;
  if (!tc::make_map(&mx, g.x, (uint64_t)g.max_rows, (uint64_t)g.d) ||
      !tc::make_map(&mw13, g.w13, (uint64_t)g.E * 2 * g.F, (uint64_t)g.d))
    return cudaErrorInvalidValue;
  Params p{};
  p.offsets = g.offsets;
  p.E = g.E;
  p.uniform_rows = g.uniform_rows;
  p.K = g.d;
  p.n_tiles = g.F / 128;
  p.b_rows = 2 * g.F;
  p.up_off = g.F;
  p.out = static_cast<__nv_bfloat16*>(g.h);
  p.ldo = g.F;
  p.order = order;
  p.st = st;
  cudaError_t e = smem_attr_once(reinterpret_cast<const void*>(grouped_gemm_dm_kernel),
                                 static_cast<int>(SMEM_BYTES));
  if (e != cudaSuccess) return e;
  const int upper = (g.uniform_rows >= 0 ? ceil_div(g.uniform_rows, TR)
                                         : ceil_div(g.max_rows, TR) + g.E) * p.n_tiles;
  int grid = num_sms();
  if (upper < grid) grid = upper;
  if (grid < 1) grid = 1;
  launch_pdl(grouped_gemm_dm_kernel, grid, THREADS, SMEM_BYTES, s, mx, mw13, p);
  return cudaGetLastError();
}

}  // namespace moe
