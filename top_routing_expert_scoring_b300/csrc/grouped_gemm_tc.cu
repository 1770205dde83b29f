// Grouped expert GEMMs on the 5th-generation tensor cores (tcgen05 + TMEM + TMA), sm_103a.
//
//   GEMM 1 (gate/up):  h = SiLU(X W1_e^T) * (X W3_e^T)     ["Systems for Mixture-of-Experts
//   GEMM 2 (down):     y = h W2_e^T                          Models" §5.2 SwiGLU experts]
//
// over expert-ordered rows (expert e owns rows [offsets[e], offsets[e+1]), ragged).
//
// Design:
//   * persistent CTAs (one per SM) walk a device-side tile list; tile -> (expert, N tile,
//     M tile) with the M tile fastest, so the CTAs running at the same time share one weight
//     tile, which is read from HBM once and from L2 by the others;
//   * warp 0 issues TMA loads (128B-swizzled, K-major, 64-element K slices) into a 4-stage
//     ring; warp 1 issues tcgen05.mma (M=128, N=256, K=16, bf16 in, fp32 accumulate in TMEM);
//     warps 2-5 drain the accumulator (tcgen05.ld) and store bf16 rows.  Two TMEM
//     accumulators (2 x 256 columns) let the epilogue of one tile overlap the MMAs of the next;
//   * GEMM 1 puts 128 gate rows and the matching 128 up rows of W13 in one B tile, so one
//     N=256 MMA yields both halves and the epilogue forms SiLU(gate) * up directly;
//   * rows of an M tile past its expert's end are computed and never stored; an expert's last
//     tile with <= 64 rows runs as an M = 64 MMA, halving its wasted tensor work;
//   * every mbarrier wait is bounded (about 2 s); on expiry the CTA records MOE_ERR_TIMEOUT in
//     the status word, stops its loops, waits (bounded) for its own copies and MMAs in flight,
//     frees TMEM and returns.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_bf16.h>

#include <cstdlib>
#include <cstring>

#include "common.cuh"
#include "kernels.h"
#include "route_thread.cuh"
#include "tc_ptx.cuh"

namespace moe {
namespace tc {

constexpr int BM = 128;
constexpr int BK = 64;                       // 64 bf16 = 128 bytes = one swizzle row
constexpr int STAGES = 4;
constexpr int A_STAGE = BM * BK * 2;         // 16 KB
constexpr int B_BOX = 128 * BK * 2;          // 16 KB, one TMA box of 128 rows
constexpr int B_STAGE = 2 * B_BOX;           // up to 256 rows
constexpr int TMEM_COLS = 512;               // 2 accumulators x 256 fp32 columns
constexpr int THREADS = 192;
// expert schedule in shared memory: the M-tile prefix in schedule order [257] and the
// expert at each schedule position [256]
constexpr int SCHED_BYTES = (257 + 256) * 4;
constexpr size_t SMEM_BYTES = 1024 + (size_t)STAGES * (A_STAGE + B_STAGE) + 256 + SCHED_BYTES;
// router (ROUTE instantiation): a 3-stage ring, 16 epilogue warps (four per TMEM lane
// quarter, each owning a quarter of a token's experts) and their shared memory (RouteSmem)
constexpr int STAGES_ROUTE = 3;
constexpr int THREADS_ROUTE = 64 + 32 * 4 * kRouteSubs;
constexpr size_t SMEM_BYTES_ROUTE = 1024 + (size_t)STAGES_ROUTE * (A_STAGE + B_STAGE) + 256 +
                                    SCHED_BYTES + sizeof(RouteSmem);
static_assert(SMEM_BYTES_ROUTE <= 232448, "router shared memory");

struct Params {
  const int32_t* offsets;   // [E+1]
  const int32_t* mtp;       // [E+1] prefix of M tiles
  int E;
  int uniform_rows;         // >= 0: one group of this many rows
  int K;                    // reduction length (multiple of 64)
  int n_tiles;              // N tiles per expert
  int bn;                   // MMA N (128 or 256)
  int swiglu;               // GEMM 1 epilogue
  int b_rows;               // rows of B per expert
  int up_off;               // GEMM 1: offset of the up rows inside an expert's B rows (F)
  void* out;                // bf16 rows, or float32 rows when out_f32
  int out_f32;
  int ldo;
  // A gathered from the token rows (GEMM 1 only): row r of the expert-ordered space is token
  // perm[r] / gk of gx [T, K]; NULL: A is read by TMA from the materialised rows
  const int32_t* gperm;
  int gk;
  const __nv_bfloat16* gx;
  // N = 256 only: the last tiles of the list may each run as two N = 128 halves, to even out
  // the final wave over the CTAs (see choose_tail_split)
  int tail_split;
  // expert order of the tile list: 0 = expert index order; 1 = interleaved by row count
  // (largest, smallest, second largest, second smallest, ...), see build_schedule
  int order;
  // 1: a tile of <= 64 rows runs as an M = 64 MMA (accumulator rows 16q..16q+15 in lanes
  // 32q..32q+15); 0: every tile is an M = 128 MMA
  int tail64;
  // float32 epilogue only: instead of storing row r, add w[perm[r]] * row into token
  // perm[r] / scat_k of scat_out [T, ldo] (float32 vector reductions); rows with perm < 0 skip
  float* scat_out;
  const int32_t* scat_perm;
  const float* scat_w;
  int scat_k;
  // router epilogue (ROUTE instantiation only): with one group of T token rows and B = W_gate
  // (N = E <= 256 in one tile), each epilogue thread routes its token from the TMEM row of
  // logits -- scoring, group limit, Top-k, weights -- writes the logits, the selection and the
  // weights, and the tile's warps add their statistics terms into one partial row per tile
  const float* r_bias;      // [E] selection bias or NULL
  float* r_logits;          // [T, E]
  int32_t* r_idx;           // [T, k]
  float* r_w;               // [T, k]
  float* r_part_P;          // [tiles, E]
  int32_t* r_part_cnt;      // [tiles, E]
  float* r_part_z;          // [tiles]
  int r_E, r_k, r_score, r_cpg, r_topk_groups, r_renorm;
  float r_scale;
  DevStatus* st;
};

// Rows of the gather producer's lag: a lane signals stage n - kGatherLag once its copies for
// that stage have landed (cp.async groups complete in order).
constexpr int kGatherLag = 2;
static_assert(kGatherLag < STAGES, "the producer must not wait on a stage it has to refill");

__device__ __forceinline__ void cp_async16(uint32_t dst, const void* src, uint32_t bytes) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(dst), "l"(src), "r"(bytes)
               : "memory");
}
__device__ __forceinline__ void cp_async_commit() {
  asm volatile("cp.async.commit_group;" ::: "memory");
}
template <int N>
__device__ __forceinline__ void cp_async_wait() {
  asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}
__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// ---------------------------------------------------------------------------------------------
// Tile list
// ---------------------------------------------------------------------------------------------
struct TileInfo {
  int e, row0, rows, nt;
  int col0, bn;             // first output column and MMA N of this tile
};

// The tile list walks the experts in schedule order: position j holds expert ord[j] (ord ==
// nullptr: expert j) and mtp[j] M tiles precede it.
struct Sched {
  const int32_t* mtp;       // [E+1] M-tile prefix in schedule order
  const int32_t* ord;       // [E] expert at each position, or nullptr for index order
};

__device__ __forceinline__ int total_tiles(const Params& p, const Sched& sc) {
  const int mt = p.uniform_rows >= 0 ? ceil_div(p.uniform_rows, BM) : sc.mtp[p.E];
  return mt * p.n_tiles;
}

__device__ __forceinline__ TileInfo decode_tile(int tile, const Params& p, const Sched& sc) {
  TileInfo ti;
  int base_m, mt_e, row_base, row_end;
  if (p.uniform_rows >= 0) {
    ti.e = 0;
    base_m = 0;
    mt_e = ceil_div(p.uniform_rows, BM);
    row_base = 0;
    row_end = p.uniform_rows;
  } else {
    int lo = 0, hi = p.E;   // largest position j in [0, E) with mtp[j] * n_tiles <= tile
    while (hi - lo > 1) {
      const int mid = (lo + hi) >> 1;
      if (sc.mtp[mid] * p.n_tiles <= tile) lo = mid; else hi = mid;
    }
    ti.e = sc.ord ? sc.ord[lo] : lo;
    base_m = sc.mtp[lo];
    mt_e = sc.mtp[lo + 1] - base_m;
    row_base = p.offsets[ti.e];
    row_end = p.offsets[ti.e + 1];
  }
  const int tt = tile - base_m * p.n_tiles;
  ti.nt = tt / mt_e;
  const int mt = tt - ti.nt * mt_e;
  ti.row0 = row_base + mt * BM;
  ti.rows = min(BM, row_end - ti.row0);
  ti.col0 = ti.nt * p.bn;
  ti.bn = p.bn;
  return ti;
}

// Interleaved expert order, built by every CTA from the offsets (E <= 256, all threads): rank
// the experts by row count (descending, ties to the lower index) and place rank r at position
// 2r for the larger half and 2(E-1-r)+1 for the smaller half.  Consecutive tiles, which run at
// the same time on neighbouring CTAs, then mix experts whose weight stream dominates (few
// rows: every weight tile read from HBM for one M tile) with experts whose tensor work does
// (many rows: one weight tile shared by many M tiles), so HBM and the tensor pipes are busy
// together rather than in turns.  The order only permutes whole experts: every tile computes
// the same rows as in index order.
__device__ void build_schedule(const Params& p, int32_t* s_mtp, int32_t* s_ord) {
  const int E = p.E;
  for (int e = threadIdx.x; e < E; e += blockDim.x) {
    const int ce = p.offsets[e + 1] - p.offsets[e];
    int rank = 0;
    for (int f = 0; f < E; ++f) {
      const int cf = p.offsets[f + 1] - p.offsets[f];
      rank += (cf > ce || (cf == ce && f < e)) ? 1 : 0;
    }
    const int half = (E + 1) >> 1;
    const int pos = rank < half ? 2 * rank : 2 * (E - 1 - rank) + 1;
    s_ord[pos] = e;
    s_mtp[pos + 1] = ceil_div(ce, BM);
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    s_mtp[0] = 0;
    for (int j = 0; j < E; ++j) s_mtp[j + 1] += s_mtp[j];
  }
  __syncthreads();
}

// With `split` tail halves, the list is total - split whole tiles followed by 2 * split half
// tiles: half tile h is the left (h even) or right half of whole tile total - split + h / 2.
__device__ __forceinline__ TileInfo decode_tile(int tile, const Params& p, const Sched& sc,
                                                int total, int split) {
  const int whole = total - split;
  if (tile < whole) return decode_tile(tile, p, sc);
  const int h = tile - whole;
  TileInfo ti = decode_tile(whole + (h >> 1), p, sc);
  ti.bn = p.bn >> 1;
  ti.col0 += (h & 1) * ti.bn;
  return ti;
}

// Number of trailing whole tiles to run as halves.  Tile t goes to CTA t mod G (persistent
// round-robin); a whole tile costs 2, a half tile 1.  With total = qG + r, the unsplit list
// costs 2(q+1) on its busiest CTA.  Splitting the r tiles of the last partial wave gives 2r
// halves after q full waves: 2q + 1 when 2r <= G.  For r > G/2, no split beats 2(q+1).
__device__ __forceinline__ int choose_tail_split(int total, int G) {
  const int r = total % G;
  return (r > 0 && 2 * r <= G) ? r : 0;
}

// ---------------------------------------------------------------------------------------------
// The kernel
// ---------------------------------------------------------------------------------------------
// GATHER: the gate/up GEMM's A rows come from the token rows through the whole producer warp
// (cp.async) instead of one TMA box over the materialised rows; a separate instantiation so the
// default kernel's code is unchanged.
// ROUTE: the router GEMM with the routing epilogue (see Params::r_*).
template <bool GATHER, bool ROUTE = false>
__global__ void __launch_bounds__(ROUTE ? THREADS_ROUTE : THREADS, 1)
    grouped_gemm_tc_kernel(const __grid_constant__ CUtensorMap tmA,
                           const __grid_constant__ CUtensorMap tmB, const Params p) {
  constexpr int STAGES = ROUTE ? STAGES_ROUTE : tc::STAGES;
  constexpr int NBARS = 2 * STAGES + 5;   // full, empty, tmem full x2, tmem empty x2, drain
  pdl_prologue();
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  uint8_t* sA = smem;
  uint8_t* sB = smem + STAGES * A_STAGE;
  uint64_t* bars = reinterpret_cast<uint64_t*>(sB + STAGES * B_STAGE);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + NBARS);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  int32_t* s_mtp = reinterpret_cast<int32_t*>(smem + STAGES * (A_STAGE + B_STAGE) + 256);
  int32_t* s_ord = s_mtp + 257;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t full0 = smem_u32(bars);
  const uint32_t empty0 = full0 + 8 * STAGES;
  const uint32_t tfull0 = empty0 + 8 * STAGES;
  const uint32_t tempty0 = tfull0 + 16;
  const uint32_t drain = tempty0 + 16;

  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      // gather mode: 32 producer lanes arrive once their copies land, plus the B expect_tx
      mbar_init(full0 + 8 * s, GATHER ? 33 : 1);
      mbar_init(empty0 + 8 * s, 1);
    }
    for (int a = 0; a < 2; ++a) {
      mbar_init(tfull0 + 8 * a, 1);
      mbar_init(tempty0 + 8 * a, ROUTE ? 4 * kRouteSubs : 4);   // epilogue warps
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
  Sched sc{p.mtp, nullptr};
  if (p.order == 1 && p.uniform_rows < 0) {
    build_schedule(p, s_mtp, s_ord);
    sc = Sched{s_mtp, s_ord};
  }
  const int total = total_tiles(p, sc);
  const int KB = p.K / BK;
  const int split = p.tail_split ? choose_tail_split(total, gridDim.x) : 0;
  const int ntiles = total + split;

  if (GATHER && warp == 0) {
    // ------------------------ gathering producer (whole warp) -------------------------------
    // A: 128 rows of 64 bf16 per stage, copied straight from the token rows with cp.async in
    // the 128-byte swizzled layout TMA would write (16-byte chunk j of row r at j ^ (r & 7)).
    // Lanes 8q..8q+7 copy one row's 128 bytes (full lines); rows past the tile are zero-filled.
    // B: lane 0's TMA, as in the TMA producer.  Each lane waits for its own copies kGatherLag
    // stages later, fences them for the tensor core (async proxy) and arrives.
    int stage = 0;
    uint32_t ph = 0;
    uint32_t issued = 0, last_par = 0;
    const int nbox = (p.swiglu || p.bn > 128) ? 2 : 1;
    const uint32_t bbytes = nbox * B_BOX;
    const int chunk = lane & 7, rsub = lane >> 3;
    int hist[kGatherLag];                 // stages of the copy groups still to be signalled
    int npend = 0;
    bool ok = true;
    for (int tile = blockIdx.x; ok && tile < ntiles; tile += gridDim.x) {
      const TileInfo ti = decode_tile(tile, p, sc, total, split);
      int tok[32];
#pragma unroll
      for (int i = 0; i < 32; ++i) {
        const int r = rsub + 4 * i;
        tok[i] = r < ti.rows ? p.gperm[ti.row0 + r] / p.gk : -1;
      }
      int b0, b1;
      if (p.swiglu) {
        b0 = ti.e * p.b_rows + ti.nt * 128;
        b1 = b0 + p.up_off;
      } else {
        b0 = ti.e * p.b_rows + ti.col0;
        b1 = b0 + 128;
      }
      for (int kb = 0; kb < KB; ++kb) {
        int okw = 1;
        if (lane == 0)
          okw = wait_bounded(empty0 + 8 * stage, ph ^ 1u, abort_flag, p.st, 1, true) ? 1 : 0;
        okw = __shfl_sync(0xffffffffu, okw, 0);
        if (!okw) {
          ok = false;
          break;
        }
        const uint32_t fb = full0 + 8 * stage;
        if (lane == 0) {
          mbar_expect_tx(fb, bbytes);
          tma_load_2d(smem_u32(sB + stage * B_STAGE), &tmB, fb, kb * BK, b0);
          if (nbox == 2) tma_load_2d(smem_u32(sB + stage * B_STAGE + B_BOX), &tmB, fb, kb * BK, b1);
        }
        const uint32_t sa = smem_u32(sA + stage * A_STAGE);
#pragma unroll
        for (int i = 0; i < 32; ++i) {
          const int r = rsub + 4 * i;
          const int t = tok[i];
          const __nv_bfloat16* src =
              p.gx + static_cast<size_t>(t < 0 ? 0 : t) * p.K + kb * BK + chunk * 8;
          cp_async16(sa + r * 128 + ((chunk ^ (r & 7)) << 4), src, t < 0 ? 0u : 16u);
        }
        cp_async_commit();
        issued |= 1u << stage;
        last_par = (last_par & ~(1u << stage)) | (ph << stage);
        if (npend == kGatherLag) {
          cp_async_wait<kGatherLag>();
          fence_proxy_async_smem();
          mbar_arrive(full0 + 8 * hist[0]);
#pragma unroll
          for (int j = 0; j + 1 < kGatherLag; ++j) hist[j] = hist[j + 1];
          --npend;
        }
        hist[npend++] = stage;
        if (++stage == STAGES) {
          stage = 0;
          ph ^= 1u;
        }
      }
    }
    // the copies still in flight: land, fence, signal
    cp_async_wait<0>();
    fence_proxy_async_smem();
    for (int j = 0; j < npend; ++j) mbar_arrive(full0 + 8 * hist[j]);
    if (!ok && lane == 0) {
      for (int s = 0; s < STAGES; ++s)
        if ((issued >> s) & 1u)
          wait_bounded(full0 + 8 * s, (last_par >> s) & 1u, abort_flag, p.st, 5, false);
    }
  } else if (warp == 0 && lane == 0) {
    // ------------------------------- TMA producer -------------------------------------------
    int stage = 0;
    uint32_t ph = 0;
    uint32_t issued = 0, last_par = 0;   // per-stage bit masks for the drain
    bool ok = true;
    // first B rows of a tile's one or two boxes
    auto b_rows_of = [&](const TileInfo& t, int& r0, int& r1) {
      if (p.swiglu) {
        r0 = t.e * p.b_rows + t.nt * 128;
        r1 = r0 + p.up_off;
      } else {
        r0 = t.e * p.b_rows + t.col0;
        r1 = r0 + 128;
      }
    };
    for (int tile = blockIdx.x; ok && tile < ntiles; tile += gridDim.x) {
      const TileInfo ti = decode_tile(tile, p, sc, total, split);
      // B: two 128-row boxes (SwiGLU gate + up, or N = 256), else one
      const int nbox = (p.swiglu || ti.bn > 128) ? 2 : 1;
      const uint32_t bytes = A_STAGE + nbox * B_BOX;
      int b0, b1;
      b_rows_of(ti, b0, b1);
      for (int kb = 0; kb < KB; ++kb) {
        if (!wait_bounded(empty0 + 8 * stage, ph ^ 1u, abort_flag, p.st, 1, true)) {
          ok = false;
          break;
        }
        const uint32_t fb = full0 + 8 * stage;
        mbar_expect_tx(fb, bytes);
        tma_load_2d(smem_u32(sA + stage * A_STAGE), &tmA, fb, kb * BK, ti.row0);
        tma_load_2d(smem_u32(sB + stage * B_STAGE), &tmB, fb, kb * BK, b0);
        if (nbox == 2) tma_load_2d(smem_u32(sB + stage * B_STAGE + B_BOX), &tmB, fb, kb * BK, b1);
        issued |= 1u << stage;
        last_par = (last_par & ~(1u << stage)) | (ph << stage);
        if (++stage == STAGES) {
          stage = 0;
          ph ^= 1u;
        }
      }
    }
    if (!ok) {
      // wait for this CTA's own copies in flight before the CTA may exit
      for (int s = 0; s < STAGES; ++s)
        if ((issued >> s) & 1u)
          wait_bounded(full0 + 8 * s, (last_par >> s) & 1u, abort_flag, p.st, 5, false);
    }
  } else if (warp == 1 && lane == 0) {
    // ------------------------------- MMA issuer ---------------------------------------------
    int stage = 0, acc = 0;
    uint32_t ph = 0, aph = 0;
    bool ok = true;
    for (int tile = blockIdx.x; ok && tile < ntiles; tile += gridDim.x) {
      // an expert's last tile with <= 64 rows runs as an M = 64 MMA (half the tensor work)
      const TileInfo tm = decode_tile(tile, p, sc, total, split);
      const uint32_t idesc = idesc_bf16_f32(p.tail64 && tm.rows <= 64 ? 64 : BM, tm.bn);
      if (!wait_bounded(tempty0 + 8 * acc, aph ^ 1u, abort_flag, p.st, 2, true)) {
        ok = false;
        break;
      }
      tc_fence_after();
      const uint32_t dt = tmem_base + static_cast<uint32_t>(acc * 256);
      for (int kb = 0; kb < KB; ++kb) {
        if (!wait_bounded(full0 + 8 * stage, ph, abort_flag, p.st, 3, true)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t a0 = smem_u32(sA + stage * A_STAGE);
        const uint32_t b0 = smem_u32(sB + stage * B_STAGE);
#pragma unroll
        for (int kk = 0; kk < BK / 16; ++kk)
          tc_mma(dt, sw128_desc(a0 + kk * 32), sw128_desc(b0 + kk * 32), idesc,
                 (kb | kk) != 0 ? 1u : 0u);
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
    // every MMA this thread issued must finish before TMEM is released
    tc_commit(drain);
    wait_bounded(drain, 0u, abort_flag, p.st, 6, false);
  } else if (ROUTE && warp >= 2) {
    // ------------------------------- routing epilogue ---------------------------------------
    // 16 warps: warp w reads TMEM lane quarter q = w % 4 (32 token slots) and owns the
    // quarter `sub` of each token's 32-expert chunks; the per-token phases meet in shared
    // memory (route_thread.cuh).  Barrier 1 spans these 512 threads; a tile's start is agreed
    // on by all of them (bar.red), so a timeout stops every warp at the same point.
    const int q = warp & 3;
    const int sub = (warp - 2) >> 2;
    const int r = q * 32 + lane;            // token slot of this thread (unique)
    const int et = threadIdx.x - 64;        // 0..511
    RouteSmem& sm = *reinterpret_cast<RouteSmem*>(smem + STAGES * (A_STAGE + B_STAGE) + 256 +
                                                  SCHED_BYTES);
    const int E = p.r_E;
    for (int e = et; e < 256; e += 512) {
      sm.bias[e] = (e < E && p.r_bias) ? p.r_bias[e] : 0.f;
      sm.cnt[e] = 0;
    }
    asm volatile("bar.sync 1, 512;" ::: "memory");
    const RouteThreadCfg rc{E / 32, p.r_k, p.r_score, p.r_cpg, p.r_topk_groups, p.r_renorm,
                            p.r_scale, 1};
    int acc = 0;
    uint32_t aph = 0;
    for (int tile = blockIdx.x; tile < ntiles; tile += gridDim.x) {
      const TileInfo ti = decode_tile(tile, p, sc, total, split);
      // one thread waits for the accumulator; the barrier below releases the other 511
      uint32_t ok = 1;
      if (warp == 2 && lane == 0)
        ok = wait_bounded(tfull0 + 8 * acc, aph, abort_flag, p.st, 4, true) ? 1 : 0;
      ok = __shfl_sync(0xffffffffu, ok, 0);
      uint32_t all_ok;
      asm volatile(
          "{\n .reg .pred p, q;\n setp.ne.u32 p, %1, 0;\n bar.red.and.pred q, 1, 512, p;\n"
          " selp.u32 %0, 1, 0, q;\n}\n"
          : "=r"(all_ok)
          : "r"(ok)
          : "memory");
      if (!all_ok) break;
      tc_fence_after();
      const uint32_t tb = tmem_base + static_cast<uint32_t>(acc * 256) +
                          (static_cast<uint32_t>(q * 32) << 16);
      const bool half = p.tail64 && ti.rows <= 64;
      const int row = half ? q * 16 + lane : r;
      const bool live = half ? (lane < 16 && row < ti.rows) : (r < ti.rows);
      const size_t t = static_cast<size_t>(ti.row0 + row);
      auto load = [&](int c, float (&v)[32]) {
        uint32_t u[32];
        tmem_ld32(tb + c * 32, u);
#pragma unroll
        for (int i = 0; i < 32; ++i) v[i] = __uint_as_float(u[i]);
      };
      // the logits, as the statistics and the backward read them
      auto each = [&](int c, const float (&v)[32]) {
        if (!live) return;
        float4* dst = reinterpret_cast<float4*>(p.r_logits + t * E + c * 32);
#pragma unroll
        for (int i = 0; i < 8; ++i)
          dst[i] = make_float4(v[4 * i], v[4 * i + 1], v[4 * i + 2], v[4 * i + 3]);
      };
      // chunk c of this thread's token row, from the logits phase A wrote (the barrier below
      // orders those writes before these reads)
      auto load_row = [&](int c, float (&v)[32]) {
        const float4* src = reinterpret_cast<const float4*>(p.r_logits + t * E + c * 32);
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          const float4 f = src[i];
          v[4 * i] = f.x;
          v[4 * i + 1] = f.y;
          v[4 * i + 2] = f.z;
          v[4 * i + 3] = f.w;
        }
      };
      route_phase_a(rc, sm, r, sub, load, each);
      asm volatile("bar.sync 1, 512;" ::: "memory");
      route_phase_b(rc, sm, r, sub, q, live, load, load_row);
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(tempty0 + 8 * acc);   // this warp is done with TMEM
      asm volatile("bar.sync 1, 512;" ::: "memory");
      if (sub == 0) {
        int idx[kRouteMaxK];
        float wv[kRouteMaxK];
        const float lse = route_phase_c(rc, sm, r, idx, wv);
        if (live) {
          for (int j = 0; j < p.r_k; ++j) {
            p.r_idx[t * p.r_k + j] = idx[j];
            p.r_w[t * p.r_k + j] = wv[j];
            atomicAdd(&sm.cnt[idx[j]], 1);
          }
        }
        const float zt = warp_sum(live ? lse * lse : 0.f);
        if (lane == 0) sm.Z[q] = zt;
      }
      asm volatile("bar.sync 1, 512;" ::: "memory");
      for (int e = et; e < E; e += 512) {
        p.r_part_P[static_cast<size_t>(tile) * E + e] =
            ((sm.P[0][e] + sm.P[1][e]) + sm.P[2][e]) + sm.P[3][e];
        p.r_part_cnt[static_cast<size_t>(tile) * E + e] = sm.cnt[e];
        sm.cnt[e] = 0;
      }
      if (et == 0) p.r_part_z[tile] = ((sm.Z[0] + sm.Z[1]) + sm.Z[2]) + sm.Z[3];
      asm volatile("bar.sync 1, 512;" ::: "memory");
      acc ^= 1;
      if (acc == 0) aph ^= 1u;
    }
  } else if (warp >= 2) {
    // ------------------------------- epilogue -----------------------------------------------
    const int q = warp & 3;                 // TMEM lanes 32q .. 32q+31 belong to this warp
    const int r = q * 32 + lane;            // row of the tile held by this thread
    int acc = 0;
    uint32_t aph = 0;
    for (int tile = blockIdx.x; tile < ntiles; tile += gridDim.x) {
      const TileInfo ti = decode_tile(tile, p, sc, total, split);
      int ok = 1;
      if (lane == 0) ok = wait_bounded(tfull0 + 8 * acc, aph, abort_flag, p.st, 4, true) ? 1 : 0;
      ok = __shfl_sync(0xffffffffu, ok, 0);
      if (!ok) break;
      tc_fence_after();
      const uint32_t tb = tmem_base + static_cast<uint32_t>(acc * 256) +
                          (static_cast<uint32_t>(q * 32) << 16);
      // M = 128: row r = 32q + lane sits in TMEM lane r.  M = 64: rows 16q .. 16q+15 sit in the
      // first 16 lanes of the warp's 32-lane quarter.
      const bool half = p.tail64 && ti.rows <= 64;
      const int row = half ? q * 16 + lane : r;
      const bool live = half ? (lane < 16 && row < ti.rows) : (r < ti.rows);
      if (p.swiglu) {
        __nv_bfloat16* orow = static_cast<__nv_bfloat16*>(p.out) +
                              static_cast<size_t>(ti.row0 + row) * p.ldo + ti.nt * 128;
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
      } else if (p.out_f32 && p.scat_out) {
        // gate weight applied here and the expert's row added into its token's output
        float* orow = nullptr;
        float wt = 0.f;
        if (live) {
          const int pair = p.scat_perm[ti.row0 + row];
          if (pair >= 0) {
            wt = p.scat_w[pair];
            orow = p.scat_out + static_cast<size_t>(pair / p.scat_k) * p.ldo + ti.col0;
          }
        }
        const int nchunks = ti.bn / 32;
#pragma unroll 1
        for (int c = 0; c < nchunks; ++c) {
          uint32_t vr[32];
          tmem_ld32(tb + c * 32, vr);
          if (orow) {
#pragma unroll
            for (int v = 0; v < 8; ++v)
              asm volatile("red.global.add.v4.f32 [%0], {%1, %2, %3, %4};" ::"l"(
                               orow + c * 32 + 4 * v),
                           "f"(wt * __uint_as_float(vr[4 * v])),
                           "f"(wt * __uint_as_float(vr[4 * v + 1])),
                           "f"(wt * __uint_as_float(vr[4 * v + 2])),
                           "f"(wt * __uint_as_float(vr[4 * v + 3]))
                           : "memory");
          }
        }
      } else if (p.out_f32) {
        float* orow = static_cast<float*>(p.out) + static_cast<size_t>(ti.row0 + row) * p.ldo +
                      ti.col0;
        const int nchunks = ti.bn / 32;
#pragma unroll 1
        for (int c = 0; c < nchunks; ++c) {
          uint32_t vr[32];
          tmem_ld32(tb + c * 32, vr);
          if (live) {
            uint4* dst = reinterpret_cast<uint4*>(orow + c * 32);
#pragma unroll
            for (int v = 0; v < 8; ++v)
              dst[v] = make_uint4(vr[4 * v], vr[4 * v + 1], vr[4 * v + 2], vr[4 * v + 3]);
          }
        }
      } else {
        __nv_bfloat16* orow = static_cast<__nv_bfloat16*>(p.out) +
                              static_cast<size_t>(ti.row0 + row) * p.ldo + ti.col0;
        const int nchunks = ti.bn / 32;
#pragma unroll 1
        for (int c = 0; c < nchunks; ++c) {
          uint32_t vr[32];
          tmem_ld32(tb + c * 32, vr);
          uint32_t packed[16];
#pragma unroll
          for (int i = 0; i < 16; ++i) {
            __nv_bfloat162 hv =
                __floats2bfloat162_rn(__uint_as_float(vr[2 * i]), __uint_as_float(vr[2 * i + 1]));
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

// A kernel whose only wait is on a flag nothing ever sets: exercises the bounded-wait failure
// path (status word set, kernel returns, context stays usable).
__global__ void timeout_probe_kernel(DevStatus* st, uint64_t limit_ns) {
  __shared__ uint64_t bar;
  __shared__ int abort_flag;
  if (threadIdx.x == 0) {
    mbar_init(smem_u32(&bar), 1);
    abort_flag = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  __syncthreads();
  if (threadIdx.x == 0) wait_bounded(smem_u32(&bar), 0u, &abort_flag, st, 99, true, limit_ns);
}

// ---------------------------------------------------------------------------------------------
// Host side
// ---------------------------------------------------------------------------------------------
static PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  if (!fn) {
    void* ptr = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(ptr);
  }
  return fn;
}

bool make_map_strided(CUtensorMap* m, const void* base, uint64_t rows, uint64_t cols,
                      uint64_t row_stride, uint32_t box_rows) {
  auto fn = encode_fn();
  if (!fn) return false;
  cuuint64_t dims[2] = {cols, rows};
  cuuint64_t strides[1] = {row_stride * 2};
  cuuint32_t box[2] = {static_cast<cuuint32_t>(BK), box_rows};
  cuuint32_t estr[2] = {1, 1};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box,
            estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

bool make_map_box(CUtensorMap* m, const void* base, uint64_t rows, uint64_t cols,
                  uint32_t box_rows) {
  return make_map_strided(m, base, rows, cols, cols, box_rows);
}

bool make_map_f32_store(CUtensorMap* m, void* base, uint64_t rows, uint64_t cols) {
  auto fn = encode_fn();
  if (!fn) return false;
  cuuint64_t dims[2] = {cols, rows};
  cuuint64_t strides[1] = {cols * 4};
  cuuint32_t box[2] = {32u, 32u};
  cuuint32_t estr[2] = {1, 1};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, base, dims, strides, box, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_NONE, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

bool make_map_u8(CUtensorMap* m, const void* base, uint64_t rows, uint64_t cols,
                 uint32_t box_rows) {
  auto fn = encode_fn();
  if (!fn) return false;
  cuuint64_t dims[2] = {cols, rows};
  cuuint64_t strides[1] = {cols};
  cuuint32_t box[2] = {128u, box_rows};
  cuuint32_t estr[2] = {1, 1};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void*>(base), dims, strides, box,
            estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// 2-D bf16 tensor [rows, cols] (cols contiguous) read in boxes of 64 columns x 128 rows.
bool make_map(CUtensorMap* m, const void* base, uint64_t rows, uint64_t cols) {
  return make_map_box(m, base, rows, cols, 128);
}

static cudaError_t launch_one(const CUtensorMap& a, const CUtensorMap& b, const Params& p,
                              int upper_tiles, cudaStream_t s) {
  const void* fn = p.gperm ? reinterpret_cast<const void*>(grouped_gemm_tc_kernel<true>)
                           : reinterpret_cast<const void*>(grouped_gemm_tc_kernel<false>);
  cudaError_t e = smem_attr_once(fn, static_cast<int>(SMEM_BYTES));
  if (e != cudaSuccess) return e;
  int grid = num_sms();
  if (upper_tiles < grid) grid = upper_tiles;
  if (grid < 1) grid = 1;
  if (p.gperm)
    launch_pdl(grouped_gemm_tc_kernel<true>, grid, THREADS, SMEM_BYTES, s, a, b, p);
  else
    launch_pdl(grouped_gemm_tc_kernel<false>, grid, THREADS, SMEM_BYTES, s, a, b, p);
  return cudaGetLastError();
}

}  // namespace tc

// Expert order of the ragged tile lists: interleaved by row count unless the environment
// variable MOE_B300_ORDER=index asks for expert index order (both compute the same rows).
static int expert_order() {
  const char* env = getenv("MOE_B300_ORDER");
  return (env && strcmp(env, "index") == 0) ? 0 : 1;
}

// M = 64 MMAs for tiles of <= 64 rows unless MOE_B300_TAIL64=0 (the same rows either way).
static int tail_m64() {
  const char* env = getenv("MOE_B300_TAIL64");
  return (env && strcmp(env, "0") == 0) ? 0 : 1;
}

static bool use_pair_kernel(const GroupedFFN& g) {
  if (g.d % 256 != 0) return false;
  const char* env = getenv("MOE_B300_GEMM");
  if (env && strcmp(env, "single") == 0) return false;
  if (env && strcmp(env, "pair") == 0) return true;
  // One group (shared experts): measured on the DeepSeekMoE-16B layer (two shared experts,
  // T = 8192) the single-CTA kernel makes the step 1% faster (its last partial wave runs as
  // N = 128 halves; the pair kernel's down GEMM has 3.5 waves of pair tiles), and on the V3
  // layer the two are within noise.  Ragged groups pay on average half a 128-row block per
  // expert for 256-row pair tiles, so pairs only win once experts average >= 2048 rows.
  if (g.uniform_rows >= 0) return false;
  return (long long)g.max_rows / g.E >= 2048;
}

bool ffn_uses_pair(const GroupedFFN& g) { return use_pair_kernel(g); }

cudaError_t launch_ffn_tc(const GroupedFFN& g, DevStatus* st, cudaStream_t s) {
  using namespace tc;
  if (use_pair_kernel(g)) {
    if (g.gather_perm) return cudaErrorInvalidValue;   // the pair kernel reads materialised rows
    return launch_ffn_tc2(g, st, s);
  }
  CUtensorMap mx, mw13, mh, mw2;
  if (!make_map(&mw13, g.w13, (uint64_t)g.E * 2 * g.F, (uint64_t)g.d) ||
      !make_map(&mh, g.h, (uint64_t)g.max_rows, (uint64_t)g.F) ||
      !make_map(&mw2, g.w2, (uint64_t)g.E * g.d, (uint64_t)g.F))
    return cudaErrorInvalidValue;
  if (g.gather_perm) mx = mw13;   // not read: A is gathered from the token rows
  else if (!make_map(&mx, g.x, (uint64_t)g.max_rows, (uint64_t)g.d))
    return cudaErrorInvalidValue;
  const int mt_upper = g.uniform_rows >= 0 ? ceil_div(g.uniform_rows, BM)
                                           : ceil_div(g.max_rows, BM) + g.E;
  Params p1{};
  p1.offsets = g.offsets;
  p1.mtp = g.mtile_prefix;
  p1.E = g.E;
  p1.uniform_rows = g.uniform_rows;
  p1.K = g.d;
  p1.n_tiles = g.F / 128;
  p1.bn = 256;
  p1.swiglu = 1;
  p1.b_rows = 2 * g.F;
  p1.up_off = g.F;
  p1.out = g.h;
  p1.out_f32 = 0;
  p1.ldo = g.F;
  p1.gperm = g.gather_perm;
  p1.gk = g.gather_k;
  p1.gx = static_cast<const __nv_bfloat16*>(g.gather_x);
  p1.order = expert_order();
  p1.tail64 = tail_m64();
  p1.st = st;
  cudaError_t err = launch_one(mx, mw13, p1, mt_upper * p1.n_tiles, s);
  if (err != cudaSuccess) return err;
  Params p2 = p1;
  p2.K = g.F;
  p2.bn = (g.d % 256 == 0) ? 256 : 128;
  p2.n_tiles = g.d / p2.bn;
  p2.swiglu = 0;
  p2.b_rows = g.d;
  p2.up_off = 0;
  p2.out = g.y;
  p2.out_f32 = (g.y_bf16 && !g.scatter_out) ? 0 : 1;
  p2.ldo = g.d;
  p2.gperm = nullptr;
  p2.tail_split = p2.bn == 256 ? 1 : 0;
  p2.scat_out = g.scatter_out;
  p2.scat_perm = g.scatter_perm;
  p2.scat_w = g.scatter_w;
  p2.scat_k = g.gather_k;
  return launch_one(mh, mw2, p2, mt_upper * p2.n_tiles, s);
}

// Router logits through the same kernel: one group of T rows, B = W_gate [E, d], fp32 output.
// N tile = E (E <= 128) or 128 (E a multiple of 128, several N tiles); rows of the B box past
// E are zero-filled by the TMA and their columns are never stored.
cudaError_t launch_router_tc(const moe_config& c, const void* x, const void* w_gate,
                             float* logits, cudaStream_t s) {
  using namespace tc;
  CUtensorMap mx, mw;
  if (!make_map(&mx, x, (uint64_t)c.T, (uint64_t)c.d_model) ||
      !make_map(&mw, w_gate, (uint64_t)c.E, (uint64_t)c.d_model))
    return cudaErrorInvalidValue;
  Params p{};
  p.offsets = nullptr;
  p.mtp = nullptr;
  p.E = 1;
  p.uniform_rows = c.T;
  p.K = c.d_model;
  p.bn = c.E <= 128 ? c.E : (c.E % 128 == 0 ? 128 : c.E);
  p.n_tiles = c.E / p.bn;
  p.swiglu = 0;
  p.b_rows = c.E;
  p.up_off = 0;
  p.out = logits;
  p.out_f32 = 1;
  p.ldo = c.E;
  p.tail64 = 1;
  p.st = nullptr;
  return launch_one(mx, mw, p, ceil_div(c.T, BM) * p.n_tiles, s);
}

// Router GEMM with the routing epilogue: one group of T rows, B = W_gate [E, d] (E % 32 == 0,
// E <= 256) in one N = E tile, 128-token tiles; one partial statistics row per tile.
cudaError_t launch_router_fused(const moe_config& c, const void* x, const void* w_gate,
                                const float* bias, float* logits, int32_t* idx, float* w,
                                float* part_P, int32_t* part_cnt, float* part_z, DevStatus* st,
                                cudaStream_t s) {
  using namespace tc;
  CUtensorMap mx, mw;
  if (!make_map(&mx, x, (uint64_t)c.T, (uint64_t)c.d_model) ||
      !make_map(&mw, w_gate, (uint64_t)c.E, (uint64_t)c.d_model))
    return cudaErrorInvalidValue;
  Params p{};
  p.E = 1;
  p.uniform_rows = c.T;
  p.K = c.d_model;
  p.bn = c.E;
  p.n_tiles = 1;
  p.b_rows = c.E;
  p.st = st;
  p.r_bias = c.score == MOE_SCORE_SIGMOID ? bias : nullptr;
  p.r_logits = logits;
  p.r_idx = idx;
  p.r_w = w;
  p.r_part_P = part_P;
  p.r_part_cnt = part_cnt;
  p.r_part_z = part_z;
  p.r_E = c.E;
  p.r_k = c.k;
  p.r_score = c.score;
  const bool limit = c.score == MOE_SCORE_SIGMOID && c.n_groups > 1 &&
                     c.topk_groups < c.n_groups;
  p.r_cpg = limit ? (c.E / c.n_groups) / 32 : 0;
  p.r_topk_groups = c.topk_groups;
  p.r_renorm = c.renormalize;
  p.r_scale = c.route_scale;
  p.tail64 = 1;
  const void* fn = reinterpret_cast<const void*>(grouped_gemm_tc_kernel<false, true>);
  cudaError_t e = smem_attr_once(fn, static_cast<int>(SMEM_BYTES_ROUTE));
  if (e != cudaSuccess) return e;
  int grid = num_sms();
  const int tiles = ceil_div(c.T, BM);
  if (tiles < grid) grid = tiles;
  launch_pdl(grouped_gemm_tc_kernel<false, true>, grid, THREADS_ROUTE, SMEM_BYTES_ROUTE, s, mx,
             mw, p);
  return cudaGetLastError();
}

cudaError_t launch_timeout_probe(DevStatus* st, int limit_us, cudaStream_t s) {
  tc::timeout_probe_kernel<<<1, 32, 0, s>>>(st, static_cast<uint64_t>(limit_us) * 1000ull);
  return cudaGetLastError();
}

}  // namespace moe
