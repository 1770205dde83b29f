// Grouped expert GEMMs on CTA pairs: tcgen05 with cta_group::2 (sm_103a).
//
// Same products as grouped_gemm_tc.cu (SwiGLU gate/up with the SiLU*up epilogue, and the down
// projection with a float32 epilogue) ["Systems for Mixture-of-Experts Models" §5.2], but one
// MMA spans two SMs of a cluster: M = 256 rows (128 per CTA) x N = 256, K = 16.  Each CTA loads
// its own 128 rows of A and its own half (128 rows) of the N = 256 B tile, so the shared-memory
// bytes per K step are 32 KB per CTA instead of 48 KB: the ring holds 6 stages, which covers
// the load latency that left the single-CTA kernel's tensor pipe idle, and L2 serves half the B
// traffic.  Both CTAs' loads complete on the leader CTA's barrier; the leader issues the MMAs
// and its commits arrive on both CTAs' barriers; each CTA drains its own 128 accumulator rows.
//
// A pair tile is 256 rows of one expert.  With `half128` set, an expert's last pair tile of at
// most 128 rows runs as an M = 128 pair MMA instead: 64 rows per CTA, the same halved B
// traffic, and the padding of a 128-row tile.  Each CTA's accumulator then holds its 64 rows
// twice over the lanes: row i's first N/2 columns in TMEM lane i, its last N/2 columns in lane
// 64 + i, both at TMEM columns 0 .. N/2-1.  For SwiGLU each CTA's B half is therefore 64 gate
// rows followed by the 64 matching up rows, so that one thread holds gate and up of the same
// 64 output columns.
//
// Every wait is bounded.  On expiry a CTA raises its own and its peer's abort flags and
// records MOE_ERR_TIMEOUT; the pair then stops, the leader reconciles and waits for every
// load still in flight to either CTA's shared memory, waits for its MMAs, and both CTAs free
// TMEM and return.
#include <cuda.h>
#include <cstdlib>
#include <cstring>
#include <cuda_bf16.h>

#include "common.cuh"
#include "kernels.h"
#include "tc_ptx.cuh"

namespace moe {
namespace tc2 {

using namespace tc;

constexpr int BM = 128;                      // rows per CTA
constexpr int PM = 256;                      // rows per pair tile
constexpr int BK = 64;
constexpr int STAGES = 6;
constexpr int A_STAGE = BM * BK * 2;         // 16 KB
constexpr int B_STAGE = 128 * BK * 2;        // 16 KB: this CTA's half of the B tile
constexpr int STAGE = A_STAGE + B_STAGE;
constexpr int TMEM_COLS = 512;
constexpr int THREADS = 192;
constexpr int MAX_E = 256;
constexpr int NBARS = 2 * STAGES + 5;        // full, empty, tmem full x2, tmem empty x2, drain
// stages | barriers | tmem slot, abort flag, issued counts | pair-tile prefix
constexpr size_t CTRL_BYTES = 8 * NBARS + 16 + 4 * STAGES;
static_assert(CTRL_BYTES <= 256, "the control block must fit its 256-byte slot");
constexpr size_t SMEM_BYTES = 1024 + (size_t)STAGES * STAGE + 256 + (MAX_E + 1) * 4;

struct Params {
  const int32_t* offsets;   // [E+1]
  int E;
  int uniform_rows;         // >= 0: one group of this many rows
  int K;
  int n_tiles;              // N tiles (of 256 columns) per expert
  int swiglu;
  int b_rows;               // rows of B per expert
  int up_off;               // SwiGLU: first up-projection row inside an expert's B rows (F)
  void* out;
  int out_f32;
  int ldo;
  int half128;              // an expert's last tile of <= 128 rows runs as an M = 128 pair
  DevStatus* st;
};

__device__ __forceinline__ uint32_t cluster_rank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}
// Address of the same shared-memory offset in CTA `rank` of the cluster.
__device__ __forceinline__ uint32_t mapa(uint32_t addr, uint32_t rank) {
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(addr), "r"(rank));
  return r;
}
__device__ __forceinline__ void cluster_sync_all() {
  asm volatile("barrier.cluster.arrive.release.aligned;\n"
               "barrier.cluster.wait.acquire.aligned;" ::: "memory");
}
__device__ __forceinline__ void st_cluster_u32(uint32_t addr, uint32_t v) {
  asm volatile("st.shared::cluster.u32 [%0], %1;" ::"r"(addr), "r"(v) : "memory");
}
__device__ __forceinline__ uint32_t ld_cluster_u32(uint32_t addr) {
  uint32_t v;
  asm volatile("ld.shared::cluster.u32 %0, [%1];" : "=r"(v) : "r"(addr) : "memory");
  return v;
}
__device__ __forceinline__ void mbar_arrive_cluster(uint32_t cluster_addr) {
  asm volatile("mbarrier.arrive.release.cluster.shared::cluster.b64 _, [%0];" ::"r"(cluster_addr)
               : "memory");
}
__device__ __forceinline__ void mbar_complete_tx(uint32_t bar, uint32_t bytes) {
  asm volatile("mbarrier.complete_tx.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(bytes) : "memory");
}
__device__ __forceinline__ bool mbar_try_wait_cl(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n .reg .pred p;\n mbarrier.try_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2;\n"
      " selp.u32 %0, 1, 0, p;\n}\n"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}

// Bounded wait with cluster-scope acquire.  On expiry raises this CTA's and the peer's abort
// flags.
__device__ __noinline__ bool wait_pair(uint32_t bar, uint32_t parity, volatile int* abort_flag,
                                       uint32_t peer_flag, DevStatus* st, int where,
                                       bool honor_abort) {
  if (mbar_try_wait_cl(bar, parity)) return true;
  const uint64_t t0 = globaltimer_ns();
  for (uint32_t it = 1;; ++it) {
    if (mbar_try_wait_cl(bar, parity)) return true;
    if ((it & 15u) == 0u) {
      if (honor_abort && *abort_flag) return false;
      if (globaltimer_ns() - t0 > kWaitLimitNs) {
        *abort_flag = 1;
        st_cluster_u32(peer_flag, 1u);
        record_error(st, MOE_ERR_TIMEOUT, where);
        return false;
      }
    }
  }
}

// TMA load whose completion is signalled on a barrier of either CTA of the pair.
__device__ __forceinline__ void tma_load_2d_pair(uint32_t dst, const CUtensorMap* map,
                                                 uint32_t bar_cluster, int c0, int c1) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes.cta_group::2"
      " [%0], [%1, {%3, %4}], [%2];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(bar_cluster), "r"(c0), "r"(c1)
      : "memory");
}
__device__ __forceinline__ void mma_pair(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc,
                                         uint32_t idesc, uint32_t accum) {
  asm volatile(
      "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n"
      " tcgen05.mma.cta_group::2.kind::f16 [%0], %1, %2, %3, p;\n}\n" ::"r"(d_tmem),
      "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accum)
      : "memory");
}
// Arrive on the barrier at this offset in both CTAs once the leader's earlier MMAs complete.
__device__ __forceinline__ void commit_pair_both(uint32_t bar) {
  asm volatile(
      "tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64"
      " [%0], %1;" ::"r"(bar),
      "h"(static_cast<uint16_t>(3))
      : "memory");
}
__device__ __forceinline__ void commit_pair_local(uint32_t bar) {
  asm volatile("tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
                   bar)
               : "memory");
}

struct PairTile {
  int e, row0, rows, nt;   // row0: first row of the pair tile; rows: valid rows in the pair
};

__device__ __forceinline__ PairTile decode_pair(int tile, const Params& p, const int* prefix) {
  PairTile ti;
  int base, mt_e, row_base, row_end;
  if (p.uniform_rows >= 0) {
    ti.e = 0;
    base = 0;
    mt_e = ceil_div(p.uniform_rows, PM);
    row_base = 0;
    row_end = p.uniform_rows;
  } else {
    int lo = 0, hi = p.E;
    while (hi - lo > 1) {
      const int mid = (lo + hi) >> 1;
      if (prefix[mid] * p.n_tiles <= tile) lo = mid; else hi = mid;
    }
    ti.e = lo;
    base = prefix[lo];
    mt_e = prefix[lo + 1] - base;
    row_base = p.offsets[lo];
    row_end = p.offsets[lo + 1];
  }
  const int tt = tile - base * p.n_tiles;
  int mt;
  if (p.uniform_rows >= 0) {
    // one group (shared experts): N fastest, so a pair tile's rows are read once from DRAM and
    // reused from L2 by all N tiles while the (small) weights stay in L2
    mt = tt / p.n_tiles;
    ti.nt = tt - mt * p.n_tiles;
  } else {
    // ragged experts: M fastest, so the CTAs of an expert's M tiles share one weight tile
    ti.nt = tt / mt_e;
    mt = tt - ti.nt * mt_e;
  }
  ti.row0 = row_base + mt * PM;
  ti.rows = min(PM, row_end - ti.row0);
  return ti;
}

__global__ void __launch_bounds__(THREADS, 1)
    grouped_gemm_tc2_kernel(const __grid_constant__ CUtensorMap tmA,
                            const __grid_constant__ CUtensorMap tmB,
                            const __grid_constant__ CUtensorMap tmB64, const Params p) {
  pdl_prologue();
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  uint8_t* stage_mem = smem;
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + STAGES * STAGE);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + NBARS);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  uint32_t* issued = tmem_slot + 4;                        // [STAGES] loads issued per stage
  int* prefix = reinterpret_cast<int*>(smem + STAGES * STAGE + 256);

  const uint32_t rank = cluster_rank();
  const bool leader = rank == 0;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t full0 = smem_u32(bars);
  const uint32_t empty0 = full0 + 8 * STAGES;
  const uint32_t tfull0 = empty0 + 8 * STAGES;
  const uint32_t tempty0 = tfull0 + 16;
  const uint32_t drain = tempty0 + 16;
  const uint32_t peer_flag = mapa(smem_u32(const_cast<int*>(abort_flag)), rank ^ 1u);

  if (p.uniform_rows < 0) {
    for (int e = threadIdx.x; e < p.E; e += blockDim.x)
      prefix[e + 1] = ceil_div(p.offsets[e + 1] - p.offsets[e], PM);
    __syncthreads();
    if (threadIdx.x == 0) {
      prefix[0] = 0;
      for (int e = 1; e <= p.E; ++e) prefix[e] += prefix[e - 1];
    }
  }
  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(full0 + 8 * s, 1);
      mbar_init(empty0 + 8 * s, 1);
      issued[s] = 0;
    }
    for (int a = 0; a < 2; ++a) {
      mbar_init(tfull0 + 8 * a, 1);
      mbar_init(tempty0 + 8 * a, 8);        // 4 epilogue warps in each CTA
    }
    mbar_init(drain, 1);
    *abort_flag = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  if (warp == 1) {
    asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                     smem_u32(tmem_slot)),
                 "r"(TMEM_COLS)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;" ::: "memory");
  }
  tc_fence_before();
  __syncthreads();
  cluster_sync_all();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;
  const int total = (p.uniform_rows >= 0 ? ceil_div(p.uniform_rows, PM) : prefix[p.E]) * p.n_tiles;
  const int KB = p.K / BK;
  const int cid = blockIdx.x >> 1, ncl = gridDim.x >> 1;

  if (warp == 0 && lane == 0) {
    // ------------------------------- TMA producer (both CTAs) -------------------------------
    const uint32_t full_leader0 = mapa(full0, 0);
    int stage = 0;
    uint32_t ph = 0;
    bool ok = true;
    for (int tile = cid; ok && tile < total; tile += ncl) {
      const PairTile ti = decode_pair(tile, p, prefix);
      // M = 128 pair tiles take 64 rows per CTA (the box still loads 128; the MMA reads 64)
      const bool half = p.half128 && ti.rows <= BM;
      const int a_row = ti.row0 + static_cast<int>(rank) * (half ? 64 : BM);
      // SwiGLU M = 128: gate rows 64*rank .. +63 of the N tile, then the matching up rows
      const int g_row = ti.e * p.b_rows + ti.nt * 128 + static_cast<int>(rank) * 64;
      const bool split_b = half && p.swiglu;
      const int b_row = p.swiglu
                            ? ti.e * p.b_rows + ti.nt * 128 + (rank ? p.up_off : 0)
                            : ti.e * p.b_rows + ti.nt * 256 + static_cast<int>(rank) * 128;
      for (int kb = 0; kb < KB; ++kb) {
        if (!wait_pair(empty0 + 8 * stage, ph ^ 1u, abort_flag, peer_flag, p.st, 11, true)) {
          ok = false;
          break;
        }
        if (leader) mbar_expect_tx(full0 + 8 * stage, 2 * STAGE);
        const uint32_t fb = full_leader0 + 8 * stage;
        const uint32_t sa = smem_u32(stage_mem + stage * STAGE);
        tma_load_2d_pair(sa, &tmA, fb, kb * BK, a_row);
        if (split_b) {
          tma_load_2d_pair(sa + A_STAGE, &tmB64, fb, kb * BK, g_row);
          tma_load_2d_pair(sa + A_STAGE + B_STAGE / 2, &tmB64, fb, kb * BK, g_row + p.up_off);
        } else {
          tma_load_2d_pair(sa + A_STAGE, &tmB, fb, kb * BK, b_row);
        }
        issued[stage] += 1;
        if (++stage == STAGES) {
          stage = 0;
          ph ^= 1u;
        }
      }
    }
  } else if (warp == 1 && lane == 0 && leader) {
    // ------------------------------- MMA issuer (leader only) -------------------------------
    const uint32_t idesc_full = idesc_bf16_f32(PM, 256);
    const uint32_t idesc_half = idesc_bf16_f32(BM, 256);
    int stage = 0, acc = 0;
    uint32_t ph = 0, aph = 0;
    bool ok = true;
    for (int tile = cid; ok && tile < total; tile += ncl) {
      const int rows = decode_pair(tile, p, prefix).rows;
      const uint32_t idesc = p.half128 && rows <= BM ? idesc_half : idesc_full;
      if (!wait_pair(tempty0 + 8 * acc, aph ^ 1u, abort_flag, peer_flag, p.st, 12, true)) {
        ok = false;
        break;
      }
      tc_fence_after();
      const uint32_t dt = tmem_base + static_cast<uint32_t>(acc * 256);
      for (int kb = 0; kb < KB; ++kb) {
        if (!wait_pair(full0 + 8 * stage, ph, abort_flag, peer_flag, p.st, 13, true)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t a0 = smem_u32(stage_mem + stage * STAGE);
        const uint32_t b0 = a0 + A_STAGE;
#pragma unroll
        for (int kk = 0; kk < BK / 16; ++kk)
          mma_pair(dt, sw128_desc(a0 + kk * 32), sw128_desc(b0 + kk * 32), idesc,
                   (kb | kk) != 0 ? 1u : 0u);
        commit_pair_both(empty0 + 8 * stage);
        if (++stage == STAGES) {
          stage = 0;
          ph ^= 1u;
        }
      }
      if (!ok) break;
      commit_pair_both(tfull0 + 8 * acc);
      acc ^= 1;
      if (acc == 0) aph ^= 1u;
    }
    commit_pair_local(drain);
    wait_pair(drain, 0u, abort_flag, peer_flag, p.st, 16, false);
  } else if (warp >= 2) {
    // ------------------------------- epilogue (both CTAs) -----------------------------------
    const int q = warp & 3;
    const int r = q * 32 + lane;
    const uint32_t tempty_leader0 = mapa(tempty0, 0);
    int acc = 0;
    uint32_t aph = 0;
    for (int tile = cid; tile < total; tile += ncl) {
      const PairTile ti = decode_pair(tile, p, prefix);
      int ok = 1;
      if (lane == 0)
        ok = wait_pair(tfull0 + 8 * acc, aph, abort_flag, peer_flag, p.st, 14, true) ? 1 : 0;
      ok = __shfl_sync(0xffffffffu, ok, 0);
      if (!ok) break;
      tc_fence_after();
      const uint32_t tb = tmem_base + static_cast<uint32_t>(acc * 256) +
                          (static_cast<uint32_t>(q * 32) << 16);
      // M = 128 pair tile: warp q holds rows 32 (q & 1) + lane of this CTA's 64, and the
      // (q >> 1)-th half of the tile's columns at TMEM columns 0 .. 127
      const bool half = p.half128 && ti.rows <= BM;
      const int hq = half ? (q >> 1) : 0;
      const int row_in_pair = half ? static_cast<int>(rank) * 64 + 32 * (q & 1) + lane
                                   : static_cast<int>(rank) * BM + r;
      const bool live = row_in_pair < ti.rows;
      const size_t grow = static_cast<size_t>(ti.row0 + row_in_pair);
      if (p.swiglu) {
        // gate column j at TMEM column j, up at j + 128 (M = 128: 64 columns, up at j + 64)
        __nv_bfloat16* orow =
            static_cast<__nv_bfloat16*>(p.out) + grow * p.ldo + ti.nt * 128 + hq * 64;
        const int nch = half ? 2 : 4;
        const uint32_t up = half ? 64 : 128;
#pragma unroll 1
        for (int c = 0; c < nch; ++c) {
          uint32_t gr[32], ur[32];
          tmem_ld32(tb + c * 32, gr);
          tmem_ld32(tb + up + c * 32, ur);
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
      } else if (p.out_f32) {
        float* orow = static_cast<float*>(p.out) + grow * p.ldo + ti.nt * 256 + hq * 128;
#pragma unroll 1
        for (int c = 0; c < (half ? 4 : 8); ++c) {
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
        __nv_bfloat16* orow =
            static_cast<__nv_bfloat16*>(p.out) + grow * p.ldo + ti.nt * 256 + hq * 128;
#pragma unroll 1
        for (int c = 0; c < (half ? 4 : 8); ++c) {
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
      if (lane == 0) mbar_arrive_cluster(tempty_leader0 + 8 * acc);
      acc ^= 1;
      if (acc == 0) aph ^= 1u;
    }
  }

  __syncthreads();
  cluster_sync_all();
  // After an abort, loads may still be in flight to either CTA.  Every load signals the
  // leader's full barrier of its stage; the last use of a stage may be armed by only one side,
  // so the leader balances the byte count (expect_tx / complete_tx) and waits for the phase.
  if (*abort_flag && leader && threadIdx.x == 0) {
    const uint32_t peer_issued0 = mapa(smem_u32(issued), 1u);
    for (int s = 0; s < STAGES; ++s) {
      const uint32_t mine = issued[s];
      const uint32_t theirs = ld_cluster_u32(peer_issued0 + 4 * s);
      const uint32_t uses = mine > theirs ? mine : theirs;
      if (uses == 0) continue;
      const uint32_t fb = full0 + 8 * s;
      if (theirs > mine) mbar_expect_tx(fb, STAGE);          // peer's bytes, never armed
      else if (mine > theirs) mbar_complete_tx(fb, STAGE);   // peer never loaded them
      wait_pair(fb, (uses - 1) & 1u, abort_flag, peer_flag, p.st, 15, false);
    }
  }
  cluster_sync_all();
  if (warp == 1) {
    __syncwarp();
    tc_fence_after();
    asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;" ::"r"(tmem_base),
                 "r"(TMEM_COLS)
                 : "memory");
  }
}

}  // namespace tc2

// Pair kernel for one GEMM; `b_rows`, `n_tiles` etc. follow tc2::Params.
cudaError_t launch_tc2(const CUtensorMap& a, const CUtensorMap& b, const CUtensorMap& b64,
                       const tc2::Params& p, int upper_pair_tiles, cudaStream_t s) {
  using namespace tc2;
  cudaError_t e0 = smem_attr_once(reinterpret_cast<const void*>(grouped_gemm_tc2_kernel),
                                  static_cast<int>(SMEM_BYTES));
  if (e0 != cudaSuccess) return e0;
  int clusters = num_sms() / 2;
  if (upper_pair_tiles < clusters) clusters = upper_pair_tiles;
  if (clusters < 1) clusters = 1;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(2 * clusters, 1, 1);
  cfg.blockDim = dim3(THREADS, 1, 1);
  cfg.dynamicSmemBytes = SMEM_BYTES;
  cfg.stream = s;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;   // see pdl_prologue
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 2;
  return cudaLaunchKernelEx(&cfg, grouped_gemm_tc2_kernel, a, b, b64, p);
}

// M = 128 pair tiles for an expert's last <= 128 rows: on unless MOE_B300_PAIR_HALF=0.
static int pair_half128() {
  const char* env = getenv("MOE_B300_PAIR_HALF");
  return (env && strcmp(env, "0") == 0) ? 0 : 1;
}

// Both SwiGLU GEMMs on CTA pairs.  Requires F % 128 == 0 and d % 256 == 0.
cudaError_t launch_ffn_tc2(const GroupedFFN& g, DevStatus* st, cudaStream_t s) {
  using namespace tc2;
  CUtensorMap mx, mw13, mw13_64, mh, mw2;
  if (!tc::make_map(&mx, g.x, (uint64_t)g.max_rows, (uint64_t)g.d) ||
      !tc::make_map(&mw13, g.w13, (uint64_t)g.E * 2 * g.F, (uint64_t)g.d) ||
      !tc::make_map_box(&mw13_64, g.w13, (uint64_t)g.E * 2 * g.F, (uint64_t)g.d, 64) ||
      !tc::make_map(&mh, g.h, (uint64_t)g.max_rows, (uint64_t)g.F) ||
      !tc::make_map(&mw2, g.w2, (uint64_t)g.E * g.d, (uint64_t)g.F))
    return cudaErrorInvalidValue;
  const int pt_upper = g.uniform_rows >= 0 ? ceil_div(g.uniform_rows, PM)
                                           : ceil_div(g.max_rows, PM) + g.E;
  Params p1{};
  p1.offsets = g.offsets;
  p1.E = g.E;
  p1.uniform_rows = g.uniform_rows;
  p1.K = g.d;
  p1.n_tiles = g.F / 128;
  p1.swiglu = 1;
  p1.b_rows = 2 * g.F;
  p1.up_off = g.F;
  p1.out = g.h;
  p1.out_f32 = 0;
  p1.ldo = g.F;
  p1.half128 = pair_half128();
  p1.st = st;
  cudaError_t err = launch_tc2(mx, mw13, mw13_64, p1, pt_upper * p1.n_tiles, s);
  if (err != cudaSuccess) return err;
  Params p2 = p1;
  p2.K = g.F;
  p2.n_tiles = g.d / 256;
  p2.swiglu = 0;
  p2.b_rows = g.d;
  p2.up_off = 0;
  p2.out = g.y;
  p2.out_f32 = g.y_bf16 ? 0 : 1;
  p2.ldo = g.d;
  return launch_tc2(mh, mw2, mw2, p2, pt_upper * p2.n_tiles, s);
}

}  // namespace moe
