// Dispatch: group the (token, choice) pairs by expert in token order, apply the expert
// capacity and gather token rows into expert order.
//   ["Systems for Mixture-of-Experts Models" §2.2 (group tokens by expert), §2.4 (capacity
//    C = ceil(cf*k*n/E), overflow dropped)]
//
// Positions come from counting, never from atomic arrival order, so every output is
// deterministic and bit-exact:
//   D1  per block of 256 tokens, a bitmap bm[e][t/32] of the tokens that chose expert e and
//       the block's count per expert;
//   D2  one CTA scans the block counts (token-block order) per expert, clamps to the
//       capacity and scans the kept counts over experts -> offsets, the M-tile schedule of
//       the expert GEMMs and the drop count;
//   D3  pos(t,j) = base[block][e] + popcount of bm[e] below t; row, perm;
//   D4  x_perm[row] = x[t] with 16-byte vector copies, one warp per row.
#include <cuda_bf16.h>
#include <cuda_fp8.h>

#include "common.cuh"
#include "kernels.h"

namespace moe {

constexpr int kWords = kDispatchBlock / 32;   // bitmap words per expert per block

__global__ void __launch_bounds__(kDispatchBlock) dispatch_count_kernel(
    const int32_t* __restrict__ idx, int T, int E, int k, uint32_t* __restrict__ bitmap,
    int32_t* __restrict__ blk_cnt, DevStatus* st) {
  pdl_prologue();
  __shared__ uint32_t bm[256 * kWords];
  const int tid = threadIdx.x;
  for (int i = tid; i < E * kWords; i += blockDim.x) bm[i] = 0u;
  __syncthreads();
  const int t = blockIdx.x * kDispatchBlock + tid;
  if (t < T) {
    int sel[8];
    for (int j = 0; j < k; ++j) {
      int e = idx[(size_t)t * k + j];
      bool bad = e < 0 || e >= E;
      for (int q = 0; q < j; ++q) bad |= (sel[q] == e);   // an expert chosen twice
      sel[j] = bad ? -1 : e;
      if (bad) {
        record_error(st, MOE_ERR_ARG, t);
        continue;
      }
      atomicOr(&bm[e * kWords + tid / 32], 1u << (tid % 32));
    }
  }
  __syncthreads();
  uint32_t* gbm = bitmap + (size_t)blockIdx.x * E * kWords;
  for (int i = tid; i < E * kWords; i += blockDim.x) gbm[i] = bm[i];
  for (int e = tid; e < E; e += blockDim.x) {
    int c = 0;
#pragma unroll
    for (int w = 0; w < kWords; ++w) c += __popc(bm[e * kWords + w]);
    blk_cnt[(size_t)blockIdx.x * E + e] = c;
  }
}

// One CTA of 256 threads (E <= 256).  blk_cnt is overwritten in place by the exclusive
// per-expert base of every block.
__global__ void __launch_bounds__(256) dispatch_scan_kernel(int32_t* __restrict__ blk_cnt,
                                                           int nblk, int E, int capacity,
                                                           int32_t* __restrict__ counts,
                                                           int32_t* __restrict__ kept,
                                                           int32_t* __restrict__ offsets,
                                                           int32_t* __restrict__ mtile_prefix,
                                                           int32_t* __restrict__ n_dropped) {
  pdl_prologue();
  __shared__ int s_kept[256];
  __shared__ int s_mt[256];
  __shared__ int s_drop[256];
  const int e = threadIdx.x;
  int total = 0;
  if (e < E) {
    // 16 blocks' counts in flight at a time, then their exclusive bases in block order
    constexpr int kBatch = 16;
    for (int b0 = 0; b0 < nblk; b0 += kBatch) {
      int c[kBatch];
#pragma unroll
      for (int j = 0; j < kBatch; ++j)
        c[j] = b0 + j < nblk ? blk_cnt[(size_t)(b0 + j) * E + e] : 0;
#pragma unroll
      for (int j = 0; j < kBatch; ++j) {
        if (b0 + j < nblk) blk_cnt[(size_t)(b0 + j) * E + e] = total;
        total += c[j];
      }
    }
  }
  const int kp = e < E ? min(total, capacity) : 0;
  s_kept[e] = kp;
  s_mt[e] = ceil_div(kp, kTileM);
  s_drop[e] = e < E ? total - kp : 0;
  if (e < E) {
    counts[e] = total;
    kept[e] = kp;
  }
  __syncthreads();
  // inclusive Hillis-Steele scans over 256 entries
  for (int s = 1; s < 256; s <<= 1) {
    int a = e >= s ? s_kept[e - s] : 0;
    int b = e >= s ? s_mt[e - s] : 0;
    int c = e >= s ? s_drop[e - s] : 0;
    __syncthreads();
    s_kept[e] += a;
    s_mt[e] += b;
    s_drop[e] += c;
    __syncthreads();
  }
  if (e < E) {
    offsets[e + 1] = s_kept[e];
    mtile_prefix[e + 1] = s_mt[e];
  }
  if (e == 0) {
    offsets[0] = 0;
    mtile_prefix[0] = 0;
    *n_dropped = s_drop[255];
  }
}

__global__ void __launch_bounds__(kDispatchBlock) dispatch_scatter_kernel(
    const int32_t* __restrict__ idx, int T, int E, int k, int capacity,
    const uint32_t* __restrict__ bitmap, const int32_t* __restrict__ blk_base,
    const int32_t* __restrict__ offsets, int32_t* __restrict__ pos, int32_t* __restrict__ row_of,
    int32_t* __restrict__ perm) {
  pdl_prologue();
  __shared__ uint32_t bm[256 * kWords];
  const int tid = threadIdx.x;
  const uint32_t* gbm = bitmap + (size_t)blockIdx.x * E * kWords;
  for (int i = tid; i < E * kWords; i += blockDim.x) bm[i] = gbm[i];
  __syncthreads();
  const int t = blockIdx.x * kDispatchBlock + tid;
  if (t >= T) return;
  const int w_me = tid / 32;
  const uint32_t below = (1u << (tid % 32)) - 1u;
  for (int j = 0; j < k; ++j) {
    const int e = idx[(size_t)t * k + j];
    int p = -1, row = -1;
    if (e >= 0 && e < E && ((bm[e * kWords + w_me] >> (tid % 32)) & 1u)) {
      int r = __popc(bm[e * kWords + w_me] & below);
      for (int w = 0; w < w_me; ++w) r += __popc(bm[e * kWords + w]);
      p = blk_base[(size_t)blockIdx.x * E + e] + r;
      if (p < capacity) {
        row = offsets[e] + p;
        perm[row] = t * k + j;
      }
    }
    pos[(size_t)t * k + j] = p;
    row_of[(size_t)t * k + j] = row;
  }
}

// T <= 256 (one token block): count, scan, scatter and the row gather in one launch.  Every
// CTA recomputes the (small) dispatch in shared memory with the same counting scheme as the
// 16-byte vectors per row segment copied by one warp in the small dispatch (2 KB)
constexpr int kSmallCopySeg = 128;
// E4M3 rows in the small dispatch: up to this many 16-byte vectors per thread (rows of up to
// kQuantVecs * kDispatchBlock * 8 bf16 values)
constexpr int kQuantVecs = 4;

// three-kernel path (bitmap of the tokens per expert, scans, popcount ranks), so the results
// are identical; CTA 0 publishes it, and all CTAs copy their share of the rows: routed rows
// [0, nkept), then (append_shared) the T token rows after them for the shared experts.
// With fin.part_P set, one extra (last) CTA finishes the load-balance statistics instead.

// The statistics' last step with 256 threads, in exactly aux_final_kernel's arithmetic and
// order: with G = the 32-expert groups (rounded up to a power of two) and W = 32 / G, expert
// e's sum is the sum over sub = 0..W-1 (in order) of the sums over rows sub, sub + W, ...
// (in order), each started from 0; f = count / T, P = sum / T; then warp 0 adds f_i P_i over
// lanes (expert x at lane x mod 32, in order) and the z partials (row b at lane b mod 32),
// each finished by the same butterfly.
__device__ void finish_stats_cta(const StatsFinal& fin, int T, int E) {
  __shared__ float prod[256];
  const int e = threadIdx.x, lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  int G = 1;
  while (G * 32 < E) G <<= 1;
  const int W = 32 / G;
  const float invT = 1.0f / (float)T;
  if (e < E) {
    float ps = 0.f;
    int cs = 0;
    for (int sub = 0; sub < W; ++sub) {
      float p = 0.f;
      int c = 0;
      for (int b0 = sub; b0 < fin.nrows; b0 += 8 * W) {   // eight rows' loads in flight
        float qp[8];
        int qc[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          const int b = b0 + i * W;
          if (b < fin.nrows) {
            qp[i] = fin.part_P[(size_t)b * E + e];
            qc[i] = fin.part_cnt[(size_t)b * E + e];
          }
        }
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          if (b0 + i * W >= fin.nrows) break;
          p += qp[i];
          c += qc[i];
        }
      }
      ps += p;
      cs += c;
    }
    const float fe = (float)cs * invT, Pe = ps * invT;
    if (fin.f) fin.f[e] = fe;
    if (fin.P) fin.P[e] = Pe;
    prod[e] = fe * Pe;
  }
  __syncthreads();
  if (warp == 0) {
    float acc = 0.f;
    for (int x = lane; x < E; x += 32) acc += prod[x];
    acc = warp_sum(acc);
    float z = 0.f;
    for (int b = lane; b < fin.nrows; b += 32) z += fin.part_z[b];
    z = warp_sum(z);
    if (lane == 0) {
      if (fin.l_balance) *fin.l_balance = (float)E * acc;
      if (fin.z_loss) *fin.z_loss = z * invT;
    }
  }
}

__global__ void __launch_bounds__(kDispatchBlock) dispatch_small_kernel(
    const int32_t* __restrict__ idx, int T, int E, int k, int capacity,
    int32_t* __restrict__ counts, int32_t* __restrict__ kept, int32_t* __restrict__ offsets,
    int32_t* __restrict__ mtile_prefix, int32_t* __restrict__ n_dropped,
    int32_t* __restrict__ pos, int32_t* __restrict__ row_of, int32_t* __restrict__ perm,
    DevStatus* st, const unsigned char* __restrict__ x, unsigned char* __restrict__ x_perm,
    int row_bytes, int append_shared, const StatsFinal fin, uint8_t* __restrict__ x8,
    float* __restrict__ sx) {
  pdl_prologue();
  const bool with_stats = fin.part_P != nullptr;
  if (with_stats && blockIdx.x == gridDim.x - 1) {
    finish_stats_cta(fin, T, E);
    return;
  }
  __shared__ uint32_t bm[256 * kWords];
  __shared__ int s_kept[256];
  __shared__ int s_mt[256];
  __shared__ int s_drop[256];
  __shared__ int s_off[257];
  __shared__ int s_perm[256 * 8];
  __shared__ int s_wsum[3][kDispatchBlock / 32];
  const bool lead = blockIdx.x == 0;
  const int tid = threadIdx.x;
  for (int i = tid; i < E * kWords; i += blockDim.x) bm[i] = 0u;
  __syncthreads();
  const int t = tid;
  if (t < T) {
    int sel[8];
    for (int j = 0; j < k; ++j) {
      const int e = idx[(size_t)t * k + j];
      bool bad = e < 0 || e >= E;
      for (int q = 0; q < j; ++q) bad |= (sel[q] == e);
      sel[j] = bad ? -1 : e;
      if (bad) {
        if (lead) record_error(st, MOE_ERR_ARG, t);
        continue;
      }
      atomicOr(&bm[e * kWords + tid / 32], 1u << (tid % 32));
    }
  }
  __syncthreads();
  const int e = tid;
  int total = 0;
  if (e < E) {
#pragma unroll
    for (int w = 0; w < kWords; ++w) total += __popc(bm[e * kWords + w]);
  }
  const int kp = e < E ? min(total, capacity) : 0;
  s_kept[e] = kp;
  s_mt[e] = ceil_div(kp, kTileM);
  s_drop[e] = e < E ? total - kp : 0;
  if (lead && e < E) {
    counts[e] = total;
    kept[e] = kp;
  }
  // inclusive scans over the 256 expert slots: within each warp by shuffles, then each warp
  // adds the totals of the warps before it
  {
    const int lane = tid & 31, wi = tid >> 5;
    int a = s_kept[e], b = s_mt[e], c = s_drop[e];
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int a2 = __shfl_up_sync(0xffffffffu, a, o);
      const int b2 = __shfl_up_sync(0xffffffffu, b, o);
      const int c2 = __shfl_up_sync(0xffffffffu, c, o);
      if (lane >= o) { a += a2; b += b2; c += c2; }
    }
    if (lane == 31) { s_wsum[0][wi] = a; s_wsum[1][wi] = b; s_wsum[2][wi] = c; }
    __syncthreads();
    for (int q = 0; q < wi; ++q) { a += s_wsum[0][q]; b += s_wsum[1][q]; c += s_wsum[2][q]; }
    s_kept[e] = a;
    s_mt[e] = b;
    s_drop[e] = c;
  }
  __syncthreads();
  if (e < E) s_off[e + 1] = s_kept[e];
  if (e == 0) s_off[0] = 0;
  if (lead) {
    if (e < E) {
      offsets[e + 1] = s_kept[e];
      mtile_prefix[e + 1] = s_mt[e];
    }
    if (e == 0) {
      offsets[0] = 0;
      mtile_prefix[0] = 0;
      *n_dropped = s_drop[255];
    }
  }
  __syncthreads();
  if (t < T) {
    const int w_me = tid / 32;
    const uint32_t below = (1u << (tid % 32)) - 1u;
    for (int j = 0; j < k; ++j) {
      const int ex = idx[(size_t)t * k + j];
      int p = -1, row = -1;
      if (ex >= 0 && ex < E && ((bm[ex * kWords + w_me] >> (tid % 32)) & 1u)) {
        int r = __popc(bm[ex * kWords + w_me] & below);
        for (int w = 0; w < w_me; ++w) r += __popc(bm[ex * kWords + w]);
        p = r;
        if (p < capacity) {
          row = s_off[ex] + p;
          s_perm[row] = t * k + j;
        }
      }
      if (lead) {
        pos[(size_t)t * k + j] = p;
        row_of[(size_t)t * k + j] = row;
      }
    }
  }
  __syncthreads();
  const int nkept = s_off[E];
  if (lead)
    for (int r = tid; r < T * k; r += blockDim.x) perm[r] = r < nkept ? s_perm[r] : -1;
  if (x == nullptr) return;
  if (x8) {
    // E4M3 rows instead of bf16 copies, one row per CTA at a time, exactly as the row
    // quantiser makes them: amax = max |v|, inv = 448 / amax, code = e4m3(v * inv) (nearest
    // even, saturating), scale = amax / 448; the row is read once (registers)
    __shared__ float red[kDispatchBlock / 32];
    const int nrows = nkept + (append_shared ? T : 0);
    const int vecs = row_bytes / 16;
    const int copy_ctas = gridDim.x - (with_stats ? 1 : 0);
    for (int r = blockIdx.x; r < nrows; r += copy_ctas) {
      const int src_t = r < nkept ? s_perm[r] / k : r - nkept;
      const uint4* src = reinterpret_cast<const uint4*>(x + (size_t)src_t * row_bytes);
      uint4 v[kQuantVecs];
      float amax = 0.f;
#pragma unroll
      for (int i = 0; i < kQuantVecs; ++i) {
        const int c = tid + i * kDispatchBlock;
        if (c < vecs) {
          v[i] = __ldg(src + c);
          const __nv_bfloat162* b = reinterpret_cast<const __nv_bfloat162*>(&v[i]);
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            const float2 f = __bfloat1622float2(b[j]);
            amax = fmaxf(amax, fmaxf(fabsf(f.x), fabsf(f.y)));
          }
        }
      }
      amax = warp_max(amax);
      if ((tid & 31) == 0) red[tid >> 5] = amax;
      __syncthreads();
      amax = red[0];
      for (int w = 1; w < kDispatchBlock / 32; ++w) amax = fmaxf(amax, red[w]);
      __syncthreads();                             // red is rewritten for the next row
      const float inv = amax > 0.f ? 448.0f / amax : 0.f;
      uint2* d = reinterpret_cast<uint2*>(x8 + (size_t)r * (row_bytes / 2));
#pragma unroll
      for (int i = 0; i < kQuantVecs; ++i) {
        const int c = tid + i * kDispatchBlock;
        if (c >= vecs) break;
        const __nv_bfloat162* b = reinterpret_cast<const __nv_bfloat162*>(&v[i]);
        uint32_t packed[2];
#pragma unroll
        for (int j = 0; j < 2; ++j) {
          const float2 f0 = __bfloat1622float2(b[2 * j]);
          const float2 f1 = __bfloat1622float2(b[2 * j + 1]);
          const uint32_t q0 = __nv_cvt_float2_to_fp8x2(make_float2(f0.x * inv, f0.y * inv),
                                                       __NV_SATFINITE, __NV_E4M3);
          const uint32_t q1 = __nv_cvt_float2_to_fp8x2(make_float2(f1.x * inv, f1.y * inv),
                                                       __NV_SATFINITE, __NV_E4M3);
          packed[j] = (q0 & 0xFFFFu) | (q1 << 16);
        }
        d[c] = make_uint2(packed[0], packed[1]);
      }
      if (tid == 0) sx[r] = amax > 0.f ? amax / 448.0f : 0.f;
    }
    return;
  }
  // row copies: one warp per 2 KB segment of a row (routed rows, then appended rows), four
  // 16-byte loads in flight per lane
  const int lane = tid & 31;
  const int nrows = nkept + (append_shared ? T : 0);
  const int n16 = row_bytes / 16;
  const int segs = ceil_div(n16, kSmallCopySeg);
  const int warps = ((gridDim.x - (with_stats ? 1 : 0)) * blockDim.x) >> 5;
  for (int item = (blockIdx.x * blockDim.x + tid) >> 5; item < nrows * segs; item += warps) {
    const int r = item / segs, sg = item - r * segs;
    const int src_t = r < nkept ? s_perm[r] / k : r - nkept;
    const uint4* src = reinterpret_cast<const uint4*>(x + (size_t)src_t * row_bytes);
    uint4* dst = reinterpret_cast<uint4*>(x_perm + (size_t)r * row_bytes);
    const int i0 = sg * kSmallCopySeg, i1 = min(n16, i0 + kSmallCopySeg);
    uint4 v[4];
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const int i = i0 + lane + 32 * u;
      if (i < i1) v[u] = __ldg(src + i);
    }
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const int i = i0 + lane + 32 * u;
      if (i < i1) dst[i] = v[u];
    }
  }
}

bool dispatch_finalizes_stats(const moe_config& c) { return c.T <= kDispatchBlock; }

bool dispatch_quantizes(const moe_config& c) {
  return c.T <= kDispatchBlock && c.dtype == MOE_DTYPE_BF16 &&
         c.d_model <= kQuantVecs * kDispatchBlock * 8;
}

// One warp per expert-ordered row; rows past offsets[E] get perm = -1.
template <int VEC_BYTES>
__global__ void __launch_bounds__(256) gather_rows_kernel(const int32_t* __restrict__ offsets,
                                                         int E, int k, int total_rows,
                                                         int row_bytes,
                                                         int32_t* __restrict__ perm,
                                                         const unsigned char* __restrict__ x,
                                                         unsigned char* __restrict__ x_perm) {
  pdl_prologue();
  const int lane = threadIdx.x & 31;
  const int warps = (gridDim.x * blockDim.x) >> 5;
  const int nkept = offsets[E];
  for (int r = (blockIdx.x * blockDim.x + threadIdx.x) >> 5; r < total_rows; r += warps) {
    if (r >= nkept) {
      if (lane == 0) perm[r] = -1;
      continue;
    }
    if (x == nullptr) continue;
    const int t = perm[r] / k;
    const uint4* src = reinterpret_cast<const uint4*>(x + (size_t)t * row_bytes);
    uint4* dst = reinterpret_cast<uint4*>(x_perm + (size_t)r * row_bytes);
    const int n16 = row_bytes / 16;
    for (int i = lane; i < n16; i += 32) dst[i] = __ldg(src + i);
  }
}

// x_perm[offsets[E] + t] = x[t]: the shared experts' rows after the routed rows (decode path).
__global__ void __launch_bounds__(256) append_rows_kernel(const int32_t* __restrict__ offsets,
                                                         int E, int T, int row_bytes,
                                                         const unsigned char* __restrict__ x,
                                                         unsigned char* __restrict__ x_perm) {
  pdl_prologue();
  const int lane = threadIdx.x & 31;
  const int warps = (gridDim.x * blockDim.x) >> 5;
  const size_t base = (size_t)offsets[E];
  for (int t = (blockIdx.x * blockDim.x + threadIdx.x) >> 5; t < T; t += warps) {
    const uint4* src = reinterpret_cast<const uint4*>(x + (size_t)t * row_bytes);
    uint4* dst = reinterpret_cast<uint4*>(x_perm + (base + t) * row_bytes);
    for (int i = lane; i < row_bytes / 16; i += 32) dst[i] = __ldg(src + i);
  }
}

cudaError_t launch_append_rows(const moe_config& c, const int32_t* offsets, const void* x,
                               void* x_perm, cudaStream_t s) {
  const int row_bytes = c.d_model * (c.dtype == MOE_DTYPE_F32 ? 4 : 2);
  int blocks = ceil_div(c.T, 8);
  if (blocks > num_sms() * 4) blocks = num_sms() * 4;
  launch_pdl(append_rows_kernel, blocks, 256, 0, s, offsets, c.E, c.T, row_bytes,
                                            (const unsigned char*)x, (unsigned char*)x_perm);
  return cudaGetLastError();
}

cudaError_t launch_dispatch(const moe_config& c, int capacity, const int32_t* idx,
                            const DispatchBufs& b, const void* x, void* x_perm, DevStatus* st,
                            cudaStream_t s, bool append_shared, const StatsFinal* fin,
                            uint8_t* x8, float* sx) {
  const int nblk = ceil_div(c.T, kDispatchBlock);
  cudaError_t err;
  const int esz = c.dtype == MOE_DTYPE_F32 ? 4 : 2;
  const int row_bytes = c.d_model * esz;
  if (nblk == 1) {
    const int rows = c.T * c.k + (append_shared ? c.T : 0);
    const int items = rows * ceil_div(row_bytes / 16, kSmallCopySeg);
    // row copies: up to one CTA per SM; E4M3 rows (one CTA per row at a time, two barriers
    // per row): up to four per SM
    int blocks = x ? (x8 ? rows : ceil_div(items, 8)) : 1;
    const int cap = x8 ? 4 * num_sms() : num_sms();
    if (blocks > cap) blocks = cap;
    const StatsFinal none{};
    const StatsFinal& sf = fin ? *fin : none;
    if (fin) ++blocks;                       // the statistics' CTA
    launch_pdl(dispatch_small_kernel, blocks, kDispatchBlock, 0, s,
        idx, c.T, c.E, c.k, capacity, b.counts, b.kept, b.offsets, b.mtile_prefix, b.n_dropped,
        b.pos, b.row_of, b.perm, st, (const unsigned char*)x, (unsigned char*)x_perm, row_bytes,
        append_shared ? 1 : 0, sf, x8, sx);
    return cudaGetLastError();
  } else {
    launch_pdl(dispatch_count_kernel, nblk, kDispatchBlock, 0, s, idx, c.T, c.E, c.k, b.bitmap,
                                                          b.blk_base, st);
    if ((err = cudaGetLastError()) != cudaSuccess) return err;
    launch_pdl(dispatch_scan_kernel, 1, 256, 0, s, b.blk_base, nblk, c.E, capacity, b.counts, b.kept,
                                           b.offsets, b.mtile_prefix, b.n_dropped);
    if ((err = cudaGetLastError()) != cudaSuccess) return err;
    launch_pdl(dispatch_scatter_kernel, nblk, kDispatchBlock, 0, s, idx, c.T, c.E, c.k, capacity,
                                                            b.bitmap, b.blk_base, b.offsets,
                                                            b.pos, b.row_of, b.perm);
    if ((err = cudaGetLastError()) != cudaSuccess) return err;
  }
  const int total_rows = c.T * c.k;
  int blocks = ceil_div(total_rows, 8);
  const int cap_blocks = num_sms() * 8;
  if (blocks > cap_blocks) blocks = cap_blocks;
  launch_pdl(gather_rows_kernel<16>, blocks, 256, 0, s, b.offsets, c.E, c.k, total_rows, row_bytes,
                                                b.perm, (const unsigned char*)x,
                                                (unsigned char*)x_perm);
  if ((err = cudaGetLastError()) != cudaSuccess) return err;
  if (append_shared && x) return launch_append_rows(c, b.offsets, x, x_perm, s);
  return cudaSuccess;
}

}  // namespace moe
