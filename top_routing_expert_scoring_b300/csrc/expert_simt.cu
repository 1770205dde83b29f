// Grouped SwiGLU expert FFN on CUDA cores (the float32 path):
//   h = SiLU(x W1^T) * (x W3^T),  y = h W2^T        ["Systems for Mixture-of-Experts Models"
//                                                     §5.2 SwiGLU]
// over expert-ordered rows: expert e owns rows [offsets[e], offsets[e+1]).  One CTA computes a
// 128-row x 64-column tile of one expert; rows past the expert's end are computed from
// whatever the buffer holds and never stored.
#include <cuda_bf16.h>

#include <type_traits>

#include "common.cuh"
#include "kernels.h"

namespace moe {

struct SimtArgs {
  const void* A;          // [rows, K]
  const void* B;          // expert e's matrix starts at B + e * b_stride (elements), rows are N
  size_t b_stride;
  int up_off;             // SwiGLU: rows of the up projection start here (F)
  void* out;              // [rows, N]
  int K, N;
  const int32_t* offsets;
  const int32_t* mtp;
  int E;
  int uniform_rows;
};

__device__ __forceinline__ void locate_tile(int tile, const int32_t* mtp, const int32_t* offsets,
                                            int E, int uniform_rows, int& e, int& row0,
                                            int& rows, bool& valid) {
  if (uniform_rows >= 0) {
    e = 0;
    row0 = tile * kTileM;
    rows = min(kTileM, uniform_rows - row0);
    valid = rows > 0;
    return;
  }
  const int total = mtp[E];
  valid = tile < total;
  if (!valid) return;
  int lo = 0, hi = E;
  while (hi - lo > 1) {
    const int mid = (lo + hi) >> 1;
    if (mtp[mid] <= tile) lo = mid; else hi = mid;
  }
  e = lo;
  row0 = offsets[e] + (tile - mtp[e]) * kTileM;
  rows = min(kTileM, offsets[e + 1] - row0);
}

template <typename T, bool SWIGLU>
__global__ void __launch_bounds__(256) ffn_simt_kernel(SimtArgs a) {
  pdl_prologue();
  using TO = typename std::conditional<SWIGLU, T, float>::type;   // h in T, y in float32
  constexpr int TM = kTileM, TN = 64, TK = 16;
  __shared__ float As[TK][TM + 4];
  __shared__ float Bs[TK][TN + 4];
  __shared__ float Us[SWIGLU ? TK : 1][TN + 4];
  int e, row0, rows;
  bool valid;
  locate_tile(blockIdx.x, a.mtp, a.offsets, a.E, a.uniform_rows, e, row0, rows, valid);
  if (!valid) return;
  const int n0 = blockIdx.y * TN;
  const T* A = (const T*)a.A;
  const T* B = (const T*)a.B + (size_t)e * a.b_stride;
  const int tid = threadIdx.x;
  const int tr = tid / 16, tc = tid % 16;        // 8 rows x 4 cols per thread
  float acc[8][4] = {}, accu[SWIGLU ? 8 : 1][4] = {};
  for (int k0 = 0; k0 < a.K; k0 += TK) {
    for (int i = tid; i < TM * TK; i += 256) {
      const int r = i / TK, kk = i % TK;
      As[kk][r] = (r < rows && k0 + kk < a.K) ? to_f32(A[(size_t)(row0 + r) * a.K + k0 + kk]) : 0.f;
    }
    for (int i = tid; i < TN * TK; i += 256) {
      const int n = i / TK, kk = i % TK;
      const bool ok = n0 + n < a.N && k0 + kk < a.K;
      Bs[kk][n] = ok ? to_f32(B[(size_t)(n0 + n) * a.K + k0 + kk]) : 0.f;
      if constexpr (SWIGLU)
        Us[kk][n] = ok ? to_f32(B[(size_t)(a.up_off + n0 + n) * a.K + k0 + kk]) : 0.f;
    }
    __syncthreads();
#pragma unroll
    for (int kk = 0; kk < TK; ++kk) {
      float av[8], bv[4], uv[4];
#pragma unroll
      for (int i = 0; i < 8; ++i) av[i] = As[kk][tr * 8 + i];
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        bv[j] = Bs[kk][tc * 4 + j];
        if constexpr (SWIGLU) uv[j] = Us[kk][tc * 4 + j];
      }
#pragma unroll
      for (int i = 0; i < 8; ++i)
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          acc[i][j] = fmaf(av[i], bv[j], acc[i][j]);
          if constexpr (SWIGLU) accu[i][j] = fmaf(av[i], uv[j], accu[i][j]);
        }
    }
    __syncthreads();
  }
  TO* out = (TO*)a.out;
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const int r = tr * 8 + i;
    if (r >= rows) continue;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const int n = n0 + tc * 4 + j;
      if (n >= a.N) continue;
      float v = acc[i][j];
      if constexpr (SWIGLU) v = (v / (1.0f + expf(-v))) * accu[i][j];
      out[(size_t)(row0 + r) * a.N + n] = from_f32<TO>(v);
    }
  }
}

cudaError_t launch_ffn_simt(const GroupedFFN& g, bool f32, DevStatus* st, cudaStream_t s) {
  (void)st;
  const int mtiles = g.uniform_rows >= 0 ? ceil_div(g.uniform_rows, kTileM)
                                         : ceil_div(g.max_rows, kTileM) + g.E;
  SimtArgs up{g.x, g.w13, (size_t)2 * g.F * g.d, g.F, g.h, g.d, g.F, g.offsets, g.mtile_prefix,
              g.E, g.uniform_rows};
  SimtArgs down{g.h, g.w2, (size_t)g.d * g.F, 0, g.y, g.F, g.d, g.offsets, g.mtile_prefix, g.E,
                g.uniform_rows};
  dim3 g1(mtiles, ceil_div(g.F, 64)), g2(mtiles, ceil_div(g.d, 64));
  if (f32) {
    launch_pdl(ffn_simt_kernel<float, true>, g1, 256, 0, s, up);
    launch_pdl(ffn_simt_kernel<float, false>, g2, 256, 0, s, down);
  } else {
    launch_pdl(ffn_simt_kernel<__nv_bfloat16, true>, g1, 256, 0, s, up);
    launch_pdl(ffn_simt_kernel<__nv_bfloat16, false>, g2, 256, 0, s, down);
  }
  return cudaGetLastError();
}

}  // namespace moe
