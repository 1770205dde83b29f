// Per-row E4M3 quantisation of bf16 rows (sm_103a): expert weights once, and the token rows
// that enter the FP8 expert GEMMs on every forward.
//
// FP8 expert weights halve the bytes a decode step streams ("Systems for Mixture-of-Experts
// Models" §1.4: DeepSeek-V3 keeps its weights in FP8; "MoE 推理优化深入" §4.2: experts may be
// quantised).  Each row (a weight's output channel, or one token's activations) gets one fp32
// scale:
//   amax = max |v|,  inv = 448 / amax,  code = e4m3(v * inv),  scale = amax / 448
// in float32, round to nearest even with saturation at +-448 (the largest finite E4M3 value);
// a row of zeros gets codes 0 and scale 0.  The row is codes * scale.
#include <cuda_bf16.h>
#include <cuda_fp8.h>

#include "common.cuh"
#include "kernels.h"

namespace moe {
namespace {

// One warp per row, 8 bf16 (16 bytes) per lane and step; the row is read twice (amax, codes).
__global__ void __launch_bounds__(256) quantize_rows_kernel(const __nv_bfloat16* __restrict__ src,
                                                           long long nrows_max, int cols,
                                                           const int32_t* nrows_base,
                                                           int nrows_extra,
                                                           uint8_t* __restrict__ dst,
                                                           float* __restrict__ scale) {
  pdl_prologue();
  long long nrows = nrows_max;
  if (nrows_base) {
    const long long n = static_cast<long long>(*nrows_base) + nrows_extra;
    nrows = n < nrows_max ? n : nrows_max;
  }
  const int lane = threadIdx.x & 31;
  const long long warps = static_cast<long long>(gridDim.x) * (blockDim.x >> 5);
  const int vecs = cols / 8;
  for (long long row = blockIdx.x * (long long)(blockDim.x >> 5) + (threadIdx.x >> 5);
       row < nrows; row += warps) {
    const uint4* s = reinterpret_cast<const uint4*>(src + row * cols);
    float amax = 0.f;
    for (int i = lane; i < vecs; i += 32) {
      const uint4 v = s[i];
      const __nv_bfloat162* b = reinterpret_cast<const __nv_bfloat162*>(&v);
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const float2 f = __bfloat1622float2(b[j]);
        amax = fmaxf(amax, fmaxf(fabsf(f.x), fabsf(f.y)));
      }
    }
    amax = warp_max(amax);
    const float inv = amax > 0.f ? 448.0f / amax : 0.f;
    uint2* d = reinterpret_cast<uint2*>(dst + row * cols);
    for (int i = lane; i < vecs; i += 32) {
      const uint4 v = s[i];
      const __nv_bfloat162* b = reinterpret_cast<const __nv_bfloat162*>(&v);
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
      d[i] = make_uint2(packed[0], packed[1]);
    }
    if (lane == 0) scale[row] = amax > 0.f ? amax / 448.0f : 0.f;
  }
}

// One CTA per row, for short lists of rows (the token rows of a decode batch): each thread keeps
// up to kRowVecs 16-byte vectors of the row in registers, so the row is read once and all its
// loads are in flight together; the amax is reduced over the CTA.  Per element the arithmetic
// is the warp kernel's, and a maximum does not depend on its order, so both give the same bytes.
constexpr int kRowVecs = 4;
__global__ void __launch_bounds__(1024) quantize_row_cta_kernel(
    const __nv_bfloat16* __restrict__ src, long long nrows_max, int cols,
    const int32_t* nrows_base, int nrows_extra, uint8_t* __restrict__ dst,
    float* __restrict__ scale) {
  pdl_prologue();
  __shared__ float red[32];
  long long nrows = nrows_max;
  if (nrows_base) {
    const long long n = static_cast<long long>(*nrows_base) + nrows_extra;
    nrows = n < nrows_max ? n : nrows_max;
  }
  const long long row = blockIdx.x;
  if (row >= nrows) return;
  const int vecs = cols / 8;
  const uint4* s = reinterpret_cast<const uint4*>(src + row * cols);
  uint4 v[kRowVecs];
  float amax = 0.f;
#pragma unroll
  for (int i = 0; i < kRowVecs; ++i) {
    const int c = threadIdx.x + i * blockDim.x;
    if (c < vecs) v[i] = s[c];
  }
#pragma unroll
  for (int i = 0; i < kRowVecs; ++i) {
    if (threadIdx.x + i * blockDim.x >= vecs) break;
    const __nv_bfloat162* b = reinterpret_cast<const __nv_bfloat162*>(&v[i]);
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const float2 f = __bfloat1622float2(b[j]);
      amax = fmaxf(amax, fmaxf(fabsf(f.x), fabsf(f.y)));
    }
  }
  amax = warp_max(amax);
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = amax;
  __syncthreads();
  amax = red[0];
  for (int w = 1; w < static_cast<int>(blockDim.x >> 5); ++w) amax = fmaxf(amax, red[w]);
  const float inv = amax > 0.f ? 448.0f / amax : 0.f;
  uint2* d = reinterpret_cast<uint2*>(dst + row * cols);
#pragma unroll
  for (int i = 0; i < kRowVecs; ++i) {
    const int c = threadIdx.x + i * blockDim.x;
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
  if (threadIdx.x == 0) scale[row] = amax > 0.f ? amax / 448.0f : 0.f;
}

}  // namespace

cudaError_t launch_quantize_rows(const void* src, long long nrows_max, int cols,
                                 const int32_t* nrows_base, int nrows_extra, uint8_t* dst,
                                 float* scale, cudaStream_t s) {
  const int vecs = cols / 8;
  if (nrows_max <= 8ll * num_sms() && vecs <= kRowVecs * 1024) {
    int threads = (vecs + 1) / 2;
    threads = (threads + 31) / 32 * 32;
    if (threads > 1024) threads = 1024;
    launch_pdl(quantize_row_cta_kernel, static_cast<int>(nrows_max), threads, 0, s,
               static_cast<const __nv_bfloat16*>(src), nrows_max, cols, nrows_base, nrows_extra,
               dst, scale);
    return cudaGetLastError();
  }
  long long blocks = (nrows_max + 7) / 8;
  const long long cap = static_cast<long long>(num_sms()) * 16;
  if (blocks > cap) blocks = cap;
  if (blocks < 1) blocks = 1;
  launch_pdl(quantize_rows_kernel, static_cast<int>(blocks), 256, 0, s,
      static_cast<const __nv_bfloat16*>(src), nrows_max, cols, nrows_base, nrows_extra, dst,
      scale);
  return cudaGetLastError();
}

}  // namespace moe

extern "C" int moe_quantize_fp8(int64_t rows, int64_t cols, const void* src, uint8_t* dst,
                                float* scale, void* stream) {
  if (!src || !dst || !scale) return MOE_ERR_ARG;
  if (rows < 1 || cols < 16 || cols % 16 || cols > (1 << 20) || rows > (1ll << 31))
    return MOE_ERR_SHAPE;
  return moe::launch_quantize_rows(src, rows, static_cast<int>(cols), nullptr, 0, dst, scale,
                                   static_cast<cudaStream_t>(stream)) == cudaSuccess
             ? MOE_OK
             : MOE_ERR_CUDA;
}
