// Weighted combine: out[t] = shared[t] + sum_j w[t,j] * y[row_of[t,j]]
//   ["MoE 路由数学" §2.1 Output = sum_{i in S} p~_i Expert_i(x), §2.2 shared experts;
//    "Systems for Mixture-of-Experts Models" §2.2 step 4 (add back in place)]
// One warp per token, 16-byte vector loads along d, fp32 accumulation in the fixed order
// j = 0..k-1 after the shared term; each token's row is written once (no atomics).  A dropped
// pair (row -1) adds nothing and the other weights keep their values.
#include <cuda_bf16.h>

#include "common.cuh"
#include "kernels.h"

namespace moe {

template <typename T>
struct Vec16 {
  static constexpr int N = 16 / sizeof(T);
};

template <typename T>
__device__ __forceinline__ void unpack16(const uint4& v, float* f) {
  if constexpr (sizeof(T) == 4) {
    f[0] = __uint_as_float(v.x); f[1] = __uint_as_float(v.y);
    f[2] = __uint_as_float(v.z); f[3] = __uint_as_float(v.w);
  } else {
    const __nv_bfloat162* h = reinterpret_cast<const __nv_bfloat162*>(&v);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      float2 p = __bfloat1622float2(h[i]);
      f[2 * i] = p.x;
      f[2 * i + 1] = p.y;
    }
  }
}

template <typename T>
__device__ __forceinline__ uint4 pack16(const float* f) {
  uint4 v;
  if constexpr (sizeof(T) == 4) {
    v.x = __float_as_uint(f[0]); v.y = __float_as_uint(f[1]);
    v.z = __float_as_uint(f[2]); v.w = __float_as_uint(f[3]);
  } else {
    __nv_bfloat162* h = reinterpret_cast<__nv_bfloat162*>(&v);
#pragma unroll
    for (int i = 0; i < 4; ++i) h[i] = __floats2bfloat162_rn(f[2 * i], f[2 * i + 1]);
  }
  return v;
}

// Token-choice combine.
template <typename T>
__global__ void __launch_bounds__(256) combine_kernel(const T* __restrict__ y,
                                                     const int32_t* __restrict__ row_of,
                                                     const float* __restrict__ w,
                                                     const T* __restrict__ shared,
                                                     T* __restrict__ out, int Tn, int d, int k) {
  constexpr int N = Vec16<T>::N;
  const int lane = threadIdx.x & 31;
  const int t = (blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  if (t >= Tn) return;
  int rows[8];
  float ws[8];
  for (int j = 0; j < k; ++j) {
    rows[j] = row_of[(size_t)t * k + j];
    ws[j] = w[(size_t)t * k + j];
  }
  const int nv = d / N;
  for (int v = lane; v < nv; v += 32) {
    float acc[N];
    if (shared) {
      uint4 s = *reinterpret_cast<const uint4*>(shared + (size_t)t * d + v * N);
      unpack16<T>(s, acc);
    } else {
#pragma unroll
      for (int i = 0; i < N; ++i) acc[i] = 0.f;
    }
    for (int j = 0; j < k; ++j) {
      if (rows[j] < 0) continue;
      uint4 q = __ldg(reinterpret_cast<const uint4*>(y + (size_t)rows[j] * d + v * N));
      float f[N];
      unpack16<T>(q, f);
#pragma unroll
      for (int i = 0; i < N; ++i) acc[i] = fmaf(ws[j], f[i], acc[i]);
    }
    *reinterpret_cast<uint4*>(out + (size_t)t * d + v * N) = pack16<T>(acc);
  }
}

cudaError_t launch_combine(const moe_config& c, const void* y_perm, const int32_t* row_of,
                           const float* w, const void* shared_out, void* out, cudaStream_t s) {
  const int blocks = ceil_div(c.T * 32, 256);
  if (c.dtype == MOE_DTYPE_F32)
    combine_kernel<float><<<blocks, 256, 0, s>>>((const float*)y_perm, row_of, w,
                                                 (const float*)shared_out, (float*)out, c.T,
                                                 c.d_model, c.k);
  else
    combine_kernel<__nv_bfloat16><<<blocks, 256, 0, s>>>(
        (const __nv_bfloat16*)y_perm, row_of, w, (const __nv_bfloat16*)shared_out,
        (__nv_bfloat16*)out, c.T, c.d_model, c.k);
  return cudaGetLastError();
}

// Expert-choice combine: token t sums the rows tok_rows[tok_ptr[t] .. tok_ptr[t+1]) (ascending
// expert order) with weights w_flat[row].
template <typename T>
__global__ void __launch_bounds__(256) combine_ec_kernel(const T* __restrict__ y,
                                                        const int32_t* __restrict__ tok_ptr,
                                                        const int32_t* __restrict__ tok_rows,
                                                        const float* __restrict__ w_flat,
                                                        const T* __restrict__ shared,
                                                        T* __restrict__ out, int Tn, int d) {
  constexpr int N = Vec16<T>::N;
  const int lane = threadIdx.x & 31;
  const int t = (blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  if (t >= Tn) return;
  const int b = tok_ptr[t], e_ = tok_ptr[t + 1];
  const int nv = d / N;
  for (int v = lane; v < nv; v += 32) {
    float acc[N];
    if (shared) {
      uint4 s = *reinterpret_cast<const uint4*>(shared + (size_t)t * d + v * N);
      unpack16<T>(s, acc);
    } else {
#pragma unroll
      for (int i = 0; i < N; ++i) acc[i] = 0.f;
    }
    for (int q = b; q < e_; ++q) {
      const int r = tok_rows[q];
      const float wt = w_flat[r];
      uint4 qv = __ldg(reinterpret_cast<const uint4*>(y + (size_t)r * d + v * N));
      float f[N];
      unpack16<T>(qv, f);
#pragma unroll
      for (int i = 0; i < N; ++i) acc[i] = fmaf(wt, f[i], acc[i]);
    }
    *reinterpret_cast<uint4*>(out + (size_t)t * d + v * N) = pack16<T>(acc);
  }
}

cudaError_t launch_combine_ec(const moe_config& c, const void* y_perm, const int32_t* tok_ptr,
                              const int32_t* tok_rows, const float* ec_w_flat,
                              const void* shared_out, void* out, cudaStream_t s) {
  const int blocks = ceil_div(c.T * 32, 256);
  if (c.dtype == MOE_DTYPE_F32)
    combine_ec_kernel<float><<<blocks, 256, 0, s>>>((const float*)y_perm, tok_ptr, tok_rows,
                                                    ec_w_flat, (const float*)shared_out,
                                                    (float*)out, c.T, c.d_model);
  else
    combine_ec_kernel<__nv_bfloat16><<<blocks, 256, 0, s>>>(
        (const __nv_bfloat16*)y_perm, tok_ptr, tok_rows, ec_w_flat,
        (const __nv_bfloat16*)shared_out, (__nv_bfloat16*)out, c.T, c.d_model);
  return cudaGetLastError();
}

}  // namespace moe
