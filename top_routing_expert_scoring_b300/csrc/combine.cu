// Weighted combine: out[t] = shared[t] + sum_j w[t,j] * y[row_of[t,j]]
// (y and shared in float32; out rounded once to bf16, or kept in float32)
//   ["MoE 路由数学" §2.1 Output = sum_{i in S} p~_i Expert_i(x), §2.2 shared experts;
//    "Systems for Mixture-of-Experts Models" §2.2 step 4 (add back in place)]
// One warp per 512-column slice of a token, 16-byte vector loads, fp32 accumulation in the fixed order
// j = 0..k-1 after the shared term; each token's row is written once (no atomics).  A dropped
// pair (row -1) adds nothing and the other weights keep their values.
#include <cuda_bf16.h>

#include "common.cuh"
#include "kernels.h"

namespace moe {

// Columns per warp: a token's row is split over ceil(d / slice) warps, slice = 512 while that
// still gives >= 2048 warps, else 256 or 128, so that decode batches still spread over the GPU
// (each lane handles 4 columns per 128-column step).
constexpr int kCombineSlice = 512;
inline int combine_slice(const moe_config& c) {
  for (int sl = kCombineSlice; sl > 128; sl >>= 1)
    if ((long long)c.T * ceil_div(c.d_model, sl) >= 2048) return sl;
  return 128;
}

// float4 of y / shared in, 4 output values out (bf16: 8 bytes, float32: 16 bytes).
template <typename TOut>
__device__ __forceinline__ void store4(TOut* dst, const float* a) {
  if constexpr (sizeof(TOut) == 4) {
    *reinterpret_cast<float4*>(dst) = make_float4(a[0], a[1], a[2], a[3]);
  } else {
    __nv_bfloat162 lo = __floats2bfloat162_rn(a[0], a[1]);
    __nv_bfloat162 hi = __floats2bfloat162_rn(a[2], a[3]);
    uint2 v;
    v.x = *reinterpret_cast<uint32_t*>(&lo);
    v.y = *reinterpret_cast<uint32_t*>(&hi);
    *reinterpret_cast<uint2*>(dst) = v;
  }
}

__device__ __forceinline__ void load_shared4(const float* shared, size_t off, float* acc) {
  if (shared) {
    const float4 q = *reinterpret_cast<const float4*>(shared + off);
    acc[0] = q.x; acc[1] = q.y; acc[2] = q.z; acc[3] = q.w;
  } else {
    acc[0] = acc[1] = acc[2] = acc[3] = 0.f;
  }
}

// Sum of nsplit partials (stride apart), in order, of 4 consecutive values.
__device__ __forceinline__ void sum_parts4(const float* p, int nsplit, size_t stride, float* v) {
  float4 q = __ldg(reinterpret_cast<const float4*>(p));
  v[0] = q.x; v[1] = q.y; v[2] = q.z; v[3] = q.w;
  for (int sl = 1; sl < nsplit; ++sl) {
    q = __ldg(reinterpret_cast<const float4*>(p + sl * stride));
    v[0] += q.x; v[1] += q.y; v[2] += q.z; v[3] += q.w;
  }
}

__device__ __forceinline__ void fma4(float wt, const float* y, float* acc) {
  const float4 q = __ldg(reinterpret_cast<const float4*>(y));
  acc[0] = fmaf(wt, q.x, acc[0]);
  acc[1] = fmaf(wt, q.y, acc[1]);
  acc[2] = fmaf(wt, q.z, acc[2]);
  acc[3] = fmaf(wt, q.w, acc[3]);
}

// Token-choice combine (y float32, shared float32, out bf16 or float32).
template <typename TOut>
__global__ void __launch_bounds__(256) combine_kernel(const float* __restrict__ y,
                                                     const int32_t* __restrict__ row_of,
                                                     const float* __restrict__ w,
                                                     const float* __restrict__ shared,
                                                     TOut* __restrict__ out, int Tn, int d,
                                                     int k, int nsplit, size_t y_stride,
                                                     size_t shared_stride, int slice) {
  pdl_prologue();
  const int lane = threadIdx.x & 31;
  const int gw = (blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const int slices = ceil_div(d, slice);
  const int t = gw / slices;
  if (t >= Tn) return;
  const int v0 = (gw - t * slices) * slice;
  const int v1 = min(d, v0 + slice);
  int rows[8];
  float ws[8];
#pragma unroll
  for (int j = 0; j < 8; ++j) {
    rows[j] = j < k ? row_of[(size_t)t * k + j] : -1;
    ws[j] = j < k ? w[(size_t)t * k + j] : 0.f;
  }
  for (int v = v0 + lane * 4; v < v1; v += 128) {
    float acc[4];
    if (nsplit == 1) {
      load_shared4(shared, (size_t)t * d + v, acc);
#pragma unroll
      for (int j = 0; j < 8; ++j)
        if (rows[j] >= 0) fma4(ws[j], y + (size_t)rows[j] * d + v, acc);
    } else {
      if (shared) sum_parts4(shared + (size_t)t * d + v, nsplit, shared_stride, acc);
      else acc[0] = acc[1] = acc[2] = acc[3] = 0.f;
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        if (rows[j] < 0) continue;
        float yv[4];
        sum_parts4(y + (size_t)rows[j] * d + v, nsplit, y_stride, yv);
#pragma unroll
        for (int i = 0; i < 4; ++i) acc[i] = fmaf(ws[j], yv[i], acc[i]);
      }
    }
    store4<TOut>(out + (size_t)t * d + v, acc);
  }
}

cudaError_t launch_combine(const moe_config& c, const float* y_perm, const int32_t* row_of,
                           const float* w, const float* shared_out, void* out, cudaStream_t s,
                           int nsplit, size_t y_stride, size_t shared_stride) {
  const int slice = combine_slice(c);
  const int blocks = ceil_div(c.T * ceil_div(c.d_model, slice) * 32, 256);
  if (c.out_dtype == MOE_DTYPE_F32)
    launch_pdl(combine_kernel<float>, blocks, 256, 0, s, y_perm, row_of, w, shared_out, (float*)out,
                                                 c.T, c.d_model, c.k, nsplit, y_stride,
                                                 shared_stride, slice);
  else
    launch_pdl(combine_kernel<__nv_bfloat16>, blocks, 256, 0, s, y_perm, row_of, w, shared_out,
                                                         (__nv_bfloat16*)out, c.T, c.d_model,
                                                         c.k, nsplit, y_stride, shared_stride,
                                                         slice);
  return cudaGetLastError();
}

// Expert-choice combine: token t sums the rows tok_rows[tok_ptr[t] .. tok_ptr[t+1]) (ascending
// expert order) with weights w_flat[row].
template <typename TOut>
__global__ void __launch_bounds__(256) combine_ec_kernel(const float* __restrict__ y,
                                                        const int32_t* __restrict__ tok_ptr,
                                                        const int32_t* __restrict__ tok_rows,
                                                        const float* __restrict__ w_flat,
                                                        const float* __restrict__ shared,
                                                        TOut* __restrict__ out, int Tn, int d) {
  pdl_prologue();
  const int lane = threadIdx.x & 31;
  const int gw = (blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const int slices = ceil_div(d, kCombineSlice);
  const int t = gw / slices;
  if (t >= Tn) return;
  const int v0 = (gw - t * slices) * kCombineSlice;
  const int v1 = min(d, v0 + kCombineSlice);
  const int b = tok_ptr[t], e_ = tok_ptr[t + 1];
  for (int v = v0 + lane * 4; v < v1; v += 128) {
    float acc[4];
    load_shared4(shared, (size_t)t * d + v, acc);
    for (int q = b; q < e_; ++q) {
      const int r = tok_rows[q];
      fma4(w_flat[r], y + (size_t)r * d + v, acc);
    }
    store4<TOut>(out + (size_t)t * d + v, acc);
  }
}

cudaError_t launch_combine_ec(const moe_config& c, const float* y_perm, const int32_t* tok_ptr,
                              const int32_t* tok_rows, const float* ec_w_flat,
                              const float* shared_out, void* out, cudaStream_t s) {
  const int blocks = ceil_div(c.T * ceil_div(c.d_model, kCombineSlice) * 32, 256);
  if (c.out_dtype == MOE_DTYPE_F32)
    launch_pdl(combine_ec_kernel<float>, blocks, 256, 0, s, y_perm, tok_ptr, tok_rows, ec_w_flat,
                                                    shared_out, (float*)out, c.T, c.d_model);
  else
    launch_pdl(combine_ec_kernel<__nv_bfloat16>, blocks, 256, 0, s, 
        y_perm, tok_ptr, tok_rows, ec_w_flat, shared_out, (__nv_bfloat16*)out, c.T, c.d_model);
  return cudaGetLastError();
}

}  // namespace moe
