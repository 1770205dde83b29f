// Weighted combine: out[t] = shared[t] + sum_j w[t,j] * y[row_of[t,j]]
// (y and shared in float32; out rounded once to bf16, or kept in float32)
//   ["MoE 路由数学" §2.1 Output = sum_{i in S} p~_i Expert_i(x), §2.2 shared experts;
//    "Systems for Mixture-of-Experts Models" §2.2 step 4 (add back in place)]
// fp32 accumulation in the fixed order j = 0..k-1 after the shared term; each token's row is
// written once (no atomics).  A dropped pair (row -1) adds nothing and the other weights keep
// their values.  Two kernels compute the same sums in the same order:
//   - combine_kernel (prefill): one warp per 512-column slice of a token, 16-byte loads;
//   - combine_rows_kernel (decode batches, or y in K-slice partials): one CTA per 128-column
//     chunk of a token with one warp per addend row, so that every load of the chunk is in
//     flight at once; warp 0 then adds the rows in the fixed order.
#include <cuda_bf16.h>

#include "common.cuh"
#include "kernels.h"

namespace moe {

// Columns per warp of the prefill kernel: a token's row is split over ceil(d / slice) warps,
// slice = 512 while that still gives >= 2048 warps, else 256 or 128, so that narrow rows still
// spread over the GPU (each lane handles 4 columns per 128-column step).
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

// Four consecutive values of y as float: 16 bytes of float32 or 8 bytes of bf16.
__device__ __forceinline__ float4 load4(const float* p) {
  return __ldg(reinterpret_cast<const float4*>(p));
}
__device__ __forceinline__ float4 load4(const __nv_bfloat16* p) {
  const uint2 v = __ldg(reinterpret_cast<const uint2*>(p));
  const float2 a = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&v.x));
  const float2 b = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&v.y));
  return make_float4(a.x, a.y, b.x, b.y);
}

__device__ __forceinline__ void load_shared4(const float* shared, size_t off, float* acc) {
  if (shared) {
    const float4 q = *reinterpret_cast<const float4*>(shared + off);
    acc[0] = q.x; acc[1] = q.y; acc[2] = q.z; acc[3] = q.w;
  } else {
    acc[0] = acc[1] = acc[2] = acc[3] = 0.f;
  }
}

// Sum of nsplit partials (stride apart), in slice order, of 4 consecutive values; the loads of
// up to eight slices are issued before the first add.
constexpr int kPartGroup = 8;
template <typename TY>
__device__ __forceinline__ float4 sum_parts4(const TY* p, int nsplit, size_t stride) {
  float4 v = make_float4(0.f, 0.f, 0.f, 0.f);
  for (int s0 = 0; s0 < nsplit; s0 += kPartGroup) {
    float4 q[kPartGroup];
#pragma unroll
    for (int i = 0; i < kPartGroup; ++i)
      if (s0 + i < nsplit) q[i] = load4(p + (s0 + i) * stride);
#pragma unroll
    for (int i = 0; i < kPartGroup; ++i) {
      if (s0 + i >= nsplit) break;
      if (s0 + i == 0) {
        v = q[0];
      } else {
        v.x += q[i].x; v.y += q[i].y; v.z += q[i].z; v.w += q[i].w;
      }
    }
  }
  return v;
}

// Eight consecutive bf16 values of y (16 bytes) into acc[0..7] with fused multiply-adds.
__device__ __forceinline__ void fma8(float wt, const __nv_bfloat16* y, float* acc) {
  const uint4 v = __ldg(reinterpret_cast<const uint4*>(y));
  const uint32_t u[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const float2 f = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&u[i]));
    acc[2 * i] = fmaf(wt, f.x, acc[2 * i]);
    acc[2 * i + 1] = fmaf(wt, f.y, acc[2 * i + 1]);
  }
}

template <typename TY>
__device__ __forceinline__ void fma4(float wt, const TY* y, float* acc) {
  const float4 q = load4(y);
  acc[0] = fmaf(wt, q.x, acc[0]);
  acc[1] = fmaf(wt, q.y, acc[1]);
  acc[2] = fmaf(wt, q.z, acc[2]);
  acc[3] = fmaf(wt, q.w, acc[3]);
}

// Token-choice combine, prefill: y (float32 or bf16) and shared (float32) hold one slice, out
// bf16 or float32.
template <typename TY, typename TOut>
__global__ void __launch_bounds__(256) combine_kernel(const TY* __restrict__ y,
                                                     const int32_t* __restrict__ row_of,
                                                     const float* __restrict__ w,
                                                     const float* __restrict__ shared,
                                                     TOut* __restrict__ out, int Tn, int d,
                                                     int k, int slice) {
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
  if constexpr (sizeof(TY) == 2) {
    // bf16 y: eight columns per lane and step, so every y load moves 16 bytes; all k row loads
    // of a step are issued before the first multiply-add (then added in the order j = 0..k-1)
    for (int v = v0 + lane * 8; v < v1; v += 256) {
      uint4 yv[8];
#pragma unroll
      for (int j = 0; j < 8; ++j)
        yv[j] = rows[j] >= 0 ? __ldg(reinterpret_cast<const uint4*>(y + (size_t)rows[j] * d + v))
                             : make_uint4(0u, 0u, 0u, 0u);
      float acc[8];
      load_shared4(shared, (size_t)t * d + v, acc);
      load_shared4(shared, (size_t)t * d + v + 4, acc + 4);
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        if (rows[j] < 0) continue;
        const uint32_t u[4] = {yv[j].x, yv[j].y, yv[j].z, yv[j].w};
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const float2 f = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&u[i]));
          acc[2 * i] = fmaf(ws[j], f.x, acc[2 * i]);
          acc[2 * i + 1] = fmaf(ws[j], f.y, acc[2 * i + 1]);
        }
      }
      store4<TOut>(out + (size_t)t * d + v, acc);
      store4<TOut>(out + (size_t)t * d + v + 4, acc + 4);
    }
  } else {
    for (int v = v0 + lane * 4; v < v1; v += 128) {
      float acc[4];
      load_shared4(shared, (size_t)t * d + v, acc);
#pragma unroll
      for (int j = 0; j < 8; ++j)
        if (rows[j] >= 0) fma4(ws[j], y + (size_t)rows[j] * d + v, acc);
      store4<TOut>(out + (size_t)t * d + v, acc);
    }
  }
}

// Token-choice combine, decode: CTA (t, chunk) has k + 1 warps; warp j < k sums the nsplit
// slices of y[row_of[t, j]] over the chunk's 128 columns, warp k those of shared[t] (when
// given), and warp 0 adds them: acc = shared (or 0), then acc = fma(w[t, j], row_j, acc) for
// j = 0..k-1, skipping dropped pairs.
template <typename TY, typename TOut>
__global__ void __launch_bounds__(288) combine_rows_kernel(const TY* __restrict__ y,
                                                          const int32_t* __restrict__ row_of,
                                                          const float* __restrict__ w,
                                                          const float* __restrict__ shared,
                                                          TOut* __restrict__ out, int d, int k,
                                                          int nsplit, size_t y_stride,
                                                          size_t shared_stride) {
  pdl_prologue();
  __shared__ float4 part[9][32];
  __shared__ float s_w[8];
  __shared__ int s_live[8];
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int chunks = ceil_div(d, 128);
  const int t = blockIdx.x / chunks;
  const int v = (blockIdx.x - t * chunks) * 128 + lane * 4;
  if (warp < k) {
    const int r = row_of[(size_t)t * k + warp];
    if (lane == 0) {
      s_live[warp] = r >= 0;
      s_w[warp] = w[(size_t)t * k + warp];
    }
    if (r >= 0 && v < d) part[warp][lane] = sum_parts4(y + (size_t)r * d + v, nsplit, y_stride);
  } else if (shared && v < d) {
    part[warp][lane] = sum_parts4(shared + (size_t)t * d + v, nsplit, shared_stride);
  }
  __syncthreads();
  if (warp != 0 || v >= d) return;
  float acc[4] = {0.f, 0.f, 0.f, 0.f};
  if (shared) {
    const float4 q = part[k][lane];
    acc[0] = q.x; acc[1] = q.y; acc[2] = q.z; acc[3] = q.w;
  }
  for (int j = 0; j < k; ++j) {
    if (!s_live[j]) continue;
    const float wt = s_w[j];
    const float4 q = part[j][lane];
    acc[0] = fmaf(wt, q.x, acc[0]);
    acc[1] = fmaf(wt, q.y, acc[1]);
    acc[2] = fmaf(wt, q.z, acc[2]);
    acc[3] = fmaf(wt, q.w, acc[3]);
  }
  store4<TOut>(out + (size_t)t * d + v, acc);
}

// y in K-slice partials, or too few (token, 128-column) slices for the prefill kernel to fill
// the GPU with warps, takes the row-parallel kernel.
constexpr int kCombineMinWarps = 2048;

template <typename TY, typename TOut>
cudaError_t launch_combine_t(const moe_config& c, const TY* y_perm, const int32_t* row_of,
                             const float* w, const float* shared_out, TOut* out, cudaStream_t s,
                             int nsplit, size_t y_stride, size_t shared_stride) {
  if (nsplit > 1 || (long long)c.T * ceil_div(c.d_model, 128) < kCombineMinWarps) {
    const int blocks = c.T * ceil_div(c.d_model, 128);
    launch_pdl(combine_rows_kernel<TY, TOut>, blocks, 32 * (c.k + 1), 0, s, y_perm, row_of, w,
               shared_out, out, c.d_model, c.k, nsplit, y_stride, shared_stride);
  } else {
    int slice = combine_slice(c);
    if (sizeof(TY) == 2 && slice < 256) slice = 256;      // a bf16 warp step covers 256 columns
    const int blocks = ceil_div(c.T * ceil_div(c.d_model, slice) * 32, 256);
    launch_pdl(combine_kernel<TY, TOut>, blocks, 256, 0, s, y_perm, row_of, w, shared_out, out,
               c.T, c.d_model, c.k, slice);
  }
  return cudaGetLastError();
}

template <typename TY>
cudaError_t launch_combine_y(const moe_config& c, const TY* y_perm, const int32_t* row_of,
                             const float* w, const float* shared_out, void* out, cudaStream_t s,
                             int nsplit, size_t y_stride, size_t shared_stride) {
  if (c.out_dtype == MOE_DTYPE_F32)
    return launch_combine_t(c, y_perm, row_of, w, shared_out, static_cast<float*>(out), s,
                            nsplit, y_stride, shared_stride);
  return launch_combine_t(c, y_perm, row_of, w, shared_out, static_cast<__nv_bfloat16*>(out), s,
                          nsplit, y_stride, shared_stride);
}

cudaError_t launch_combine(const moe_config& c, const float* y_perm, const int32_t* row_of,
                           const float* w, const float* shared_out, void* out, cudaStream_t s,
                           int nsplit, size_t y_stride, size_t shared_stride) {
  return launch_combine_y(c, y_perm, row_of, w, shared_out, out, s, nsplit, y_stride,
                          shared_stride);
}

cudaError_t launch_combine_bf16y(const moe_config& c, const void* y_perm, const int32_t* row_of,
                                 const float* w, const float* shared_out, void* out,
                                 cudaStream_t s) {
  return launch_combine_y(c, static_cast<const __nv_bfloat16*>(y_perm), row_of, w, shared_out,
                          out, s, 1, 0, 0);
}

// Expert-choice combine: token t sums the rows tok_rows[tok_ptr[t] .. tok_ptr[t+1]) (ascending
// expert order) with weights w_flat[row].
template <typename TY, typename TOut>
__global__ void __launch_bounds__(256) combine_ec_kernel(const TY* __restrict__ y,
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
  // the warp's whole slice is accumulated at once (each row's index and weight read once per
  // row, all of the row's loads in flight); per element: shared first, then the rows in order
  constexpr int VEC = sizeof(TY) == 2 ? 8 : 4;
  constexpr int NSTEP = kCombineSlice / (32 * VEC);
  float acc[NSTEP][VEC];
#pragma unroll
  for (int st = 0; st < NSTEP; ++st) {
    const int v = v0 + st * 32 * VEC + lane * VEC;
#pragma unroll
    for (int i = 0; i < VEC; i += 4) {
      if (v < v1) load_shared4(shared, (size_t)t * d + v + i, &acc[st][i]);
      else acc[st][i] = acc[st][i + 1] = acc[st][i + 2] = acc[st][i + 3] = 0.f;
    }
  }
  for (int q = b; q < e_; ++q) {
    const int r = tok_rows[q];
    const float wt = w_flat[r];
    const TY* yr = y + (size_t)r * d;
#pragma unroll
    for (int st = 0; st < NSTEP; ++st) {
      const int v = v0 + st * 32 * VEC + lane * VEC;
      if (v >= v1) continue;
      if constexpr (VEC == 8) fma8(wt, yr + v, acc[st]);
      else fma4(wt, yr + v, acc[st]);
    }
  }
#pragma unroll
  for (int st = 0; st < NSTEP; ++st) {
    const int v = v0 + st * 32 * VEC + lane * VEC;
    if (v >= v1) continue;
#pragma unroll
    for (int i = 0; i < VEC; i += 4) store4<TOut>(out + (size_t)t * d + v + i, &acc[st][i]);
  }
}

template <typename TY>
cudaError_t launch_combine_ec_y(const moe_config& c, const TY* y_perm, const int32_t* tok_ptr,
                                const int32_t* tok_rows, const float* ec_w_flat,
                                const float* shared_out, void* out, cudaStream_t s) {
  const int blocks = ceil_div(c.T * ceil_div(c.d_model, kCombineSlice) * 32, 256);
  if (c.out_dtype == MOE_DTYPE_F32)
    launch_pdl(combine_ec_kernel<TY, float>, blocks, 256, 0, s, y_perm, tok_ptr, tok_rows,
               ec_w_flat, shared_out, (float*)out, c.T, c.d_model);
  else
    launch_pdl(combine_ec_kernel<TY, __nv_bfloat16>, blocks, 256, 0, s, y_perm, tok_ptr,
               tok_rows, ec_w_flat, shared_out, (__nv_bfloat16*)out, c.T, c.d_model);
  return cudaGetLastError();
}

cudaError_t launch_combine_ec(const moe_config& c, const void* y_perm, bool y_bf16,
                              const int32_t* tok_ptr, const int32_t* tok_rows,
                              const float* ec_w_flat, const float* shared_out, void* out,
                              cudaStream_t s) {
  if (y_bf16)
    return launch_combine_ec_y(c, static_cast<const __nv_bfloat16*>(y_perm), tok_ptr, tok_rows,
                               ec_w_flat, shared_out, out, s);
  return launch_combine_ec_y(c, static_cast<const float*>(y_perm), tok_ptr, tok_rows, ec_w_flat,
                             shared_out, out, s);
}

}  // namespace moe
