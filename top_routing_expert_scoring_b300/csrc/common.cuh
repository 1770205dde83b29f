// Shared device helpers of the MoE layer kernels (sm_103a).
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "moe_b300.h"

namespace moe {

// Device-side bounded waits give up after this long and record MOE_ERR_TIMEOUT.
constexpr uint64_t kWaitLimitNs = 2000ull * 1000ull * 1000ull;   // 2 s

struct DevStatus {
  int32_t code;       // first error recorded (0 = none)
  int32_t detail;     // kernel-specific detail of the first error
};

__device__ __forceinline__ void record_error(DevStatus* st, int code, int detail) {
  if (st && atomicCAS(&st->code, 0, code) == 0) st->detail = detail;
}

__device__ __forceinline__ uint64_t globaltimer_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

__device__ __forceinline__ float to_f32(float v) { return v; }
__device__ __forceinline__ float to_f32(__nv_bfloat16 v) { return __bfloat162float(v); }

template <typename T> __device__ __forceinline__ T from_f32(float v);
template <> __device__ __forceinline__ float from_f32<float>(float v) { return v; }
template <> __device__ __forceinline__ __nv_bfloat16 from_f32<__nv_bfloat16>(float v) {
  return __float2bfloat16_rn(v);
}

// (key, index) ordering used by every Top-k: larger key first, equal keys -> lower index.
// -0.0 and +0.0 compare equal.
__device__ __forceinline__ bool ranks_before(float ka, int ia, float kb, int ib) {
  return ka > kb || (ka == kb && ia < ib);
}

__device__ __forceinline__ void warp_best(float& key, int& idx) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    float k2 = __shfl_xor_sync(0xffffffffu, key, o);
    int i2 = __shfl_xor_sync(0xffffffffu, idx, o);
    if (ranks_before(k2, i2, key, idx)) { key = k2; idx = i2; }
  }
}

__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
  return v;
}

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

__host__ __device__ __forceinline__ int ceil_div(int a, int b) { return (a + b - 1) / b; }

// Programmatic dependent launch.  Every kernel of the layer starts with this: it waits until the
// grids it depends on have completed and their writes are visible (a no-op when the kernel was
// launched without the programmatic-serialization attribute), then lets the next kernel's CTAs
// be scheduled, so its launch overlaps this kernel's run.  No global memory is touched before
// the wait, so neither read-after-write nor write-after-read across kernels can race.
__device__ __forceinline__ void pdl_prologue() {
  asm volatile("griddepcontrol.wait;" ::: "memory");
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// Rows of one M tile of the expert GEMMs.
constexpr int kTileM = 128;
// Tokens per dispatch block (one thread per token).
constexpr int kDispatchBlock = 256;

}  // namespace moe
