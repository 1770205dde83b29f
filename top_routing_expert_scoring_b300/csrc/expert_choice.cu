// Expert-choice routing ["MoE混合专家模型深度解析：路由机制与负载均衡" §2.2 Expert Choice]:
// transpose the logits and let every expert take the C = T*k/E tokens with the largest logit
// in its column (ties -> lower token index).  The weight of a chosen (token, expert) pair is
// the token's softmax probability of that expert.
//
//   K1  per expert (one CTA): radix select of the C-th largest key over the column, then the
//       chosen tokens in ascending token order (block prefix sums, no atomics in the order);
//   K2  per token: how many experts chose it;  K3: exclusive scan -> tok_ptr;
//   K4  per token: its rows e*C + i in ascending expert order (CSR used by the combine).
#include "common.cuh"
#include "kernels.h"

namespace moe {

constexpr int kEcThreads = 1024;

__device__ __forceinline__ uint32_t orderable(float f) {
  if (f == 0.0f) f = 0.0f;                 // -0.0 ranks equal to +0.0
  const uint32_t b = __float_as_uint(f);
  return (b & 0x80000000u) ? ~b : (b | 0x80000000u);
}

// Block-wide exclusive scan of one int per thread (kEcThreads threads); returns the total.
__device__ int block_exclusive_scan(int v, int* s_warp, int& total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  int x = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int y = __shfl_up_sync(0xffffffffu, x, o);
    if (lane >= o) x += y;
  }
  if (lane == 31) s_warp[warp] = x;
  __syncthreads();
  if (warp == 0) {
    int w = lane < (kEcThreads / 32) ? s_warp[lane] : 0;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int y = __shfl_up_sync(0xffffffffu, w, o);
      if (lane >= o) w += y;
    }
    s_warp[32 + lane] = w;   // inclusive prefix over warps
  }
  __syncthreads();
  const int before = (warp > 0 ? s_warp[32 + warp - 1] : 0) + x - v;
  total = s_warp[32 + kEcThreads / 32 - 1];
  __syncthreads();
  return before;
}

// Per-token softmax normaliser (max, sum of exp) used for the weights.
__global__ void __launch_bounds__(256) token_softmax_stats(const float* __restrict__ g, int T,
                                                          int E, float2* __restrict__ ms) {
  pdl_prologue();
  const int lane = threadIdx.x & 31;
  const int t = (blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  if (t >= T) return;
  float m = -INFINITY;
  for (int e = lane; e < E; e += 32) m = fmaxf(m, g[(size_t)t * E + e]);
  m = warp_max(m);
  float s = 0.f;
  for (int e = lane; e < E; e += 32) s += expf(g[(size_t)t * E + e] - m);
  s = warp_sum(s);
  if (lane == 0) ms[t] = make_float2(m, s);
}

__global__ void __launch_bounds__(kEcThreads) ec_select_kernel(const float* __restrict__ g, int T,
                                                              int E, int C,
                                                              const float2* __restrict__ ms,
                                                              int32_t* __restrict__ ec_tokens,
                                                              float* __restrict__ ec_w,
                                                              int32_t* __restrict__ posmap) {
  pdl_prologue();
  __shared__ int hist[256];
  __shared__ int s_warp[64];
  __shared__ int s_sel[2];
  const int e = blockIdx.x;
  const int tid = threadIdx.x;
  uint32_t prefix = 0, mask = 0;
  int remaining = C;
  for (int shift = 24; shift >= 0; shift -= 8) {
    for (int i = tid; i < 256; i += kEcThreads) hist[i] = 0;
    __syncthreads();
    for (int t = tid; t < T; t += kEcThreads) {
      const uint32_t u = orderable(g[(size_t)t * E + e]);
      if ((u & mask) == prefix) atomicAdd(&hist[(u >> shift) & 0xFFu], 1);
    }
    __syncthreads();
    if (tid == 0) {
      int acc = 0, b = 255;
      for (; b > 0; --b) {
        if (acc + hist[b] >= remaining) break;
        acc += hist[b];
      }
      s_sel[0] = b;
      s_sel[1] = remaining - acc;
    }
    __syncthreads();
    prefix |= static_cast<uint32_t>(s_sel[0]) << shift;
    mask |= 0xFFu << shift;
    remaining = s_sel[1];
    __syncthreads();
  }
  // prefix = key of the C-th largest; `remaining` tokens equal to it are taken (lowest index)
  int eq_before = 0, sel_before = 0;
  for (int base = 0; base < T; base += kEcThreads) {
    const int t = base + tid;
    uint32_t u = 0;
    if (t < T) u = orderable(g[(size_t)t * E + e]);
    const int is_eq = (t < T && u == prefix) ? 1 : 0;
    int eq_total;
    const int eq_rank = eq_before + block_exclusive_scan(is_eq, s_warp, eq_total);
    const int chosen = (t < T && (u > prefix || (is_eq && eq_rank < remaining))) ? 1 : 0;
    int sel_total;
    const int pos = sel_before + block_exclusive_scan(chosen, s_warp, sel_total);
    if (t < T) {
      posmap[(size_t)e * T + t] = chosen ? pos : -1;
      if (chosen) {
        ec_tokens[(size_t)e * C + pos] = t;
        const float2 st = ms[t];
        ec_w[(size_t)e * C + pos] = expf(g[(size_t)t * E + e] - st.x) / st.y;
      }
    }
    eq_before += eq_total;
    sel_before += sel_total;
  }
}

__global__ void __launch_bounds__(256) ec_count_kernel(const int32_t* __restrict__ posmap, int T,
                                                      int E, int32_t* __restrict__ cnt) {
  pdl_prologue();
  const int t = blockIdx.x * blockDim.x + threadIdx.x;
  if (t >= T) return;
  int c = 0;
  for (int e = 0; e < E; ++e) c += posmap[(size_t)e * T + t] >= 0;
  cnt[t] = c;
}

__global__ void __launch_bounds__(kEcThreads) ec_scan_kernel(const int32_t* __restrict__ cnt,
                                                            int T, int32_t* __restrict__ ptr) {
  pdl_prologue();
  __shared__ int s_warp[64];
  int run = 0;
  for (int base = 0; base < T; base += kEcThreads) {
    const int t = base + threadIdx.x;
    const int v = t < T ? cnt[t] : 0;
    int tot;
    const int ex = block_exclusive_scan(v, s_warp, tot);
    if (t < T) ptr[t] = run + ex;
    run += tot;
  }
  if (threadIdx.x == 0) ptr[T] = run;
}

__global__ void __launch_bounds__(256) ec_fill_kernel(const int32_t* __restrict__ posmap, int T,
                                                     int E, int C,
                                                     const int32_t* __restrict__ ptr,
                                                     int32_t* __restrict__ rows) {
  pdl_prologue();
  const int t = blockIdx.x * blockDim.x + threadIdx.x;
  if (t >= T) return;
  int o = ptr[t];
  for (int e = 0; e < E; ++e) {
    const int p = posmap[(size_t)e * T + t];
    if (p >= 0) rows[o++] = e * C + p;
  }
}

cudaError_t launch_expert_choice(const moe_config& c, const float* logits, int32_t* ec_tokens,
                                 float* ec_w, int32_t* tok_cnt, int32_t* tok_ptr,
                                 int32_t* tok_rows, int32_t* posmap, float2* ms, DevStatus* st,
                                 cudaStream_t s) {
  (void)st;
  const int C = (int)((long long)c.T * c.k / c.E);
  launch_pdl(token_softmax_stats, ceil_div(c.T * 32, 256), 256, 0, s, logits, c.T, c.E, ms);
  launch_pdl(ec_select_kernel, c.E, kEcThreads, 0, s, logits, c.T, c.E, C, ms, ec_tokens, ec_w, posmap);
  launch_pdl(ec_count_kernel, ceil_div(c.T, 256), 256, 0, s, posmap, c.T, c.E, tok_cnt);
  launch_pdl(ec_scan_kernel, 1, kEcThreads, 0, s, tok_cnt, c.T, tok_ptr);
  launch_pdl(ec_fill_kernel, ceil_div(c.T, 256), 256, 0, s, posmap, c.T, c.E, C, tok_ptr, tok_rows);
  return cudaGetLastError();
}

__global__ void ec_offsets_kernel(int E, int C, int32_t* offsets, int32_t* mtp) {
  pdl_prologue();
  for (int e = threadIdx.x; e <= E; e += blockDim.x) {
    offsets[e] = e * C;
    mtp[e] = e * ceil_div(C, kTileM);
  }
}

__global__ void __launch_bounds__(256) gather_by_token_kernel(const int32_t* __restrict__ tok,
                                                             int rows, int row_bytes,
                                                             const unsigned char* __restrict__ x,
                                                             unsigned char* __restrict__ xp) {
  pdl_prologue();
  const int lane = threadIdx.x & 31;
  const int warps = (gridDim.x * blockDim.x) >> 5;
  for (int r = (blockIdx.x * blockDim.x + threadIdx.x) >> 5; r < rows; r += warps) {
    const int t = tok[r];
    const uint4* src = reinterpret_cast<const uint4*>(x + (size_t)t * row_bytes);
    uint4* dst = reinterpret_cast<uint4*>(xp + (size_t)r * row_bytes);
    for (int i = lane; i < row_bytes / 16; i += 32) dst[i] = __ldg(src + i);
  }
}

cudaError_t launch_gather_ec(const moe_config& c, const int32_t* ec_tokens, const void* x,
                             void* x_perm, int32_t* offsets, int32_t* mtile_prefix,
                             cudaStream_t s) {
  const int C = (int)((long long)c.T * c.k / c.E);
  launch_pdl(ec_offsets_kernel, 1, 256, 0, s, c.E, C, offsets, mtile_prefix);
  const int rows = c.E * C;
  const int esz = c.dtype == MOE_DTYPE_F32 ? 4 : 2;
  int blocks = ceil_div(rows, 8);
  if (blocks > num_sms() * 8) blocks = num_sms() * 8;
  launch_pdl(gather_by_token_kernel, blocks, 256, 0, s, ec_tokens, rows, c.d_model * esz,
                                                (const unsigned char*)x, (unsigned char*)x_perm);
  return cudaGetLastError();
}

}  // namespace moe
