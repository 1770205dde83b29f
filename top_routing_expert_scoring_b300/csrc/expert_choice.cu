// Expert-choice routing ["MoE混合专家模型深度解析：路由机制与负载均衡" §2.2 Expert Choice]:
// transpose the logits and let every expert take the C = T*k/E tokens with the largest logit
// in its column (ties -> lower token index).  The weight of a chosen (token, expert) pair is
// the token's softmax probability of that expert.
//
//   K1  per expert (one CTA): radix select of the C-th largest key over the column (kept in
//       shared memory), then the chosen tokens in ascending token order (block prefix sums,
//       no atomics in the order);
//   K2  per token: how many experts chose it;  K3: exclusive scan -> tok_ptr;
//   K4  per token: its rows e*C + i in ascending expert order (CSR used by the combine).
#include "common.cuh"
#include "kernels.h"

namespace moe {

constexpr int kEcThreads = 1024;
constexpr int kEcSmemT = 40960;        // tokens whose keys the selection keeps in shared memory

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

// The bin of the 256-bin histogram `hist` that holds the `remaining`-th largest key, counting
// from the top bin, and how many keys of that bin are still to be taken.  All threads call it;
// the first 256 threads scan the bins from the top (a suffix sum) in parallel.
__device__ __forceinline__ void ec_pick_bin(const int* hist, int remaining, int* s_scan,
                                            int* s_sel) {
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  int v = 0, incl = 0;
  if (tid < 256) {
    v = hist[255 - tid];                   // thread j holds bin 255 - j
    incl = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int y = __shfl_up_sync(0xffffffffu, incl, o);
      if (lane >= o) incl += y;
    }
    if (lane == 31) s_scan[warp] = incl;
  }
  __syncthreads();
  if (tid < 256) {
    int before = 0;
    for (int w = 0; w < warp; ++w) before += s_scan[w];
    incl += before;
    // keys in bins above this one: incl - v; the wanted key lies here when they fall short
    // of `remaining` and this bin reaches it (the lowest bin takes whatever is left)
    const int above = incl - v;
    if (above < remaining && (incl >= remaining || tid == 255)) {
      s_sel[0] = 255 - tid;
      s_sel[1] = remaining - above;
    }
  }
  __syncthreads();
}

// Expert choice, one CTA per expert: the C largest keys of the expert's logit column (ties to
// the lower token index) by a 4-pass radix select on the orderable bits, then the chosen
// tokens in ascending token order.  With T <= kEcSmemT the column is read from global memory
// once and kept in shared memory as keys; the histograms aggregate equal bins within a warp
// (one shared atomic per distinct bin), since the top byte of the keys falls into few bins.
template <bool CACHED>
__global__ void __launch_bounds__(kEcThreads) ec_select_kernel(const float* __restrict__ g, int T,
                                                              int E, int C,
                                                              const float2* __restrict__ ms,
                                                              int32_t* __restrict__ ec_tokens,
                                                              float* __restrict__ ec_w,
                                                              int32_t* __restrict__ posmap) {
  pdl_prologue();
  extern __shared__ uint32_t s_keys[];     // [T] when CACHED
  __shared__ int hist[256];
  __shared__ int s_warp[64];
  __shared__ int s_sel[2];
  const int e = blockIdx.x;
  const int tid = threadIdx.x, lane = tid & 31;
  auto key_of = [&](int t) -> uint32_t {
    return CACHED ? s_keys[t] : orderable(g[(size_t)t * E + e]);
  };
  if (CACHED) {
    for (int t = tid; t < T; t += kEcThreads) s_keys[t] = orderable(g[(size_t)t * E + e]);
  }
  uint32_t prefix = 0, mask = 0;
  int remaining = C;
  for (int shift = 24; shift >= 0; shift -= 8) {
    for (int i = tid; i < 256; i += kEcThreads) hist[i] = 0;
    __syncthreads();
    for (int base = 0; base < T; base += kEcThreads) {
      const int t = base + tid;
      int bin = -1;
      if (t < T) {
        const uint32_t u = key_of(t);
        if ((u & mask) == prefix) bin = static_cast<int>((u >> shift) & 0xFFu);
      }
      const uint32_t same = __match_any_sync(0xffffffffu, bin);
      if (bin >= 0 && lane == __ffs(same) - 1) atomicAdd(&hist[bin], __popc(same));
    }
    __syncthreads();
    ec_pick_bin(hist, remaining, s_warp, s_sel);
    prefix |= static_cast<uint32_t>(s_sel[0]) << shift;
    mask |= 0xFFu << shift;
    remaining = s_sel[1];
    __syncthreads();
  }
  // prefix = key of the C-th largest; `remaining` tokens equal to it are taken (lowest index).
  // Warp w owns the contiguous token range [w * per, (w + 1) * per): it counts its keys above
  // and equal to the prefix, one scan over the 32 warps places each warp's equal keys and
  // chosen tokens, and each warp then writes its range in token order (ballot prefixes), so
  // the chosen set and its order are those of a sequential walk over the tokens.
  constexpr int kWarps = kEcThreads / 32;
  __shared__ int s_eqb[kWarps], s_selb[kWarps];
  const int warp = tid >> 5;
  const int per = (T + kWarps - 1) / kWarps;
  const int t_lo = warp * per, t_hi = min(T, t_lo + per);
  int n_gt = 0, n_eq = 0;
  for (int b = t_lo; b < t_hi; b += 32) {
    const int t = b + lane;
    const uint32_t u = t < t_hi ? key_of(t) : 0u;
    n_gt += __popc(__ballot_sync(0xffffffffu, t < t_hi && u > prefix));
    n_eq += __popc(__ballot_sync(0xffffffffu, t < t_hi && u == prefix));
  }
  if (lane == 0) {
    s_eqb[warp] = n_eq;
    s_selb[warp] = n_gt;
  }
  __syncthreads();
  if (warp == 0) {
    // equal keys before each warp, then the chosen count of each warp, both scanned in order
    const int eq_w = s_eqb[lane];
    int incl = eq_w;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int y = __shfl_up_sync(0xffffffffu, incl, o);
      if (lane >= o) incl += y;
    }
    const int eq_before = incl - eq_w;
    const int take_eq = max(0, min(eq_w, remaining - eq_before));
    const int sel_w = s_selb[lane] + take_eq;
    int sincl = sel_w;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int y = __shfl_up_sync(0xffffffffu, sincl, o);
      if (lane >= o) sincl += y;
    }
    s_eqb[lane] = eq_before;
    s_selb[lane] = sincl - sel_w;
  }
  __syncthreads();
  int eq_seen = s_eqb[warp], pos_base = s_selb[warp];
  const uint32_t below = (1u << lane) - 1u;
  for (int b = t_lo; b < t_hi; b += 32) {
    const int t = b + lane;
    const bool live = t < t_hi;
    const uint32_t u = live ? key_of(t) : 0u;
    const bool is_eq = live && u == prefix;
    const uint32_t eq_mask = __ballot_sync(0xffffffffu, is_eq);
    const int eq_rank = eq_seen + __popc(eq_mask & below);
    const bool chosen = live && (u > prefix || (is_eq && eq_rank < remaining));
    const uint32_t ch_mask = __ballot_sync(0xffffffffu, chosen);
    const int pos = pos_base + __popc(ch_mask & below);
    if (live) {
      posmap[(size_t)e * T + t] = chosen ? pos : -1;
      if (chosen) {
        ec_tokens[(size_t)e * C + pos] = t;
        const float2 st = ms[t];
        ec_w[(size_t)e * C + pos] = expf(g[(size_t)t * E + e] - st.x) / st.y;
      }
    }
    eq_seen += __popc(eq_mask);
    pos_base += __popc(ch_mask);
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
  // each thread takes kPer consecutive tokens per round: their counts are loaded together,
  // summed, and the block scan of the sums places each thread's run
  constexpr int kPer = 8;
  int run = 0;
  for (int base = 0; base < T; base += kEcThreads * kPer) {
    const int t0 = base + threadIdx.x * kPer;
    int v[kPer];
    int sum = 0;
#pragma unroll
    for (int j = 0; j < kPer; ++j) {
      v[j] = t0 + j < T ? cnt[t0 + j] : 0;
      sum += v[j];
    }
    int tot;
    int ex = run + block_exclusive_scan(sum, s_warp, tot);
#pragma unroll
    for (int j = 0; j < kPer; ++j) {
      if (t0 + j < T) ptr[t0 + j] = ex;
      ex += v[j];
    }
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
  if (c.T <= kEcSmemT) {
    const int smem = c.T * 4;
    cudaError_t e = smem_attr_once(reinterpret_cast<const void*>(ec_select_kernel<true>),
                                   kEcSmemT * 4);
    if (e != cudaSuccess) return e;
    launch_pdl(ec_select_kernel<true>, c.E, kEcThreads, smem, s, logits, c.T, c.E, C, ms,
               ec_tokens, ec_w, posmap);
  } else {
    launch_pdl(ec_select_kernel<false>, c.E, kEcThreads, 0, s, logits, c.T, c.E, C, ms,
               ec_tokens, ec_w, posmap);
  }
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
