// Host-side launchers of the MoE layer kernels.  Each returns cudaSuccess or the launch error.
#pragma once

#include <mutex>
#include <set>
#include <utility>

#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include "common.cuh"

namespace moe {

// ---- router ----------------------------------------------------------------------------------
// part (nullable): router_split_bytes(c) of workspace for the K-sliced decode router.
cudaError_t launch_router_logits(const moe_config& c, const void* x, const void* w_gate,
                                 float* logits, cudaStream_t s, float* part = nullptr,
                                 DevStatus* st = nullptr);
// K-sliced router for decode batches of a wide router (E % 256 == 0, 16 < T <= 512); 0 = off.
constexpr int kRouterSplitMaxT = 512;
int router_split(const moe_config& c);
size_t router_split_bytes(const moe_config& c);
cudaError_t launch_router_split(const moe_config& c, const void* x, const void* w_gate,
                                float* part, float* logits, DevStatus* st, cudaStream_t s);
// Router logits on the tensor cores (bf16, E a multiple of 32): g = x W_gate^T in fp32.
cudaError_t launch_router_tc(const moe_config& c, const void* x, const void* w_gate,
                             float* logits, cudaStream_t s);
// With part_P/part_cnt/part_z the kernel also writes the load-balance partials, aux_rows(c)
// rows: one per fixed token set, or one per token for decode batches with E > 32 (route_cta);
// launch_aux_stats' first kernel writes the same values, and launch_aux_final reduces them.
cudaError_t launch_route_topk(const moe_config& c, const float* logits, const float* bias,
                              int32_t* idx, float* w, DevStatus* st, cudaStream_t s,
                              float* part_P = nullptr, int32_t* part_cnt = nullptr,
                              float* part_z = nullptr);
cudaError_t launch_aux_final(const moe_config& c, const float* part_P, const int32_t* part_cnt,
                             const float* part_z, int nblocks, float* f, float* P,
                             float* l_balance, float* z_loss, cudaStream_t s);
cudaError_t launch_aux_stats(const moe_config& c, const float* logits, const int32_t* idx,
                             const int32_t* ec_counts, float* part_P, int32_t* part_cnt,
                             float* part_z, int nblocks, float* f, float* P, float* l_balance,
                             float* z_loss, DevStatus* st, cudaStream_t s);
int aux_blocks(const moe_config& c);
bool route_cta(const moe_config& c);
int aux_rows(const moe_config& c);
// Prefill router with the routing in the GEMM epilogue (router_fused(c)): writes the logits,
// the selection, the weights and one statistics partial row per 128-token tile (aux_rows(c)).
bool router_fused(const moe_config& c);
cudaError_t launch_router_fused(const moe_config& c, const void* x, const void* w_gate,
                                const float* bias, float* logits, int32_t* idx, float* w,
                                float* part_P, int32_t* part_cnt, float* part_z, DevStatus* st,
                                cudaStream_t s);

// ---- dispatch --------------------------------------------------------------------------------
struct DispatchBufs {
  uint32_t* bitmap;     // [nblk][E][kDispatchBlock/32]
  int32_t* blk_base;    // [nblk][E]
  int32_t* counts;      // [E]
  int32_t* kept;        // [E]
  int32_t* offsets;     // [E+1]
  int32_t* mtile_prefix;// [E+1] prefix of ceil(kept/kTileM)
  int32_t* n_dropped;   // [1]
  int32_t* pos;         // [T,k]
  int32_t* row_of;      // [T,k]
  int32_t* perm;        // [T*k]
};
// The last step of the load-balance statistics (launch_aux_final's arithmetic and order), for
// the small dispatch to run in one extra CTA: partial rows in, f / P / l_balance / z_loss out
// (each nullable).
struct StatsFinal {
  const float* part_P;
  const int32_t* part_cnt;
  const float* part_z;
  int nrows;
  float* f;
  float* P;
  float* l_balance;
  float* z_loss;
};
// append_shared: also copy the T token rows after the kept rows (decode path's shared rows).
// fin (nullable): with T <= kDispatchBlock (one launch; dispatch_finalizes_stats) the launch
// also finishes the statistics, so no launch_aux_final is needed.
// x8 / sx (nullable, only where dispatch_quantizes): the rows go out as E4M3 codes with their
// per-row scales (the row quantiser's bytes) instead of bf16 copies into x_perm.
cudaError_t launch_dispatch(const moe_config& c, int capacity, const int32_t* idx,
                            const DispatchBufs& b, const void* x, void* x_perm, DevStatus* st,
                            cudaStream_t s, bool append_shared = false,
                            const StatsFinal* fin = nullptr, uint8_t* x8 = nullptr,
                            float* sx = nullptr);
bool dispatch_finalizes_stats(const moe_config& c);
bool dispatch_quantizes(const moe_config& c);

// x_perm[offsets[E] + t] = x[t] for t < T (rows of the shared experts on the decode path).
cudaError_t launch_append_rows(const moe_config& c, const int32_t* offsets, const void* x,
                               void* x_perm, cudaStream_t s);

// ---- expert FFN ------------------------------------------------------------------------------
// Grouped SwiGLU over expert-ordered rows.  offsets/mtile_prefix describe the E groups; with
// uniform_rows >= 0 there is one group of uniform_rows rows and the device arrays are unused.
struct GroupedFFN {
  const void* x;            // [rows, d]
  const int32_t* offsets;   // [E+1]
  const int32_t* mtile_prefix;  // [E+1]
  int uniform_rows;
  int E, d, F;
  int max_rows;             // rows allocated in x / h / y
  const void* w13;          // [E, 2F, d]
  const void* w2;           // [E, d, F]
  void* h;                  // [max_rows, F] scratch
  float* y;                 // [max_rows, d] float32, or bf16 when y_bf16
  int y_bf16;               // the down GEMM rounds y to bf16 (tensor-core kernels only)
  // Optional (single-CTA kernel only): gather the gate/up GEMM's A rows straight from the
  // token rows, row r = token gather_perm[r] / gather_k of gather_x [T, d]; x is then unused.
  const int32_t* gather_perm;
  int gather_k;             // k of the layer (pair index / k = token)
  const void* gather_x;
  // Optional (single-CTA kernel only): the down GEMM adds w[perm[r]] * y_r into the float32
  // output row of token perm[r] / k instead of storing y (y is then unused); the output must be
  // zeroed first.  Deterministic only with at most two addends per output element.
  float* scatter_out;
  const int32_t* scatter_perm;
  const float* scatter_w;
};
// true when launch_ffn_tc would run the CTA-pair kernel for g (which needs materialised rows)
bool ffn_uses_pair(const GroupedFFN& g);
// Tensor-core path.  Picks the CTA-pair kernel (cta_group::2, 256-row tiles) for ragged
// experts averaging >= 2048 rows (d % 256 == 0), else the single-CTA kernel (always for one
// group of rows, the shared experts); the environment variable MOE_B300_GEMM=single|pair|auto
// overrides the choice (pair falls back to single when d % 256 != 0).
cudaError_t launch_ffn_tc(const GroupedFFN& g, DevStatus* st, cudaStream_t s);
cudaError_t launch_ffn_tc2(const GroupedFFN& g, DevStatus* st, cudaStream_t s);
cudaError_t launch_ffn_simt(const GroupedFFN& g, bool f32, DevStatus* st, cudaStream_t s);

// Decode-sized batches: swap-AB tensor-core GEMMs (weights on M, tokens on N) over the routed
// experts plus the shared experts in one tile list.  x holds the expert-ordered token rows
// with the T shared rows appended after offsets[E]; h has ldo = max(F, F_shared).
struct DecodeFFN {
  const void* x;            // [max_rows, d] bf16
  const int32_t* offsets;   // [E+1]
  int E, T, d, F, F_shared;
  int max_rows;
  int np, np_shared;        // token rows per chunk (16, 32, 64, 128)
  const void* w13;
  const void* w2;
  const void* ws13;
  const void* ws2;
  void* h;                  // [max_rows, max(F, F_shared)] bf16
  float* y;                 // [ksplit2][max_rows, d] f32 partials (routed rows)
  float* shared_out;        // [ksplit2][T, d] f32 partials
  int ksplit1, ksplit2;     // K slices of the gate/up and down GEMMs (1 = no split)
  float* gu;                // [ksplit1][max_rows, 2 max(F, F_shared)] f32 when ksplit1 > 1
  size_t y_part_stride;     // elements between y partials (max_rows * d)
  size_t shared_part_stride;// elements between shared partials (T * d)
  // E4M3 operands: x, h, w13, w2, ws13, ws2 hold one-byte codes and these hold the per-row
  // scales; gu must be set: the gate/up GEMM writes its float32 partials there (with one K
  // slice, h = SiLU(g) * u itself as [max_rows, max(F, F_shared)]), then h is quantised per
  // row into h / hs
  int fp8;
  const float* s13;         // [E * 2F]
  const float* s2;          // [E * d]
  const float* ss13;        // [2 Fs]
  const float* ss2;         // [d]
  const float* sx;          // [max_rows] token-row scales of x
  float* hs;                // [max_rows] token-row scales of h (written)
};
cudaError_t launch_ffn_decode(const DecodeFFN& g, DevStatus* st, cudaStream_t s);
// Per-row E4M3 quantisation of bf16 rows (see moe_quantize_fp8); rows read from *nrows_base +
// nrows_extra when nrows_base is set (device-side count), else nrows_max.
cudaError_t launch_quantize_rows(const void* src, long long nrows_max, int cols,
                                 const int32_t* nrows_base, int nrows_extra, uint8_t* dst,
                                 float* scale, cudaStream_t s);

// ---- combine ---------------------------------------------------------------------------------
// y_perm and shared_out (or NULL) are float32 [*, d]; out follows c.out_dtype.  With nsplit > 1
// they hold nsplit K-slice partials, y_stride / shared_stride elements apart, summed in order.
cudaError_t launch_combine(const moe_config& c, const float* y_perm, const int32_t* row_of,
                           const float* w, const float* shared_out, void* out, cudaStream_t s,
                           int nsplit = 1, size_t y_stride = 0, size_t shared_stride = 0);
// The same with y_perm in bf16 (one slice), as the fused forward's down GEMM writes it.
cudaError_t launch_combine_bf16y(const moe_config& c, const void* y_perm, const int32_t* row_of,
                                 const float* w, const float* shared_out, void* out,
                                 cudaStream_t s);
// y_perm float32, or bf16 when y_bf16.
cudaError_t launch_combine_ec(const moe_config& c, const void* y_perm, bool y_bf16,
                              const int32_t* tok_ptr, const int32_t* tok_rows,
                              const float* ec_w_flat, const float* shared_out, void* out,
                              cudaStream_t s);

// ---- expert choice ---------------------------------------------------------------------------
// posmap [E][T]: position of token t in expert e's list or -1; ms [T]: softmax (max, sum).
cudaError_t launch_expert_choice(const moe_config& c, const float* logits, int32_t* ec_tokens,
                                 float* ec_w, int32_t* tok_cnt, int32_t* tok_ptr,
                                 int32_t* tok_rows, int32_t* posmap, float2* ms, DevStatus* st,
                                 cudaStream_t s);
cudaError_t launch_gather_ec(const moe_config& c, const int32_t* ec_tokens, const void* x,
                             void* x_perm, int32_t* offsets, int32_t* mtile_prefix,
                             cudaStream_t s);

// ---- failure-path self test ------------------------------------------------------------------
cudaError_t launch_timeout_probe(DevStatus* st, int limit_us, cudaStream_t s);

int num_sms();

// Launch with the programmatic-serialization attribute: the kernel may be scheduled while the
// previous kernel in the stream still runs; it waits for it in pdl_prologue() before touching
// global memory.
template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem,
                       cudaStream_t s, Args... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, args...);
}

// cudaFuncSetAttribute(MaxDynamicSharedMemorySize) once per (device, kernel): a process that
// drives several GPUs gets the attribute on each of them.
inline cudaError_t smem_attr_once(const void* func, int bytes) {
  static std::mutex mu;
  static std::set<std::pair<int, const void*>> done;
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  std::lock_guard<std::mutex> lock(mu);
  if (done.count({dev, func})) return cudaSuccess;
  e = cudaFuncSetAttribute(func, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
  if (e == cudaSuccess) done.insert({dev, func});
  return e;
}

}  // namespace moe
