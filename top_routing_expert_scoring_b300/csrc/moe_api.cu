// C ABI of the MoE layer forward: argument checks, workspace layout and the launch sequence.
// Every entry point validates on the host, enqueues on the caller's stream and returns; the
// library allocates no memory and never synchronises (except moe_sync_status, which exists
// to).  The fused forward forks its shared experts onto a side stream and joins them back.
#include <cuda_runtime.h>

#include <algorithm>
#include <cmath>
#include <cstdlib>
#include <cstring>

#include "common.cuh"
#include "kernels.h"

namespace moe {

int num_sms() {
  static int n = 0;
  if (n == 0) {
    int dev = 0;
    cudaGetDevice(&dev);
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n < 1)
      n = 148;
  }
  return n;
}

namespace {

constexpr size_t kAlign = 256;

size_t align_up(size_t v) { return (v + kAlign - 1) & ~(kAlign - 1); }

// Workspace layout.  Offsets are relative to the 256-byte aligned workspace base.
struct Layout {
  size_t status, logits, idx, w, bitmap, blk_base, counts, kept, offsets, mtp, n_dropped, pos,
      row_of, perm, part_P, part_cnt, part_z, f, P, lb, z, x_perm, h, y_perm, shared_out,
      ec_tokens, ec_w, tok_cnt, tok_ptr, tok_rows, posmap, tokstat, dec_gu, dec_y, dec_sh,
      router_part, total;
};

// K-split of the decode GEMMs: up to kMaxSplit slices, partial buffers only for small batches.
constexpr int kMaxSplit = 8;
constexpr long long kSplitRows = 1024;

int rows_max(const moe_config& c) { return c.T * c.k; }

// Decode regime: bf16 with few rows per expert (<= 64 on average); the swap-AB kernel streams
// each touched expert's weights once with the tokens on the MMA's N side.
// The environment variable MOE_B300_PATH=prefill|decode|auto overrides the choice (decode
// still needs bf16, token choice and d % 256 == 0).
bool decode_regime(const moe_config& c) {
  if (c.dtype != MOE_DTYPE_BF16 || c.routing != MOE_ROUTE_TOKEN_CHOICE || c.d_model % 256 != 0)
    return false;
  const char* env = getenv("MOE_B300_PATH");
  if (env && strcmp(env, "decode") == 0) return true;
  if (env && strcmp(env, "prefill") == 0) return false;
  return (long long)c.T * c.k <= 64ll * c.E;
}

// Prefill gate/up GEMM reading its A rows straight from x (no materialised x_perm), on the
// single-CTA kernel.  Off by default: the warp-wide cp.async gather costs the GEMM more than
// the separate row copy it saves (measured on Mixtral-, DeepSeekMoE- and V3-shaped layers).
// MOE_B300_GATHER=fused turns it on.
bool gather_fused(const moe_config& c, bool dec) {
  if (dec || c.dtype != MOE_DTYPE_BF16 || c.routing != MOE_ROUTE_TOKEN_CHOICE) return false;
  const char* env0 = getenv("MOE_B300_GATHER");
  if (!env0 || strcmp(env0, "fused") != 0) return false;
  GroupedFFN probe{};
  probe.uniform_rows = -1;
  probe.E = c.E;
  probe.d = c.d_model;
  probe.F = c.d_ff;
  probe.max_rows = rows_max(c);
  return !ffn_uses_pair(probe);
}

// Prefill down GEMM adding w * y straight into the float32 layer output (no y rows, no combine
// pass).  Deterministic because a token receives at most two addends (0 + a = a and a + b =
// b + a exactly), so only for k <= 2 without shared experts; single-CTA kernel only.  The
// environment variable MOE_B300_COMBINE=separate turns it off.
bool combine_fused(const moe_config& c, bool dec) {
  if (dec || c.dtype != MOE_DTYPE_BF16 || c.routing != MOE_ROUTE_TOKEN_CHOICE) return false;
  if (c.k > 2 || c.d_ff_shared > 0 || c.out_dtype != MOE_DTYPE_F32) return false;
  GroupedFFN probe{};
  probe.uniform_rows = -1;
  probe.E = c.E;
  probe.d = c.d_model;
  probe.F = c.d_ff;
  probe.max_rows = rows_max(c);
  if (ffn_uses_pair(probe)) return false;
  const char* env = getenv("MOE_B300_COMBINE");
  return !(env && strcmp(env, "separate") == 0);
}

// Prefill shared experts on a side stream, forked before the router and joined before the
// routed GEMMs: the shared experts' two GEMMs read only x, so they run while the router (one
// CTA per 128 tokens), the dispatch and the row gather hold few SMs or no tensor pipes.  Their
// h rows sit after the routed rows' h in the workspace, so the two never share bytes.
// MOE_B300_SHARED=serial runs them after the routed GEMMs on the caller's stream instead.
bool shared_overlap(const moe_config& c, bool dec) {
  if (dec || c.d_ff_shared <= 0 || c.dtype != MOE_DTYPE_BF16) return false;
  const char* env = getenv("MOE_B300_SHARED");
  return !(env && strcmp(env, "serial") == 0);
}

// The side stream and its fork and join events: one set per device and host thread, created on
// first use and never destroyed (no CUDA call runs from a destructor at thread or process
// exit, when the runtime may already be gone).  They are not created while the caller's
// stream is being captured into a graph (creation could end a global-mode capture); the call
// then runs the shared experts on the caller's stream (same kernels, same results).
struct SideStream {
  cudaStream_t s = nullptr;
  cudaEvent_t fork = nullptr, join = nullptr;
};

SideStream* side_stream(cudaStream_t caller) {
  constexpr int kMaxDevices = 64;
  thread_local SideStream per_dev[kMaxDevices];
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
  SideStream& ss = per_dev[dev];
  if (!ss.s) {
    // a failed query or creation leaves no error behind for the launches that follow
    auto give_up = []() -> SideStream* {
      (void)cudaGetLastError();
      return nullptr;
    };
    cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
    if (cudaStreamIsCapturing(caller, &cs) != cudaSuccess || cs != cudaStreamCaptureStatusNone)
      return give_up();
    cudaStream_t st = nullptr;
    cudaEvent_t a = nullptr, b = nullptr;
    if (cudaStreamCreateWithFlags(&st, cudaStreamNonBlocking) != cudaSuccess) return give_up();
    if (cudaEventCreateWithFlags(&a, cudaEventDisableTiming) != cudaSuccess ||
        cudaEventCreateWithFlags(&b, cudaEventDisableTiming) != cudaSuccess) {
      if (a) cudaEventDestroy(a);
      cudaStreamDestroy(st);
      return give_up();
    }
    ss.fork = a;
    ss.join = b;
    ss.s = st;
  }
  return &ss;
}

bool decode_split_possible(const moe_config& c) {
  return decode_regime(c) && (long long)c.T * c.k <= kSplitRows;
}

// K slices of a decode GEMM.  The expected experts touched by T tokens, E(1 - (1 - k/E)^T)
// ("Systems for MoE Models" §1.4), plus the shared experts, give the tile count; each slice
// count ks is costed in units of one K block streamed by every SM at the HBM rate.  The
// kernel streams weights, so a round of n < SMs active CTAs (the last, partial one) runs each
// CTA faster than a full round, up to kSmRate times an SM's share of the HBM rate (one CTA's
// ring of TMA loads in flight sets that ceiling; fitted to Mixtral-shaped down GEMMs, whose
// one unsplit round of 32 CTAs ran ~1.5x an SM's share):
//   full rounds x blocks per tile + blocks per tile / min(kSmRate, SMs / n)   the weight stream
//   + 1                                                                       the ring's fill
//   + (ks - 1) * 2 * partial_bytes / (SMs * 32 KB)                            extra partials
// and the cheapest (fewest slices on ties) is taken, at most kMaxSplit.  A round that already
// holds most of the SMs thus gains nothing from slicing.  With 8 or more rounds unsplit the
// tail is a small share of the stream: one slice.  MOE_B300_SPLITMODEL=waves restores the
// earlier cost, rounds x (blocks per tile + 1), which charges every round as a full one.
constexpr double kSmRate = 1.5;

int split_by_waves(const moe_config& c, int tiles_per_entry, int kblocks, double partial_bytes) {
  const double touched = c.E * (1.0 - std::pow(1.0 - (double)c.k / c.E, (double)c.T));
  const double entries = touched + (c.d_ff_shared > 0 ? 1.0 : 0.0);
  const long long tiles = (long long)std::ceil(entries * tiles_per_entry);
  const int sms = num_sms();
  if (tiles >= 8ll * sms) return 1;
  const char* env = getenv("MOE_B300_SPLITMODEL");
  const bool waves_model = env && strcmp(env, "waves") == 0;
  const double unit = (double)sms * 32768.0;     // one 256-row weight K block on every SM
  int best = 1;
  double best_cost = 1e300;
  for (int ks = 1; ks <= kMaxSplit && ks <= kblocks; ++ks) {
    const long long n = tiles * ks;
    const double kb = (double)((kblocks + ks - 1) / ks);
    double stream;
    if (waves_model) {
      stream = (double)((n + sms - 1) / sms) * (kb + 1.0);
    } else {
      const long long rest = n % sms;
      stream = (double)(n / sms) * kb + 1.0;
      if (rest) stream += kb / std::min(kSmRate, (double)sms / (double)rest);
    }
    const double cost = stream + (ks - 1) * 2.0 * partial_bytes / unit;
    if (cost < best_cost - 1e-9) {
      best_cost = cost;
      best = ks;
    }
  }
  return best;
}

// K slices of the bf16 decode gate/up (which = 1) or down (which = 2) GEMM.  The environment
// variables MOE_B300_KSPLIT1 / MOE_B300_KSPLIT2 fix the count (clamped to 1..kMaxSplit and the
// K blocks), for measuring the cost model against other choices.
int decode_split(const moe_config& c, int tiles_per_entry, int kblocks, double partial_bytes,
                 int which) {
  if (!decode_split_possible(c)) return 1;
  const char* env = getenv(which == 1 ? "MOE_B300_KSPLIT1" : "MOE_B300_KSPLIT2");
  if (env && *env) {
    int ks = atoi(env);
    if (ks > kMaxSplit) ks = kMaxSplit;
    if (ks > kblocks) ks = kblocks;
    return ks < 1 ? 1 : ks;
  }
  return split_by_waves(c, tiles_per_entry, kblocks, partial_bytes);
}

int pow2_clamp(long long v, int lo, int hi) {
  int p = lo;
  while (p < v && p < hi) p <<= 1;
  return p;
}

Layout layout(const moe_config& c) {
  Layout L{};
  size_t o = 0;
  auto take = [&](size_t bytes) {
    size_t at = o;
    o = align_up(o + (bytes ? bytes : 1));
    return at;
  };
  const size_t T = c.T, E = c.E, k = c.k, d = c.d_model, F = c.d_ff, Fs = c.d_ff_shared;
  const size_t esz = c.dtype == MOE_DTYPE_F32 ? 4 : 2;
  const size_t nblk = (T + kDispatchBlock - 1) / kDispatchBlock;
  const size_t naux = aux_rows(c);
  const size_t R = rows_max(c);
  L.status = take(sizeof(DevStatus));
  L.logits = take(T * E * 4);
  L.idx = take(T * k * 4);
  L.w = take(T * k * 4);
  L.bitmap = take(nblk * E * (kDispatchBlock / 32) * 4);
  L.blk_base = take(nblk * E * 4);
  L.counts = take(E * 4);
  L.kept = take(E * 4);
  L.offsets = take((E + 1) * 4);
  L.mtp = take((E + 1) * 4);
  L.n_dropped = take(4);
  L.pos = take(T * k * 4);
  L.row_of = take(T * k * 4);
  L.perm = take(T * k * 4);
  L.part_P = take(naux * E * 4);
  L.part_cnt = take(naux * E * 4);
  L.part_z = take(naux * 4);
  L.f = take(E * 4);
  L.P = take(E * 4);
  L.lb = take(4);
  L.z = take(4);
  // the decode path appends the T shared-expert rows after the routed rows
  L.x_perm = take((R + T) * d * esz);
  const size_t hrows = R + T;
  const size_t hcols = F > Fs ? F : Fs;
  L.h = take(hrows * hcols * esz);
  L.y_perm = take(R * d * 4);          // float32 expert outputs
  L.shared_out = take(Fs ? T * d * 4 : 0);   // float32 for both activation types
  if (c.routing == MOE_ROUTE_EXPERT_CHOICE) {
    const size_t C = (T * k) / E;
    L.ec_tokens = take(E * C * 4);
    L.ec_w = take(E * C * 4);
    L.tok_cnt = take(T * 4);
    L.tok_ptr = take((T + 1) * 4);
    L.tok_rows = take(E * C * 4);
    L.posmap = take(E * T * 4);
    L.tokstat = take(T * 8);
  }
  if (decode_split_possible(c)) {
    const size_t Fmax = F > Fs ? F : Fs;
    L.dec_gu = take((size_t)kMaxSplit * (R + T) * 2 * Fmax * 4);
    L.dec_y = take((size_t)kMaxSplit * R * d * 4);
    L.dec_sh = take((size_t)kMaxSplit * T * d * 4);
  }
  L.router_part = take(router_split_bytes(c));
  L.total = o;
  return L;
}

template <typename P>
P* at(void* ws, size_t off) {
  return reinterpret_cast<P*>(static_cast<unsigned char*>(ws) + off);
}

int check_ws(void* ws) {
  if (!ws) return MOE_ERR_WORKSPACE;
  if (reinterpret_cast<uintptr_t>(ws) % kAlign) return MOE_ERR_WORKSPACE;
  return MOE_OK;
}

int cuda_status(cudaError_t e) { return e == cudaSuccess ? MOE_OK : MOE_ERR_CUDA; }

int capacity_of(const moe_config& c) {
  if (!(c.capacity_factor > 0.0f)) return c.T * c.k;
  const double C = std::ceil(static_cast<double>(c.capacity_factor) * c.k * c.T / c.E);
  const double lim = static_cast<double>(c.T) * c.k;
  return static_cast<int>(C < lim ? C : lim);
}

bool bf16(const moe_config& c) { return c.dtype == MOE_DTYPE_BF16; }

}  // namespace
}  // namespace moe

using namespace moe;

extern "C" {

const char* moe_status_string(int status) {
  switch (status) {
    case MOE_OK: return "ok";
    case MOE_ERR_ARG: return "invalid argument (NULL pointer, bad enum or bad index)";
    case MOE_ERR_SHAPE: return "unsupported or inconsistent sizes";
    case MOE_ERR_UNSUPPORTED: return "request not implemented by this library";
    case MOE_ERR_WORKSPACE: return "workspace missing, too small or not 256-byte aligned";
    case MOE_ERR_CUDA: return "CUDA runtime error";
    case MOE_ERR_TIMEOUT: return "a bounded device-side wait ran out";
    default: return "unknown status";
  }
}

const char* moe_version(void) { return "moe_b300 1.0 sm_103a"; }

int moe_check_config(const moe_config* c) {
  if (!c) return MOE_ERR_ARG;
  if (c->score != MOE_SCORE_SOFTMAX && c->score != MOE_SCORE_SIGMOID) return MOE_ERR_ARG;
  if (c->routing != MOE_ROUTE_TOKEN_CHOICE && c->routing != MOE_ROUTE_EXPERT_CHOICE)
    return MOE_ERR_ARG;
  if (c->dtype != MOE_DTYPE_BF16 && c->dtype != MOE_DTYPE_F32) return MOE_ERR_ARG;
  if (c->out_dtype != MOE_DTYPE_BF16 && c->out_dtype != MOE_DTYPE_F32) return MOE_ERR_ARG;
  if (c->renormalize != 0 && c->renormalize != 1) return MOE_ERR_ARG;
  if (!std::isfinite(c->route_scale) || !std::isfinite(c->capacity_factor)) return MOE_ERR_ARG;
  if (c->T < 1 || c->T > (1 << 20)) return MOE_ERR_SHAPE;
  if (c->E < 1 || c->E > 256) return MOE_ERR_SHAPE;
  if (c->k < 1 || c->k > 8 || c->k > c->E) return MOE_ERR_SHAPE;
  if (c->d_model < 1 || c->d_ff < 1 || c->d_ff_shared < 0) return MOE_ERR_SHAPE;
  if ((long long)c->T * c->k * (c->d_model > c->d_ff ? c->d_model : c->d_ff) > (1ll << 40))
    return MOE_ERR_SHAPE;
  if (c->n_groups < 1 || c->n_groups > 32 || c->E % c->n_groups) return MOE_ERR_SHAPE;
  if (c->topk_groups < 1 || c->topk_groups > c->n_groups) return MOE_ERR_SHAPE;
  if (c->topk_groups < c->n_groups) {
    if (c->score != MOE_SCORE_SIGMOID) return MOE_ERR_UNSUPPORTED;
    if (c->E / c->n_groups < 2) return MOE_ERR_SHAPE;   // group score = sum of the top two
    if (c->topk_groups * (c->E / c->n_groups) < c->k) return MOE_ERR_SHAPE;
  }
  if (c->dtype == MOE_DTYPE_BF16) {
    if (c->d_model % 128 || c->d_ff % 128 || c->d_ff_shared % 128) return MOE_ERR_SHAPE;
  } else {
    if (c->d_model % 4) return MOE_ERR_SHAPE;
  }
  if (c->routing == MOE_ROUTE_EXPERT_CHOICE) {
    if (c->score != MOE_SCORE_SOFTMAX) return MOE_ERR_UNSUPPORTED;
    const long long C = (long long)c->T * c->k / c->E;
    if (C < 1 || C > c->T) return MOE_ERR_SHAPE;
  }
  return MOE_OK;
}

int moe_capacity(const moe_config* c, int32_t* capacity) {
  int st = moe_check_config(c);
  if (st) return st;
  if (!capacity) return MOE_ERR_ARG;
  *capacity = capacity_of(*c);
  return MOE_OK;
}

int moe_workspace_size(const moe_config* c, size_t* bytes) {
  int st = moe_check_config(c);
  if (st) return st;
  if (!bytes) return MOE_ERR_ARG;
  *bytes = layout(*c).total;
  return MOE_OK;
}

int moe_sync_status(void* ws, void* stream) {
  if (check_ws(ws)) return MOE_ERR_WORKSPACE;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  DevStatus h{};
  DevStatus* d = at<DevStatus>(ws, 0);
  if (cudaMemcpyAsync(&h, d, sizeof(h), cudaMemcpyDeviceToHost, s) != cudaSuccess)
    return MOE_ERR_CUDA;
  if (cudaStreamSynchronize(s) != cudaSuccess) return MOE_ERR_CUDA;
  if (h.code != 0) {
    if (cudaMemsetAsync(d, 0, sizeof(DevStatus), s) != cudaSuccess) return MOE_ERR_CUDA;
    if (cudaStreamSynchronize(s) != cudaSuccess) return MOE_ERR_CUDA;
  }
  return h.code;
}

int moe_router_topk(const moe_config* c, const void* x, const void* w_gate, const float* bias,
                    float* logits, int32_t* topk_idx, float* topk_w, void* ws, void* stream) {
  int st = moe_check_config(c);
  if (st) return st;
  if (c->routing != MOE_ROUTE_TOKEN_CHOICE) return MOE_ERR_UNSUPPORTED;
  if (!x || !w_gate || !topk_idx || !topk_w) return MOE_ERR_ARG;
  if ((st = check_ws(ws))) return st;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const Layout L = layout(*c);
  float* g = logits ? logits : at<float>(ws, L.logits);
  if (router_fused(*c))
    return cuda_status(launch_router_fused(*c, x, w_gate, bias, g, topk_idx, topk_w,
                                           at<float>(ws, L.part_P), at<int32_t>(ws, L.part_cnt),
                                           at<float>(ws, L.part_z), at<DevStatus>(ws, L.status),
                                           s));
  cudaError_t e = launch_router_logits(*c, x, w_gate, g, s, at<float>(ws, L.router_part),
                                       at<DevStatus>(ws, L.status));
  if (e == cudaSuccess)
    e = launch_route_topk(*c, g, bias, topk_idx, topk_w, at<DevStatus>(ws, L.status), s);
  return cuda_status(e);
}

int moe_aux_stats(const moe_config* c, const float* logits, const int32_t* topk_idx, float* f,
                  float* P, float* l_balance, float* z_loss, void* ws, void* stream) {
  int st = moe_check_config(c);
  if (st) return st;
  if (!logits) return MOE_ERR_ARG;
  if (c->routing == MOE_ROUTE_TOKEN_CHOICE && !topk_idx) return MOE_ERR_ARG;
  if ((st = check_ws(ws))) return st;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const Layout L = layout(*c);
  return cuda_status(launch_aux_stats(
      *c, logits, topk_idx, nullptr, at<float>(ws, L.part_P), at<int32_t>(ws, L.part_cnt),
      at<float>(ws, L.part_z), aux_rows(*c), f, P, l_balance, z_loss,
      at<DevStatus>(ws, L.status), s));
}

int moe_dispatch(const moe_config* c, const int32_t* topk_idx, const void* x, int32_t* counts,
                 int32_t* kept, int32_t* offsets, int32_t* pos, int32_t* row_of, int32_t* perm,
                 void* x_perm, int32_t* n_dropped, void* ws, void* stream) {
  int st = moe_check_config(c);
  if (st) return st;
  if (c->routing != MOE_ROUTE_TOKEN_CHOICE) return MOE_ERR_UNSUPPORTED;
  if (!topk_idx || !counts || !kept || !offsets || !pos || !row_of || !perm || !n_dropped)
    return MOE_ERR_ARG;
  if ((x == nullptr) != (x_perm == nullptr)) return MOE_ERR_ARG;
  if ((st = check_ws(ws))) return st;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const Layout L = layout(*c);
  DispatchBufs b{at<uint32_t>(ws, L.bitmap), at<int32_t>(ws, L.blk_base), counts, kept,
                 offsets, at<int32_t>(ws, L.mtp), n_dropped, pos, row_of, perm};
  return cuda_status(launch_dispatch(*c, capacity_of(*c), topk_idx, b, x, x_perm,
                                     at<DevStatus>(ws, L.status), s));
}

}  // extern "C"

namespace moe {
namespace {

int run_ffn(const moe_config& c, const void* xin, const int32_t* offsets, const int32_t* mtp,
            int uniform_rows, int E, int F, int max_rows, const void* w13, const void* w2,
            float* y, void* ws, const Layout& L, cudaStream_t s,
            const int32_t* gather_perm = nullptr, const void* gather_x = nullptr,
            float* scatter_out = nullptr, const int32_t* scatter_perm = nullptr,
            const float* scatter_w = nullptr, bool y_bf16 = false, void* h = nullptr) {
  GroupedFFN g{};
  g.y_bf16 = y_bf16 && bf16(c) ? 1 : 0;
  g.gather_perm = gather_perm;
  g.gather_k = c.k;
  g.gather_x = gather_x;
  g.scatter_out = scatter_out;
  g.scatter_perm = scatter_perm;
  g.scatter_w = scatter_w;
  g.x = xin;
  g.offsets = offsets;
  g.mtile_prefix = mtp;
  g.uniform_rows = uniform_rows;
  g.E = E;
  g.d = c.d_model;
  g.F = F;
  g.max_rows = max_rows;
  g.w13 = w13;
  g.w2 = w2;
  g.h = h ? h : at<void>(ws, L.h);
  g.y = y;
  DevStatus* st = at<DevStatus>(ws, L.status);
  cudaError_t e = bf16(c) ? launch_ffn_tc(g, st, s) : launch_ffn_simt(g, true, st, s);
  return cuda_status(e);
}

// offsets [E+1] given by the caller: the M-tile prefix the GEMM scheduler needs is rebuilt
// on the device from them.
__global__ void mtp_from_offsets(const int32_t* offsets, int E, int32_t* mtp) {
  pdl_prologue();
  __shared__ int s[256];
  const int e = threadIdx.x;
  int v = 0;
  if (e < E) v = ceil_div(offsets[e + 1] - offsets[e], kTileM);
  s[e] = v;
  __syncthreads();
  for (int o = 1; o < 256; o <<= 1) {
    int a = e >= o ? s[e - o] : 0;
    __syncthreads();
    s[e] += a;
    __syncthreads();
  }
  if (e < E) mtp[e + 1] = s[e];
  if (e == 0) mtp[0] = 0;
}

}  // namespace
}  // namespace moe

extern "C" {

int moe_expert_ffn(const moe_config* c, const void* x_perm, const int32_t* offsets,
                   const void* w13, const void* w2, float* y_perm, void* ws, void* stream) {
  int st = moe_check_config(c);
  if (st) return st;
  if (!x_perm || !offsets || !w13 || !w2 || !y_perm) return MOE_ERR_ARG;
  if ((st = check_ws(ws))) return st;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const Layout L = layout(*c);
  if (decode_regime(*c)) {
    DecodeFFN g{};
    g.x = x_perm;
    g.offsets = offsets;
    g.E = c->E;
    g.T = c->T;
    g.d = c->d_model;
    g.F = c->d_ff;
    g.F_shared = 0;
    g.max_rows = rows_max(*c);
    g.np = pow2_clamp(2ll * c->T * c->k / c->E, 16, 128);
    g.np_shared = 16;
    g.w13 = w13;
    g.w2 = w2;
    g.h = at<void>(ws, L.h);
    g.y = y_perm;
    g.ksplit1 = decode_split(*c, c->d_ff / 128, c->d_model / 64,
                             (double)g.max_rows * 2 * c->d_ff * 4, 1);
    g.ksplit2 = 1;                          // the caller's y_perm holds one slice
    g.gu = g.ksplit1 > 1 ? at<float>(ws, L.dec_gu) : nullptr;
    g.y_part_stride = (size_t)rows_max(*c) * c->d_model;
    g.shared_part_stride = 0;
    return launch_ffn_decode(g, at<DevStatus>(ws, L.status), s) == cudaSuccess ? MOE_OK
                                                                             : MOE_ERR_CUDA;
  }
  int32_t* mtp = at<int32_t>(ws, L.mtp);
  launch_pdl(mtp_from_offsets, 1, 256, 0, s, offsets, c->E, mtp);
  if (cudaGetLastError() != cudaSuccess) return MOE_ERR_CUDA;
  return run_ffn(*c, x_perm, offsets, mtp, -1, c->E, c->d_ff, rows_max(*c), w13, w2, y_perm, ws,
                 L, s);
}

int moe_shared_ffn(const moe_config* c, const void* x, const void* ws13, const void* ws2,
                   float* shared_out, void* ws, void* stream) {
  int st = moe_check_config(c);
  if (st) return st;
  if (c->d_ff_shared <= 0) return MOE_ERR_SHAPE;
  if (!x || !ws13 || !ws2 || !shared_out) return MOE_ERR_ARG;
  if ((st = check_ws(ws))) return st;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const Layout L = layout(*c);
  return run_ffn(*c, x, nullptr, nullptr, c->T, 1, c->d_ff_shared, c->T, ws13, ws2, shared_out,
                 ws, L, s);
}

int moe_combine(const moe_config* c, const float* y_perm, const int32_t* row_of,
                const float* topk_w, const float* shared_out, void* out, void* stream) {
  int st = moe_check_config(c);
  if (st) return st;
  if (c->routing != MOE_ROUTE_TOKEN_CHOICE) return MOE_ERR_UNSUPPORTED;
  if (!y_perm || !row_of || !topk_w || !out) return MOE_ERR_ARG;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  return cuda_status(launch_combine(*c, y_perm, row_of, topk_w, shared_out, out, s));
}

int moe_expert_choice(const moe_config* c, const float* logits, int32_t* ec_tokens, float* ec_w,
                      int32_t* tok_ptr, int32_t* tok_rows, void* ws, void* stream) {
  int st = moe_check_config(c);
  if (st) return st;
  if (c->routing != MOE_ROUTE_EXPERT_CHOICE) return MOE_ERR_ARG;
  if (!logits || !ec_tokens || !ec_w || !tok_ptr || !tok_rows) return MOE_ERR_ARG;
  if ((st = check_ws(ws))) return st;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const Layout L = layout(*c);
  return cuda_status(launch_expert_choice(*c, logits, ec_tokens, ec_w, at<int32_t>(ws, L.tok_cnt),
                                          tok_ptr, tok_rows, at<int32_t>(ws, L.posmap),
                                          at<float2>(ws, L.tokstat), at<DevStatus>(ws, L.status),
                                          s));
}

}  // extern "C"

namespace moe {
namespace {

int forward_impl(const moe_config* c, const void* x, const void* w_gate, const float* bias,
                 const void* w13, const void* w2, const void* ws13, const void* ws2, void* out,
                 int32_t* topk_idx, float* topk_w, float* f, float* P, float* l_balance,
                 float* z_loss, int32_t* n_dropped, void* ws, cudaStream_t s,
                 cudaEvent_t ev_begin, cudaEvent_t ev_end) {
  int st = moe_check_config(c);
  if (st) return st;
  if (!x || !w_gate || !w13 || !w2 || !out) return MOE_ERR_ARG;
  if (c->d_ff_shared > 0 && (!ws13 || !ws2)) return MOE_ERR_ARG;
  if ((st = check_ws(ws))) return st;
  const Layout L = layout(*c);
  DevStatus* dst = at<DevStatus>(ws, L.status);
  float* g = at<float>(ws, L.logits);
  f = f ? f : at<float>(ws, L.f);
  P = P ? P : at<float>(ws, L.P);
  l_balance = l_balance ? l_balance : at<float>(ws, L.lb);
  z_loss = z_loss ? z_loss : at<float>(ws, L.z);
  float* shared = c->d_ff_shared > 0 ? at<float>(ws, L.shared_out) : nullptr;
  float* part_P = at<float>(ws, L.part_P);
  int32_t* part_cnt = at<int32_t>(ws, L.part_cnt);
  float* part_z = at<float>(ws, L.part_z);
  auto mark = [&](cudaEvent_t ev) {
    return ev ? cudaEventRecord(ev, s) : cudaSuccess;
  };

  cudaError_t e = cudaSuccess;
  const bool tc = c->routing == MOE_ROUTE_TOKEN_CHOICE;
  SideStream* side = shared && shared_overlap(*c, tc && decode_regime(*c)) ? side_stream(s)
                                                                           : nullptr;
  const bool side_ffn = side != nullptr;
  if (side_ffn && cudaEventRecord(side->fork, s) != cudaSuccess) return MOE_ERR_CUDA;
  // the shared experts' h rows sit after the routed rows' h, so the two never share bytes
  void* shared_h = at<uint8_t>(ws, L.h) + (size_t)rows_max(*c) * c->d_ff * 2;
  // the shared experts' GEMMs on the side stream, issued right after the router's first launch
  // so that the router's CTAs take their SMs first
  auto launch_side = [&]() -> int {
    if (!side_ffn) return MOE_OK;
    if (cudaStreamWaitEvent(side->s, side->fork, 0) != cudaSuccess) return MOE_ERR_CUDA;
    const int r = run_ffn(*c, x, nullptr, nullptr, c->T, 1, c->d_ff_shared, c->T, ws13, ws2,
                          shared, ws, L, side->s, nullptr, nullptr, nullptr, nullptr, nullptr,
                          false, shared_h);
    if (r) return r;
    return cudaEventRecord(side->join, side->s) == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
  };
  auto join_side = [&]() {
    return side ? cudaStreamWaitEvent(s, side->join, 0) : cudaSuccess;
  };
  // without the side stream the shared FFN runs after the routed GEMMs
  auto shared_after = [&]() -> int {
    if (!shared || side_ffn) return MOE_OK;
    return run_ffn(*c, x, nullptr, nullptr, c->T, 1, c->d_ff_shared, c->T, ws13, ws2, shared,
                   ws, L, s);
  };
  if (!(tc && router_fused(*c))) {
    e = launch_router_logits(*c, x, w_gate, g, s, at<float>(ws, L.router_part), dst);
    if (e != cudaSuccess) return MOE_ERR_CUDA;
    if ((st = launch_side())) return st;
  }

  if (c->routing == MOE_ROUTE_TOKEN_CHOICE) {
    int32_t* idx = topk_idx ? topk_idx : at<int32_t>(ws, L.idx);
    float* w = topk_w ? topk_w : at<float>(ws, L.w);
    // Top-k with the load-balance partials of the same pass (in the router GEMM's epilogue for
    // prefill batches of a wide router); the partials are reduced by an extra CTA of the small
    // dispatch (T <= 256), else after the combine, off the path to the output
    if (router_fused(*c)) {
      e = launch_router_fused(*c, x, w_gate, bias, g, idx, w, part_P, part_cnt, part_z, dst, s);
      if (e != cudaSuccess) return MOE_ERR_CUDA;
      if ((st = launch_side())) return st;
    } else {
      e = launch_route_topk(*c, g, bias, idx, w, dst, s, part_P, part_cnt, part_z);
    }
    if (e != cudaSuccess) return MOE_ERR_CUDA;
    const bool dec = decode_regime(*c);
    const bool fuse = gather_fused(*c, dec);
    DispatchBufs b{at<uint32_t>(ws, L.bitmap), at<int32_t>(ws, L.blk_base),
                   at<int32_t>(ws, L.counts), at<int32_t>(ws, L.kept),
                   at<int32_t>(ws, L.offsets), at<int32_t>(ws, L.mtp),
                   n_dropped ? n_dropped : at<int32_t>(ws, L.n_dropped), at<int32_t>(ws, L.pos),
                   at<int32_t>(ws, L.row_of), at<int32_t>(ws, L.perm)};
    // small batches: the dispatch launch also finishes the statistics (one extra CTA)
    const bool fin_in_dispatch = dispatch_finalizes_stats(*c);
    const StatsFinal fin{part_P, part_cnt, part_z, aux_rows(*c), f, P, l_balance, z_loss};
    if ((e = launch_dispatch(*c, capacity_of(*c), idx, b, fuse ? nullptr : x,
                             fuse ? nullptr : at<void>(ws, L.x_perm), dst, s,
                             dec && shared != nullptr, fin_in_dispatch ? &fin : nullptr)) !=
        cudaSuccess)
      return MOE_ERR_CUDA;
    if (dec) {
      DecodeFFN g{};
      g.x = at<void>(ws, L.x_perm);
      g.offsets = b.offsets;
      g.E = c->E;
      g.T = c->T;
      g.d = c->d_model;
      g.F = c->d_ff;
      g.F_shared = c->d_ff_shared;
      g.max_rows = rows_max(*c) + c->T;
      g.np = pow2_clamp(2ll * c->T * c->k / c->E, 16, 128);
      g.np_shared = pow2_clamp(c->T, 16, 128);
      g.w13 = w13;
      g.w2 = w2;
      g.ws13 = ws13;
      g.ws2 = ws2;
      g.h = at<void>(ws, L.h);
      const int Fmx = c->d_ff > c->d_ff_shared ? c->d_ff : c->d_ff_shared;
      g.ksplit1 = decode_split(*c, c->d_ff / 128, c->d_model / 64,
                               (double)g.max_rows * 2 * Fmx * 4, 1);
      // every K slice must hold at least one 64-wide block of both the routed and shared K
      const int kb2 = (c->d_ff_shared > 0 && c->d_ff_shared < c->d_ff ? c->d_ff_shared
                                                                      : c->d_ff) / 64;
      g.ksplit2 = decode_split(*c, c->d_model / 256, kb2,
                               (double)(rows_max(*c) + (shared ? c->T : 0)) * c->d_model * 4, 2);
      g.gu = g.ksplit1 > 1 ? at<float>(ws, L.dec_gu) : nullptr;
      g.y = g.ksplit2 > 1 ? at<float>(ws, L.dec_y) : at<float>(ws, L.y_perm);
      g.shared_out = g.ksplit2 > 1 ? at<float>(ws, L.dec_sh) : shared;
      g.y_part_stride = (size_t)rows_max(*c) * c->d_model;
      g.shared_part_stride = (size_t)c->T * c->d_model;
      if (mark(ev_begin) != cudaSuccess || launch_ffn_decode(g, dst, s) != cudaSuccess ||
          mark(ev_end) != cudaSuccess)
        return MOE_ERR_CUDA;
      if ((e = launch_combine(*c, g.y, b.row_of, w, shared ? g.shared_out : nullptr, out, s,
                              g.ksplit2, g.y_part_stride, g.shared_part_stride)) != cudaSuccess)
        return MOE_ERR_CUDA;
    } else {
      const bool scat = combine_fused(*c, dec);
      if (scat && cudaMemsetAsync(out, 0, (size_t)c->T * c->d_model * 4, s) != cudaSuccess)
        return MOE_ERR_CUDA;
      if (join_side() != cudaSuccess || mark(ev_begin) != cudaSuccess) return MOE_ERR_CUDA;
      // y leaves the down GEMM in bf16 when a combine pass reads it back
      const bool ybf = !scat && bf16(*c);
      if ((st = run_ffn(*c, at<void>(ws, L.x_perm), b.offsets, b.mtile_prefix, -1, c->E,
                        c->d_ff, rows_max(*c), w13, w2, at<float>(ws, L.y_perm), ws, L, s,
                        fuse ? b.perm : nullptr, fuse ? x : nullptr,
                        scat ? static_cast<float*>(out) : nullptr, scat ? b.perm : nullptr,
                        scat ? w : nullptr, ybf)))
        return st;
      if ((st = shared_after())) return st;
      if (mark(ev_end) != cudaSuccess) return MOE_ERR_CUDA;
      if (!scat) {
        e = ybf ? launch_combine_bf16y(*c, at<void>(ws, L.y_perm), b.row_of, w, shared, out, s)
                : launch_combine(*c, at<float>(ws, L.y_perm), b.row_of, w, shared, out, s);
        if (e != cudaSuccess) return MOE_ERR_CUDA;
      }
    }
    if (fin_in_dispatch) return MOE_OK;
    return cuda_status(launch_aux_final(*c, part_P, part_cnt, part_z, aux_rows(*c), f, P,
                                        l_balance, z_loss, s));
  }

  // expert choice
  const int C = (int)((long long)c->T * c->k / c->E);
  int32_t* ec_tokens = at<int32_t>(ws, L.ec_tokens);
  float* ec_w = at<float>(ws, L.ec_w);
  if ((e = launch_expert_choice(*c, g, ec_tokens, ec_w, at<int32_t>(ws, L.tok_cnt),
                                at<int32_t>(ws, L.tok_ptr), at<int32_t>(ws, L.tok_rows),
                                at<int32_t>(ws, L.posmap), at<float2>(ws, L.tokstat), dst, s)) !=
      cudaSuccess)
    return MOE_ERR_CUDA;
  if ((e = launch_gather_ec(*c, ec_tokens, x, at<void>(ws, L.x_perm), at<int32_t>(ws, L.offsets),
                            at<int32_t>(ws, L.mtp), s)) != cudaSuccess)
    return MOE_ERR_CUDA;
  if (join_side() != cudaSuccess || mark(ev_begin) != cudaSuccess) return MOE_ERR_CUDA;
  const bool ybf = bf16(*c);
  if ((st = run_ffn(*c, at<void>(ws, L.x_perm), at<int32_t>(ws, L.offsets),
                    at<int32_t>(ws, L.mtp), -1, c->E, c->d_ff, c->E * C, w13, w2,
                    at<float>(ws, L.y_perm), ws, L, s, nullptr, nullptr, nullptr, nullptr,
                    nullptr, ybf)))
    return st;
  if ((st = shared_after())) return st;
  if (mark(ev_end) != cudaSuccess) return MOE_ERR_CUDA;
  if ((e = launch_combine_ec(*c, at<void>(ws, L.y_perm), ybf, at<int32_t>(ws, L.tok_ptr),
                             at<int32_t>(ws, L.tok_rows), ec_w, shared, out, s)) != cudaSuccess)
    return MOE_ERR_CUDA;
  return cuda_status(launch_aux_stats(*c, g, nullptr, nullptr, part_P, part_cnt, part_z,
                                      aux_rows(*c), f, P, l_balance, z_loss, dst, s));
}

}  // namespace
}  // namespace moe

extern "C" {

int moe_forward(const moe_config* c, const void* x, const void* w_gate, const float* bias,
                const void* w13, const void* w2, const void* ws13, const void* ws2, void* out,
                int32_t* topk_idx, float* topk_w, float* f, float* P, float* l_balance,
                float* z_loss, int32_t* n_dropped, void* ws, void* stream) {
  return forward_impl(c, x, w_gate, bias, w13, w2, ws13, ws2, out, topk_idx, topk_w, f, P,
                      l_balance, z_loss, n_dropped, ws, static_cast<cudaStream_t>(stream),
                      nullptr, nullptr);
}

int moe_forward_timed(const moe_config* c, const void* x, const void* w_gate, const float* bias,
                      const void* w13, const void* w2, const void* ws13, const void* ws2,
                      void* out, int32_t* topk_idx, float* topk_w, float* f, float* P,
                      float* l_balance, float* z_loss, int32_t* n_dropped, void* ws,
                      void* stream, void* ev_expert_begin, void* ev_expert_end) {
  if (!ev_expert_begin || !ev_expert_end) return MOE_ERR_ARG;
  return forward_impl(c, x, w_gate, bias, w13, w2, ws13, ws2, out, topk_idx, topk_w, f, P,
                      l_balance, z_loss, n_dropped, ws, static_cast<cudaStream_t>(stream),
                      static_cast<cudaEvent_t>(ev_expert_begin),
                      static_cast<cudaEvent_t>(ev_expert_end));
}

int moe_workspace_views(const moe_config* c, void* ws, float** logits, int32_t** row_of,
                        int32_t** offsets, void** x_perm, float** y_perm) {
  int st = moe_check_config(c);
  if (st) return st;
  if ((st = check_ws(ws))) return st;
  const Layout L = layout(*c);
  if (logits) *logits = at<float>(ws, L.logits);
  if (row_of) *row_of = at<int32_t>(ws, L.row_of);
  if (offsets) *offsets = at<int32_t>(ws, L.offsets);
  if (x_perm) *x_perm = at<void>(ws, L.x_perm);
  if (y_perm) *y_perm = at<float>(ws, L.y_perm);
  return MOE_OK;
}

int moe_workspace_views_ec(const moe_config* c, void* ws, int32_t** ec_tokens, float** ec_w,
                           int32_t** tok_ptr, int32_t** tok_rows) {
  int st = moe_check_config(c);
  if (st) return st;
  if (c->routing != MOE_ROUTE_EXPERT_CHOICE) return MOE_ERR_ARG;
  if ((st = check_ws(ws))) return st;
  const Layout L = layout(*c);
  if (ec_tokens) *ec_tokens = at<int32_t>(ws, L.ec_tokens);
  if (ec_w) *ec_w = at<float>(ws, L.ec_w);
  if (tok_ptr) *tok_ptr = at<int32_t>(ws, L.tok_ptr);
  if (tok_rows) *tok_rows = at<int32_t>(ws, L.tok_rows);
  return MOE_OK;
}

int moe_selftest_timeout(void* ws, int32_t limit_us, void* stream) {
  int st = check_ws(ws);
  if (st) return st;
  if (limit_us < 1 || limit_us > 2000000) return MOE_ERR_ARG;
  return cuda_status(launch_timeout_probe(at<DevStatus>(ws, 0), limit_us,
                                          static_cast<cudaStream_t>(stream)));
}

}  // extern "C"

// ---------------------------------------------------------------------------------------------
// FP8 (E4M3) expert weights: the decode kernels on one-byte codes with per-row scales
// ---------------------------------------------------------------------------------------------
namespace moe {
namespace {



struct Fp8Layout {
  Layout base;
  size_t x8, sx, h8, hs, gu, y, sh, total;
  int ks1, ks2;
};

Fp8Layout fp8_layout(const moe_config& c) {
  Fp8Layout L{};
  L.base = layout(c);
  size_t o = L.base.total;
  auto take = [&](size_t bytes) {
    size_t at = o;
    o = align_up(o + (bytes ? bytes : 1));
    return at;
  };
  const size_t R = rows_max(c), T = c.T, d = c.d_model, F = c.d_ff, Fs = c.d_ff_shared;
  const size_t rows = R + T, Fmax = F > Fs ? F : Fs;
  // K slices as on the bf16 decode path (split_by_waves), on 128-element E4M3 K blocks
  L.ks1 = split_by_waves(c, c.d_ff / 128, c.d_model / 128, (double)rows * 2 * Fmax * 4);
  const int kf = (int)((Fs > 0 && Fs < F ? Fs : F) / 128);
  L.ks2 = split_by_waves(c, c.d_model / 256, kf, (double)(R + (Fs ? T : 0)) * d * 4);
  L.x8 = take(rows * d);
  L.sx = take(rows * 4);
  L.h8 = take(rows * Fmax);
  L.hs = take(rows * 4);
  L.gu = take((size_t)L.ks1 * rows * 2 * Fmax * 4);
  L.y = take((size_t)L.ks2 * R * d * 4);
  L.sh = take(Fs ? (size_t)L.ks2 * T * d * 4 : 0);
  L.total = o;
  return L;
}

int check_fp8_config(const moe_config* c) {
  int st = moe_check_config(c);
  if (st) return st;
  if (c->dtype != MOE_DTYPE_BF16 || c->routing != MOE_ROUTE_TOKEN_CHOICE)
    return MOE_ERR_UNSUPPORTED;
  if (c->d_model % 256) return MOE_ERR_SHAPE;
  return MOE_OK;
}

}  // namespace
}  // namespace moe

extern "C" {

int moe_fp8_workspace_size(const moe_config* c, size_t* bytes) {
  int st = check_fp8_config(c);
  if (st) return st;
  if (!bytes) return MOE_ERR_ARG;
  *bytes = fp8_layout(*c).total;
  return MOE_OK;
}

int moe_forward_fp8(const moe_config* c, const void* x, const void* w_gate, const float* bias,
                    const uint8_t* w13_q, const float* w13_scale, const uint8_t* w2_q,
                    const float* w2_scale, const uint8_t* ws13_q, const float* ws13_scale,
                    const uint8_t* ws2_q, const float* ws2_scale, void* out, int32_t* topk_idx,
                    float* topk_w, float* f, float* P, float* l_balance, float* z_loss,
                    int32_t* n_dropped, void* ws, void* stream) {
  int st = check_fp8_config(c);
  if (st) return st;
  if (!x || !w_gate || !w13_q || !w13_scale || !w2_q || !w2_scale || !out) return MOE_ERR_ARG;
  const bool has_sh = c->d_ff_shared > 0;
  if (has_sh && (!ws13_q || !ws13_scale || !ws2_q || !ws2_scale)) return MOE_ERR_ARG;
  if ((st = check_ws(ws))) return st;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const Fp8Layout F8 = fp8_layout(*c);
  const Layout& L = F8.base;
  DevStatus* dst = at<DevStatus>(ws, L.status);
  float* g = at<float>(ws, L.logits);
  f = f ? f : at<float>(ws, L.f);
  P = P ? P : at<float>(ws, L.P);
  l_balance = l_balance ? l_balance : at<float>(ws, L.lb);
  z_loss = z_loss ? z_loss : at<float>(ws, L.z);
  int32_t* idx = topk_idx ? topk_idx : at<int32_t>(ws, L.idx);
  float* w = topk_w ? topk_w : at<float>(ws, L.w);
  float* part_P = at<float>(ws, L.part_P);
  int32_t* part_cnt = at<int32_t>(ws, L.part_cnt);
  float* part_z = at<float>(ws, L.part_z);

  if (router_fused(*c)) {
    if (launch_router_fused(*c, x, w_gate, bias, g, idx, w, part_P, part_cnt, part_z, dst, s) !=
        cudaSuccess)
      return MOE_ERR_CUDA;
  } else if (launch_router_logits(*c, x, w_gate, g, s, at<float>(ws, L.router_part), dst) !=
                 cudaSuccess ||
             launch_route_topk(*c, g, bias, idx, w, dst, s, part_P, part_cnt, part_z) !=
                 cudaSuccess) {
    return MOE_ERR_CUDA;
  }
  DispatchBufs b{at<uint32_t>(ws, L.bitmap), at<int32_t>(ws, L.blk_base),
                 at<int32_t>(ws, L.counts), at<int32_t>(ws, L.kept), at<int32_t>(ws, L.offsets),
                 at<int32_t>(ws, L.mtp), n_dropped ? n_dropped : at<int32_t>(ws, L.n_dropped),
                 at<int32_t>(ws, L.pos), at<int32_t>(ws, L.row_of), at<int32_t>(ws, L.perm)};
  // routed rows in expert order, then (with shared experts) the T token rows; small batches
  // finish the statistics in the same launch
  // (and, for small batches, write the rows straight as E4M3 codes)
  const bool fin_in_dispatch = dispatch_finalizes_stats(*c);
  const StatsFinal fin{part_P, part_cnt, part_z, aux_rows(*c), f, P, l_balance, z_loss};
  const int R = rows_max(*c);
  uint8_t* x8 = at<uint8_t>(ws, F8.x8);
  float* sx = at<float>(ws, F8.sx);
  const bool q_in_dispatch = dispatch_quantizes(*c);
  if (launch_dispatch(*c, capacity_of(*c), idx, b, x, at<void>(ws, L.x_perm), dst, s, has_sh,
                      fin_in_dispatch ? &fin : nullptr, q_in_dispatch ? x8 : nullptr,
                      q_in_dispatch ? sx : nullptr) != cudaSuccess)
    return MOE_ERR_CUDA;
  if (!q_in_dispatch &&
      launch_quantize_rows(at<void>(ws, L.x_perm), (long long)R + c->T, c->d_model,
                           b.offsets + c->E, has_sh ? c->T : 0, x8, sx, s) != cudaSuccess)
    return MOE_ERR_CUDA;
  DecodeFFN gd{};
  gd.x = x8;
  gd.offsets = b.offsets;
  gd.E = c->E;
  gd.T = c->T;
  gd.d = c->d_model;
  gd.F = c->d_ff;
  gd.F_shared = c->d_ff_shared;
  gd.max_rows = R + c->T;
  gd.np = pow2_clamp(2ll * c->T * c->k / c->E, 16, 128);
  gd.np_shared = pow2_clamp(c->T, 16, 128);
  gd.w13 = w13_q;
  gd.w2 = w2_q;
  gd.ws13 = ws13_q;
  gd.ws2 = ws2_q;
  gd.h = at<void>(ws, F8.h8);
  gd.ksplit1 = F8.ks1;
  gd.ksplit2 = F8.ks2;
  gd.gu = at<float>(ws, F8.gu);
  gd.y = at<float>(ws, F8.y);
  gd.shared_out = has_sh ? at<float>(ws, F8.sh) : nullptr;
  gd.y_part_stride = (size_t)R * c->d_model;
  gd.shared_part_stride = (size_t)c->T * c->d_model;
  gd.fp8 = 1;
  gd.s13 = w13_scale;
  gd.s2 = w2_scale;
  gd.ss13 = ws13_scale;
  gd.ss2 = ws2_scale;
  gd.sx = sx;
  gd.hs = at<float>(ws, F8.hs);
  if (launch_ffn_decode(gd, dst, s) != cudaSuccess) return MOE_ERR_CUDA;
  if (launch_combine(*c, gd.y, b.row_of, w, gd.shared_out, out, s, F8.ks2, gd.y_part_stride,
                     gd.shared_part_stride) != cudaSuccess)
    return MOE_ERR_CUDA;
  if (fin_in_dispatch) return MOE_OK;
  return cuda_status(launch_aux_final(*c, part_P, part_cnt, part_z, aux_rows(*c), f, P,
                                      l_balance, z_loss, s));
}

}  // extern "C"

