// Dispatch for callers that cannot allocate device memory.
//
// Some callers of this library may not call cudaMalloc at all: code running inside another
// framework's memory pool that forbids allocations outside it, plugin hosts that hand a plugin
// only the tensors they own, and embedded runtimes whose allocator is locked down.  moe_dispatch
// needs per-block scratch (a bitmap of the tokens each expert received, the per-block bases of
// the token-order scan and the M-tile prefix) that normally lives in a caller-allocated
// workspace.  moe_dispatch_noalloc keeps that scratch in one fixed array compiled into this
// library instead, so such callers pass only their inputs and outputs.
//
// The array is a file-scope __device__ variable: every GPU that loads the library holds it
// (kNoAllocScratchBytes, about 2.3 MB) until the process exits.  Its size fixes the largest
// call: T <= 65536 tokens and E <= 256 experts; larger calls are refused with MOE_ERR_SHAPE.
// Every call shares the same array and it keeps the previous call's contents, so two calls
// that overlap on the GPU (two streams, or two host threads) race on it; issue them one after
// another.  Each call rewrites every scratch word before reading it, and clears the caller's
// two status words first.
//
// Every call made outside stream capture looks up the array's device address
// (cudaGetSymbolAddress, with the calling device current) and caches it per device, so the
// address stays right after a device reset or a context torn down and created again.  A call
// made while its stream is being captured uses the cached address instead (no lookup during
// capture): make one call on that device before capturing.
#include <cuda_runtime.h>

#include <mutex>

#include "common.cuh"
#include "kernels.h"

namespace moe {
namespace {

constexpr int kNoAllocMaxTokens = 65536;
constexpr int kNoAllocMaxExperts = 256;
constexpr int kNoAllocMaxBlocks = kNoAllocMaxTokens / kDispatchBlock;       // 256
constexpr size_t kBitmapWords = (size_t)kNoAllocMaxBlocks * kNoAllocMaxExperts * (kDispatchBlock / 32);
constexpr size_t kBaseWords = (size_t)kNoAllocMaxBlocks * kNoAllocMaxExperts;
constexpr size_t kMtpWords = kNoAllocMaxExperts + 1;
constexpr size_t kNoAllocScratchBytes = (kBitmapWords + kBaseWords + kMtpWords) * 4;

static __device__ __align__(256) uint32_t g_dispatch_scratch[kBitmapWords + kBaseWords + kMtpWords];
static_assert(sizeof(g_dispatch_scratch) == kNoAllocScratchBytes, "scratch size");

constexpr int kMaxDevices = 128;
std::mutex g_mu;
void* g_scratch_addr[kMaxDevices] = {};

// Device address of g_dispatch_scratch on the current device.  In host code the symbol name is
// only a host-side handle, so the address is looked up with the device current: afresh on
// every call outside stream capture (a reset device or a re-created context may place the
// array elsewhere), from the per-device cache while `s` is capturing.
int scratch_address(cudaStream_t s, void** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return MOE_ERR_CUDA;
  if (dev < 0 || dev >= kMaxDevices) return MOE_ERR_UNSUPPORTED;
  cudaStreamCaptureStatus cap = cudaStreamCaptureStatusNone;
  if (cudaStreamIsCapturing(s, &cap) != cudaSuccess) return MOE_ERR_CUDA;
  std::lock_guard<std::mutex> lock(g_mu);
  if (cap == cudaStreamCaptureStatusNone) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_dispatch_scratch) != cudaSuccess || !p) return MOE_ERR_CUDA;
    g_scratch_addr[dev] = p;
  } else if (!g_scratch_addr[dev]) {
    return MOE_ERR_UNSUPPORTED;       // no uncaptured call on this device yet
  }
  *out = g_scratch_addr[dev];
  return MOE_OK;
}

}  // namespace
}  // namespace moe

using namespace moe;

extern "C" int moe_dispatch_noalloc(const moe_config* c, const int32_t* topk_idx, const void* x,
                                    int32_t* counts, int32_t* kept, int32_t* offsets,
                                    int32_t* pos, int32_t* row_of, int32_t* perm, void* x_perm,
                                    int32_t* n_dropped, int32_t* status, void* stream) {
  int st = moe_check_config(c);
  if (st) return st;
  if (c->routing != MOE_ROUTE_TOKEN_CHOICE) return MOE_ERR_UNSUPPORTED;
  if (!topk_idx || !counts || !kept || !offsets || !pos || !row_of || !perm || !n_dropped ||
      !status)
    return MOE_ERR_ARG;
  if ((x == nullptr) != (x_perm == nullptr)) return MOE_ERR_ARG;
  if (c->T > kNoAllocMaxTokens || c->E > kNoAllocMaxExperts) return MOE_ERR_SHAPE;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  void* base = nullptr;
  if ((st = scratch_address(s, &base))) return st;
  uint32_t* words = static_cast<uint32_t*>(base);
  DispatchBufs b{words,
                 reinterpret_cast<int32_t*>(words + kBitmapWords),
                 counts,
                 kept,
                 offsets,
                 reinterpret_cast<int32_t*>(words + kBitmapWords + kBaseWords),
                 n_dropped,
                 pos,
                 row_of,
                 perm};
  if (cudaMemsetAsync(status, 0, sizeof(DevStatus), s) != cudaSuccess) return MOE_ERR_CUDA;
  int32_t capacity = 0;
  if ((st = moe_capacity(c, &capacity))) return st;
  return launch_dispatch(*c, capacity, topk_idx, b, x, x_perm,
                         reinterpret_cast<DevStatus*>(status), s) == cudaSuccess
             ? MOE_OK
             : MOE_ERR_CUDA;
}
