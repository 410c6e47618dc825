// dispatch_noalloc.cu - moe_dispatch without a caller workspace.
//
// moe_dispatch needs scratch memory for its per-chunk histogram and prefix
// tables, which normally lives in a workspace the caller allocates. Some
// callers cannot allocate device memory at the point where they dispatch:
// code running under an allocator that forbids new allocations (a memory
// pool that is already sized and locked, a region being replayed), plugins
// that only receive pre-allocated input and output buffers from their host
// framework, or code that must not call cudaMalloc because it would
// synchronise the device. For them this file provides moe_dispatch_noalloc,
// which keeps its scratch in a fixed array compiled into the library
// instead.
//
// The array is a file-scope __device__ variable: every GPU that loads this
// library holds it (4 MiB + 256 B) until the process exits. Its size caps the
// problem: E * ceil(T / 8) must not exceed kNoAllocTableEntries (524288,
// enough for T = 16384 tokens over 256 experts). Larger requests are
// rejected on the host with MOE_ERR_WORKSPACE_TOO_SMALL before any work is
// enqueued.
//
// All calls share the one array and it keeps whatever the last call left in
// it. The tables are fully rewritten by every call (no stale value is ever
// read) and the error word is cleared at the start of each call. Two calls
// whose kernels overlap on the GPU (different streams with no ordering
// between them, or different host threads) race on the array and produce
// wrong results: serialise them.
//
// Host code cannot use the array's name as a device address (it refers to a
// host-side stand-in). The first call on each device, with that device
// current, looks up the real device address with cudaGetSymbolAddress and
// caches it; make that first call before any stream capture begins. The
// cached address belongs to the device's primary context and is never looked
// up again, so it is stale once that context is destroyed (cudaDeviceReset):
// a process that resets the device must not call this entry point again.
#include <cstdint>
#include <mutex>

#include <cuda_runtime.h>

#include "common.cuh"
#include "moe.h"

namespace moe {
namespace {

constexpr size_t kNoAllocTableEntries = static_cast<size_t>(1) << 19;
constexpr size_t kNoAllocHeader = 256;  // error word, padded to 256 bytes
constexpr size_t kNoAllocBytes = kNoAllocHeader + 2 * kNoAllocTableEntries * sizeof(int32_t);
constexpr int kMaxDevices = 64;

static __device__ __align__(256) unsigned char g_dispatch_scratch[kNoAllocBytes];

std::mutex g_scratch_mu;
void* g_scratch_addr[kMaxDevices] = {};

// Device address of g_dispatch_scratch on the current device (looked up once
// per device).
int scratch_address(void** out) {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess) return MOE_ERR_LAUNCH;
  if (dev < 0 || dev >= kMaxDevices) return MOE_ERR_UNSUPPORTED;
  std::lock_guard<std::mutex> lock(g_scratch_mu);
  if (g_scratch_addr[dev] == nullptr) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_dispatch_scratch) != cudaSuccess || p == nullptr)
      return MOE_ERR_LAUNCH;
    g_scratch_addr[dev] = p;
  }
  *out = g_scratch_addr[dev];
  return MOE_OK;
}

bool aligned16(const void* p) { return p != nullptr && (reinterpret_cast<uintptr_t>(p) % 16) == 0; }

}  // namespace
}  // namespace moe

using namespace moe;

extern "C" MOE_API int moe_dispatch_noalloc(const moe_config_t* cfg, const void* x,
                                            const int32_t* topk_idx, int32_t* counts,
                                            int32_t* offsets, int32_t* pos, int32_t* src,
                                            void* x_perm, float* x_scale, void* stream) {
  const int st = moe_check_config(cfg);
  if (st != MOE_OK) return st;
  if (counts == nullptr || offsets == nullptr) return MOE_ERR_INVALID_ARG;
  const bool soft = cfg->router == MOE_ROUTER_SOFT_GUMBEL;
  if (cfg->T > 0 && (pos == nullptr || src == nullptr ||
                     (!soft && (!aligned16(x) || topk_idx == nullptr || !aligned16(x_perm) ||
                                (cfg->payload_fp8 && x_scale == nullptr)))))
    return MOE_ERR_INVALID_ARG;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (cfg->T == 0)
    return launch_dispatch_empty(cfg->E, counts, offsets, s) == cudaSuccess ? MOE_OK
                                                                             : MOE_ERR_LAUNCH;
  if (soft)  // every token to every expert: no tables needed
    return launch_dense_layout(cfg->T, cfg->E, counts, offsets, pos, src, nullptr, 0, s) ==
                   cudaSuccess
               ? MOE_OK
               : MOE_ERR_LAUNCH;
  const int nchunk = ceil_div(cfg->T, kDispatchTokensPerChunk);
  if (static_cast<size_t>(cfg->E) * static_cast<size_t>(nchunk) > kNoAllocTableEntries)
    return MOE_ERR_WORKSPACE_TOO_SMALL;
  void* base = nullptr;
  const int sa = scratch_address(&base);
  if (sa != MOE_OK) return sa;
  uint32_t* err = static_cast<uint32_t*>(base);
  int32_t* hist = reinterpret_cast<int32_t*>(static_cast<char*>(base) + kNoAllocHeader);
  int32_t* tbase = hist + kNoAllocTableEntries;
  if (cudaMemsetAsync(err, 0, sizeof(uint32_t), s) != cudaSuccess) return MOE_ERR_LAUNCH;
  cudaError_t e = launch_dispatch_count(topk_idx, cfg->T, cfg->k, cfg->E, nchunk, hist, err,
                                        nullptr, 0, s);
  if (e == cudaSuccess) e = launch_dispatch_scan(hist, nchunk, cfg->E, tbase, counts, s);
  if (e == cudaSuccess)
    e = launch_dispatch_scatter(cfg->dtype, cfg->payload_fp8 != 0,
                                cfg->payload_fp8 == 2 ? cfg->payload_scale : 0.f, x, topk_idx,
                                cfg->T, cfg->d,
                                cfg->k, cfg->E, nchunk, counts, tbase, offsets, pos, src, x_perm,
                                x_scale, err, s);
  return e == cudaSuccess ? MOE_OK : MOE_ERR_LAUNCH;
}
