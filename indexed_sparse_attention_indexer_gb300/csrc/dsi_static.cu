// dsi_indexed_attention_static: the fused layer for callers that cannot
// allocate device memory.
//
// Some callers have no way to hand the library a workspace: a plugin hosted
// by a runtime that owns every device allocation and gives its kernels no
// scratch API, or a latency-critical path where cudaMalloc's implicit device
// synchronisation cannot be tolerated.  For them the scratch the fused layer
// needs (score rows, selected indices, split-K partials) lives in one
// file-scope device array of fixed size, DSI_STATIC_SCRATCH_BYTES, that every
// GPU which loads this library keeps until the process exits.
//
// Host code must not pass the array's name to a kernel (on the host it is
// only a stand-in symbol, not a device address).  The first call on each
// device, with that device current, looks up the array's device address with
// cudaGetSymbolAddress and caches it; that first call should therefore come
// before any stream capture.  The cache is an atomic per device, so host
// threads that make their first calls at once both store the same address.
// The address belongs to the device's primary context: after
// cudaDeviceReset() the library must not be called again in the process.
// Nothing here calls cudaMalloc, cudaFree or an allocating library routine.
//
// Every call shares the one array and leaves its contents behind: calls whose
// kernels overlap on the GPU (different streams, or different host threads on
// one device without ordering) race on it.  No part of the scratch needs to
// start at zero: each kernel writes every element it later reads.
#include "dsi.h"

#include <cuda_runtime.h>

#include <atomic>

namespace {

__device__ __align__(256) unsigned char g_static_scratch[DSI_STATIC_SCRATCH_BYTES];

constexpr int kMaxDevices = 64;
std::atomic<void*> g_scratch_addr[kMaxDevices];  // device address of g_static_scratch, per device

// Device address of the scratch array on the current device (looked up once).
void* scratch_address(dsi_status* st) {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) {
    *st = DSI_ERR_CUDA;
    return nullptr;
  }
  void* p = g_scratch_addr[dev].load(std::memory_order_acquire);
  if (!p) {
    if (cudaGetSymbolAddress(&p, g_static_scratch) != cudaSuccess || p == nullptr) {
      *st = DSI_ERR_CUDA;
      return nullptr;
    }
    g_scratch_addr[dev].store(p, std::memory_order_release);
  }
  *st = DSI_OK;
  return p;
}

}  // namespace

extern "C" dsi_status dsi_indexed_attention_static(const void* q_idx, const float* w, const void* q,
                                                   const dsi_cache* cache, int32_t rows,
                                                   int32_t n_heads_idx, int32_t n_heads, int32_t K,
                                                   int64_t q_offset, float scale, int32_t decode,
                                                   int32_t* idx_out, int32_t* count_out, void* out,
                                                   float* lse, void* stream) {
  if (!cache) return DSI_ERR_INVALID_ARG;
  if (rows > 0 && K > 0 && n_heads > 0) {
    const size_t need =
        dsi_layer_workspace_size(cache, rows, n_heads_idx, n_heads, K, q_offset, decode);
    if (need > (size_t)DSI_STATIC_SCRATCH_BYTES) return DSI_ERR_WORKSPACE;
  }
  dsi_status st;
  void* scratch = scratch_address(&st);
  if (!scratch) return st;
  return dsi_indexed_attention(q_idx, w, q, cache, rows, n_heads_idx, n_heads, K, q_offset, scale,
                               decode, idx_out, count_out, out, lse, scratch,
                               (size_t)DSI_STATIC_SCRATCH_BYTES, stream);
}
