// hs_resolve_topk_noalloc: the resolver for callers that cannot allocate device memory.
//
// Some callers of this library cannot call cudaMalloc.  Examples:
//   - plug-ins loaded into a serving engine that has already reserved nearly all device memory for
//     its own KV cache, where a cudaMalloc fails or takes memory the engine has accounted for;
//   - latency-sensitive decode loops, where cudaMalloc may synchronise the device;
//   - plain C callers that have no device allocator of their own.
// hs_resolve_topk needs caller-owned scratch (the workspace holding the per-unit miss lists that the
// resolver kernel hands to the miss-copy kernel).  This entry point instead uses a scratch array
// compiled into the library: a file-scope static __device__ array of HS_STATIC_SCRATCH_BYTES.
// Every GPU that loads this library's code holds that array until the process exits.
//
// In host code the array's name is only a host-side stand-in, not a device address; the device
// address comes from cudaGetSymbolAddress, taken once per device with that device current, and is
// then passed to the kernels like any caller workspace.
#include <cuda_runtime.h>

#include <mutex>

#include "hs.h"

namespace {

static __device__ __align__(256) unsigned char g_resolve_scratch[HS_STATIC_SCRATCH_BYTES];

std::mutex g_scratch_mu;
void* g_scratch_addr[64] = {};

// Device address of g_resolve_scratch on device `dev` (which must be current), set up on first use.
hs_status scratch_address(int dev, void** out) {
  if (dev < 0 || dev >= 64) return HS_ERR_INVALID_ARG;
  std::lock_guard<std::mutex> lock(g_scratch_mu);
  if (!g_scratch_addr[dev]) {
    void* p = nullptr;
    const cudaError_t e = cudaGetSymbolAddress(&p, g_resolve_scratch);
    if (e != cudaSuccess || p == nullptr) {
      cudaGetLastError();
      return HS_ERR_CUDA;
    }
    g_scratch_addr[dev] = p;
  }
  *out = g_scratch_addr[dev];
  return HS_OK;
}

}  // namespace

extern "C" hs_status hs_resolve_topk_noalloc(const hs_pool* pool, int32_t layer_begin, int32_t nl, int32_t R,
                                             int32_t P, int32_t K, const int32_t* topk_ids,
                                             const int32_t* block_table, const int32_t* host_block_table,
                                             const int32_t* ctx_len, int32_t max_pages, const hs_hot_state* hot,
                                             int32_t step, int32_t* out_rows, int32_t* out_stats,
                                             hs_stream_t stream) {
  if (!pool || !hot) return HS_ERR_INVALID_ARG;
  // Shapes whose scratch would exceed the built-in array are refused before anything else (units are
  // index groups: nl / G of them per request).
  const int32_t G = hot->layers_per_index > 1 ? hot->layers_per_index : 1;
  const size_t need = hs_resolve_workspace_bytes_min(nl / G, R, P, K, hot->capacity);
  if (need > (size_t)HS_STATIC_SCRATCH_BYTES) return HS_ERR_INVALID_ARG;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) {
    cudaGetLastError();
    return HS_ERR_CUDA;
  }
  void* scratch = nullptr;
  const hs_status st = scratch_address(dev, &scratch);
  if (st != HS_OK) return st;
  return hs_resolve_topk(pool, layer_begin, nl, R, P, K, topk_ids, block_table, host_block_table, ctx_len,
                         max_pages, hot, step, out_rows, out_stats, scratch, (size_t)HS_STATIC_SCRATCH_BYTES, stream);
}
