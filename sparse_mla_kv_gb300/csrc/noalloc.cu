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
// address comes from cudaGetSymbolAddress, taken with the pool's device current, and is then passed
// to the kernels like any caller workspace.  The address belongs to the CUDA context that loaded the
// module: it is cached per context, keyed on the context's unique id (a context created after
// cudaDeviceReset has a new id, so its address is looked up again).
#include <cuda.h>
#include <cuda_runtime.h>

#include <mutex>

#include "hs_internal.cuh"

namespace {

static __device__ __align__(256) unsigned char g_resolve_scratch[HS_STATIC_SCRATCH_BYTES];

// The driver's context queries, reached through the runtime so that the library does not link the
// driver library directly.
typedef CUresult(CUDAAPI* CtxGetCurrentFn)(CUcontext*);
typedef CUresult(CUDAAPI* CtxGetIdFn)(CUcontext, unsigned long long*);

struct ScratchCache {
  unsigned long long ctx_id = 0;  // 0: nothing cached (context ids start at 1)
  void* addr = nullptr;
};

std::mutex g_scratch_mu;
CtxGetCurrentFn g_ctx_get_current = nullptr;
CtxGetIdFn g_ctx_get_id = nullptr;
bool g_ctx_fns_tried = false;
ScratchCache g_scratch[64];

// The unique id of the current context (0 if it cannot be read).  Caller holds g_scratch_mu.
unsigned long long current_ctx_id() {
  if (!g_ctx_fns_tried) {
    g_ctx_fns_tried = true;
    void* f = nullptr;
    cudaDriverEntryPointQueryResult q{};
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &f, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      g_ctx_get_current = reinterpret_cast<CtxGetCurrentFn>(f);
    f = nullptr;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &f, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      g_ctx_get_id = reinterpret_cast<CtxGetIdFn>(f);
    cudaGetLastError();
  }
  if (!g_ctx_get_current || !g_ctx_get_id) return 0;
  CUcontext ctx = nullptr;
  unsigned long long id = 0;
  if (g_ctx_get_current(&ctx) != CUDA_SUCCESS || !ctx) return 0;
  if (g_ctx_get_id(ctx, &id) != CUDA_SUCCESS) return 0;
  return id;
}

// Device address of g_resolve_scratch in the current context of device `dev` (which must be
// current).  Looked up on the first call in each context.
hs_status scratch_address(int dev, void** out) {
  if (dev < 0 || dev >= 64) return HS_ERR_INVALID_ARG;
  std::lock_guard<std::mutex> lock(g_scratch_mu);
  const unsigned long long id = current_ctx_id();
  ScratchCache& c = g_scratch[dev];
  if (id == 0 || c.ctx_id != id || !c.addr) {
    void* p = nullptr;
    const cudaError_t e = cudaGetSymbolAddress(&p, g_resolve_scratch);
    if (e != cudaSuccess || p == nullptr) {
      cudaGetLastError();
      c = ScratchCache{};
      return HS_ERR_CUDA;
    }
    c.addr = p;
    c.ctx_id = id;  // id 0 (context id unreadable): looked up again on every call
  }
  *out = c.addr;
  return HS_OK;
}

}  // namespace

extern "C" hs_status hs_resolve_topk_noalloc(const hs_pool* pool, int32_t layer_begin, int32_t nl, int32_t R,
                                             int32_t P, int32_t K, const int32_t* topk_ids,
                                             const int32_t* block_table, const int32_t* host_block_table,
                                             const int32_t* ctx_len, int32_t max_pages, const hs_hot_state* hot,
                                             int32_t step, int32_t* out_rows, int32_t* out_stats,
                                             hs_stream_t stream) {
  HS_RANGE("hs_resolve_topk_noalloc");
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
  // the scratch must live on the pool's GPU: its array is looked up in the current device's context
  if (dev != hs::pool_device(pool)) return HS_ERR_INVALID_ARG;
  void* scratch = nullptr;
  const hs_status st = scratch_address(dev, &scratch);
  if (st != HS_OK) return st;
  return hs_resolve_topk(pool, layer_begin, nl, R, P, K, topk_ids, block_table, host_block_table, ctx_len,
                         max_pages, hot, step, out_rows, out_stats, scratch, (size_t)HS_STATIC_SCRATCH_BYTES, stream);
}
