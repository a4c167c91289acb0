// Internal declarations shared by the library's translation units (not part of the ABI).
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include <utility>

#include "hs.h"

namespace hs {

// Per-layer base pointers, passed to kernels by value (kernel parameter space, no device
// allocation).  host[] holds device-usable addresses of the pinned host pool.
struct LayerPtrs {
  uint8_t* gpu[HS_MAX_LAYERS];
  uint8_t* host[HS_MAX_LAYERS];
};

struct PoolGeom {
  int32_t num_layers, page_size, row_bytes, num_gpu_blocks, num_host_blocks;
};

// Resolver launch configuration.
constexpr int kResolveThreads = 1024;
constexpr int kResolveWarps = kResolveThreads / 32;
constexpr int kRadixBins = 256;
constexpr int kSortWarps = 8;  // warps that own chunks in the victim sort
// Miss-copy work item: this many consecutive misses of one unit.
constexpr int kMissRowsPerItem = 4;
// Workspace layout shared by the resolve entry points.
inline size_t ws_counts_bytes(int64_t units) { return (4 * (size_t)units + 15) & ~size_t(15); }
inline size_t ws_msrc_offset(int64_t units, int64_t n, int64_t C) {
  const int64_t max_m = n < C ? n : C;
  return ws_counts_bytes(units) + 16 * (size_t)units * (size_t)max_m;
}

// Error bits collected inside one resolver CTA; the reported code follows the precedence
// STEP_ORDER > ID_RANGE > TABLE_RANGE > MISSING_ROW > CAPACITY.
enum : uint32_t {
  kErrStep = 1u,
  kErrId = 2u,
  kErrTable = 4u,
  kErrMissing = 8u,
  kErrCapacity = 16u,
  kErrHot = 32u,  // a hot-block entry outside the pool: TABLE_RANGE only if the unit has a hit or a miss
};

// A resolver unit is (index group, request); `group` = G layers share one top-K list and one hot
// state.  layer_begin and nl count groups: the group's layers are [g*G, (g+1)*G).
struct ResolveParams {
  int32_t layer_begin, nl, group, R, n /* P*K */, C, S, max_pages, step;
  int32_t num_gpu_blocks, num_host_blocks;
  int32_t id_hash_bits;
  int32_t max_m;  // miss-list capacity per unit = min(n, C)
  const int32_t* topk;
  const int32_t* bt;
  const int32_t* hbt;
  const int32_t* ctx_len;
  const int32_t* hot_blocks;
  int32_t* slot_token;
  int32_t* slot_stamp;
  int32_t* out_rows;
  int32_t* out_stats;
  int32_t* miss_count;  // workspace [nl*R] (units)
  int4* miss_list;      // workspace [nl*R][max_m] = (host row, pool row, position r*n+i, 0)
  // Fused mode (non-null): per output position, the fused gather's source:
  //   >= 0 pool row; -1 zero row (padding / failed unit); INT_MIN the first occurrence of a miss
  //   (written by the gather's miss warps from the miss list); other values <= -2: host row
  //   (-2 - value), a repeated position of a miss.
  int32_t* msrc;
};

struct ResolveSmem {
  // byte offsets into dynamic shared memory
  size_t stamp, ids, val, cls, slot, hot, idh /* id hash, later radix buffers */, total;
  int32_t id_hash_bits;
  int32_t id_hash_wide;  // 1: 64-bit (id, position) entries; 0: 32-bit position entries
  int32_t threads;       // threads per resolver CTA (1024, or 512: two units per SM)
  size_t tbl;         // staged block-table + host-table rows (when tbl_pages > 0)
  int32_t tbl_pages;
};

// Shared-memory plan of one resolver CTA for (n = P*K ids, C slots, page size S); total = 0 if out
// of limits.  The narrow plan is the smallest footprint.
ResolveSmem resolve_smem_plan(int64_t n, int64_t C, int64_t S, bool wide = false);
// The plan to launch: the wide id table and the request's two table rows staged in shared memory
// (when max_pages is at most kMaxStagedPages) as far as they fit within `limit`.
constexpr int64_t kMaxStagedPages = 8192;
ResolveSmem resolve_smem_plan_staged(int64_t n, int64_t C, int64_t S, int64_t max_pages, size_t limit);
size_t resolve_workspace_bytes(int64_t units, int64_t n, int64_t C);
// Largest dynamic shared memory a resolver CTA may use on device `dev` (0 on failure).
size_t resolve_smem_limit(int dev);
// Threads per resolver CTA for this plan: 512 when two CTAs fit in an SM and the units outnumber the
// SMs or a unit is small, else 1024.  resolve_smem_limit(dev) must have been called.
int resolve_threads(const ResolveSmem& sm, int64_t units, int64_t n, int sms, int dev);

// Launchers (return cudaGetLastError() of the launch).
cudaError_t launch_resolve(const ResolveParams& p, const ResolveSmem& sm, cudaStream_t s);
cudaError_t launch_miss_copy(const ResolveParams& p, const LayerPtrs& ptrs, int32_t row_bytes, int sms,
                             cudaStream_t s);
cudaError_t launch_gather(const LayerPtrs& ptrs, int32_t layer_begin, int32_t nl, const int32_t* rows, int64_t n,
                          uint8_t* out, int32_t row_bytes, int64_t num_rows, int32_t* status, int sms,
                          cudaStream_t s);
// The fused gather: rows of layers [layer_begin, layer_begin+nl), R requests x n positions each; miss
// rows come from the pinned host pool through the resolver's miss lists (dedicated warps) and are
// also stored into their hot slots; msrc marks positions the miss warps own.  Layer layer_begin + l
// reads the plan of unit group (l / group); layer_begin is a multiple of group.
cudaError_t launch_gather_fused(const LayerPtrs& ptrs, int32_t layer_begin, int32_t nl, int32_t group, int32_t R,
                                int32_t n, int32_t max_m, const int32_t* rows, const int32_t* miss_count,
                                const int4* miss_list, const int32_t* msrc, uint8_t* out, int32_t row_bytes,
                                int64_t num_rows, int sms,
                                cudaStream_t s);
cudaError_t launch_offload(const LayerPtrs& ptrs, const PoolGeom& g, const int32_t* gpu_blocks,
                           const int32_t* host_blocks, int32_t n, int32_t* status, int sms, cudaStream_t s);
cudaError_t launch_fill_i32(int32_t* a, int64_t count, int32_t value, int sms, cudaStream_t s);
cudaError_t launch_reset_requests(int32_t* tok, int32_t* stamp, int32_t groups, int32_t R, int32_t C,
                                  const int32_t* requests, int32_t n, int sms, cudaStream_t s);

void count_launch(int k = 1);

// Programmatic dependent launch.  A kernel that follows another of this library's kernels on the
// same stream is launched with programmatic stream serialization: its CTAs may be placed as soon as
// the previous kernel has started (and signalled), and wait in hardware for the previous grid to
// complete and its memory to be visible before reading anything it wrote.
__device__ __forceinline__ void pdl_allow_dependents() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }
__device__ __forceinline__ void pdl_wait_prerequisites() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

template <typename... KArgs, typename... Args>
cudaError_t launch_dependent(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t s,
                             Args&&... args) {
  cudaLaunchConfig_t cfg{};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
}
// Per-device launch configuration (occupancy, shared-memory limits) is computed once, at pool
// creation, so that no later call needs a CUDA attribute query.
void warm_gather_launch_configs();

}  // namespace hs
