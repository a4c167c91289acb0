// C ABI of the resolver library: argument validation, the pool handle, and kernel launches.
// Every entry point is asynchronous on the caller's stream and allocates no device memory.
#include <atomic>
#include <cstdint>
#include <cstring>
#include <new>

#include "hs_internal.cuh"

struct hs_pool {
  hs::PoolGeom g;
  hs::LayerPtrs ptrs;
  int device;
  int32_t miss_order;   // HS_MISS_ORDER_*
  int32_t gather_copy;  // HS_GATHER_COPY_*
  int32_t miss_warps;   // fused gather: -1 default, 0 SM partition, 1 or 2 miss warps in every CTA
  int32_t miss_sm_div;  // SM partition: every miss_sm_div-th SM copies misses (0 = the library's default, -1 none)
  int32_t miss_prefetch;  // HS_MISS_PREFETCH_*
  hs::OutPlanes planes;   // output layout of the gathers (planes.n = 0: rows)
  unsigned long long* phase_ts;  // optional device timestamps of the SM-partition gather
};

namespace hs {
namespace {

std::atomic<int64_t> g_launches{0};

int sm_count(int dev) {
  static std::atomic<int> cache[64];
  if (dev < 0 || dev >= 64) return 0;
  int v = cache[dev].load();
  if (v > 0) return v;
  if (cudaDeviceGetAttribute(&v, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || v <= 0) return 0;
  cache[dev].store(v);
  return v;
}

bool aligned16(const void* p) { return ((uintptr_t)p & 15u) == 0; }

// Layers per index group (IndexShare) of a hot state; 0 if the value does not fit the pool.
int32_t layers_per_index(const hs_hot_state* hot, const hs::PoolGeom& g) {
  const int32_t G = hot->layers_per_index <= 1 ? 1 : hot->layers_per_index;
  if (hot->layers_per_index < 0 || G > HS_MAX_LAYERS || g.num_layers % G) return 0;
  return G;
}

hs_status cuda_status(cudaError_t e) { return e == cudaSuccess ? HS_OK : HS_ERR_CUDA; }

// Whether a resolve call on nl layers (ng = nl / G index groups) files its misses in address order.
// Both halves of a planned call decide it alike.
bool use_miss_order(const hs_pool* pool, int32_t nl, int64_t ng, int32_t R, int64_t n, int32_t C,
                    size_t workspace_bytes) {
  const PoolGeom& g = pool->g;
  if (pool->miss_order == HS_MISS_ORDER_OFF || g.num_host_blocks == 0 || n == 0 || ng * R == 0) return false;
  const int64_t max_m = n < C ? n : C;
  if (2 * (int64_t)R * max_m > INT32_MAX) return false;
  if (workspace_bytes < resolve_workspace_bytes_ordered(ng, R, n, C)) return false;
  const int64_t host_bytes = (int64_t)g.num_host_blocks * g.page_size * g.row_bytes * nl;
  return pool->miss_order >= HS_MISS_ORDER_ON || host_bytes >= kMissOrderAutoBytes;
}

// The ordered layout's pointers within `workspace`, or cnt = nullptr for per-unit lists.
MissOrder call_miss_order(const hs_pool* pool, int32_t nl, int64_t ng, int32_t R, int64_t n, int32_t C,
                          void* workspace, size_t workspace_bytes) {
  if (!use_miss_order(pool, nl, ng, R, n, C, workspace_bytes)) return MissOrder{};
  MissOrder o = miss_order_layout(workspace, ng, R, n, C, (int64_t)pool->g.num_host_blocks * pool->g.page_size);
  const PoolGeom& g = pool->g;
  o.ranges = pool->miss_order == HS_MISS_ORDER_RANGES ||
             (pool->miss_order != HS_MISS_ORDER_SPREAD &&
              (int64_t)g.num_host_blocks * g.page_size * g.row_bytes * nl >= kMissRangesBytes) ? 1 : 0;
  return o;
}

}  // namespace

void count_launch(int k) { g_launches.fetch_add(k, std::memory_order_relaxed); }

int pool_device(const hs_pool* pool) { return pool ? pool->device : -1; }

}  // namespace hs

extern "C" {

const char* hs_status_str(hs_status s) {
  switch (s) {
    case HS_OK: return "ok";
    case HS_ERR_INVALID_ARG: return "invalid argument";
    case HS_ERR_ID_RANGE: return "top-K id or row id out of range";
    case HS_ERR_MISSING_ROW: return "miss on a placeholder page without a host copy";
    case HS_ERR_CAPACITY: return "more misses than evictable hot slots";
    case HS_ERR_STEP_ORDER: return "step older than the hot state";
    case HS_ERR_CUDA: return "CUDA error";
    case HS_ERR_TIMEOUT: return "device wait timed out";
    case HS_ERR_TABLE_RANGE: return "table entry outside the pool";
  }
  return "unknown status";
}

int64_t hs_launch_count(void) { return hs::g_launches.load(); }

int32_t hs_check_status(void) {
#if HS_CHECKED
  if (cudaDeviceSynchronize() != cudaSuccess) {
    cudaGetLastError();
    return -2;
  }
  const uint32_t a = hs::check_take_resolve();
  const uint32_t b = hs::check_take_gather();
  if (a == 0xFFFFFFFFu || b == 0xFFFFFFFFu) return -2;
  return (int32_t)(a ? a : b);
#else
  return -1;
#endif
}

hs_status hs_pool_create(const hs_pool_desc* d, hs_pool** out) {
  if (!out) return HS_ERR_INVALID_ARG;
  *out = nullptr;
  if (!d) return HS_ERR_INVALID_ARG;
  if (d->num_layers < 1 || d->num_layers > HS_MAX_LAYERS) return HS_ERR_INVALID_ARG;
  if (d->page_size < 1 || d->page_size > HS_MAX_PAGE_SIZE) return HS_ERR_INVALID_ARG;
  if (d->row_bytes <= 0 || d->row_bytes % 16 != 0) return HS_ERR_INVALID_ARG;
  if ((int64_t)d->page_size * d->row_bytes >= (int64_t(1) << 31)) return HS_ERR_INVALID_ARG;
  if (d->num_gpu_blocks < 1 || d->num_host_blocks < 0) return HS_ERR_INVALID_ARG;
  if ((int64_t)d->num_gpu_blocks * d->page_size >= (int64_t(1) << 31)) return HS_ERR_INVALID_ARG;
  if ((int64_t)d->num_host_blocks * d->page_size >= (int64_t(1) << 31)) return HS_ERR_INVALID_ARG;
  if (!d->gpu_layer_base) return HS_ERR_INVALID_ARG;
  if (d->num_host_blocks > 0 && !d->host_layer_base) return HS_ERR_INVALID_ARG;
  for (int l = 0; l < d->num_layers; ++l) {
    if (!d->gpu_layer_base[l] || !hs::aligned16(d->gpu_layer_base[l])) return HS_ERR_INVALID_ARG;
    if (d->num_host_blocks > 0 && (!d->host_layer_base[l] || !hs::aligned16(d->host_layer_base[l])))
      return HS_ERR_INVALID_ARG;
  }
  hs_pool* p = new (std::nothrow) hs_pool;
  if (!p) return HS_ERR_INVALID_ARG;
  std::memset(p, 0, sizeof(*p));
  p->miss_warps = -1;
  p->g = {d->num_layers, d->page_size, d->row_bytes, d->num_gpu_blocks, d->num_host_blocks};
  if (cudaGetDevice(&p->device) != cudaSuccess) {
    cudaGetLastError();
    delete p;
    return HS_ERR_CUDA;
  }
  for (int l = 0; l < d->num_layers; ++l) {
    cudaPointerAttributes a{};
    if (cudaPointerGetAttributes(&a, d->gpu_layer_base[l]) != cudaSuccess ||
        (a.type != cudaMemoryTypeDevice && a.type != cudaMemoryTypeManaged)) {
      cudaGetLastError();
      delete p;
      return HS_ERR_INVALID_ARG;
    }
    p->ptrs.gpu[l] = static_cast<uint8_t*>(d->gpu_layer_base[l]);
    if (d->num_host_blocks > 0) {
      void* dp = nullptr;
      if (cudaHostGetDevicePointer(&dp, d->host_layer_base[l], 0) != cudaSuccess || !dp || !hs::aligned16(dp)) {
        cudaGetLastError();
        delete p;
        return HS_ERR_INVALID_ARG;  // not pinned / not mapped into the device address space
      }
      p->ptrs.host[l] = static_cast<uint8_t*>(dp);
    }
  }
  // settle the lazily computed launch configuration now, once, outside any later stream work
  if (hs::sm_count(p->device) <= 0 || hs::resolve_smem_limit(p->device) == 0) {
    cudaGetLastError();
    delete p;
    return HS_ERR_CUDA;
  }
  hs::warm_gather_launch_configs();
  *out = p;
  return HS_OK;
}

void hs_pool_destroy(hs_pool* p) { delete p; }

hs_status hs_pool_set_miss_order(hs_pool* pool, int32_t mode) {
  if (!pool || mode < HS_MISS_ORDER_AUTO || mode > HS_MISS_ORDER_SPREAD) return HS_ERR_INVALID_ARG;
  pool->miss_order = mode;
  return HS_OK;
}

hs_status hs_pool_set_gather_copy(hs_pool* pool, int32_t mode) {
  if (!pool || mode < HS_GATHER_COPY_LOADS || mode > HS_GATHER_COPY_BULK) return HS_ERR_INVALID_ARG;
  pool->gather_copy = mode;
  return HS_OK;
}

hs_status hs_pool_set_miss_warps(hs_pool* pool, int32_t warps) {
  if (!pool || warps < -1 || warps > 2) return HS_ERR_INVALID_ARG;
  pool->miss_warps = warps;
  return HS_OK;
}

hs_status hs_pool_set_gather_planes(hs_pool* pool, int32_t nplanes, const int32_t* plane_bytes) {
  if (!pool || nplanes < 0 || nplanes > HS_MAX_PLANES || (nplanes > 0 && !plane_bytes)) return HS_ERR_INVALID_ARG;
  hs::OutPlanes pl{};
  int64_t sum = 0;
  for (int p = 0; p < nplanes; ++p) {
    if (plane_bytes[p] <= 0 || plane_bytes[p] % 16) return HS_ERR_INVALID_ARG;
    pl.start[p] = (int32_t)(sum >> 4);
    pl.width[p] = plane_bytes[p] >> 4;
    sum += plane_bytes[p];
  }
  if (nplanes > 0 && sum != pool->g.row_bytes) return HS_ERR_INVALID_ARG;
  for (int p = nplanes; p < HS_MAX_PLANES; ++p) pl.start[p] = INT32_MAX;  // no chunk reaches a missing plane
  pl.start[0] = 0;
  pl.n = nplanes;
  pool->planes = pl;
  return HS_OK;
}

hs_status hs_pool_set_phase_timestamps(hs_pool* pool, unsigned long long* device_ts) {
  if (!pool || (device_ts && !hs::aligned16(device_ts))) return HS_ERR_INVALID_ARG;
  pool->phase_ts = device_ts;
  return HS_OK;
}

hs_status hs_pool_set_miss_prefetch(hs_pool* pool, int32_t mode) {
  if (!pool || mode < HS_MISS_PREFETCH_OFF || mode > HS_MISS_PREFETCH_ON) return HS_ERR_INVALID_ARG;
  pool->miss_prefetch = mode;
  return HS_OK;
}

hs_status hs_pool_set_miss_sm_divisor(hs_pool* pool, int32_t divisor) {
  if (!pool || divisor < -1 || divisor == 1 || divisor > 32) return HS_ERR_INVALID_ARG;
  pool->miss_sm_div = divisor;
  return HS_OK;
}

hs_status hs_hot_reset(const hs_pool* pool, const hs_hot_state* hot, int32_t R, hs_stream_t stream) {
  HS_RANGE("hs_hot_reset");
  if (!pool || !hot || R < 0) return HS_ERR_INVALID_ARG;
  if (hot->capacity < pool->g.page_size || hot->capacity > HS_MAX_CAPACITY || hot->capacity % pool->g.page_size)
    return HS_ERR_INVALID_ARG;
  const int32_t G = hs::layers_per_index(hot, pool->g);
  if (G == 0) return HS_ERR_INVALID_ARG;
  const int64_t count = (int64_t)(pool->g.num_layers / G) * R * hot->capacity;
  if (count == 0) return HS_OK;
  if (!hot->slot_token || !hot->slot_stamp) return HS_ERR_INVALID_ARG;
  const int sms = hs::sm_count(pool->device);
  cudaError_t e = hs::launch_fill_i32(hot->slot_token, count, -1, sms, stream);
  if (e == cudaSuccess) e = hs::launch_fill_i32(hot->slot_stamp, count, -1, sms, stream);
  return hs::cuda_status(e);
}

hs_status hs_hot_reset_requests(const hs_pool* pool, const hs_hot_state* hot, int32_t R, const int32_t* requests,
                                int32_t n, hs_stream_t stream) {
  HS_RANGE("hs_hot_reset_requests");
  if (!pool || !hot || R < 0 || n < 0) return HS_ERR_INVALID_ARG;
  if (hot->capacity < pool->g.page_size || hot->capacity > HS_MAX_CAPACITY || hot->capacity % pool->g.page_size)
    return HS_ERR_INVALID_ARG;
  const int32_t G = hs::layers_per_index(hot, pool->g);
  if (G == 0) return HS_ERR_INVALID_ARG;
  if (n == 0 || R == 0) return HS_OK;
  if (!requests || !hot->slot_token || !hot->slot_stamp) return HS_ERR_INVALID_ARG;
  const int sms = hs::sm_count(pool->device);
  if (sms <= 0) return HS_ERR_CUDA;
  return hs::cuda_status(hs::launch_reset_requests(hot->slot_token, hot->slot_stamp, pool->g.num_layers / G, R,
                                                   hot->capacity, requests, n, sms, stream));
}

size_t hs_resolve_workspace_bytes_min(int32_t nl, int32_t R, int32_t P, int32_t K, int32_t capacity) {
  if (nl < 0 || R < 0 || P < 1 || K < 0 || capacity < 1) return 0;
  const int64_t n = (int64_t)P * K;
  if (n > HS_MAX_PLAN || capacity > HS_MAX_CAPACITY) return 0;
  return hs::resolve_workspace_bytes((int64_t)nl * R, n, capacity);
}

size_t hs_resolve_workspace_bytes(int32_t nl, int32_t R, int32_t P, int32_t K, int32_t capacity) {
  if (hs_resolve_workspace_bytes_min(nl, R, P, K, capacity) == 0) return 0;
  return hs::resolve_workspace_bytes_ordered(nl, R, (int64_t)P * K, capacity);
}

int32_t hs_resolve_miss_order(const hs_pool* pool, int32_t layer_begin, int32_t nl, int32_t R, int32_t P, int32_t K,
                              const hs_hot_state* hot, size_t workspace_bytes) {
  if (!pool || !hot || layer_begin < 0 || nl < 0 || (int64_t)layer_begin + nl > pool->g.num_layers || R < 0 ||
      P < 1 || K < 0 || hot->capacity < 1 || hot->capacity > HS_MAX_CAPACITY || (int64_t)P * K > HS_MAX_PLAN)
    return -1;
  const int32_t G = hs::layers_per_index(hot, pool->g);
  if (G == 0 || layer_begin % G || nl % G) return -1;
  return hs::use_miss_order(pool, nl, nl / G, R, (int64_t)P * K, hot->capacity, workspace_bytes) ? 1 : 0;
}

size_t hs_resolve_smem_bytes(int32_t P, int32_t K, int32_t capacity, int32_t page_size) {
  if (P < 1 || K < 0) return 0;
  return hs::resolve_smem_plan((int64_t)P * K, capacity, page_size).total;
}

}  // extern "C"

namespace {

// Validates a resolve call and fills the launch parameters; shared by both resolve entry points.
hs_status prepare_resolve(const hs_pool* pool, int32_t layer_begin, int32_t nl, int32_t R, int32_t P, int32_t K,
                          const int32_t* topk_ids, const int32_t* block_table, const int32_t* host_block_table,
                          const int32_t* ctx_len, int32_t max_pages, const hs_hot_state* hot, int32_t step,
                          int32_t* out_rows, int32_t* out_stats, void* workspace, size_t workspace_bytes,
                          hs::ResolveParams& p, hs::ResolveSmem& sm, int& sms, bool& nothing) {
  nothing = false;
  if (!pool || !hot) return HS_ERR_INVALID_ARG;
  const hs::PoolGeom& g = pool->g;
  if (layer_begin < 0 || nl < 0 || (int64_t)layer_begin + nl > g.num_layers) return HS_ERR_INVALID_ARG;
  if (R < 0 || P < 1 || K < 0 || step < 0 || max_pages < 1) return HS_ERR_INVALID_ARG;
  const int64_t n = (int64_t)P * K;
  const int32_t C = hot->capacity;
  if (n > HS_MAX_PLAN || C < g.page_size || C > HS_MAX_CAPACITY || C % g.page_size) return HS_ERR_INVALID_ARG;
  const int32_t G = hs::layers_per_index(hot, g);
  if (G == 0 || layer_begin % G || nl % G) return HS_ERR_INVALID_ARG;
  const int32_t ng = nl / G;  // index groups in this call: the resolver's units are (group, request)
  if ((int64_t)ng * R > INT32_MAX) return HS_ERR_INVALID_ARG;
  if (nl == 0 || R == 0) {
    nothing = true;
    return HS_OK;
  }
  if (!block_table || !host_block_table || !ctx_len || !hot->hot_blocks || !hot->slot_token || !hot->slot_stamp ||
      !out_stats || !workspace)
    return HS_ERR_INVALID_ARG;
  if (n > 0 && (!topk_ids || !out_rows)) return HS_ERR_INVALID_ARG;
  if (!hs::aligned16(workspace) || workspace_bytes < hs::resolve_workspace_bytes((int64_t)ng * R, n, C))
    return HS_ERR_INVALID_ARG;
  const size_t smem_limit = hs::resolve_smem_limit(pool->device);
  sm = hs::resolve_smem_plan(n, C, g.page_size);
  if (sm.total == 0 || sm.total > smem_limit) return HS_ERR_INVALID_ARG;
  sm = hs::resolve_smem_plan_staged(n, C, g.page_size, max_pages, smem_limit);
  sms = hs::sm_count(pool->device);
  if (sms <= 0) return HS_ERR_CUDA;
  sm.threads = hs::resolve_threads(sm, (int64_t)ng * R, n, sms, pool->device);

  p = hs::ResolveParams{};
  p.layer_begin = layer_begin / G;
  p.nl = ng;
  p.group = G;
  p.R = R;
  p.n = (int32_t)n;
  p.C = C;
  p.S = g.page_size;
  p.max_pages = max_pages;
  p.step = step;
  p.num_gpu_blocks = g.num_gpu_blocks;
  p.num_host_blocks = g.num_host_blocks;
  p.id_hash_bits = sm.id_hash_bits;
  p.max_m = (int32_t)(n < C ? n : C);
  p.topk = topk_ids;
  p.bt = block_table;
  p.hbt = host_block_table;
  p.ctx_len = ctx_len;
  p.hot_blocks = hot->hot_blocks;
  p.slot_token = hot->slot_token;
  p.slot_stamp = hot->slot_stamp;
  p.out_rows = out_rows;
  p.out_stats = out_stats;
  p.miss_count = static_cast<int32_t*>(workspace);
  p.miss_list = reinterpret_cast<int4*>(static_cast<uint8_t*>(workspace) + hs::ws_counts_bytes((int64_t)ng * R));
  p.ord = hs::call_miss_order(pool, nl, ng, R, n, C, workspace, workspace_bytes);
  p.msrc = nullptr;
  p.queues = reinterpret_cast<int32_t*>(static_cast<uint8_t*>(workspace) + hs::ws_queue_offset((int64_t)ng * R, n, C));
  if (pool->miss_prefetch != HS_MISS_PREFETCH_OFF && g.num_host_blocks > 0) {
    p.row_bytes = g.row_bytes;
    for (int l = 0; l < g.num_layers; ++l) p.host[l] = pool->ptrs.host[l];
  }
  return HS_OK;
}

}  // namespace

extern "C" {

hs_status hs_resolve_topk(const hs_pool* pool, int32_t layer_begin, int32_t nl, int32_t R, int32_t P, int32_t K,
                          const int32_t* topk_ids, const int32_t* block_table, const int32_t* host_block_table,
                          const int32_t* ctx_len, int32_t max_pages, const hs_hot_state* hot, int32_t step,
                          int32_t* out_rows, int32_t* out_stats, void* workspace, size_t workspace_bytes,
                          hs_stream_t stream) {
  HS_RANGE("hs_resolve_topk");
  hs::ResolveParams p;
  hs::ResolveSmem sm;
  int sms = 0;
  bool nothing = false;
  hs_status st = prepare_resolve(pool, layer_begin, nl, R, P, K, topk_ids, block_table, host_block_table, ctx_len,
                                 max_pages, hot, step, out_rows, out_stats, workspace, workspace_bytes, p, sm, sms,
                                 nothing);
  if (st != HS_OK || nothing) return st;
  cudaError_t e = hs::launch_resolve(p, sm, stream);
  if (e == cudaSuccess && p.max_m > 0) e = hs::launch_miss_copy(p, pool->ptrs, pool->g.row_bytes, sms, stream);
  return hs::cuda_status(e);
}

hs_status hs_resolve_plan(const hs_pool* pool, int32_t layer_begin, int32_t nl, int32_t R, int32_t P, int32_t K,
                          const int32_t* topk_ids, const int32_t* block_table, const int32_t* host_block_table,
                          const int32_t* ctx_len, int32_t max_pages, const hs_hot_state* hot, int32_t step,
                          int32_t* out_rows, int32_t* out_stats, void* workspace, size_t workspace_bytes,
                          hs_stream_t stream) {
  HS_RANGE("hs_resolve_plan");
  hs::ResolveParams p;
  hs::ResolveSmem sm;
  int sms = 0;
  bool nothing = false;
  hs_status st = prepare_resolve(pool, layer_begin, nl, R, P, K, topk_ids, block_table, host_block_table, ctx_len,
                                 max_pages, hot, step, out_rows, out_stats, workspace, workspace_bytes, p, sm, sms,
                                 nothing);
  if (st != HS_OK || nothing) return st;
  p.msrc = reinterpret_cast<int32_t*>(static_cast<uint8_t*>(workspace) +
                                      hs::ws_msrc_offset((int64_t)p.nl * R, p.n, p.C));
  return hs::cuda_status(hs::launch_resolve(p, sm, stream));
}

hs_status hs_gather_planned(const hs_pool* pool, int32_t layer_begin, int32_t nl, int32_t R, int32_t P, int32_t K,
                            const hs_hot_state* hot, const int32_t* out_rows, const void* workspace,
                            size_t workspace_bytes, void* out, hs_stream_t stream) {
  HS_RANGE("hs_gather_planned");
  if (!pool || !hot) return HS_ERR_INVALID_ARG;
  const hs::PoolGeom& g = pool->g;
  if (layer_begin < 0 || nl < 0 || (int64_t)layer_begin + nl > g.num_layers || R < 0 || P < 1 || K < 0)
    return HS_ERR_INVALID_ARG;
  const int64_t n = (int64_t)P * K;
  const int32_t capacity = hot->capacity;
  const int32_t G = hs::layers_per_index(hot, g);
  if (G == 0 || layer_begin % G || nl % G) return HS_ERR_INVALID_ARG;
  if (n > HS_MAX_PLAN || (int64_t)nl * R > INT32_MAX || capacity < 1 || capacity > HS_MAX_CAPACITY)
    return HS_ERR_INVALID_ARG;
  if (nl == 0 || R == 0 || n == 0) return HS_OK;
  const int64_t units = (int64_t)(nl / G) * R;
  if (!out_rows || !workspace || !out || !hs::aligned16(out) || !hs::aligned16(workspace) ||
      workspace_bytes < hs::resolve_workspace_bytes(units, n, capacity))
    return HS_ERR_INVALID_ARG;
  const int sms = hs::sm_count(pool->device);
  if (sms <= 0) return HS_ERR_CUDA;
  const uint8_t* ws = static_cast<const uint8_t*>(workspace);
  const int32_t max_m = (int32_t)(n < capacity ? n : capacity);
  const hs::MissOrder ord =
      hs::call_miss_order(pool, nl, nl / G, R, n, capacity, const_cast<void*>(workspace), workspace_bytes);
  // The SM partition numbers its miss units with 32-bit counters: shapes whose unit count could come near
  // 2^31 (per layer: 1024 buckets and 64-miss overflow slices, or 16-miss chunks of every unit's list) take
  // one miss warp per CTA instead.
  const int64_t miss_units =
      (int64_t)nl * (ord.cnt ? 1024 + ((int64_t)R * max_m + 63) / 64 : (int64_t)R * ((max_m + 15) / 16));
  const int32_t miss_warps = miss_units > (int64_t(1) << 30) && pool->miss_warps <= 0 ? 1 : pool->miss_warps;
  return hs::cuda_status(hs::launch_gather_fused(
      pool->ptrs, layer_begin, nl, G, R, (int32_t)n, max_m, out_rows, reinterpret_cast<const int32_t*>(ws),
      reinterpret_cast<const int4*>(ws + hs::ws_counts_bytes(units)), ord,
      reinterpret_cast<const int32_t*>(ws + hs::ws_msrc_offset(units, n, capacity)), static_cast<uint8_t*>(out),
      g.row_bytes, (int64_t)g.num_gpu_blocks * g.page_size, (int64_t)g.num_host_blocks * g.page_size,
      miss_warps, pool->miss_sm_div, pool->planes,
      reinterpret_cast<int32_t*>(const_cast<uint8_t*>(ws) + hs::ws_queue_offset(units, n, capacity)), pool->phase_ts,
      sms, stream));
}

hs_status hs_resolve_gather(const hs_pool* pool, int32_t layer_begin, int32_t nl, int32_t R, int32_t P, int32_t K,
                            const int32_t* topk_ids, const int32_t* block_table, const int32_t* host_block_table,
                            const int32_t* ctx_len, int32_t max_pages, const hs_hot_state* hot, int32_t step,
                            int32_t* out_rows, int32_t* out_stats, void* out, void* workspace,
                            size_t workspace_bytes, hs_stream_t stream) {
  HS_RANGE("hs_resolve_gather");
  if ((int64_t)P * K > 0 && nl > 0 && R > 0 && (!out || !hs::aligned16(out))) return HS_ERR_INVALID_ARG;
  hs_status st = hs_resolve_plan(pool, layer_begin, nl, R, P, K, topk_ids, block_table, host_block_table, ctx_len,
                                 max_pages, hot, step, out_rows, out_stats, workspace, workspace_bytes, stream);
  if (st != HS_OK) return st;
  return hs_gather_planned(pool, layer_begin, nl, R, P, K, hot, out_rows, workspace, workspace_bytes, out, stream);
}

hs_status hs_gather_rows(const hs_pool* pool, int32_t layer_begin, int32_t nl, const int32_t* rows, int64_t n,
                         void* out, int32_t* out_status, hs_stream_t stream) {
  HS_RANGE("hs_gather_rows");
  if (!pool) return HS_ERR_INVALID_ARG;
  const hs::PoolGeom& g = pool->g;
  if (layer_begin < 0 || nl < 0 || (int64_t)layer_begin + nl > g.num_layers || n < 0) return HS_ERR_INVALID_ARG;
  if (nl == 0 || n == 0) return HS_OK;
  if (!rows || !out || !hs::aligned16(out)) return HS_ERR_INVALID_ARG;
  if (n > (INT64_MAX / 2) / g.row_bytes) return HS_ERR_INVALID_ARG;
  const int sms = hs::sm_count(pool->device);
  if (sms <= 0) return HS_ERR_CUDA;
  return hs::cuda_status(hs::launch_gather(pool->ptrs, layer_begin, nl, rows, n, static_cast<uint8_t*>(out),
                                           g.row_bytes, (int64_t)g.num_gpu_blocks * g.page_size, out_status, sms,
                                           stream, pool->gather_copy == HS_GATHER_COPY_BULK, pool->planes));
}

hs_status hs_offload_pages(const hs_pool* pool, const int32_t* gpu_blocks, const int32_t* host_blocks, int32_t n,
                           int32_t* out_status, hs_stream_t stream) {
  HS_RANGE("hs_offload_pages");
  if (!pool || n < 0) return HS_ERR_INVALID_ARG;
  if (n == 0) return HS_OK;
  if (!gpu_blocks || !host_blocks || pool->g.num_host_blocks == 0) return HS_ERR_INVALID_ARG;
  const int sms = hs::sm_count(pool->device);
  if (sms <= 0) return HS_ERR_CUDA;
  return hs::cuda_status(hs::launch_offload(pool->ptrs, pool->g, gpu_blocks, host_blocks, n, out_status, sms, stream));
}

}  // extern "C"
