// Internal declarations shared by the library's translation units (not part of the ABI).
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include <utility>

#include "hs.h"

// NVTX ranges: every entry point that launches work opens one range named after itself in the "hs"
// domain, so that a timeline of a decode step attributes its time to resolve, gather and offload.
// Header-only NVTX (v3): with no tool attached a range costs a load and a branch.  HS_NVTX=0 builds
// without them.
#ifndef HS_NVTX
#define HS_NVTX 1
#endif
#if HS_NVTX
#include <nvtx3/nvToolsExt.h>
namespace hs {
inline nvtxDomainHandle_t nvtx_domain() {
  static const nvtxDomainHandle_t d = nvtxDomainCreateA("hs");
  return d;
}
struct NvtxRange {
  explicit NvtxRange(const char* name) {
    nvtxEventAttributes_t a{};
    a.version = NVTX_VERSION;
    a.size = NVTX_EVENT_ATTRIB_STRUCT_SIZE;
    a.messageType = NVTX_MESSAGE_TYPE_ASCII;
    a.message.ascii = name;
    nvtxDomainRangePushEx(nvtx_domain(), &a);
  }
  ~NvtxRange() { nvtxDomainRangePop(nvtx_domain()); }
  NvtxRange(const NvtxRange&) = delete;
  NvtxRange& operator=(const NvtxRange&) = delete;
};
}  // namespace hs
#define HS_RANGE(name) const ::hs::NvtxRange hs_nvtx_range_(name)
#else
#define HS_RANGE(name) ((void)0)
#endif

// Bounds-checked build.  Compiled with HS_CHECKED=1, every address a kernel computes from data it read
// (a table entry, a slot index, a miss-list entry, a chain link, an output position) is checked
// against the extent of the buffer it points into before the access; a violation skips the access and
// records the site of the first failing check in a device word of the kernel's file, which
// hs_check_status reads and clears.  The normal build (HS_CHECKED=0) compiles the checks away and keeps
// the data checks the ABI documents (status words).
#ifndef HS_CHECKED
#define HS_CHECKED 0
#endif
#if HS_CHECKED
#define HS_CHECK_WORD static __device__ unsigned int hs_check_word_ = 0u;
#define HS_CHECK(cond, site) ((cond) ? true : (atomicCAS(&hs_check_word_, 0u, (unsigned)(site)), false))
#else
#define HS_CHECK_WORD
#define HS_CHECK(cond, site) true
#endif

namespace hs {

// Sites of the bounds-checked build's checks (the value hs_check_status returns).
enum CheckSite : uint32_t {
  kChkTablePage = 1,  // resolver: a page index outside the request's table row
  kChkStateSlot = 2,  // resolver: a slot index outside the unit's hot state
  kChkMissList = 3,   // resolver: a miss-list index outside the unit's list
  kChkPoolRow = 4,    // a GPU pool row outside the pool (miss destination)
  kChkHostRow = 5,    // a host pool row outside the pinned pool (miss source)
  kChkOutPos = 6,     // an output position outside the call's output
  kChkChain = 7,      // a repeat-chain link outside the unit's positions
};
// Reads and clears the check word of each kernel file (0 in the normal build).
uint32_t check_take_resolve();
uint32_t check_take_gather();

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
// Miss-copy work item: this many consecutive misses of one unit (or of one bucket, below).
constexpr int kMissRowsPerItem = 4;

// Address-ordered miss layout.  Misses scattered over tens of GB of pinned host memory are limited
// by the device's address translation for host memory, not by the link: a step whose in-flight
// reads span the whole pool misses the translation caches on nearly every row.  In this layout the
// resolver files each miss of an index group into one of kMissBuckets buckets by host row range
// (bucket = host row >> shift), and the copy warps take the buckets in one of two schedules (below).
// Results do not depend on it: every miss writes its own hot slot and output row.
constexpr int kMissBuckets = 1024;  // enough host ranges that every copy warp of a large step owns some
constexpr int kBucketsPerLane = kMissBuckets / 32;
// the resolver counts a unit's misses per bucket in the victim sort's histogram memory
static_assert(kMissBuckets <= kRadixBins * kSortWarps, "bucket counters must fit the sort histograms");
// Output layout of gathered rows.  n = 0: rows, [positions][row_bytes].  n = 1..4: the row is cut into
// n planes of width[p] 16-byte chunks (start[p] = the plane's first chunk within the row; start[q] for
// q >= n lies past any chunk), stored one after the other: [plane 0 of every position][plane 1 ...].
struct OutPlanes {
  int32_t n;
  int32_t start[4];
  int32_t width[4];
};
// One layer's output: `rows` positions from `base`, in the pool's layout.
struct OutMap {
  uint8_t* base;
  int64_t rows;
  int32_t row_bytes;
  OutPlanes pl;
};
// Address of 16-byte chunk j of output position i in the plane layout.
__device__ __forceinline__ uint4* plane_chunk(uint8_t* base, const OutPlanes& pl, int64_t rows, int64_t i, int j) {
  const int p = (j >= pl.start[1]) + (j >= pl.start[2]) + (j >= pl.start[3]);
  return reinterpret_cast<uint4*>(base) + rows * pl.start[p] + i * pl.width[p] + (j - pl.start[p]);
}
// Address of 16-byte chunk j of output position i in either layout.
__device__ __forceinline__ uint4* out_chunk(const OutMap& om, int64_t i, int j) {
  return om.pl.n ? plane_chunk(om.base, om.pl, om.rows, i, j)
                 : reinterpret_cast<uint4*>(om.base + i * om.row_bytes) + j;
}

struct MissOrder {
  int32_t* cnt;       // [groups][kMissBuckets + 1]: entries filed per bucket, then the overflow count;
                      // zeroed before the resolver runs.  nullptr: per-unit lists instead.
  int4* buckets;      // [groups][kMissBuckets][cap]
  int4* overflow;     // [groups][per_group]: misses whose bucket was full (in no particular order)
  int32_t shift;      // bucket of host row h: h >> shift
  int32_t cap;        // entries per bucket
  int32_t per_group;  // misses an index group can have: R * max_m
  int32_t ranges;     // 1: each copy warp takes whole buckets (ranges); 0: 4-entry items in bucket order,
                      // spread over all copy warps
};
// The SM partition's work counters (miss units, finished CTAs, HBM chunks, registered miss CTAs), at the
// end of the per-unit workspace layout.  The resolver zeroes them; the partition gather's last CTA
// zeroes them again, so that the plan's gather can be replayed.
constexpr int kQueueInts = 4;
constexpr size_t kQueueBytes = 256;
// Host pools at least this large (over the layers of a call) are copied bucket by bucket, each bucket by
// one warp; smaller ones with the items of all buckets spread over every copy warp.  Measured with the
// library's miss path (131K misses per step, one layer): over spans up to 20 GB the spread items keep
// more rows in flight (185 against 145 GB/s at 4 GB); from 40 GB on, where the device's translation of
// host addresses binds, whole buckets per warp are faster (118 against 50 GB/s at 40 GB, 54 against 39
// at 72 GB).
constexpr int64_t kMissRangesBytes = int64_t(40) << 30;
// Bucket capacity: twice the even share, so that only strongly skewed steps overflow.
inline int32_t miss_bucket_cap(int64_t per_group) {
  return (int32_t)((2 * per_group + kMissBuckets - 1) / kMissBuckets);
}
// Smallest shift that maps every host row below num_host_rows into the buckets.
inline int32_t miss_bucket_shift(int64_t num_host_rows) {
  int32_t s = 0;
  while (num_host_rows > 0 && ((num_host_rows - 1) >> s) >= kMissBuckets) ++s;
  return s;
}
// Host pools at least this large (over the layers of a call) use the ordered layout by default.
constexpr int64_t kMissOrderAutoBytes = int64_t(16) << 30;
// Workspace layout shared by the resolve entry points.
inline size_t ws_counts_bytes(int64_t units) { return (4 * (size_t)units + 15) & ~size_t(15); }
inline size_t ws_msrc_offset(int64_t units, int64_t n, int64_t C) {
  const int64_t max_m = n < C ? n : C;
  return ws_counts_bytes(units) + 16 * (size_t)units * (size_t)max_m;
}
// [miss counts][miss lists][per-position sources][work counters]: the counters' offset.
inline size_t ws_queue_offset(int64_t units, int64_t n, int64_t C) {
  return ws_msrc_offset(units, n, C) + ((4 * (size_t)units * (size_t)n + 15) & ~size_t(15));
}
// The ordered layout's extra areas follow the per-unit layout (resolve_workspace_bytes): bucket
// counters, then the buckets; its overflow lists reuse the per-unit miss lists (group g's at unit
// (g, 0)).  resolve_workspace_bytes_ordered is the whole size with them.
inline size_t ws_order_cnt_bytes(int64_t groups) { return (4 * (size_t)groups * (kMissBuckets + 1) + 15) & ~size_t(15); }
size_t resolve_workspace_bytes_ordered(int64_t groups, int64_t R, int64_t n, int64_t C);
// The ordered layout for a call, or cnt = nullptr when the per-unit layout is used.
MissOrder miss_order_layout(void* workspace, int64_t groups, int64_t R, int64_t n, int64_t C, int64_t num_host_rows);

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
  int4* miss_list;      // workspace [nl*R][max_m] = (host row, pool row, position r*n+i, first repeat)
  MissOrder ord;        // ord.cnt != nullptr: misses are filed by host row range instead
  // Fused mode (non-null): per output position, the fused gather's source:
  //   >= 0 pool row; -1 zero row (padding / failed unit); <= -2 written by the miss warps: INT_MIN the
  //   first occurrence of a missed id, -3 - next a repeated position of it (next: the unit-local
  //   position of the following repeat, -1 after the last).  A miss entry's fourth field is its first
  //   repeat (-1: none), so the repeats form a chain that starts at the entry.
  int32_t* msrc;
  int32_t* queues;  // the SM partition's work counters, zeroed by the resolver (kQueueInts ints)
  // Miss prefetch (row_bytes > 0): each miss's host row is prefetched into L2, in every layer of its
  // index group, as soon as the resolver classifies it (host[l] is layer l's host pool).
  int32_t row_bytes;
  const uint8_t* host[HS_MAX_LAYERS];
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
// With the ordered layout (p.ord.cnt set) launch_resolve first clears its counters with a small
// kernel, on which the resolver depends programmatically.
cudaError_t launch_resolve(const ResolveParams& p, const ResolveSmem& sm, cudaStream_t s);
cudaError_t launch_miss_copy(const ResolveParams& p, const LayerPtrs& ptrs, int32_t row_bytes, int sms,
                             cudaStream_t s);
// bulk: move the rows with one-dimensional bulk copies through shared memory (HS_GATHER_COPY_BULK)
// when the stages fit the device's shared memory, else with 16-byte loads and stores.
// planes: the output layout (rows when planes.n = 0; the bulk mode writes rows only and falls back to
// loads for planes).
cudaError_t launch_gather(const LayerPtrs& ptrs, int32_t layer_begin, int32_t nl, const int32_t* rows, int64_t n,
                          uint8_t* out, int32_t row_bytes, int64_t num_rows, int32_t* status, int sms,
                          cudaStream_t s, bool bulk, const OutPlanes& planes);
bool gather_bulk_fits(int32_t row_bytes);
// The fused gather: rows of layers [layer_begin, layer_begin+nl), R requests x n positions each; miss
// rows come from the pinned host pool through the resolver's miss lists (dedicated warps) and are
// also stored into their hot slots; msrc marks positions the miss warps own.  Layer layer_begin + l
// reads the plan of unit group (l / group); layer_begin is a multiple of group.
cudaError_t launch_gather_fused(const LayerPtrs& ptrs, int32_t layer_begin, int32_t nl, int32_t group, int32_t R,
                                int32_t n, int32_t max_m, const int32_t* rows, const int32_t* miss_count,
                                const int4* miss_list, const MissOrder& ord, const int32_t* msrc, uint8_t* out,
                                int32_t row_bytes, int64_t num_rows, int64_t num_host_rows, int range_miss_warps,
                                int miss_sm_div, const OutPlanes& planes, int32_t* queues,
                                unsigned long long* phase_ts, int sms, cudaStream_t s);
cudaError_t launch_offload(const LayerPtrs& ptrs, const PoolGeom& g, const int32_t* gpu_blocks,
                           const int32_t* host_blocks, int32_t n, int32_t* status, int sms, cudaStream_t s);
cudaError_t launch_fill_i32(int32_t* a, int64_t count, int32_t value, int sms, cudaStream_t s);
cudaError_t launch_reset_requests(int32_t* tok, int32_t* stamp, int32_t groups, int32_t R, int32_t C,
                                  const int32_t* requests, int32_t n, int sms, cudaStream_t s);

void count_launch(int k = 1);
// The device a pool was created on (its device pointers belong to it).
int pool_device(const hs_pool* pool);

// The index of an index group's ordered misses, kept in shared memory (one per copy warp or CTA):
// entries filed in each bucket (at most cap) and in the overflow list, and the item numbering of the
// spread schedule -- item i (up to kMissRowsPerItem consecutive entries of one bucket, or of the
// overflow list) -> its first entry and its row count.  load() is called by one whole warp; other
// warps read after a barrier.
struct MissItems {
  int32_t cnt[kMissBuckets];       // entries in each bucket (at most cap)
  int32_t pref[kMissBuckets + 1];  // items before each bucket; pref[kMissBuckets]: all bucket items
  int32_t overflow;                // overflow entries (at most per_group)
  int32_t items;                   // bucket items plus overflow items

  __device__ __forceinline__ void load(const MissOrder& o, int g) {
    const int lane = threadIdx.x & 31;
    const int32_t* c = o.cnt + (int64_t)g * (kMissBuckets + 1);
    int32_t sum = 0;
#pragma unroll 4
    for (int k = 0; k < kBucketsPerLane; ++k) {
      const int32_t x = __ldcg(c + lane * kBucketsPerLane + k);
      const int32_t v = x < o.cap ? x : o.cap;
      cnt[lane * kBucketsPerLane + k] = v;
      sum += (v + kMissRowsPerItem - 1) / kMissRowsPerItem;
    }
    int32_t incl = sum;
#pragma unroll
    for (int d = 1; d < 32; d <<= 1) {
      const int32_t x = __shfl_up_sync(0xffffffffu, incl, d);
      if (lane >= d) incl += x;
    }
    int32_t base = incl - sum;
    for (int k = 0; k < kBucketsPerLane; ++k) {
      pref[lane * kBucketsPerLane + k] = base;
      base += (cnt[lane * kBucketsPerLane + k] + kMissRowsPerItem - 1) / kMissRowsPerItem;
    }
    if (lane == 31) {
      pref[kMissBuckets] = incl;
      const int32_t ov = __ldcg(c + kMissBuckets);
      overflow = ov < o.per_group ? ov : o.per_group;
      items = incl + (overflow + kMissRowsPerItem - 1) / kMissRowsPerItem;
    }
    __syncwarp();
  }
  // Spread schedule, item i < items: its first entry (relative to the group's buckets, or to its
  // overflow list when in_overflow) and its row count.
  __device__ __forceinline__ void locate(const MissOrder& o, int32_t i, int64_t& start, bool& in_overflow,
                                         int& nrows) const {
    const int32_t nb = pref[kMissBuckets];
    int32_t first, count;
    if (i >= nb) {
      first = (i - nb) * kMissRowsPerItem;
      count = overflow - first;
      start = first;
      in_overflow = true;
    } else {
      int lo = 0, hi = kMissBuckets - 1;  // the last bucket b with pref[b] <= i (it has items)
      while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (pref[mid] <= i) lo = mid;
        else hi = mid - 1;
      }
      first = (i - pref[lo]) * kMissRowsPerItem;
      count = cnt[lo] - first;
      start = (int64_t)lo * o.cap + first;
      in_overflow = false;
    }
    nrows = count < kMissRowsPerItem ? count : kMissRowsPerItem;
  }
};

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
