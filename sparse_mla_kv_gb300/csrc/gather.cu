// Single-stride gather of resolved pool rows, and the fused gather that carries the miss copies.
//
// Source: Japanese article (news.ainew.jp), section "仕組み" (How it works): whether a row sits in a
// resident page or in the hot buffer, the resolver hands back pool (HMA) row ids and the rows are
// gathered with one stride; hot pages live in the same KV tensor, so the consumer sees them as
// ordinary pages.  "vLLM GLM 5.3 Optimizations: Hybrid HiSparse Offloading", "Technical
// Implementation of Hybrid HiSparse": a miss copies a single row from pinned host memory.
//
// gather_kernel        HBM-bound byte copy.  The output is a flat array of 16-byte chunks;
//                      consecutive threads take consecutive chunks, so a warp stores 512 contiguous
//                      bytes and reads one or two source rows contiguously.  blockIdx.y selects the
//                      layer; the grid is exactly one resident wave, and each thread keeps
//                      kGatherUnroll loads in flight.
// gather_fused_kernel  the same gather for the rows a resolve plan left in the pool (resident and
//                      hit rows), run by 7 of every 8 warps, while the other warp of each CTA copies
//                      the plan's misses: one read of each host row over the host link, stored into
//                      its hot slot and into every output position of its id.  Host-link and HBM traffic overlap in
//                      one launch, and HBM warps never wait on host latency.  Under IndexShare
//                      the G layers of an index group read the same plan (rows, sources, miss
//                      list); each layer's CTAs copy the misses into that layer's tensor.  With the
//                      ordered miss layout each miss warp takes whole host-row ranges (buckets) and
//                      reads them in address order.
// gather_partition_kernel  the fused gather's SM partition: the CTAs on every sixth SM copy the misses,
//                      the others stream the HBM rows (the default with the range schedule).
// gather_bulk_kernel   the plain gather with one-dimensional bulk copies through shared memory.
// Every gather writes rows, or the planes the pool asks for (hs_pool_set_gather_planes).
#include "hs_internal.cuh"

namespace hs {
namespace {

HS_CHECK_WORD

constexpr unsigned kFull = 0xffffffffu;
constexpr int kGatherThreads = 256;
constexpr int kGatherUnroll = 8;
// Miss warps per CTA of the fused gather when every CTA carries misses: one keeps the host link busy on
// small pools (two were slower on the mixed batch); with the range schedule of large pools the pool may
// ask for two (hs_pool_set_miss_warps) instead of the SM partition.
constexpr int kMaxMissWarps = 2;

template <int CPR, bool kPlanes>
__global__ void __launch_bounds__(kGatherThreads) gather_kernel(const LayerPtrs ptrs, int32_t layer_begin,
                                                                const int32_t* __restrict__ rows, int64_t n,
                                                                uint8_t* __restrict__ out, int32_t row_bytes,
                                                                int64_t num_rows, int32_t* status,
                                                                const OutPlanes pl) {
  const int cpr = CPR ? CPR : (row_bytes >> 4);
  const int lr = blockIdx.y;
  const uint8_t* __restrict__ pool = ptrs.gpu[layer_begin + lr];
  const int32_t* __restrict__ lrows = rows + (int64_t)lr * n;
  uint4* __restrict__ lout = reinterpret_cast<uint4*>(out + (int64_t)lr * n * row_bytes);
  const int64_t total = n * cpr;
  const int64_t stride = (int64_t)gridDim.x * blockDim.x;
  bool bad = false;
  for (int64_t c0 = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; c0 < total; c0 += stride * kGatherUnroll) {
    uint4 v[kGatherUnroll];
#pragma unroll
    for (int k = 0; k < kGatherUnroll; ++k) {
      const int64_t c = c0 + k * stride;
      v[k] = make_uint4(0u, 0u, 0u, 0u);
      if (c < total) {
        const int64_t i = c / cpr;
        const int j = (int)(c - i * cpr);
        const int row = __ldg(lrows + i);
        if (row >= 0 && row < num_rows)
          v[k] = __ldg(reinterpret_cast<const uint4*>(pool + (int64_t)row * row_bytes) + j);
        else if (row != -1)
          bad = true;
      }
    }
#pragma unroll
    for (int k = 0; k < kGatherUnroll; ++k) {
      const int64_t c = c0 + k * stride;
      if (c < total) {
        if constexpr (kPlanes) {
          const int64_t i = c / cpr;
          *plane_chunk(reinterpret_cast<uint8_t*>(lout), pl, n, i, (int)(c - i * cpr)) = v[k];
        } else {
          lout[c] = v[k];
        }
      }
    }
  }
  if (bad && status) *status = HS_ERR_ID_RANGE;
}

// ---- the plain gather with one-dimensional bulk copies (cp.async.bulk), selected per pool by
// hs_pool_set_gather_copy.  Each warp owns kBulkStages row-sized stages of shared memory and one
// mbarrier per stage; lane 0 moves the warp's rows i = w, w + warps, ... from HBM into the stages
// (global -> shared, completing on the stage's mbarrier) kBulkAhead rows ahead, and from each
// completed stage into its output row (shared -> global, one bulk group per row).  A stage is
// reloaded only after the bulk store that read it has finished reading (wait_group.read).  Rows -1
// (and rows outside the pool) are zero-filled by the warp's lanes with ordinary stores.  Every wait
// is bounded: a load that has not completed after kBulkSpinLimit polls sets HS_ERR_TIMEOUT in the
// status word (when given), and the warp stops issuing, waits (bounded again) for the copies it
// has in flight and returns.
constexpr int kBulkThreads = 256;
constexpr int kBulkWarps = kBulkThreads / 32;
constexpr int kBulkStages = 16;
constexpr int kBulkAhead = 12;  // loads in flight per warp; the stores of the other stages drain meanwhile
constexpr uint32_t kBulkSpinLimit = 1u << 22;

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}
__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\tmbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\tselp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0u;
}
// Polls a stage's mbarrier for the phase `parity`; false after kBulkSpinLimit polls.
__device__ __forceinline__ bool mbar_wait_bounded(uint32_t bar, uint32_t parity) {
  for (uint32_t it = 0; it < kBulkSpinLimit; ++it)
    if (mbar_try_wait(bar, parity)) return true;
  return false;
}

__global__ void __launch_bounds__(kBulkThreads) gather_bulk_kernel(const LayerPtrs ptrs, int32_t layer_begin,
                                                                   const int32_t* __restrict__ rows, int64_t n,
                                                                   uint8_t* __restrict__ out, int32_t row_bytes,
                                                                   int64_t num_rows, int32_t* status) {
  extern __shared__ __align__(128) unsigned char bulk_smem[];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int lr = blockIdx.y;
  const uint8_t* __restrict__ pool = ptrs.gpu[layer_begin + lr];
  const int32_t* __restrict__ lrows = rows + (int64_t)lr * n;
  uint8_t* __restrict__ lout = out + (int64_t)lr * n * row_bytes;
  uint64_t* bars = reinterpret_cast<uint64_t*>(bulk_smem) + warp * kBulkStages;
  unsigned char* stages =
      bulk_smem + sizeof(uint64_t) * kBulkStages * kBulkWarps + (size_t)warp * kBulkStages * row_bytes;
  const int64_t gw = (int64_t)blockIdx.x * kBulkWarps + warp;
  const int64_t nw = (int64_t)gridDim.x * kBulkWarps;
  const int64_t cnt = gw < n ? (n - gw + nw - 1) / nw : 0;  // rows of this warp: gw + k * nw, k < cnt
  if (lane == 0) {
    for (int st = 0; st < kBulkStages; ++st)
      asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" ::"r"(smem_u32(bars + st)) : "memory");
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  __syncwarp();
  uint32_t phase = 0u;     // lane 0: parity bit per stage of the next completion to wait for
  uint32_t loaded = 0u;    // lane 0: stages with a load in flight
  bool bad = false, timed_out = false;
  auto row_of = [&](int64_t k) { return __ldg(lrows + gw + k * nw); };
  auto issue = [&](int64_t k) {  // lane 0: the load of the warp's k-th row into its stage
    const int row = row_of(k);
    if (row < 0 || row >= num_rows) return;
    const int st = (int)(k % kBulkStages);
    const uint32_t bar = smem_u32(bars + st);
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(row_bytes) : "memory");
    asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
                     smem_u32(stages + (size_t)st * row_bytes)),
                 "l"(pool + (int64_t)row * row_bytes), "r"(row_bytes), "r"(bar)
                 : "memory");
    loaded |= 1u << st;
  };
  if (lane == 0)
    for (int64_t k = 0; k < cnt && k < kBulkAhead; ++k) issue(k);
  for (int64_t k = 0; k < cnt; ++k) {
    const int row = row_of(k);
    const int64_t i = gw + k * nw;
    if (row >= 0 && row < num_rows) {
      if (lane == 0 && !timed_out) {
        const int st = (int)(k % kBulkStages);
        if (mbar_wait_bounded(smem_u32(bars + st), (phase >> st) & 1u)) {
          phase ^= 1u << st;
          loaded &= ~(1u << st);
          asm volatile("cp.async.bulk.global.shared::cta.bulk_group [%0], [%1], %2;" ::"l"(lout + i * row_bytes),
                       "r"(smem_u32(stages + (size_t)st * row_bytes)), "r"(row_bytes)
                       : "memory");
        } else {
          timed_out = true;
        }
      }
    } else {
      if (row != -1) bad = true;
      uint4* dst = reinterpret_cast<uint4*>(lout + i * row_bytes);
      for (int c = lane; c < (row_bytes >> 4); c += 32) dst[c] = make_uint4(0u, 0u, 0u, 0u);
    }
    if (lane == 0 && !timed_out) {
      asm volatile("cp.async.bulk.commit_group;" ::: "memory");  // one group per row (empty for zero rows)
      const int64_t kk = k + kBulkAhead;
      if (kk < cnt) {
        // the stage of row kk last served row kk - kBulkStages, whose store group was committed
        // kBulkStages - kBulkAhead groups ago: it must have finished reading the stage
        asm volatile("cp.async.bulk.wait_group.read %0;" ::"n"(kBulkStages - kBulkAhead) : "memory");
        issue(kk);
      }
    }
    if (__shfl_sync(0xffffffffu, (int)timed_out, 0)) break;
  }
  timed_out = __shfl_sync(0xffffffffu, (int)timed_out, 0) != 0;
  if (lane == 0) {
    if (timed_out) {
      // bounded drain of the loads still in flight, so that no copy lands in shared memory after exit
      for (int st = 0; st < kBulkStages; ++st)
        if (loaded & (1u << st)) mbar_wait_bounded(smem_u32(bars + st), (phase >> st) & 1u);
      if (status) *status = HS_ERR_TIMEOUT;
    }
    asm volatile("cp.async.bulk.wait_group 0;" ::: "memory");
  }
  if (bad && status && !timed_out) *status = HS_ERR_ID_RANGE;
}

constexpr int kRepeatRegs = 3;  // repeat positions per entry followed before the stores (P - 1 for MTP3)

// Where the miss copies write a layer's output.  The row-size-specialised kernels (CPR > 0) write rows
// only and carry just the base; the generic kernels (CPR = 0) carry the layout, rows or planes (the
// launchers send plane layouts to the generic kernels).
// at(i, b, row_bytes): the 16 bytes at byte b (a multiple of 16) of position i's row.
template <int CPR>
struct MissOut {
  uint8_t* base;
  __device__ __forceinline__ uint4* at(int64_t i, int64_t b, int row_bytes) const {
    return reinterpret_cast<uint4*>(base + i * row_bytes + b);
  }
};
template <>
struct MissOut<0> {
  OutMap om;
  __device__ __forceinline__ uint4* at(int64_t i, int64_t b, int) const { return out_chunk(om, i, (int)(b >> 4)); }
};
template <int CPR>
__device__ __forceinline__ MissOut<CPR> miss_out(uint8_t* base, int64_t rows, int row_bytes, const OutPlanes& pl) {
  if constexpr (CPR > 0) return MissOut<CPR>{base};
  else return MissOut<0>{OutMap{base, rows, row_bytes, pl}};
}

// Copies the rows of up to kMissRowsPerItem miss entries (lane j < nrows holds entry j) from the
// host pool into their hot slots, their output positions and the output positions of their repeats
// (the chain that starts at the entry's fourth field and continues through lmsrc, the plan's
// per-position sources).  The host loads are issued first; the first kRepeatRegs links of each chain
// are read while they are in flight, then everything is stored.  n: positions per request.
template <int CPR>
__device__ __forceinline__ void copy_miss_item(const uint8_t* __restrict__ host, uint8_t* __restrict__ pool,
                                               const MissOut<CPR>& om, const int32_t* __restrict__ lmsrc,
                                               int n, int4 ent, int nrows, int row_bytes, int64_t per_layer,
                                               int64_t gpu_rows, int64_t host_rows) {
  constexpr int kU = CPR ? (kMissRowsPerItem * CPR + 31) / 32 : 4;
  const int cpr = CPR ? CPR : (row_bytes >> 4);
  const int lane = threadIdx.x & 31;
  const int total = nrows * cpr;
  // checked build: an entry whose host row, pool row or output position lies outside its buffer is
  // skipped (lanes past nrows hold no entry)
  const int ok = lane >= nrows || (HS_CHECK(ent.x >= 0 && ent.x < host_rows, kChkHostRow) &&
                                   HS_CHECK(ent.y >= 0 && ent.y < gpu_rows, kChkPoolRow) &&
                                   HS_CHECK(ent.z >= 0 && ent.z < per_layer, kChkOutPos));
  (void)ok;
  (void)per_layer;
  (void)gpu_rows;
  (void)host_rows;
  const int rq = lane < nrows && ok ? ent.z / n : 0;  // the entry's request
  for (int f0 = 0; f0 < total; f0 += 32 * kU) {
    uint4 v[kU];
#pragma unroll
    for (int k = 0; k < kU; ++k) {
      const int f = f0 + k * 32 + lane;
      const int rr = f < total ? f / cpr : 0;
      const int src = __shfl_sync(kFull, ent.x, rr);
      const bool row_ok = HS_CHECKED ? __shfl_sync(kFull, ok, rr) != 0 : true;
      if (f < total && row_ok)
        v[k] = __ldcg(reinterpret_cast<const uint4*>(host + (int64_t)src * row_bytes) + (f - rr * cpr));
    }
    int d = lane < nrows && ok ? ent.w : -1;
    int rep[kRepeatRegs];
#pragma unroll
    for (int t = 0; t < kRepeatRegs; ++t) {
      if (d >= 0 && !HS_CHECK(d < n, kChkChain)) d = -1;
      rep[t] = d;
      if (d >= 0) d = -3 - __ldcg(lmsrc + (int64_t)rq * n + d);
    }
#pragma unroll
    for (int k = 0; k < kU; ++k) {
      const int f = f0 + k * 32 + lane;
      const bool in = f < total;
      const int rr = in ? f / cpr : 0;
      const int64_t cc16 = (int64_t)(f - rr * cpr) * 16;
      const int dst = __shfl_sync(kFull, ent.y, rr);
      const int pos = __shfl_sync(kFull, ent.z, rr);
      const int q = __shfl_sync(kFull, rq, rr);
      int rp[kRepeatRegs];
#pragma unroll
      for (int t = 0; t < kRepeatRegs; ++t) rp[t] = __shfl_sync(kFull, rep[t], rr);
      const bool row_ok = HS_CHECKED ? __shfl_sync(kFull, ok, rr) != 0 : true;
      if (in && row_ok) {
        *reinterpret_cast<uint4*>(pool + (int64_t)dst * row_bytes + cc16) = v[k];
        *om.at(pos, cc16, row_bytes) = v[k];
#pragma unroll
        for (int t = 0; t < kRepeatRegs; ++t)
          if (rp[t] >= 0) *om.at((int64_t)q * n + rp[t], cc16, row_bytes) = v[k];
      }
    }
    if (d >= 0 && !HS_CHECK(d < n, kChkChain)) d = -1;
    while (__any_sync(kFull, d >= 0)) {  // longer chains: one link per round
#pragma unroll
      for (int k = 0; k < kU; ++k) {
        const int f = f0 + k * 32 + lane;
        const int rr = f < total ? f / cpr : 0;
        const int q = __shfl_sync(kFull, rq, rr);
        const int dd = __shfl_sync(kFull, d, rr);
        if (f < total && dd >= 0)
          *om.at((int64_t)q * n + dd, (int64_t)(f - rr * cpr) * 16, row_bytes) = v[k];
      }
      if (d >= 0) d = -3 - __ldcg(lmsrc + (int64_t)rq * n + d);
      if (d >= 0 && !HS_CHECK(d < n, kChkChain)) d = -1;
    }
  }
}

// The miss warps of the fused gather (the CTA's first warps), outside the kernel body (not inlined) so
// that their registers do not add to the HBM warps' streaming loop.
//
// Range schedule (ordered layout on large host pools): the layer's nmw miss warps split its group's
// buckets into contiguous blocks -- warp w takes buckets [w * kMissBuckets / nmw, (w + 1) * kMissBuckets
// / nmw), a range of the host pool -- and copies their entries in 4-entry items as filed, then one
// slice of the overflow list.  Every warp thus reads its own range of the pool.  Measured on the
// full-size MTP3 miss pattern (4 pools of 18 GB, 94.5K misses each) with a standalone read: 134 GB/s
// with 304 warps per pool reading contiguous blocks of 17.6 MB buckets, against 113 GB/s with 152
// warps, 85-120 GB/s fully address-sorted, and 39 GB/s in random order; rows staged in shared memory
// with cp.async were no faster than rows held in registers.
template <int CPR>
__device__ __noinline__ void miss_warp_ranges(const MissOrder ord, int pu, int mw, int nmw,
                                              const uint8_t* __restrict__ host, uint8_t* __restrict__ pool,
                                              const MissOut<CPR> om, const int32_t* __restrict__ lmsrc, int n,
                                              int row_bytes, int64_t per_layer, int64_t num_rows,
                                              int64_t num_host_rows) {
  const int lane = threadIdx.x & 31;
  const int32_t* cntg = ord.cnt + (int64_t)pu * (kMissBuckets + 1);  // counts read from L2 where needed
  const int4* bk = ord.buckets + (int64_t)pu * kMissBuckets * ord.cap;
  const int b0 = (int)((int64_t)mw * kMissBuckets / nmw), b1 = (int)((int64_t)(mw + 1) * kMissBuckets / nmw);
  for (int b = b0; b < b1; ++b) {
    const int nb = min(__ldcg(cntg + b), ord.cap);
    const int4* src = bk + (int64_t)b * ord.cap;
    for (int i = 0; i < nb; i += kMissRowsPerItem) {
      const int nrows = min(kMissRowsPerItem, nb - i);
      const int4 ent = lane < nrows ? src[i + lane] : make_int4(0, 0, 0, 0);
      copy_miss_item<CPR>(host, pool, om, lmsrc, n, ent, nrows, row_bytes, per_layer, num_rows, num_host_rows);
    }
  }
  const int ovn = min(__ldcg(cntg + kMissBuckets), ord.per_group);
  const int ov_per = (ovn + nmw - 1) / nmw;
  const int o0 = mw * ov_per, o1 = min(ovn, o0 + ov_per);
  const int4* ovl = ord.overflow + (int64_t)pu * ord.per_group;
  for (int i = o0; i < o1; i += kMissRowsPerItem) {
    const int nrows = min(kMissRowsPerItem, o1 - i);
    const int4 ent = lane < nrows ? ovl[i + lane] : make_int4(0, 0, 0, 0);
    copy_miss_item<CPR>(host, pool, om, lmsrc, n, ent, nrows, row_bytes, per_layer, num_rows, num_host_rows);
  }
}

// ---- SM partition (the default with the range schedule, on large host pools; optional with per-unit
// lists).  Host reads and HBM rows slow each other down when warps of both kinds share an SM, and the host
// reads are bound by the device's translation of host addresses, which favours fewer host ranges in flight
// at a time.  So the CTAs on every kMissSmDivisor-th SM (by %smid) copy misses with all their warps, one
// work unit per warp at a time (a bucket of the range schedule, in address order, or a chunk of a unit's
// miss list), layer after layer, while the CTAs on the other SMs stream the HBM rows.  Work comes from
// counters shared by every layer of the launch: one of miss units and one of HBM chunks.  A miss CTA
// that finds no miss work left joins the HBM rows; an HBM CTA joins the misses only if no CTA has
// registered as a miss CTA, so the misses are always drained, whichever SMs the CTAs land on.
//
// Measured on the full-size MTP3 batch (4 layers over 18 GB host pools each, 378K misses and 8.4M HBM
// rows per step; medians of 20 replays of one planned gather in one process): one miss warp in every CTA
// 3.20-3.32 ms, this layout 2.60-2.66 ms; every fifth, sixth, seventh or eighth SM for the misses 2.83,
// 2.77, 2.79 and 2.86 ms.  In instrumented copies: buckets handed out over all layers at once 2.83 ms
// (against 2.68), across 64 stripes of every pool 2.9-3.9 ms, a bucket split between 4 or 8 warps 3.8-4.0
// ms, the HBM CTAs' first warp joining the misses 2.82 ms.  Its own timestamps put the end of the HBM rows
// at 2.04 ms and the end of the misses at 2.76 ms: the misses set the time.
constexpr int kMissSmDivisor = 6;
constexpr int kOvUnit = 64;          // overflow entries per work unit
constexpr int kListChunk = 16;       // per-unit lists: misses per work unit
constexpr int kHbmChunk = 8192;      // 16-byte output chunks per HBM work unit (128 KB)

// What the partition's miss warps copy: the range schedule's buckets (ord.cnt set), else the resolver's
// per-unit miss lists; and the work counters.
struct PartitionWork {
  MissOrder ord;
  const int32_t* miss_count;  // per-unit lists: misses of each (index group, request) unit
  const int4* miss_list;      // [units][max_m] entries
  int32_t max_m;
  int32_t* queues;            // kQueueInts counters: miss units, finished CTAs, HBM chunks, miss CTAs
  unsigned long long* phase_ts;  // optional (hs_pool_set_phase_timestamps): start, HBM rows done, misses done, end
};

__device__ __forceinline__ unsigned long long global_ns() {
  unsigned long long t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

__device__ __forceinline__ unsigned sm_id() {
  unsigned r;
  asm volatile("mov.u32 %0, %%smid;" : "=r"(r));
  return r;
}

// Miss work units per layer: kMissBuckets buckets, then as many overflow slices of kOvUnit entries as
// the fullest group's overflow list needs.
__device__ __forceinline__ int partition_layer_units(const MissOrder& ord, int nl, int group) {
  int ov_units = 0;
  for (int pu = 0; pu * group < nl; ++pu) {
    const int ovn = min(__ldcg(ord.cnt + (int64_t)pu * (kMissBuckets + 1) + kMissBuckets), ord.per_group);
    ov_units = max(ov_units, (ovn + kOvUnit - 1) / kOvUnit);
  }
  return kMissBuckets + ov_units;
}

// The entries of range-schedule unit i of group pu: bucket i (address order), or overflow slice
// i - kMissBuckets, as src[0, nb).
__device__ __forceinline__ void partition_unit_range(const MissOrder& ord, int i, int pu, const int4*& src, int& nb) {
  const int32_t* cntg = ord.cnt + (int64_t)pu * (kMissBuckets + 1);
  if (i < kMissBuckets) {
    nb = min(__ldcg(cntg + i), ord.cap);
    src = ord.buckets + ((int64_t)pu * kMissBuckets + i) * ord.cap;
  } else {
    const int o0 = (i - kMissBuckets) * kOvUnit;
    nb = max(0, min(kOvUnit, min(__ldcg(cntg + kMissBuckets), ord.per_group) - o0));
    src = ord.overflow + (int64_t)pu * ord.per_group + o0;
  }
}

// The whole CTA: HBM chunks until the queue is empty.  Chunk unit c covers 16-byte output chunks
// [(c / nl) * kHbmChunk, ...) of layer c % nl; every position the miss warps do not own is written.
template <int CPR, bool kPlanes>
__device__ __forceinline__ bool partition_hbm(const LayerPtrs& ptrs, int32_t layer_begin, int32_t group, int nl,
                                              int32_t* queues, const int32_t* __restrict__ msrc,
                                              uint8_t* __restrict__ out, int64_t per_layer, int row_bytes,
                                              int64_t num_rows, const OutPlanes& pl) {
  const int cpr = CPR ? CPR : (row_bytes >> 4);
  const int64_t total = per_layer * cpr;  // 16-byte chunks per layer
  const int64_t units = (total + kHbmChunk - 1) / kHbmChunk * nl;
  __shared__ int64_t s_unit;
  bool worked = false;
  for (;;) {
    __syncthreads();  // every thread has read the previous unit
    if (threadIdx.x == 0) s_unit = (int64_t)atomicAdd(reinterpret_cast<unsigned int*>(queues + 2), 1u);
    __syncthreads();
    const int64_t c = s_unit;
    if (c >= units) break;
    worked = true;
    const int l = (int)(c % nl);
    const int64_t c0 = (c / nl) * kHbmChunk, c1 = min(total, c0 + kHbmChunk);
    const uint8_t* __restrict__ pool = ptrs.gpu[layer_begin + l];
    uint4* __restrict__ lout4 = reinterpret_cast<uint4*>(out + (int64_t)l * per_layer * row_bytes);
    const int32_t* __restrict__ lmsrc = msrc + (int64_t)(l / group) * per_layer;
    for (int64_t cb = c0 + threadIdx.x; cb < c1; cb += (int64_t)kGatherThreads * kGatherUnroll) {
      uint4 v[kGatherUnroll];
      bool st[kGatherUnroll];
#pragma unroll
      for (int k = 0; k < kGatherUnroll; ++k) {
        const int64_t cc = cb + (int64_t)k * kGatherThreads;
        v[k] = make_uint4(0u, 0u, 0u, 0u);
        st[k] = false;
        if (cc < c1) {
          const int64_t i = cc / cpr;
          const int j = (int)(cc - i * cpr);
          const int ms = __ldg(lmsrc + i);
          if (ms >= 0) {
            if (ms < num_rows) v[k] = __ldg(reinterpret_cast<const uint4*>(pool + (int64_t)ms * row_bytes) + j);
            st[k] = true;
          } else if (ms == -1) {
            st[k] = true;
          }
        }
      }
#pragma unroll
      for (int k = 0; k < kGatherUnroll; ++k) {
        if (!st[k]) continue;
        const int64_t cc = cb + (int64_t)k * kGatherThreads;
        if constexpr (kPlanes) {
          const int64_t i = cc / cpr;
          *plane_chunk(reinterpret_cast<uint8_t*>(lout4), pl, per_layer, i, (int)(cc - i * cpr)) = v[k];
        } else {
          lout4[cc] = v[k];
        }
      }
    }
  }
  return worked;
}

// A warp's share of the miss units: it takes units until the counter passes the end, layer after layer.
// Range schedule: unit u is unit u % upl (a bucket, then an overflow slice) of layer u / upl.  Per-unit
// lists: the units of a layer are chunks of kListChunk misses of its group's lists, chunk-major (chunk
// c of request r is unit c * R + r), up to the most misses any list of the call holds.
template <int CPR>
__device__ __forceinline__ void partition_misses(const LayerPtrs& ptrs, int32_t layer_begin, int32_t group, int nl,
                                                 int R, const PartitionWork& pw, const int32_t* __restrict__ msrc,
                                                 uint8_t* __restrict__ out, int n, int64_t per_layer, int row_bytes,
                                                 int64_t num_rows, int64_t num_host_rows, const OutPlanes& pl) {
  const int lane = threadIdx.x & 31;
  const bool lists = pw.ord.cnt == nullptr;
  int upl;
  if (lists) {
    int m = 0;
    const int ngroups = (nl + group - 1) / group;
    for (int k = lane; k < ngroups * R; k += 32) m = max(m, __ldcg(pw.miss_count + k));
    m = min(__reduce_max_sync(kFull, m), pw.max_m);
    upl = R * ((m + kListChunk - 1) / kListChunk);
  } else {
    upl = partition_layer_units(pw.ord, nl, group);
  }
  const int units = nl * upl;
  for (;;) {
    int u = 0;
    if (lane == 0) u = atomicAdd(pw.queues, 1);
    u = __shfl_sync(kFull, u, 0);
    if (u >= units) break;
    const int l = u / upl, pu = l / group, i = u - l * upl;
    // the unit's entries: src[0, nb)
    const int4* src;
    int nb;
    if (lists) {
      const int c = i / R, r = i - c * R;
      const int cnt = min(__ldcg(pw.miss_count + (int64_t)pu * R + r), pw.max_m);
      const int j0 = c * kListChunk;
      nb = max(0, min(kListChunk, cnt - j0));
      src = pw.miss_list + ((int64_t)pu * R + r) * pw.max_m + j0;
    } else {
      partition_unit_range(pw.ord, i, pu, src, nb);
    }
    const MissOut<CPR> om = miss_out<CPR>(out + (int64_t)l * per_layer * row_bytes, per_layer, row_bytes, pl);
    const int32_t* lmsrc = msrc + (int64_t)pu * per_layer;
    for (int j = 0; j < nb; j += kMissRowsPerItem) {
      const int nrows = min(kMissRowsPerItem, nb - j);
      const int4 ent = lane < nrows ? src[j + lane] : make_int4(0, 0, 0, 0);
      copy_miss_item<CPR>(ptrs.host[layer_begin + l], ptrs.gpu[layer_begin + l], om, lmsrc, n, ent, nrows, row_bytes,
                          per_layer, num_rows, num_host_rows);
    }
  }
}

// Spread schedule (ordered layout on smaller host pools): the layer's miss warps take its group's
// 4-entry items in bucket order (warp w: items w, w + nmw, ...), so that all copy warps work on
// neighbouring host ranges at once and every warp has an item in flight.
template <int CPR>
__device__ __noinline__ void miss_warp_spread(const MissOrder ord, int pu, int mw, int nmw,
                                              const uint8_t* __restrict__ host, uint8_t* __restrict__ pool,
                                              const MissOut<CPR> om, const int32_t* __restrict__ lmsrc, int n,
                                              int row_bytes, int64_t per_layer, int64_t num_rows,
                                              int64_t num_host_rows, MissItems& mi) {
  const int lane = threadIdx.x & 31;
  mi.load(ord, pu);
  const int4* bk = ord.buckets + (int64_t)pu * kMissBuckets * ord.cap;
  const int4* ovl = ord.overflow + (int64_t)pu * ord.per_group;
  for (int32_t i = mw; i < mi.items; i += nmw) {
    int64_t start;
    bool in_ov;
    int nrows;
    mi.locate(ord, i, start, in_ov, nrows);
    int4 ent = make_int4(0, 0, 0, 0);
    if (lane < nrows) ent = (in_ov ? ovl : bk)[start + lane];
    copy_miss_item<CPR>(host, pool, om, lmsrc, n, ent, nrows, row_bytes, per_layer, num_rows, num_host_rows);
  }
}

// Per-unit lists: items (request, chunk of kMissRowsPerItem misses) of this layer, numbered chunk-major
// so live items are the low numbers; lane j of miss-warp w tests item w + j * nmw.
template <int CPR>
__device__ __noinline__ void miss_warp_lists(const int32_t* __restrict__ miss_count, const int4* __restrict__ miss_list,
                                             int pu, int R, int max_m, int64_t mw, int64_t nmw,
                                             const uint8_t* __restrict__ host, uint8_t* __restrict__ pool,
                                             const MissOut<CPR> om, const int32_t* __restrict__ lmsrc, int n,
                                             int row_bytes, int64_t per_layer, int64_t num_rows,
                                             int64_t num_host_rows) {
  const int lane = threadIdx.x & 31;
  const int items_per_unit = (max_m + kMissRowsPerItem - 1) / kMissRowsPerItem;
  const int64_t items = (int64_t)R * items_per_unit;
  for (int64_t base = mw; base < items; base += nmw * 32) {
    const int64_t item = base + (int64_t)lane * nmw;
    int r = 0, chunk = 0, cnt = 0;
    bool live = false;
    if (item < items) {
      chunk = (int)(item / R);
      r = (int)(item - (int64_t)chunk * R);
      cnt = miss_count[pu * R + r];
      live = chunk * kMissRowsPerItem < cnt;
    }
    uint32_t todo = __ballot_sync(kFull, live);
    while (todo) {
      const int src_lane = __ffs(todo) - 1;
      todo &= todo - 1u;
      const int rq = __shfl_sync(kFull, r, src_lane);
      const int ch = __shfl_sync(kFull, chunk, src_lane);
      const int c = __shfl_sync(kFull, cnt, src_lane);
      const int r0 = ch * kMissRowsPerItem;
      const int nrows = min(kMissRowsPerItem, c - r0);
      int4 ent = make_int4(0, 0, 0, 0);
      if (lane < nrows) ent = miss_list[((int64_t)pu * R + rq) * max_m + r0 + lane];
      copy_miss_item<CPR>(host, pool, om, lmsrc, n, ent, nrows, row_bytes, per_layer, num_rows, num_host_rows);
    }
  }
}

// The fused gather with the range schedule's SM partition (see partition_misses): the same outputs as
// gather_fused_kernel, in a kernel of its own so that neither layout's registers constrain the other's.
// The CTAs on SMs whose %smid is a multiple of miss_sm_div (kMissSmDivisor unless the pool sets another)
// copy the misses; miss_sm_div = 0 names no miss SM, so every CTA streams HBM rows first and then takes
// misses (the path a launch whose CTAs miss every miss SM takes).
template <int CPR, bool kPlanes>
__global__ void __launch_bounds__(kGatherThreads, 4) gather_partition_kernel(
    const LayerPtrs ptrs, int32_t layer_begin, int32_t group, int32_t R, int32_t n, const PartitionWork pw,
    const int32_t* __restrict__ msrc, uint8_t* __restrict__ out, int32_t row_bytes, int64_t num_rows,
    int64_t num_host_rows, int miss_sm_div, const OutPlanes pl) {
  pdl_wait_prerequisites();   // per-unit lists: launched early, the plan must be complete and visible
  const int nl = gridDim.y;
  const int64_t per_layer = (int64_t)R * n;
  // CTAs on a miss SM register, copy misses, then help with the HBM rows; the others stream HBM rows and
  // take misses only when no miss CTA has registered (queues[3] counts them)
  const bool miss_sm = miss_sm_div > 0 && sm_id() % (unsigned)miss_sm_div == 0;
  if (pw.phase_ts && threadIdx.x == 0) atomicMin(pw.phase_ts, global_ns());
  if (miss_sm) {
    if (threadIdx.x == 0) atomicAdd(pw.queues + 3, 1);
    partition_misses<CPR>(ptrs, layer_begin, group, nl, R, pw, msrc, out, n, per_layer, row_bytes, num_rows,
                          num_host_rows, pl);
    if (pw.phase_ts && (threadIdx.x & 31) == 0) atomicMax(pw.phase_ts + 2, global_ns());
  }
  const bool hbm = partition_hbm<CPR, kPlanes>(ptrs, layer_begin, group, nl, pw.queues, msrc, out, per_layer,
                                               row_bytes, num_rows, pl);
  if (pw.phase_ts && hbm && threadIdx.x == 0) atomicMax(pw.phase_ts + 1, global_ns());
  if (!miss_sm) {
    int no_miss_cta = 0;  // decided once per warp: the miss loop below is warp-synchronous
    if ((threadIdx.x & 31) == 0) no_miss_cta = *reinterpret_cast<volatile int32_t*>(pw.queues + 3) == 0;
    if (__shfl_sync(kFull, no_miss_cta, 0)) {
      partition_misses<CPR>(ptrs, layer_begin, group, nl, R, pw, msrc, out, n, per_layer, row_bytes, num_rows,
                            num_host_rows, pl);
      if (pw.phase_ts && (threadIdx.x & 31) == 0) atomicMax(pw.phase_ts + 2, global_ns());
    }
  }
  // the last CTA to finish zeroes the counters, so that the next launch on this workspace (a replay of
  // the same plan) starts from zero; every other CTA is done with them when it counts itself finished
  __syncthreads();
  if (threadIdx.x == 0) {
    if (pw.phase_ts) atomicMax(pw.phase_ts + 3, global_ns());
    __threadfence();
    if (atomicAdd(pw.queues + 1, 1) == (int)(gridDim.x * gridDim.y) - 1) {
      pw.queues[0] = 0;
      pw.queues[2] = 0;
      pw.queues[3] = 0;
      __threadfence();
      pw.queues[1] = 0;
    }
  }
}

template <int CPR, bool kPlanes>
__global__ void __launch_bounds__(kGatherThreads, 4) gather_fused_kernel(
    const LayerPtrs ptrs, int32_t layer_begin, int32_t group, int32_t R, int32_t n, int32_t max_m,
    const int32_t* __restrict__ rows, const int32_t* __restrict__ miss_count, const int4* __restrict__ miss_list,
    const MissOrder ord, const int32_t* __restrict__ msrc, uint8_t* __restrict__ out, int32_t row_bytes,
    int64_t num_rows, int64_t num_host_rows, int32_t nmiss, const OutPlanes pl) {
  pdl_wait_prerequisites();   // the resolve plan (rows, sources, miss lists) must be complete and visible
  const int cpr = CPR ? CPR : (row_bytes >> 4);
  const int lr = blockIdx.y;
  const int pu = lr / group;  // the index group (plan) this layer reads
  const int warp = threadIdx.x >> 5;
  uint8_t* __restrict__ pool = ptrs.gpu[layer_begin + lr];
  const uint8_t* __restrict__ host = ptrs.host[layer_begin + lr];
  const int64_t per_layer = (int64_t)R * n;
  uint8_t* __restrict__ lout = out + (int64_t)lr * per_layer * row_bytes;
  const MissOut<CPR> om = miss_out<CPR>(lout, per_layer, row_bytes, pl);
  const int32_t* __restrict__ lmsrc = msrc + (int64_t)pu * per_layer;

  if (warp < nmiss) {
    // CTA-major numbering: consecutive buckets (or items) go to different CTAs, spread over the SMs
    const int64_t mw = (int64_t)warp * gridDim.x + blockIdx.x;
    const int64_t nmw = (int64_t)gridDim.x * nmiss;
    __shared__ MissItems s_mi;  // spread schedule (one miss warp)
    if (ord.cnt && !ord.ranges)
      miss_warp_spread<CPR>(ord, pu, (int)mw, (int)nmw, host, pool, om, lmsrc, n, row_bytes, per_layer, num_rows,
                            num_host_rows, s_mi);
    else if (ord.cnt)
      miss_warp_ranges<CPR>(ord, pu, (int)mw, (int)nmw, host, pool, om, lmsrc, n, row_bytes, per_layer, num_rows,
                            num_host_rows);
    else
      miss_warp_lists<CPR>(miss_count, miss_list, pu, R, max_m, mw, nmw, host, pool, om, lmsrc, n, row_bytes,
                           per_layer, num_rows, num_host_rows);
    return;
  }

  // ---- HBM warps: every position the miss warps do not own (resident rows, hit rows, padding);
  // one source word per position
  const int hbm_threads = kGatherThreads - nmiss * 32;
  uint4* __restrict__ lout4 = reinterpret_cast<uint4*>(lout);
  const int64_t total = per_layer * cpr;
  const int64_t stride = (int64_t)gridDim.x * hbm_threads;
  for (int64_t c0 = (int64_t)blockIdx.x * hbm_threads + (threadIdx.x - nmiss * 32); c0 < total;
       c0 += stride * kGatherUnroll) {
    uint4 v[kGatherUnroll];
    bool st[kGatherUnroll];
#pragma unroll
    for (int k = 0; k < kGatherUnroll; ++k) {
      const int64_t c = c0 + k * stride;
      v[k] = make_uint4(0u, 0u, 0u, 0u);
      st[k] = false;
      if (c < total) {
        const int64_t i = c / cpr;
        const int j = (int)(c - i * cpr);
        const int ms = __ldg(lmsrc + i);
        if (ms >= 0) {
          if (ms < num_rows) v[k] = __ldg(reinterpret_cast<const uint4*>(pool + (int64_t)ms * row_bytes) + j);
          st[k] = true;
        } else if (ms == -1) {
          st[k] = true;
        }  // <= -2: a missed id's position, stored by the miss warps
      }
    }
#pragma unroll
    for (int k = 0; k < kGatherUnroll; ++k) {
      if (!st[k]) continue;
      const int64_t c = c0 + k * stride;
      if constexpr (kPlanes) {
        const int64_t i = c / cpr;
        *plane_chunk(lout, pl, per_layer, i, (int)(c - i * cpr)) = v[k];
      } else {
        lout4[c] = v[k];
      }
    }
  }
}

// resident CTAs per SM of each kernel: [0] 656-byte rows, [1] any row size, [2] any row size in planes
int g_occ_plain[3] = {0, 0, 0};
int g_occ_fused[3] = {0, 0, 0};
int g_occ_partition[3] = {0, 0, 0};
int g_occ_bulk = 0;          // resident bulk-gather CTAs per SM for the 656-byte rows' footprint
size_t g_bulk_smem_max = 0;  // dynamic shared memory the bulk gather may use (the opt-in maximum)

size_t bulk_smem_bytes(int32_t row_bytes) {
  return sizeof(uint64_t) * kBulkStages * kBulkWarps + (size_t)kBulkStages * kBulkWarps * (size_t)row_bytes;
}

template <typename Kern>
int resident_blocks(Kern kern, int* cache, size_t smem = 0) {
  if (*cache <= 0 && cudaOccupancyMaxActiveBlocksPerMultiprocessor(cache, kern, kGatherThreads, smem) != cudaSuccess)
    *cache = 2;
  if (*cache <= 0) *cache = 1;
  return *cache;
}

dim3 wave_grid(int sms, int occ, int64_t want, int nl) {
  int64_t cap = ((int64_t)sms * occ) / (nl > 0 ? nl : 1);
  if (cap < 1) cap = 1;
  const int64_t gx = want < cap ? (want > 0 ? want : 1) : cap;
  return dim3((unsigned)gx, (unsigned)nl);
}

}  // namespace

uint32_t check_take_gather() {
#if HS_CHECKED
  unsigned v = 0u, z = 0u;
  if (cudaMemcpyFromSymbol(&v, hs_check_word_, sizeof(v)) != cudaSuccess ||
      cudaMemcpyToSymbol(hs_check_word_, &z, sizeof(z)) != cudaSuccess) {
    cudaGetLastError();
    return 0xFFFFFFFFu;
  }
  return v;
#else
  return 0u;
#endif
}

void warm_gather_launch_configs() {
  resident_blocks(gather_kernel<41, false>, &g_occ_plain[0]);
  resident_blocks(gather_kernel<0, false>, &g_occ_plain[1]);
  resident_blocks(gather_kernel<0, true>, &g_occ_plain[2]);
  resident_blocks(gather_fused_kernel<41, false>, &g_occ_fused[0]);
  resident_blocks(gather_fused_kernel<0, false>, &g_occ_fused[1]);
  resident_blocks(gather_fused_kernel<0, true>, &g_occ_fused[2]);
  resident_blocks(gather_partition_kernel<41, false>, &g_occ_partition[0]);
  resident_blocks(gather_partition_kernel<0, false>, &g_occ_partition[1]);
  resident_blocks(gather_partition_kernel<0, true>, &g_occ_partition[2]);
  if (g_bulk_smem_max == 0) {
    int dev = 0, optin = 0;
    if (cudaGetDevice(&dev) == cudaSuccess &&
        cudaDeviceGetAttribute(&optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev) == cudaSuccess && optin > 0 &&
        cudaFuncSetAttribute(gather_bulk_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, optin) == cudaSuccess) {
      g_bulk_smem_max = (size_t)optin;
      if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&g_occ_bulk, gather_bulk_kernel, kBulkThreads,
                                                        bulk_smem_bytes(656)) != cudaSuccess || g_occ_bulk < 1)
        g_occ_bulk = 1;
    }
    cudaGetLastError();
  }
}

bool gather_bulk_fits(int32_t row_bytes) {
  return g_bulk_smem_max > 0 && bulk_smem_bytes(row_bytes) <= g_bulk_smem_max;
}

cudaError_t launch_gather(const LayerPtrs& ptrs, int32_t layer_begin, int32_t nl, const int32_t* rows, int64_t n,
                          uint8_t* out, int32_t row_bytes, int64_t num_rows, int32_t* status, int sms,
                          cudaStream_t s, bool bulk, const OutPlanes& planes) {
  if (bulk && planes.n == 0 && gather_bulk_fits(row_bytes)) {
    const size_t smem = bulk_smem_bytes(row_bytes);
    const int occ = row_bytes == 656 ? g_occ_bulk : 1;
    const int64_t want = (n + kBulkWarps * kBulkStages - 1) / (kBulkWarps * kBulkStages);
    const dim3 grid = wave_grid(sms, occ, want, nl);
    gather_bulk_kernel<<<grid, kBulkThreads, smem, s>>>(ptrs, layer_begin, rows, n, out, row_bytes, num_rows, status);
    count_launch();
    return cudaGetLastError();
  }
  // kernel variant: 656-byte rows, any row size, any row size in planes
  const int var = planes.n ? 2 : (row_bytes == 656 ? 0 : 1);
  auto kern = var == 0 ? gather_kernel<41, false> : (var == 1 ? gather_kernel<0, false> : gather_kernel<0, true>);
  const int64_t want = (n * (row_bytes >> 4) + (int64_t)kGatherThreads * kGatherUnroll - 1) /
                       ((int64_t)kGatherThreads * kGatherUnroll);
  const dim3 grid = wave_grid(sms, resident_blocks(kern, &g_occ_plain[var]), want, nl);
  kern<<<grid, kGatherThreads, 0, s>>>(ptrs, layer_begin, rows, n, out, row_bytes, num_rows, status, planes);
  count_launch();
  return cudaGetLastError();
}

cudaError_t launch_gather_fused(const LayerPtrs& ptrs, int32_t layer_begin, int32_t nl, int32_t group, int32_t R,
                                int32_t n, int32_t max_m, const int32_t* rows, const int32_t* miss_count,
                                const int4* miss_list, const MissOrder& ord, const int32_t* msrc, uint8_t* out,
                                int32_t row_bytes, int64_t num_rows, int64_t num_host_rows, int range_miss_warps,
                                int miss_sm_div, const OutPlanes& planes, int32_t* queues,
                                unsigned long long* phase_ts, int sms, cudaStream_t s) {
  // kernel variant: 656-byte rows, any row size, any row size in planes
  const int var = planes.n ? 2 : (row_bytes == 656 ? 0 : 1);
  auto kern = var == 0 ? gather_fused_kernel<41, false>
                       : (var == 1 ? gather_fused_kernel<0, false> : gather_fused_kernel<0, true>);
  // the pool's choice (range_miss_warps): -1 (default) the SM partition with the range schedule and one miss
  // warp in every CTA otherwise; 0 the SM partition with the range schedule or per-unit lists; 1 or 2
  // miss warps in every CTA with the range schedule (one with lists: two were slower on the mixed batch).
  // The spread schedule keeps one miss warp in every CTA.
  const bool ranges = ord.cnt && ord.ranges, lists = !ord.cnt;
  const int mw = range_miss_warps;
  const int nmiss = ((ranges && mw <= 0) || (lists && mw == 0)) ? 0 : (ranges && mw >= kMaxMissWarps ? kMaxMissWarps : 1);
  const int64_t per_layer = (int64_t)R * n * (row_bytes >> 4);
  const int64_t want_hbm = (per_layer + (int64_t)kGatherThreads * kGatherUnroll - 1) /
                           ((int64_t)kGatherThreads * kGatherUnroll);
  // enough CTAs that each miss warp can take one item (kMissRowsPerItem misses) of the most a layer can
  // have, so a small batch does not queue its host round trips on a few warps
  const int64_t want_miss =
      ((int64_t)R * ((max_m + kMissRowsPerItem - 1) / kMissRowsPerItem) + nmiss - 1) / (nmiss > 0 ? nmiss : 1);
  const dim3 grid = wave_grid(sms, resident_blocks(kern, &g_occ_fused[var]), want_hbm > want_miss ? want_hbm : want_miss,
                              nl);
  // With the ordered layout (large host pools) the gather is not launched early: CTAs placed while
  // the resolver still runs made the whole gather's host reads slower there (measured: agentic
  // decode over a 29 GB pool, 684 us per step against 333 us with the launch held back).
  cudaError_t e;
  if (nmiss == 0) {
    // SM partition: one full wave; its work counters were zeroed by the resolver (and again by the last
    // CTA of the previous launch on this workspace).  Launched early only with per-unit lists.
    auto pkern = var == 0 ? gather_partition_kernel<41, false>
                          : (var == 1 ? gather_partition_kernel<0, false> : gather_partition_kernel<0, true>);
    const dim3 pgrid = wave_grid(sms, resident_blocks(pkern, &g_occ_partition[var]), (int64_t)1 << 40, nl);
    const PartitionWork pw{ord, miss_count, miss_list, max_m, queues, phase_ts};
    const int div = miss_sm_div >= 2 ? miss_sm_div : (miss_sm_div < 0 ? 0 : kMissSmDivisor);
    if (lists) {
      e = launch_dependent(pkern, pgrid, dim3(kGatherThreads), 0, s, ptrs, layer_begin, group, R, n, pw, msrc, out,
                           row_bytes, num_rows, num_host_rows, div, planes);
    } else {
      pkern<<<pgrid, kGatherThreads, 0, s>>>(ptrs, layer_begin, group, R, n, pw, msrc, out, row_bytes, num_rows,
                                             num_host_rows, div, planes);
      e = cudaGetLastError();
    }
  } else if (ord.cnt) {
    kern<<<grid, kGatherThreads, 0, s>>>(ptrs, layer_begin, group, R, n, max_m, rows, miss_count, miss_list, ord, msrc,
                                         out, row_bytes, num_rows, num_host_rows, nmiss, planes);
    e = cudaGetLastError();
  } else {
    e = launch_dependent(kern, grid, dim3(kGatherThreads), 0, s, ptrs, layer_begin, group, R, n, max_m, rows,
                         miss_count, miss_list, ord, msrc, out, row_bytes, num_rows, num_host_rows, 1, planes);
  }
  if (e != cudaSuccess) return e;
  count_launch();
  return cudaGetLastError();
}

}  // namespace hs
