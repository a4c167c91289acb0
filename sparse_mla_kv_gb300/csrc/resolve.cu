// Fused per-step top-K resolver and the miss-copy kernel.
//
// Source: "vLLM GLM 5.3 Optimizations: Hybrid HiSparse Offloading", section "Technical
// Implementation of Hybrid HiSparse", item 2 (Mixed residency): resident tokens are read in place,
// hot tokens are read and their LRU entry refreshed, a miss copies a single row from pinned host
// memory into an LRU slot.  Japanese article (news.ainew.jp), section "仕組み" (How it works): the
// block table mixes real blocks and null placeholders; the resolver hands back pool row ids; no
// step waits for the CPU (CUDA-graph capturable).  Section "vLLM の他の部分との統合"
// (Integration): speculative decoding uses one replayable per-step plan sharing the hot state.
//
// Design (sm_103a):
//   resolve_kernel   one CTA (1024 threads) per (index group, request) unit.  The unit's slot stamps,
//                    ids and their pages' table entries are staged in shared memory; an
//                    open-addressing hash table (32-bit entries) maps id -> first position, and each
//                    slot's token is looked up in it once, so that every plan entry learns the lowest
//                    slot holding its token (an atomicMin) without a second table over the slots.
//                    The plan, hit/miss classification and the miss ranks come from block-wide scans;
//                    victims are the candidates sorted by (stamp, slot) with a stable LSD radix sort
//                    (8-bit digits, per-warp histograms, __match_any_sync ranking) whose buffers reuse
//                    the hash table's memory.  Misses go to a per-unit list in the caller's
//                    workspace (or, for large host pools, filed by host row range: the ordered
//                    layout).  For the fused gather, the repeated positions of a missed id are
//                    chained so that the row read once serves all of them.  A unit with a data error
//                    writes nothing but -1 rows and its status.
//                    The footprint, 4*C + 13*P*K bytes plus the hash table, fits the pages' MTP sizing
//                    (num_spec + 2) * K = 10240 slots with P*K = 8192 ids in one CTA.
//   miss_copy_kernel a persistent grid spreads every unit's misses over all SMs: each warp takes
//                    batches of 32 (unit, 4-row) items, skips empty ones with one ballot, and copies
//                    the rows as 16-byte zero-copy loads from the mapped pinned host pool, once for
//                    each layer of the unit's index group.  Spreading keeps enough loads in flight on
//                    the host link even when few units miss a lot.  With the ordered layout each
//                    index group gets its own CTAs, whose warps take the group's buckets (host row
//                    ranges) whole, each read in address order.
//   order_clear_kernel zeroes the ordered layout's bucket counters before the resolver, which is its
//                    programmatic dependent and waits for it only where it first needs them.
//
// IndexShare (one indexer per group of G sparse-MLA layers): the group's layers resolve the same ids
// against the same tables at the same step, so one unit per (group, request) decides for all of
// them, and only the byte copies are repeated per layer.
#include <atomic>
#include <climits>

#include "hs_internal.cuh"

namespace hs {
namespace {

HS_CHECK_WORD

constexpr unsigned kFull = 0xffffffffu;
constexpr int kEmpty = -1;
constexpr int kBadHost = INT_MIN;
constexpr int kGatherOwnedByMissWarps = INT_MIN;
constexpr int kNoSlot = INT_MAX;
constexpr int kTokRegs = 4;  // slot tokens and stamps per thread loaded first and held in registers
constexpr int kIdRegs = 2;   // ids per thread loaded first
constexpr int kTblRegs = 2;  // staged block-table / host-table entries per thread loaded first

// A load issued where it is written: the asm statement (with a memory clobber) keeps the compiler from
// sinking it to the value's first use, so a thread's independent loads are all in flight together.
__device__ __forceinline__ int ld_early(const int32_t* ptr) {
  int v;
  asm volatile("ld.global.s32 %0, [%1];" : "=r"(v) : "l"(ptr) : "memory");
  return v;
}
// kNone: padding; kDup: a repeated id (s_val holds its first occurrence's position)
enum : uint8_t { kNone = 0, kResident = 1, kHit = 2, kMiss = 3, kDup = 4 };

__device__ __forceinline__ uint32_t fib_hash(int32_t key, int bits) {
  return ((uint32_t)key * 0x9E3779B1u) >> (32 - bits);
}

// Open addressing with linear probing; an entry is an index e into keys[] (the key is keys[e]).
// Insert e under key k = keys[e]; when the key is already present keep the smallest entry (lowest
// slot / first position).
__device__ __forceinline__ void hash_insert_min(int* tab, int bits, const int32_t* keys, int32_t k, int e) {
  const uint32_t mask = (1u << bits) - 1u;
  uint32_t h = fib_hash(k, bits);
  for (uint32_t it = 0; it <= mask; ++it, h = (h + 1u) & mask) {
    int cur = atomicCAS(&tab[h], kEmpty, e);
    if (cur == kEmpty) return;
    if (keys[cur] == k) {
      atomicMin(&tab[h], e);
      return;
    }
  }
}

__device__ __forceinline__ int hash_find(const int* tab, int bits, const int32_t* keys, int32_t k) {
  const uint32_t mask = (1u << bits) - 1u;
  uint32_t h = fib_hash(k, bits);
  for (uint32_t it = 0; it <= mask; ++it, h = (h + 1u) & mask) {
    const int cur = tab[h];
    if (cur == kEmpty) return -1;
    if (keys[cur] == k) return cur;
  }
  return -1;
}

// The id -> first position table.  Narrow: 32-bit entries holding a position (the key is read from
// the ids array: two dependent shared-memory reads per probe).  Wide: 64-bit entries packing
// (id << 32 | position), one read per probe; since the id is the high half, atomicMin on an entry
// keeps the smallest position of that id.  Wide is used when its shared memory fits.
template <bool kWide>
struct IdHash;

template <>
struct IdHash<false> {
  int* tab;
  int bits;
  const int32_t* keys;
  __device__ void clear() {
    for (int i = threadIdx.x; i < (1 << bits); i += blockDim.x) tab[i] = kEmpty;
  }
  __device__ void insert_min(int32_t k, int e) { hash_insert_min(tab, bits, keys, k, e); }
  __device__ int find(int32_t k) const { return hash_find(tab, bits, keys, k); }
};

template <>
struct IdHash<true> {
  unsigned long long* tab;
  int bits;
  static constexpr unsigned long long kVoid = ~0ull;
  __device__ void clear() {
    for (int i = threadIdx.x; i < (1 << bits); i += blockDim.x) tab[i] = kVoid;
  }
  __device__ void insert_min(int32_t k, int e) {
    const uint32_t mask = (1u << bits) - 1u;
    const unsigned long long packed = ((unsigned long long)(uint32_t)k << 32) | (uint32_t)e;
    uint32_t h = fib_hash(k, bits);
    for (uint32_t it = 0; it <= mask; ++it, h = (h + 1u) & mask) {
      const unsigned long long cur = atomicCAS(&tab[h], kVoid, packed);
      if (cur == kVoid) return;
      if ((uint32_t)(cur >> 32) == (uint32_t)k) {
        atomicMin(&tab[h], packed);
        return;
      }
    }
  }
  __device__ int find(int32_t k) const {
    const uint32_t mask = (1u << bits) - 1u;
    uint32_t h = fib_hash(k, bits);
    for (uint32_t it = 0; it <= mask; ++it, h = (h + 1u) & mask) {
      const unsigned long long cur = tab[h];
      if (cur == kVoid) return -1;
      if ((uint32_t)(cur >> 32) == (uint32_t)k) return (int)(uint32_t)cur;
    }
    return -1;
  }
};

// Exclusive block-wide scan of two ints at once over kW warps.  Contains __syncthreads: call uniformly.
template <int kW>
__device__ __forceinline__ void block_scan2(int a, int b, int& ea, int& eb, int& ta, int& tb, int* s_tmp) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  int ia = a, ib = b;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int xa = __shfl_up_sync(kFull, ia, o);
    const int xb = __shfl_up_sync(kFull, ib, o);
    if (lane >= o) { ia += xa; ib += xb; }
  }
  if (lane == 31) { s_tmp[warp] = ia; s_tmp[kW + warp] = ib; }
  __syncthreads();
  if (warp == 0) {
    int va = lane < kW ? s_tmp[lane] : 0;
    int vb = lane < kW ? s_tmp[kW + lane] : 0;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int xa = __shfl_up_sync(kFull, va, o);
      const int xb = __shfl_up_sync(kFull, vb, o);
      if (lane >= o) { va += xa; vb += xb; }
    }
    if (lane < kW) { s_tmp[lane] = va; s_tmp[kW + lane] = vb; }
  }
  __syncthreads();
  ea = (warp ? s_tmp[warp - 1] : 0) + ia - a;
  eb = (warp ? s_tmp[kW + warp - 1] : 0) + ib - b;
  ta = s_tmp[kW - 1];
  tb = s_tmp[2 * kW - 1];
  __syncthreads();
}

// Stable LSD radix sort of slot ids a[0..nc) by key stamp[slot] - lo over `passes` 8-bit digits.
// kSortWarps warps own contiguous chunks (per-warp histograms keep the scatter stable); all threads
// take part in the histogram scan.  Returns the buffer holding the result (a or b).  Call uniformly
// (contains __syncthreads).
template <int kT>
__device__ unsigned short* radix_sort_slots(unsigned short* a, unsigned short* b, int nc, const int32_t* s_stamp,
                                            int lo, int passes, int* hist, int* s_tmp) {
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int per_warp = (nc + kSortWarps - 1) / kSortWarps;
  const int w0 = warp < kSortWarps ? min(nc, warp * per_warp) : nc;
  const int w1 = warp < kSortWarps ? min(nc, w0 + per_warp) : nc;
  constexpr int kEntries = kRadixBins * kSortWarps;
  constexpr int kPerThread = kEntries / kT;
  static_assert(kEntries % kT == 0, "histogram split");
  for (int pass = 0; pass < passes; ++pass) {
    const int shift = pass * 8;
    for (int i = tid; i < kEntries; i += kT) hist[i] = 0;
    __syncthreads();
    for (int e = w0 + lane; e < w1; e += 32) {
      const uint32_t d = (((uint32_t)s_stamp[a[e]] - (uint32_t)lo) >> shift) & 0xFFu;
      atomicAdd(&hist[d * kSortWarps + warp], 1);
    }
    __syncthreads();
    int loc[kPerThread];
    int sum = 0;
#pragma unroll
    for (int k = 0; k < kPerThread; ++k) { loc[k] = hist[tid * kPerThread + k]; sum += loc[k]; }
    int base, dummy_e, total, dummy_t;
    block_scan2<kT / 32>(sum, 0, base, dummy_e, total, dummy_t, s_tmp);
#pragma unroll
    for (int k = 0; k < kPerThread; ++k) { hist[tid * kPerThread + k] = base; base += loc[k]; }
    __syncthreads();
    for (int e0 = w0; e0 < w1; e0 += 32) {  // warp-uniform trip count
      const int e = e0 + lane;
      const bool valid = e < w1;
      const unsigned short slot = valid ? a[e] : (unsigned short)0;
      const uint32_t d = valid ? ((((uint32_t)s_stamp[slot] - (uint32_t)lo) >> shift) & 0xFFu) : 0u;
      const uint32_t key = valid ? d : (0x100u + (uint32_t)lane);
      const uint32_t peers = __match_any_sync(kFull, key);
      const int rank = __popc(peers & ((1u << lane) - 1u));
      int* ctr = &hist[d * kSortWarps + warp];
      if (valid) b[*ctr + rank] = slot;
      __syncwarp();
      if (valid && rank == 0) *ctr += __popc(peers);
      __syncwarp();
    }
    __syncthreads();
    unsigned short* t = a; a = b; b = t;
  }
  return a;
}

// kS: the page size when it is a compile-time constant (64 in the pages' FP8 MLA setup), else 0.
// kWide: the id table's entry width (see IdHash).  kT: threads per CTA -- 1024, or 512 so that two
// units share an SM when there are more units than SMs or a unit is small.  Results do not depend on it.
// Starts moving a missed row into L2 in every layer of the unit's index group (lr: the group within
// the call), so that the copy that follows finds it there: one bulk prefetch per layer, with no
// completion to wait for.  The row is inside the host pool (its block was checked) and 16-byte aligned.
__device__ __forceinline__ void prefetch_host_row(const ResolveParams& p, int lr, int row) {
  const int l0 = (p.layer_begin + lr) * p.group;
  for (int g = 0; g < p.group; ++g) {
    const uint8_t* a = p.host[l0 + g] + (int64_t)row * p.row_bytes;
    asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(a), "r"(p.row_bytes) : "memory");
  }
}

template <int kS, bool kWide, int kT>
__global__ void __launch_bounds__(kT, kResolveThreads / kT) resolve_kernel(const ResolveParams p, const ResolveSmem sm) {
  extern __shared__ __align__(16) unsigned char smem[];
  int32_t* s_stamp = reinterpret_cast<int32_t*>(smem + sm.stamp);
  int32_t* s_ids = reinterpret_cast<int32_t*>(smem + sm.ids);
  int32_t* s_val = reinterpret_cast<int32_t*>(smem + sm.val);
  uint8_t* s_cls = reinterpret_cast<uint8_t*>(smem + sm.cls);
  int32_t* s_slot = reinterpret_cast<int32_t*>(smem + sm.slot);  // lowest slot holding position i's id

  int32_t* s_hot = reinterpret_cast<int32_t*>(smem + sm.hot);
  // the request's block-table and host-table rows, staged when they are small (sm.tbl_pages > 0)
  const bool staged = sm.tbl_pages > 0;
  int32_t* s_bt = reinterpret_cast<int32_t*>(smem + sm.tbl);
  int32_t* s_hbt = s_bt + sm.tbl_pages;
  __shared__ uint32_t s_err;
  __shared__ int s_cnt[3];
  __shared__ int s_lo, s_hi;
  __shared__ int s_any_dup;  // some plan entry repeats an earlier id
  __shared__ int s_tmp[2 * (kT / 32)];

  const int tid = threadIdx.x, lane = tid & 31;
  pdl_allow_dependents();   // the following gather / miss-copy kernel may place its CTAs now
  const int unit = blockIdx.x;
  const int lr = unit / p.R, r = unit - lr * p.R;
  if (unit == 0 && tid < kQueueInts && p.queues) p.queues[tid] = 0;  // the fused gather's work counters
  const int grp = p.layer_begin + lr;  // index group (a layer when no layers share an indexer)
  const int n = p.n, C = p.C, step = p.step;
  const int S = kS ? kS : p.S;
  const int64_t state_off = ((int64_t)grp * p.R + r) * C;
  const int32_t* ids_g = p.topk + (int64_t)unit * n;
  const int32_t* bt = p.bt + (int64_t)r * p.max_pages;
  const int32_t* hbt = p.hbt + (int64_t)r * p.max_pages;
  const int32_t* hot = p.hot_blocks + (int64_t)r * (C / S);
  int32_t* rows_g = p.out_rows + (int64_t)unit * n;
  int32_t* msrc_g = p.msrc ? p.msrc + (int64_t)unit * n : nullptr;
  const int ctx = p.ctx_len[r];
  IdHash<kWide> idh;
  if constexpr (kWide) {
    idh = IdHash<kWide>{reinterpret_cast<unsigned long long*>(smem + sm.idh), sm.id_hash_bits};
  } else {
    idh = IdHash<kWide>{reinterpret_cast<int*>(smem + sm.idh), sm.id_hash_bits, s_ids};
  }

  // ---- phase 0: every independent load of the unit is issued first (their latencies overlap), then
  // staged in shared memory; checks that need no classification.  With the wide id table the ids are
  // inserted as they are staged (an entry carries its key, so no other position must be staged first).
  if (tid == 0) {
    s_err = 0u;
    s_cnt[0] = s_cnt[1] = s_cnt[2] = 0;
    s_lo = INT_MAX;
    s_hi = INT_MIN;
    s_any_dup = 0;
  }
  const int32_t* tok_g = p.slot_token + state_off;
  const int32_t* stamp_g = p.slot_stamp + state_off;
  int idr[kIdRegs], tokr[kTokRegs], str[kTokRegs], btr[kTblRegs], hbtr[kTblRegs];
#pragma unroll
  for (int k = 0; k < kIdRegs; ++k) {
    const int i = tid + k * kT;
    idr[k] = i < n ? ld_early(ids_g + i) : -1;
  }
#pragma unroll
  for (int k = 0; k < kTokRegs; ++k) {
    const int s = tid + k * kT;
    tokr[k] = s < C ? ld_early(tok_g + s) : -1;
    str[k] = s < C ? ld_early(stamp_g + s) : -1;
  }
#pragma unroll
  for (int k = 0; k < kTblRegs; ++k) {
    const int j = tid + k * kT;
    btr[k] = (staged && j < sm.tbl_pages) ? ld_early(bt + j) : -1;
    hbtr[k] = (staged && j < sm.tbl_pages) ? ld_early(hbt + j) : -1;
  }
  const int hotr = tid < C / S ? ld_early(hot + tid) : 0;
  idh.clear();
  __syncthreads();  // the status words are reset and the table empty before any thread uses them
  uint32_t err = 0u;
  // ids, and (unstaged tables) their page's table entries.  Combined entry in s_val:
  //   e >= 0      resident block e;      e == -1   placeholder without a host copy;
  //   e == kBadHost  placeholder whose host block is outside the pool;  else host block -2 - e.
  auto stage_id = [&](int i, int id) {
    s_ids[i] = id;
    int e = -1;
    if (id != -1) {
      if (id < -1 || id >= ctx || (unsigned)id / S >= (unsigned)p.max_pages) {
        err |= kErrId;
      } else {
        if constexpr (kWide) idh.insert_min(id, i);
        const int page = (unsigned)id / S;
        if (!staged && HS_CHECK((unsigned)page < (unsigned)p.max_pages, kChkTablePage)) {
          const int b = bt[page];
          const int h = hbt[page];
          e = b >= 0 ? b : (h < 0 ? -1 : (h >= p.num_host_blocks ? kBadHost : -2 - h));
        }
      }
    }
    s_val[i] = e;
    s_slot[i] = kNoSlot;
  };
#pragma unroll
  for (int k = 0; k < kIdRegs; ++k) {
    const int i = tid + k * kT;
    if (i < n) stage_id(i, idr[k]);
  }
  for (int i = tid + kIdRegs * kT; i < n; i += kT) stage_id(i, ids_g[i]);
  if (staged) {
#pragma unroll
    for (int k = 0; k < kTblRegs; ++k) {
      const int j = tid + k * kT;
      if (j < sm.tbl_pages) {
        s_bt[j] = btr[k];
        s_hbt[j] = hbtr[k];
      }
    }
    for (int j = tid + kTblRegs * kT; j < sm.tbl_pages; j += kT) {
      s_bt[j] = bt[j];
      s_hbt[j] = hbt[j];
    }
  }
  if (tid < C / S) {
    s_hot[tid] = hotr;
    if (hotr < 0 || hotr >= p.num_gpu_blocks) err |= kErrHot;
  }
  for (int b = tid + kT; b < C / S; b += kT) {
    const int hb = hot[b];
    s_hot[b] = hb;
    if (hb < 0 || hb >= p.num_gpu_blocks) err |= kErrHot;
  }
#pragma unroll
  for (int k = 0; k < kTokRegs; ++k) {
    const int s = tid + k * kT;
    if (s < C) {
      s_stamp[s] = str[k];
      if (str[k] > step) err |= kErrStep;
    }
  }
  for (int s = tid + kTokRegs * kT; s < C; s += kT) {
    const int st = stamp_g[s];
    s_stamp[s] = st;
    if (st > step) err |= kErrStep;
  }
  if (err) atomicOr(&s_err, err);
  __syncthreads();
  const bool early = (s_err & (kErrStep | kErrId)) != 0u;

  // ---- phase 1 (narrow id table only): inserts, once every id is staged (a probe reads other keys)
  if constexpr (!kWide) {
    if (!early) {
      for (int i = tid; i < n; i += kT) {
        const int id = s_ids[i];
        if (id >= 0) idh.insert_min(id, i);
      }
    }
    __syncthreads();
  }

  // ---- phase 1a: each id's table entry (from the staged rows when staged), and whether the unit reads
  // any page that is not resident (or a table entry outside the pool): one barrier with an OR decides
  // for the whole unit.
  bool other = false;
  if (!early) {
    for (int i = tid; i < n; i += kT) {
      const int id = s_ids[i];
      if (id >= 0) {
        int e = s_val[i];
        const int page = (unsigned)id / S;
        if (staged && HS_CHECK((unsigned)page < (unsigned)sm.tbl_pages, kChkTablePage)) {
          const int b = s_bt[page];
          const int h = s_hbt[page];
          e = b >= 0 ? b : (h < 0 ? -1 : (h >= p.num_host_blocks ? kBadHost : -2 - h));
          s_val[i] = e;
        }
        other |= (e < 0 || e >= p.num_gpu_blocks);
      }
    }
  }
  const bool fully_resident = !__syncthreads_or(other) && !early;

  if (fully_resident) {
    // Full residency (Japanese article, "仕組み"): every id is read in place, nothing is hit or copied,
    // and the hot state is not touched -- the same results as the phases below, without them.
    int c = 0;
    for (int i = tid; i < n; i += kT) {
      const int id = s_ids[i];
      int row = -1;
      if (id >= 0) {
        row = s_val[i] * S + (int)((unsigned)id % S);
        c += idh.find(id) == i;  // distinct ids: first occurrences
      }
      rows_g[i] = row;
      if (msrc_g) msrc_g[i] = row;
    }
    c = __reduce_add_sync(kFull, c);
    if (lane == 0 && c) atomicAdd(&s_cnt[0], c);
    __syncthreads();
    if (tid == 0) {
      int32_t* st = p.out_stats + (int64_t)unit * 4;
      st[0] = HS_OK;
      st[1] = s_cnt[0];
      st[2] = st[3] = 0;
      p.miss_count[unit] = 0;
    }
    // ordered layout: no unit of the grid ends before the counters' clearing kernel has, so the
    // kernels after this one never see a counter of an earlier step
    if (p.ord.cnt) pdl_wait_prerequisites();
    return;
  }

  // ---- phase 1b: each slot's token, looked up among the ids: the plan entry of that id learns the
  // lowest slot holding it
  if (!early) {
#pragma unroll
    for (int k = 0; k < kTokRegs; ++k) {
      const int t = tokr[k];
      if (t >= 0) {
        const int f = idh.find(t);
        if (f >= 0) atomicMin(&s_slot[f], tid + k * kT);
      }
    }
    for (int s = tid + kTokRegs * kT; s < C; s += kT) {
      const int t = tok_g[s];
      if (t >= 0) {
        const int f = idh.find(t);
        if (f >= 0) atomicMin(&s_slot[f], s);
      }
    }
  }
  __syncthreads();

  // ---- phase 2: classify each plan entry (first occurrences); hits get stamp = step in smem;
  // repeated ids record their first occurrence
  int c_res = 0, c_hit = 0, c_miss = 0;
  if (!early) {
    for (int i = tid; i < n; i += kT) {
      const int id = s_ids[i];
      uint8_t cls = kNone;
      int val = 0;
      const int f = id >= 0 ? idh.find(id) : -1;
      if (f >= 0 && f != i) {
        cls = kDup;
        val = f;
        s_any_dup = 1;
      } else if (f == i) {
        const int off = (unsigned)id % S;
        const int e = s_val[i];
        if (e >= 0) {
          if (e >= p.num_gpu_blocks) err |= kErrTable;
          else val = e * S + off;
          cls = kResident;
          ++c_res;
        } else {
          const int s = s_slot[i];
          if (s != kNoSlot) {
            cls = kHit;
            val = s;
            s_stamp[s] = step;
            ++c_hit;
          } else {
            if (e == -1) err |= kErrMissing;
            else if (e == kBadHost) err |= kErrTable;
            else {
              val = (-2 - e) * S + off;
              if (p.row_bytes) prefetch_host_row(p, lr, val);
            }
            cls = kMiss;
            ++c_miss;
          }
        }
      }
      s_cls[i] = cls;
      s_val[i] = val;
    }
  }
  c_res = __reduce_add_sync(kFull, c_res);
  c_hit = __reduce_add_sync(kFull, c_hit);
  c_miss = __reduce_add_sync(kFull, c_miss);
  if (lane == 0 && (c_res | c_hit | c_miss)) {
    atomicAdd(&s_cnt[0], c_res);
    atomicAdd(&s_cnt[1], c_hit);
    atomicAdd(&s_cnt[2], c_miss);
  }
  if (err) atomicOr(&s_err, err);
  __syncthreads();

  uint32_t e = s_err;
  if (e & kErrHot) {  // hot blocks matter only to a unit that hits or misses (uniform: block totals)
    e &= ~kErrHot;
    if (s_cnt[1] + s_cnt[2] > 0) e |= kErrTable;
  }
  // per-thread contiguous chunks: positions [i0, i1) and slots [q0, q1)
  const int ipt = (n + kT - 1) / kT;
  const int i0 = min(n, tid * ipt), i1 = min(n, i0 + ipt);
  const int spt = (C + kT - 1) / kT;
  const int q0 = min(C, tid * spt), q1 = min(C, q0 + spt);
  int miss_base = 0, cand_base = 0, tot_miss = 0, tot_cand = 0;
  unsigned short* sorted = nullptr;

  if (e == 0u) {
    // ---- phase 3: miss ranks (plan order) and candidate positions (slot order); capacity
    int my_miss = 0;
    for (int i = i0; i < i1; ++i) my_miss += (s_cls[i] == kMiss);
    int my_cand = 0, lo = INT_MAX, hi = INT_MIN;
    for (int s = q0; s < q1; ++s) {
      const int st = s_stamp[s];
      if (st < step) { ++my_cand; lo = min(lo, st); hi = max(hi, st); }
    }
    lo = __reduce_min_sync(kFull, lo);
    hi = __reduce_max_sync(kFull, hi);
    if (lane == 0 && lo != INT_MAX) { atomicMin(&s_lo, lo); atomicMax(&s_hi, hi); }
    block_scan2<kT / 32>(my_miss, my_cand, miss_base, cand_base, tot_miss, tot_cand, s_tmp);
    if (tot_miss > tot_cand) e = kErrCapacity;  // uniform: totals are block-wide
    if (e == 0u && tot_miss > 0) {
      // ---- phase 4: victims = candidates in ascending (stamp, slot)
      unsigned short* buf_a = reinterpret_cast<unsigned short*>(smem + sm.idh);
      unsigned short* buf_b = buf_a + ((C + 7) & ~7);
      int* hist = reinterpret_cast<int*>(buf_b + ((C + 7) & ~7));
      __syncthreads();  // the id hash (same memory) is dead from here on
      int k = cand_base;
      for (int s = q0; s < q1; ++s)
        if (s_stamp[s] < step) buf_a[k++] = (unsigned short)s;
      __syncthreads();
      // the span of the candidates' stamps, in unsigned arithmetic: any two int32 stamps differ by less
      // than 2^32, so keys stamp - lo are exact as uint32 (up to four 8-bit passes)
      const uint32_t span = (uint32_t)s_hi - (uint32_t)s_lo;
      const int bits = span ? 32 - __clz((int)span) : 0;
      sorted = radix_sort_slots<kT>(buf_a, buf_b, tot_cand, s_stamp, s_lo, (bits + 7) / 8, hist, s_tmp);
    }
  }

  // ---- phase 4b (ordered miss layout): the unit counts its misses per host row range, reserves
  // that many entries in each of its group's buckets (one global atomic per bucket it uses), and
  // phase 5 files each miss at the next reserved entry of its bucket (the overflow list once a
  // bucket is full).  s_bk reuses the victim sort's histogram memory.
  const bool ordered = p.ord.cnt != nullptr && e == 0u && tot_miss > 0;  // uniform
  int* s_bk = reinterpret_cast<int*>(smem + sm.idh) + ((C + 7) & ~7);    // after the two slot buffers
  int32_t* ord_cnt = ordered ? p.ord.cnt + (int64_t)lr * (kMissBuckets + 1) : nullptr;
  // ---- phase 4c (fused plans with misses): the repeated positions of a missed id are chained, so that
  // the gather's miss warps store the row they read once into every position of the id.  s_slot (dead
  // since phase 2) becomes the chain heads: s_slot[f] = the last-linked repeat of first occurrence f;
  // a repeat's per-position source holds the link to the next one, -3 - next (-2 ends the chain).
  const bool chains = msrc_g != nullptr && e == 0u && tot_miss > 0 && s_any_dup;  // uniform
  if (chains) {
    for (int i = tid; i < n; i += kT) s_slot[i] = -1;
    __syncthreads();
    for (int i = tid; i < n; i += kT) {
      if (s_cls[i] == kDup) {
        const int f = s_val[i];
        if (s_cls[f] == kMiss) msrc_g[i] = -3 - atomicExch(&s_slot[f], i);
      }
    }
    __syncthreads();
  }

  // every unit of an ordered launch waits for the counters' clearing kernel (launched just before
  // this one): those that file misses need the counters zero, and none may end before it has
  if (p.ord.cnt) pdl_wait_prerequisites();
  if (ordered) {
    __syncthreads();  // the sort's histogram is dead
    for (int b = tid; b < kMissBuckets; b += kT) s_bk[b] = 0;
    __syncthreads();
    for (int i = i0; i < i1; ++i)
      if (s_cls[i] == kMiss) atomicAdd(&s_bk[min(kMissBuckets - 1, (int)((uint32_t)s_val[i] >> p.ord.shift))], 1);
    __syncthreads();
    for (int b = tid; b < kMissBuckets; b += kT) {
      const int c = s_bk[b];
      s_bk[b] = c ? atomicAdd(ord_cnt + b, c) : 0;
    }
    __syncthreads();
  }

  if (e == 0u) {
    // ---- phase 5: hits refresh their stamp; the j-th miss takes the j-th victim and one row
    int j = miss_base;
    for (int i = i0; i < i1; ++i) {
      const uint8_t cls = s_cls[i];
      if (cls == kMiss) {
        const int v = sorted[j];
        if (!HS_CHECK((unsigned)v < (unsigned)C, kChkStateSlot) ||
            !HS_CHECK(ordered || (unsigned)j < (unsigned)p.max_m, kChkMissList)) {
          ++j;
          continue;
        }
        const int vb = (unsigned)v / S;
        const int dst = s_hot[vb] * S + (v - vb * S);
        if (!HS_CHECK((unsigned)dst < (unsigned)p.num_gpu_blocks * (unsigned)S, kChkPoolRow)) {
          ++j;
          continue;
        }
        const int4 ent = make_int4(s_val[i], dst, r * n + i, chains ? s_slot[i] : -1);
        if (ordered) {
          const int b = min(kMissBuckets - 1, (int)((uint32_t)s_val[i] >> p.ord.shift));
          const int q = atomicAdd(&s_bk[b], 1);
          if (q < p.ord.cap) {
            p.ord.buckets[((int64_t)lr * kMissBuckets + b) * p.ord.cap + q] = ent;
          } else {
            const int o = atomicAdd(ord_cnt + kMissBuckets, 1);
            if (o < p.ord.per_group) p.ord.overflow[(int64_t)lr * p.ord.per_group + o] = ent;
          }
        } else {
          p.miss_list[(int64_t)unit * p.max_m + j] = ent;
        }
        if (msrc_g) msrc_g[i] = kGatherOwnedByMissWarps;
        p.slot_token[state_off + v] = s_ids[i];
        p.slot_stamp[state_off + v] = step;
        s_val[i] = dst;
        ++j;
      } else if (cls == kHit) {
        const int v = s_val[i];
        if (!HS_CHECK((unsigned)v < (unsigned)C, kChkStateSlot)) continue;
        const int vb = (unsigned)v / S;
        p.slot_stamp[state_off + v] = step;
        s_val[i] = s_hot[vb] * S + (v - vb * S);
        if (msrc_g) msrc_g[i] = s_val[i];
      } else if (msrc_g && cls == kResident) {
        msrc_g[i] = s_val[i];
      }
    }
    __syncthreads();
    // ---- phase 6: emit rows (duplicates read their first occurrence's row)
    for (int i = tid; i < n; i += kT) {
      const int id = s_ids[i];
      int row = -1;
      if (id >= 0) {
        if (s_cls[i] != kDup) {
          row = s_val[i];
        } else {  // a repeated id: share the first occurrence's row
          const int f = s_val[i];
          row = s_val[f];
          if (msrc_g && s_cls[f] != kMiss) msrc_g[i] = row;  // a miss's repeats are chained (phase 4c)
        }
      } else if (msrc_g) {
        msrc_g[i] = -1;
      }
      rows_g[i] = row;
    }
    if (tid == 0) {
      int32_t* st = p.out_stats + (int64_t)unit * 4;
      st[0] = HS_OK;
      st[1] = s_cnt[0];
      st[2] = s_cnt[1];
      st[3] = s_cnt[2];
      p.miss_count[unit] = tot_miss;
    }
  } else {
    const int code = (e & kErrStep) ? HS_ERR_STEP_ORDER
                   : (e & kErrId) ? HS_ERR_ID_RANGE
                   : (e & kErrTable) ? HS_ERR_TABLE_RANGE
                   : (e & kErrMissing) ? HS_ERR_MISSING_ROW
                   : HS_ERR_CAPACITY;
    for (int i = tid; i < n; i += kT) {
      rows_g[i] = -1;
      if (msrc_g) msrc_g[i] = -1;
    }
    if (tid == 0) {
      int32_t* st = p.out_stats + (int64_t)unit * 4;
      st[0] = code;
      st[1] = st[2] = st[3] = 0;
      p.miss_count[unit] = 0;
    }
  }
}

constexpr int kCopyThreads = 256;

// Copies the rows of up to kMissRowsPerItem entries (lane j < nrows holds entry j) from the host pool
// into their hot slots, in every layer [l0, l0 + group), all of a layer's 16-byte loads before its
// stores.
template <int CPR>
__device__ __forceinline__ void copy_miss_rows(const LayerPtrs& ptrs, int l0, int group, int4 ent, int nrows,
                                               int row_bytes, int gpu_rows, int host_rows) {
  constexpr int kU = CPR ? (kMissRowsPerItem * CPR + 31) / 32 : 4;
  const int cpr = CPR ? CPR : (row_bytes >> 4);
  const int lane = threadIdx.x & 31;
  const int total = nrows * cpr;
  // checked build: a lane whose entry points outside either pool has its row skipped
  const int ok = lane >= nrows || (HS_CHECK((unsigned)ent.x < (unsigned)host_rows, kChkHostRow) &&
                                   HS_CHECK((unsigned)ent.y < (unsigned)gpu_rows, kChkPoolRow));
  (void)ok;
  for (int l = l0; l < l0 + group; ++l) {
    const uint8_t* host = ptrs.host[l];
    uint8_t* pool = ptrs.gpu[l];
    for (int f0 = 0; f0 < total; f0 += 32 * kU) {
      uint4 v[kU];
      int64_t dst_off[kU];
#pragma unroll
      for (int k = 0; k < kU; ++k) {
        const int f = f0 + k * 32 + lane;
        const bool ok_f = f < total;
        const int rr = ok_f ? f / cpr : 0;
        const int cc = f - rr * cpr;
        const int src = __shfl_sync(kFull, ent.x, rr);
        const int dst = __shfl_sync(kFull, ent.y, rr);
        const bool row_ok = HS_CHECKED ? __shfl_sync(kFull, ok, rr) != 0 : true;
        dst_off[k] = -1;
        if (ok_f && row_ok) {
          v[k] = __ldcg(reinterpret_cast<const uint4*>(host + (int64_t)src * row_bytes) + cc);
          dst_off[k] = (int64_t)dst * row_bytes + (int64_t)cc * 16;
        }
      }
#pragma unroll
      for (int k = 0; k < kU; ++k)
        if (dst_off[k] >= 0) *reinterpret_cast<uint4*>(pool + dst_off[k]) = v[k];
    }
  }
}

// Copies the misses of every unit.  Per-unit lists: items (unit, group of kMissRowsPerItem
// consecutive misses) are numbered chunk-major (item = group * units + unit), so the live items are
// the low numbers; lane j of warp w tests item w + j * nwarps, which spreads the live items over all
// warps of the grid.  Ordered layout: blockIdx.y is the index group, and each warp of its CTAs takes
// whole buckets and reads them in address order, so every warp walks its own host range upward.  A
// live item's rows are copied with all its 16-byte loads issued before any store.
template <int CPR>
__global__ void __launch_bounds__(kCopyThreads) miss_copy_kernel(const ResolveParams p, const LayerPtrs ptrs,
                                                                 int32_t row_bytes) {
  pdl_wait_prerequisites();   // the resolver's miss lists must be complete and visible
  const int lane = threadIdx.x & 31;
  __shared__ MissItems mi;  // the ordered layout's index of this CTA's index group
  if (p.ord.cnt && !p.ord.ranges) {
    // ordered layout, spread schedule: the group's warps take its 4-entry items in bucket order (warp w:
    // items w, w + nwarps, ...)
    const int g = blockIdx.y;
    const int64_t warp = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
    const int64_t nwarps = ((int64_t)gridDim.x * blockDim.x) >> 5;
    if (threadIdx.x < 32) mi.load(p.ord, g);
    __syncthreads();
    const int4* bk = p.ord.buckets + (int64_t)g * kMissBuckets * p.ord.cap;
    const int4* ov = p.ord.overflow + (int64_t)g * p.ord.per_group;
    const int l0 = (p.layer_begin + g) * p.group;
    for (int32_t i = (int32_t)warp; i < mi.items; i += (int32_t)nwarps) {
      int64_t start;
      bool in_ov;
      int nrows;
      mi.locate(p.ord, i, start, in_ov, nrows);
      int4 ent = make_int4(0, 0, 0, 0);
      if (lane < nrows) ent = (in_ov ? ov : bk)[start + lane];
      copy_miss_rows<CPR>(ptrs, l0, p.group, ent, nrows, row_bytes, p.num_gpu_blocks * p.S, p.num_host_blocks * p.S);
    }
    return;
  }
  if (p.ord.cnt) {
    // ordered layout on large host pools (range schedule): the group's warps split its buckets into
    // contiguous blocks (warp w: buckets [w * kMissBuckets / nwarps, (w + 1) * kMissBuckets / nwarps),
    // numbered CTA-major so that neighbouring blocks run on different SMs), copy their entries as filed,
    // then one slice of the overflow list each
    const int g = blockIdx.y;
    const int warp = (int)(threadIdx.x >> 5) * (int)gridDim.x + (int)blockIdx.x;
    const int nwarps = (int)(((int64_t)gridDim.x * blockDim.x) >> 5);
    const int4* bk = p.ord.buckets + (int64_t)g * kMissBuckets * p.ord.cap;
    const int32_t* cntg = p.ord.cnt + (int64_t)g * (kMissBuckets + 1);
    const int l0 = (p.layer_begin + g) * p.group;
    const int gpu_rows = p.num_gpu_blocks * p.S, host_rows = p.num_host_blocks * p.S;
    const int b0 = (int)((int64_t)warp * kMissBuckets / nwarps), b1 = (int)((int64_t)(warp + 1) * kMissBuckets / nwarps);
    for (int b = b0; b < b1; ++b) {
      const int nb = min(__ldcg(cntg + b), p.ord.cap);
      for (int i = 0; i < nb; i += kMissRowsPerItem) {
        const int nrows = min(kMissRowsPerItem, nb - i);
        const int4 ent = lane < nrows ? bk[(int64_t)b * p.ord.cap + i + lane] : make_int4(0, 0, 0, 0);
        copy_miss_rows<CPR>(ptrs, l0, p.group, ent, nrows, row_bytes, gpu_rows, host_rows);
      }
    }
    const int ovn = min(__ldcg(cntg + kMissBuckets), p.ord.per_group);
    const int ov_per = (ovn + nwarps - 1) / nwarps;
    const int o0 = warp * ov_per, o1 = min(ovn, o0 + ov_per);
    const int4* ov = p.ord.overflow + (int64_t)g * p.ord.per_group;
    for (int i = o0; i < o1; i += kMissRowsPerItem) {
      const int nrows = min(kMissRowsPerItem, o1 - i);
      const int4 ent = lane < nrows ? ov[i + lane] : make_int4(0, 0, 0, 0);
      copy_miss_rows<CPR>(ptrs, l0, p.group, ent, nrows, row_bytes, gpu_rows, host_rows);
    }
    return;
  }
  const int units = p.nl * p.R;
  const int items_per_unit = (p.max_m + kMissRowsPerItem - 1) / kMissRowsPerItem;
  const int64_t items = (int64_t)units * items_per_unit;
  const int64_t warp = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const int64_t nwarps = ((int64_t)gridDim.x * blockDim.x) >> 5;
  for (int64_t base = warp; base < items; base += nwarps * 32) {
    const int64_t item = base + (int64_t)lane * nwarps;
    int unit = 0, chunk = 0, cnt = 0;
    bool live = false;
    if (item < items) {
      chunk = (int)(item / units);
      unit = (int)(item - (int64_t)chunk * units);
      cnt = p.miss_count[unit];
      live = chunk * kMissRowsPerItem < cnt;
    }
    uint32_t todo = __ballot_sync(kFull, live);
    while (todo) {
      const int src_lane = __ffs(todo) - 1;
      todo &= todo - 1u;
      const int u = __shfl_sync(kFull, unit, src_lane);
      const int ch = __shfl_sync(kFull, chunk, src_lane);
      const int c = __shfl_sync(kFull, cnt, src_lane);
      const int r0 = ch * kMissRowsPerItem;
      const int nrows = min(kMissRowsPerItem, c - r0);
      int4 ent = make_int4(0, 0, 0, 0);
      if (lane < nrows) ent = p.miss_list[(int64_t)u * p.max_m + r0 + lane];
      copy_miss_rows<CPR>(ptrs, (p.layer_begin + u / p.R) * p.group, p.group, ent, nrows, row_bytes,
                          p.num_gpu_blocks * p.S, p.num_host_blocks * p.S);
    }
  }
}

// Zeroes the ordered layout's counters; the resolver launched after it waits for it only where it
// first touches them.
__global__ void order_clear_kernel(int32_t* __restrict__ cnt, int32_t count) {
  pdl_allow_dependents();
  for (int i = blockIdx.x * blockDim.x + threadIdx.x; i < count; i += gridDim.x * blockDim.x) cnt[i] = 0;
}

int ceil_log2(int64_t x) {
  int b = 0;
  while ((int64_t(1) << b) < x) ++b;
  return b;
}

size_t align16(size_t x) { return (x + 15) & ~size_t(15); }

}  // namespace

uint32_t check_take_resolve() {
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

ResolveSmem resolve_smem_plan(int64_t n, int64_t C, int64_t S, bool wide) {
  ResolveSmem sm{};
  if (n < 0 || n > HS_MAX_PLAN || C < 1 || C > HS_MAX_CAPACITY || S < 1 || C % S) return sm;
  sm.id_hash_bits = ceil_log2(2 * (n > 16 ? n : 16));
  sm.id_hash_wide = wide ? 1 : 0;
  size_t off = 0;
  sm.stamp = off; off = align16(off + 4 * (size_t)C);
  sm.ids = off;   off = align16(off + 4 * (size_t)n);
  sm.val = off;   off = align16(off + 4 * (size_t)n);
  sm.cls = off;   off = align16(off + (size_t)n);
  sm.slot = off;  off = align16(off + 4 * (size_t)n);
  sm.hot = off;   off = align16(off + 4 * (size_t)(C / S));
  sm.idh = off;   // the id hash, later the victim sort's buffers
  const size_t id_hash = (wide ? 8 : 4) * ((size_t)1 << sm.id_hash_bits);
  const size_t cbuf = 2 * (size_t)((C + 7) & ~int64_t(7));
  const size_t radix = 2 * cbuf + 4 * (size_t)kRadixBins * kSortWarps;
  off = align16(off + (id_hash > radix ? id_hash : radix));
  sm.total = off;
  return sm;
}

ResolveSmem resolve_smem_plan_staged(int64_t n, int64_t C, int64_t S, int64_t max_pages, size_t limit) {
  // preference: wide id table with staged table rows, narrow with staged rows, wide, narrow
  const size_t tbl = align16(8 * (size_t)max_pages);
  for (int k = 0; k < 4; ++k) {
    const bool wide = (k % 2) == 0, staged = k < 2;
    if (staged && max_pages > kMaxStagedPages) continue;
    ResolveSmem sm = resolve_smem_plan(n, C, S, wide);
    if (sm.total == 0) return sm;
    if (staged) {
      sm.tbl = sm.total;
      sm.tbl_pages = (int32_t)max_pages;
      sm.total += tbl;
    }
    if (sm.total <= limit) return sm;
  }
  return resolve_smem_plan(n, C, S, false);
}

size_t resolve_workspace_bytes(int64_t units, int64_t n, int64_t C) {
  // [miss counts, 16-byte aligned] [miss lists: units x min(n, C) int4] [per-position sources: units x n]
  // [the fused gather's work counters]
  return ws_queue_offset(units, n, C) + kQueueBytes;
}

size_t resolve_workspace_bytes_ordered(int64_t groups, int64_t R, int64_t n, int64_t C) {
  const int64_t max_m = n < C ? n : C;
  return resolve_workspace_bytes(groups * R, n, C) + ws_order_cnt_bytes(groups) +
         16 * (size_t)groups * kMissBuckets * (size_t)miss_bucket_cap(R * max_m);
}

MissOrder miss_order_layout(void* workspace, int64_t groups, int64_t R, int64_t n, int64_t C, int64_t num_host_rows) {
  MissOrder o{};
  const int64_t max_m = n < C ? n : C;
  const int64_t per_group = R * max_m;
  if (!workspace || per_group <= 0 || 2 * per_group > INT32_MAX) return o;
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  const size_t base = resolve_workspace_bytes(groups * R, n, C);
  o.cnt = reinterpret_cast<int32_t*>(ws + base);
  o.buckets = reinterpret_cast<int4*>(ws + base + ws_order_cnt_bytes(groups));
  o.overflow = reinterpret_cast<int4*>(ws + ws_counts_bytes(groups * R));
  o.shift = miss_bucket_shift(num_host_rows);
  o.cap = miss_bucket_cap(per_group);
  o.per_group = (int32_t)per_group;
  return o;
}

namespace {

// every resolver instantiation, in the order (page size 64?, wide table?, 512 threads?) -> index
const void* resolver_kernels[8] = {
    (const void*)resolve_kernel<0, false, 1024>, (const void*)resolve_kernel<0, false, 512>,
    (const void*)resolve_kernel<0, true, 1024>,  (const void*)resolve_kernel<0, true, 512>,
    (const void*)resolve_kernel<64, false, 1024>, (const void*)resolve_kernel<64, false, 512>,
    (const void*)resolve_kernel<64, true, 1024>,  (const void*)resolve_kernel<64, true, 512>};

std::atomic<long long> g_smem_limit[64];
std::atomic<long long> g_smem_per_sm[64];
std::atomic<int> g_static_smem{0};

}  // namespace

size_t resolve_smem_limit(int dev) {
  // Dynamic shared memory one resolver CTA may use on this device (opt-in maximum minus the
  // kernels' static shared memory).  Also raises the kernels' attribute to that limit, once.
  if (dev < 0 || dev >= 64) return 0;
  long long v = g_smem_limit[dev].load();
  if (v > 0) return (size_t)v;
  int optin = 0, per_sm = 0;
  if (cudaDeviceGetAttribute(&optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev) != cudaSuccess) return 0;
  if (cudaDeviceGetAttribute(&per_sm, cudaDevAttrMaxSharedMemoryPerMultiprocessor, dev) != cudaSuccess) return 0;
  size_t st = 0;
  for (const void* k : resolver_kernels) {
    cudaFuncAttributes fa{};
    if (cudaFuncGetAttributes(&fa, k) != cudaSuccess) return 0;
    if (fa.sharedSizeBytes > st) st = fa.sharedSizeBytes;
  }
  const long long dyn = (long long)optin - (long long)st;
  if (dyn <= 0) return 0;
  for (const void* k : resolver_kernels)
    if (cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)dyn) != cudaSuccess) return 0;
  g_static_smem.store((int)st);
  g_smem_per_sm[dev].store(per_sm);
  g_smem_limit[dev].store(dyn);
  return (size_t)dyn;
}

int resolve_threads(const ResolveSmem& sm, int64_t units, int64_t n, int sms, int dev) {
  // 512 threads when two CTAs fit in one SM's shared memory (with the 1 KB the hardware reserves per
  // CTA) and either the units outnumber the SMs or a unit is small; 1024 otherwise
  if (dev < 0 || dev >= 64) return kResolveThreads;
  const long long per_sm = g_smem_per_sm[dev].load();
  const long long need = 2 * ((long long)sm.total + g_static_smem.load() + 1024);
  if (per_sm <= 0 || need > per_sm) return kResolveThreads;
  return (units > sms || n <= 1024) ? kResolveThreads / 2 : kResolveThreads;
}

cudaError_t launch_resolve(const ResolveParams& p, const ResolveSmem& sm, cudaStream_t s) {
  const int idx = (p.S == 64 ? 4 : 0) + (sm.id_hash_wide ? 2 : 0) + (sm.threads == kResolveThreads / 2 ? 1 : 0);
  const dim3 grid(p.nl * p.R), block(sm.threads == kResolveThreads / 2 ? kResolveThreads / 2 : kResolveThreads);
  void* args[] = {(void*)&p, (void*)&sm};
  if (!p.ord.cnt) {
    cudaError_t e = cudaLaunchKernel(resolver_kernels[idx], grid, block, args, sm.total, s);
    count_launch();
    return e;
  }
  const int count = p.nl * (kMissBuckets + 1);
  order_clear_kernel<<<(count + 255) / 256, 256, 0, s>>>(p.ord.cnt, count);
  count_launch();
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg{};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = sm.total;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  e = cudaLaunchKernelExC(&cfg, resolver_kernels[idx], args);
  count_launch();
  return e;
}

cudaError_t launch_miss_copy(const ResolveParams& p, const LayerPtrs& ptrs, int32_t row_bytes, int sms,
                             cudaStream_t s) {
  const int64_t units = (int64_t)p.nl * p.R;
  const int64_t items = units * ((p.max_m + kMissRowsPerItem - 1) / kMissRowsPerItem);
  // one warp per item at most, capped at a full resident grid (split over the index groups when
  // the ordered layout gives each group its own CTAs)
  int64_t blocks = (items + kCopyThreads / 32 - 1) / (kCopyThreads / 32);
  // the range schedule: two CTAs per SM over all index groups (about 2,400 warps, each owning a block of
  // buckets, spread over every SM); the others up to eight CTAs per SM
  const int64_t cap = p.ord.cnt ? (p.ord.ranges ? ((int64_t)sms * 2 + p.nl - 1) / p.nl
                                                : ((int64_t)sms * 8 + p.nl - 1) / p.nl)
                                : (int64_t)sms * 8;
  if (p.ord.cnt) blocks = (blocks + p.nl - 1) / p.nl;
  if (blocks > cap) blocks = cap;
  if (blocks < 1) blocks = 1;
  const dim3 grid((unsigned)blocks, p.ord.cnt ? (unsigned)p.nl : 1u);
  auto kern = row_bytes == 656 ? miss_copy_kernel<41> : miss_copy_kernel<0>;
  cudaError_t e;
  if (p.ord.cnt) {  // large host pools: no early launch (as for the fused gather)
    kern<<<grid, kCopyThreads, 0, s>>>(p, ptrs, row_bytes);
    e = cudaGetLastError();
  } else {
    e = launch_dependent(kern, grid, dim3(kCopyThreads), 0, s, p, ptrs, row_bytes);
  }
  if (e != cudaSuccess) return e;
  count_launch();
  return cudaGetLastError();
}

}  // namespace hs
