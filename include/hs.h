/*
 * hs.h -- C ABI of the Hybrid HiSparse top-K resolver for sparse-MLA decode.
 *
 * Operations (each one cites the passage of the source pages that defines it):
 *
 *   hs_resolve_topk   the fused per-step top-K resolver.  "vLLM GLM 5.3 Optimizations: Hybrid
 *                     HiSparse Offloading", section "Technical Implementation of Hybrid HiSparse",
 *                     item 2 (Mixed residency): resident tokens are read in place, hot tokens are read
 *                     and their LRU entry refreshed, a miss copies a single row from pinned host memory
 *                     into an LRU slot; the same article in Japanese (news.ainew.jp), section
 *                     "仕組み" (How it works), which adds that nothing on the decode path waits for a
 *                     CPU decision, so the step stays CUDA-graph capturable.
 *   hs_gather_rows    the single-stride gather by pool row id.  Japanese article, section "仕組み":
 *                     whether a row sits in a resident page or in the hot buffer, the resolver hands
 *                     back pool (HMA) row ids and they are gathered with one stride.
 *   hs_offload_pages  the post-forward proactive copy.  English page, section "Key Architectural
 *                     Details" (Proactive Copying, Lightweight Execution): completed prefix pages are
 *                     copied to CPU memory while the GPU keeps serving them, all sparse-MLA layers in a
 *                     single launch after the forward pass, ordered on the model's GPU stream.
 *   hs_hot_reset      empties hot buffers (the buffer is leased empty for a new request: Japanese
 *                     article, section "仕組み", "No residency" state).
 *
 * Conventions shared by every call
 *   - The caller owns all memory (device buffers, pinned host pool, workspace) and all streams.
 *     No call allocates device or pinned memory; hs_pool_create allocates only its small host struct.
 *   - resolve / gather / offload / reset are asynchronous on the given stream: they validate what the
 *     host can see, launch, and return.  They never synchronise the device.
 *   - The return value reports host-checkable argument errors (HS_ERR_INVALID_ARG) and launch
 *     failures (HS_ERR_CUDA).  Data errors found on the device are written to device status words
 *     (out_stats for the resolver, an optional status word for gather/offload); they never trap.
 *   - Stream ordering is the only synchronisation: gather after resolve on the same stream; reuse of a
 *     GPU block after hs_offload_pages on the same stream; readers of host copies on another stream
 *     wait for an event recorded after the offload.
 *   - Layout: row id = gpu_block * page_size + offset (int32); the bytes of a row in layer l live at
 *     gpu_layer_base[l] + (int64)row * row_bytes.  Host pool rows likewise with host blocks.
 *   - Data-error precedence inside one (layer, request) unit, highest first:
 *     HS_ERR_STEP_ORDER, HS_ERR_ID_RANGE, HS_ERR_TABLE_RANGE, HS_ERR_MISSING_ROW, HS_ERR_CAPACITY.
 */
#ifndef HS_H_
#define HS_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* A CUDA stream (ABI-identical to cudaStream_t / CUstream).  NULL = the legacy default stream. */
typedef struct CUstream_st* hs_stream_t;

typedef enum {
  HS_OK = 0,
  HS_ERR_INVALID_ARG = 1,  /* host-visible argument error; nothing was launched                  */
  HS_ERR_ID_RANGE = 2,     /* a top-K id < -1, >= ctx_len[r], or on a page >= max_pages;
                              gather: a row id outside [-1, num_gpu_blocks*page_size)            */
  HS_ERR_MISSING_ROW = 3,  /* a miss on a placeholder page that has no host copy                  */
  HS_ERR_CAPACITY = 4,     /* more misses than evictable hot slots this step                      */
  HS_ERR_STEP_ORDER = 5,   /* step is older than a stamp already in the hot state                 */
  HS_ERR_CUDA = 6,         /* a CUDA runtime call or launch failed                                */
  HS_ERR_TIMEOUT = 7,      /* a bounded device wait gave up (the bulk-copy gather's loads)        */
  HS_ERR_TABLE_RANGE = 8   /* a block-table, host-block-table or hot-block entry that the step
                              dereferences lies outside the pool; offload: a pair out of range    */
} hs_status;

/* Compile-time limits of the library.  Each launch's shared-memory footprint is also checked (see
 * hs_resolve_smem_bytes); a shape that does not fit returns HS_ERR_INVALID_ARG. */
#define HS_MAX_LAYERS 128
#define HS_MAX_PAGE_SIZE 1024
#define HS_MAX_CAPACITY 16384   /* hot rows per (layer, request) */
#define HS_MAX_PLAN 16384       /* P * K ids per (layer, request) */

typedef struct hs_pool hs_pool; /* opaque: geometry and the per-layer base pointers only */

typedef struct {
  int32_t num_layers;      /* sparse-MLA layers, 1..HS_MAX_LAYERS                                   */
  int32_t page_size;       /* tokens per page (block), 1..HS_MAX_PAGE_SIZE                          */
  int32_t row_bytes;       /* bytes of one KV row, > 0 and a multiple of 16 (656 for FP8 MLA rows)  */
  int32_t num_gpu_blocks;  /* blocks per layer in the GPU pool; num_gpu_blocks*page_size < 2^31     */
  int32_t num_host_blocks; /* blocks per layer in the pinned host pool (may be 0)                   */
  /* [num_layers] device pointers, each to [num_gpu_blocks][page_size][row_bytes] bytes,
   * 16-byte aligned.  Resident pages and leased hot blocks live in these same tensors. */
  void* const* gpu_layer_base;
  /* [num_layers] pinned (page-locked, device-mapped) host pointers, each to
   * [num_host_blocks][page_size][row_bytes] bytes, 16-byte aligned.  May be NULL when
   * num_host_blocks == 0. */
  void* const* host_layer_base;
} hs_pool_desc;

/* Per-request LRU hot buffers.  The blocks are ordinary pool blocks leased by the caller and are
 * shared by all layers (each layer's copy lives in that layer's tensor); the token/stamp state is
 * per (index group, request): an index group is the set of consecutive layers that read one top-K
 * list.  Slot v of request r is pool row hot_blocks[r][v / page_size] * page_size + v % page_size.
 *
 * layers_per_index (G) selects the grouping:
 *   0 or 1  every layer has its own top-K list and its own state (G = 1);
 *   G > 1   IndexShare: one indexer serves G consecutive sparse-MLA layers (Japanese article
 *           (news.ainew.jp), section "必要な時にスパーシティを活用する" (Using sparsity when it is
 *           needed): GLM 5.3 places one indexer layer per four sparse-MLA layers).  The layers of
 *           a group see the same ids, tables and step, so their LRU decisions are identical: the
 *           resolver runs once per (group, request), and each miss copies the token's row of every
 *           layer of the group into that layer's tensor (same slot, same pool row).
 * num_layers must be a multiple of G; groups are layers [g*G, (g+1)*G). */
typedef struct {
  int32_t capacity;          /* C rows per (group, request): a multiple of page_size,
                                page_size..HS_MAX_CAPACITY; the pages' default is 2*K            */
  const int32_t* hot_blocks; /* device int32 [R][capacity/page_size]; pool blocks in
                                [0, num_gpu_blocks), disjoint across requests and from every
                                resident block (not checked for overlap).  A request whose ids are
                                all resident needs none (entries may be -1); a unit with a hit or a
                                miss and an entry outside the pool gets HS_ERR_TABLE_RANGE        */
  int32_t* slot_token;       /* device int32 [num_layers/G][R][capacity]; -1 = empty slot        */
  int32_t* slot_stamp;       /* device int32 [num_layers/G][R][capacity]; last step that used the
                                slot, -1 = never                                                  */
  int32_t layers_per_index;  /* G, 0..HS_MAX_LAYERS (0 reads as 1)                                */
} hs_hot_state;

/* Validates the geometry and the pointers (device pointers must be device memory, host pointers
 * pinned and device-mapped), copies the pointer arrays, and returns a handle in *out.  Needs a
 * current CUDA device.  Returns HS_ERR_INVALID_ARG or HS_ERR_CUDA on failure (*out = NULL). */
hs_status hs_pool_create(const hs_pool_desc* desc, hs_pool** out);
void hs_pool_destroy(hs_pool* pool);

/* Sets slot_token and slot_stamp of all (num_layers/G) x R x capacity slots to -1 (async). */
hs_status hs_hot_reset(const hs_pool* pool, const hs_hot_state* hot, int32_t R, hs_stream_t stream);

/* Sets slot_token and slot_stamp to -1 for the listed requests only, in every index group (async):
 * the requests that just leased a hot buffer (hs_res_take_resets in hs_residency.h) start with empty
 * slots, while the other requests keep theirs.
 *   requests  device int32 [n]; entries outside [0, R) are skipped. */
hs_status hs_hot_reset_requests(const hs_pool* pool, const hs_hot_state* hot, int32_t R, const int32_t* requests,
                                int32_t n, hs_stream_t stream);

/* Bytes of caller-owned device workspace for hs_resolve_topk and hs_resolve_gather with this shape
 * (per-unit miss lists handed from the resolver kernel to the miss-copy kernel, per-position host
 * sources handed to the fused gather, 256 bytes of the fused gather's work counters, which the
 * resolver zeroes), including the room the address-ordered miss layout needs
 * (hs_pool_set_miss_order).  nl counts resolver units per request: layers when G = 1, index groups
 * (layers / G) under IndexShare; passing the layer count there over-sizes the workspace, which is
 * harmless.  0 on a bad shape. */
size_t hs_resolve_workspace_bytes(int32_t nl, int32_t R, int32_t P, int32_t K, int32_t capacity);

/* The smallest workspace resolve calls accept for this shape: the same without the ordered layout's
 * room (calls given less than hs_resolve_workspace_bytes use per-unit miss lists).  0 on a bad shape. */
size_t hs_resolve_workspace_bytes_min(int32_t nl, int32_t R, int32_t P, int32_t K, int32_t capacity);

/* How resolve calls hand a step's misses to the kernels that copy them.  Results are identical in
 * every mode; only the order of the host reads differs.
 *   HS_MISS_ORDER_AUTO (default)  address-ordered when the host pools of the call's layers hold at
 *                                 least 16 GiB together and the workspace has room for it;
 *   HS_MISS_ORDER_OFF             per-unit lists, copied unit by unit;
 *   HS_MISS_ORDER_ON              address-ordered whenever the workspace has room for it;
 *   HS_MISS_ORDER_RANGES          address-ordered with the range schedule (below) whatever the pool size;
 *   HS_MISS_ORDER_SPREAD          address-ordered with the spread schedule (below) whatever the pool size.
 * Address-ordered: the resolver files each index group's misses into 1024 buckets by host row range.
 * The copy warps then take them in one of two schedules: on host pools under 40 GiB (over the call's
 * layers) the 4-entry items of all buckets in bucket order, spread over every copy warp; from 40 GiB
 * on (or with HS_MISS_ORDER_RANGES; HS_MISS_ORDER_SPREAD keeps the spread schedule on any pool) one
 * contiguous block of buckets per warp, so that every warp reads its own range of the pool.  The pages
 * copy single rows from pinned host memory
 * ("vLLM GLM 5.3 Optimizations: Hybrid HiSparse Offloading", "Technical Implementation of Hybrid
 * HiSparse") and say nothing of their order; this is the library's choice.  Zero-copy reads spread
 * over tens of GB of host memory are bound by the device's address translation for host memory, not
 * by the link, and the same rows read in address order arrive several times faster.  It costs one
 * more small kernel per resolve call and workspace of 2 x R x min(P*K, capacity) x 16 bytes per index
 * group.  A plan and its hs_gather_planned must see the same mode and workspace size.  Set it
 * between calls, not while another thread is calling with the same pool.  HS_ERR_INVALID_ARG for an
 * unknown mode. */
#define HS_MISS_ORDER_AUTO 0
#define HS_MISS_ORDER_OFF 1
#define HS_MISS_ORDER_ON 2
#define HS_MISS_ORDER_RANGES 3
#define HS_MISS_ORDER_SPREAD 4
hs_status hs_pool_set_miss_order(hs_pool* pool, int32_t mode);

/* Diagnostics of the fused gather's SM partition.  With device_ts set (device memory, 4 x uint64,
 * 16-byte aligned; NULL turns it off, the default) every partition launch records %globaltimer
 * nanoseconds there: [0] the earliest CTA start (atomic min), [1] the latest end of a CTA that streamed HBM
 * rows, [2] the latest end of a miss warp's misses, [3] the latest CTA end (atomic max).  The caller sets
 * [0] to all ones and [1..3] to zero before a launch and reads them after it; [2] - [0] against [1] - [0]
 * shows which kind of traffic sets the gather's time.  The pages have no counterpart; results are
 * unchanged.  HS_ERR_INVALID_ARG for a misaligned pointer. */
hs_status hs_pool_set_phase_timestamps(hs_pool* pool, unsigned long long* device_ts);

/* Miss prefetch: with HS_MISS_PREFETCH_ON the resolver starts moving each miss's host row into L2
 * (one bulk L2 prefetch per row and layer of its index group) as soon as it classifies the id, before
 * it picks the victims, so that the copy that follows (the miss-copy kernel, or the fused gather's miss
 * warps) may find the row in L2.  HS_MISS_PREFETCH_OFF (default): no prefetch.  Results are identical.
 * Measured on one GB300, whole timed passes alternating in one process: no gain on the mixed-residency
 * batch (83 against 82.6 us per step) and slower on the agentic batch (0.75 against 0.34 ms), so it
 * stays off.
 * The pages copy single rows from pinned host memory ("vLLM GLM 5.3 Optimizations: Hybrid HiSparse
 * Offloading", "Technical Implementation of Hybrid HiSparse"); when the read starts is this library's
 * choice.  HS_ERR_INVALID_ARG for an unknown mode. */
#define HS_MISS_PREFETCH_OFF 0
#define HS_MISS_PREFETCH_ON 1
hs_status hs_pool_set_miss_prefetch(hs_pool* pool, int32_t mode);

/* Output layout of the gathers (hs_gather_rows, hs_gather_planned, hs_resolve_gather).  nplanes = 0
 * (the default): rows, out[layer][position][row_bytes].  nplanes = 1..HS_MAX_PLANES: each row is cut
 * into planes of plane_bytes[p] bytes (each > 0 and a multiple of 16, summing to row_bytes), and each
 * layer's output holds the planes one after the other: plane p of position i at
 *   out + layer_bytes * layer + positions * (plane_bytes[0] + ... + plane_bytes[p-1]) + i * plane_bytes[p],
 * layer_bytes = positions * row_bytes (the same buffer size as rows).  The FP8 MLA row of the pages'
 * benchmark configs is 512 B of latent, 16 B of scales and 128 B of rope: {512, 16, 128} gives a
 * sparse-MLA consumer each part as its own dense array.  The pages gather whole rows with one stride
 * ("vLLM GLM 5.3 Optimizations: Hybrid HiSparse Offloading", "Technical Implementation of Hybrid
 * HiSparse"); the split is this library's option.  The bulk copy mode writes rows only: with planes
 * set, hs_gather_rows uses loads.  Results are the same bytes in either layout.  HS_ERR_INVALID_ARG
 * for a bad count or plane size (plane_bytes is read during the call only). */
#define HS_MAX_PLANES 4
hs_status hs_pool_set_gather_planes(hs_pool* pool, int32_t nplanes, const int32_t* plane_bytes);

/* How hs_gather_rows moves its HBM rows.  Results are identical in both modes; only the speed
 * differs.
 *   HS_GATHER_COPY_LOADS (default)  every lane moves 16-byte chunks with ordinary loads and stores,
 *                                   eight chunks in flight per thread;
 *   HS_GATHER_COPY_BULK             one-dimensional bulk copies (cp.async.bulk) of whole rows, global
 *                                   -> shared -> global, issued by one lane per warp through a ring of
 *                                   16 row-sized shared-memory stages (12 loads in flight per warp);
 *                                   falls back to loads when the stages do not fit the device's
 *                                   shared memory.  Its waits are bounded: a load that never completes
 *                                   sets HS_ERR_TIMEOUT in the gather's status word.
 * The pages say only that the rows are gathered with one stride ([JA] "仕組み"); the copy mechanism
 * is this library's choice.  HS_ERR_INVALID_ARG for an unknown mode. */
#define HS_GATHER_COPY_LOADS 0
#define HS_GATHER_COPY_BULK 1
hs_status hs_pool_set_gather_copy(hs_pool* pool, int32_t mode);

/* How the fused gather (hs_gather_planned, hs_resolve_gather) places its miss copies.
 *   0   SM partition: the CTAs on one SM in six (hs_pool_set_miss_sm_divisor) copy misses, a bucket of
 *       host rows (range schedule) or a chunk of a unit's miss list (per-unit lists) per warp at a time,
 *       and the others stream the HBM rows; a CTA that runs out of its own kind of work takes the other.
 *   1, 2  with the range schedule, that many miss warps in every CTA beside the HBM warps, each reading a
 *       contiguous block of buckets; with per-unit lists, one miss warp in every CTA.
 *   -1  the default: the SM partition with the range schedule (host pools from 40 GiB), one miss warp in
 *       every CTA with per-unit lists.  Measured in one process (the planned gather replayed): full-size
 *       MTP3 batch 2.62 ms partitioned against 3.32 ms with one miss warp per CTA; mixed-residency batch
 *       63.1 against 61.1 us, cold start 127.7 against 126.6 us, tiny decode 21.1 against 10.9 us.
 * The spread schedule always uses one miss warp in every CTA.  Results are identical.
 * HS_ERR_INVALID_ARG for another value. */
hs_status hs_pool_set_miss_warps(hs_pool* pool, int32_t warps);

/* The SM partition's share of miss SMs: the CTAs on every divisor-th SM (by SM id) copy the misses, the
 * others stream the HBM rows.  divisor 2..32, or 0 for the library's default (6: on the full-size MTP3
 * batch the misses, read over the host link, end last; fewer miss SMs leave them slower, more slow the
 * HBM rows), or -1 for no miss SM: every CTA streams HBM rows, then copies misses.  Results are identical
 * for every divisor.  HS_ERR_INVALID_ARG for another value. */
hs_status hs_pool_set_miss_sm_divisor(hs_pool* pool, int32_t divisor);

/* 1 if a resolve call on layers [layer_begin, layer_begin + nl) with this shape, hot state and
 * workspace size uses the address-ordered miss layout, 0 if it uses per-unit lists, -1 on bad
 * arguments. */
int32_t hs_resolve_miss_order(const hs_pool* pool, int32_t layer_begin, int32_t nl, int32_t R, int32_t P, int32_t K,
                              const hs_hot_state* hot, size_t workspace_bytes);

/* Dynamic shared memory one resolver CTA needs for this shape, or 0 if the shape exceeds a limit.
 * Resolve calls reject shapes whose footprint exceeds the device's per-block opt-in maximum. */
size_t hs_resolve_smem_bytes(int32_t P, int32_t K, int32_t capacity, int32_t page_size);

/* The fused top-K resolver for layers [layer_begin, layer_begin + nl) and R requests at decode
 * step `step`.  One (index group, request) pair is one independent unit (with G = 1 a group is one
 * layer); g below indexes the call's groups, g < nl/G:
 *   plan      the distinct non-padding ids of topk_ids[g][r][0..P)[0..K) in first-occurrence order
 *             (position-major, then top-K order); all P query positions of a step share it;
 *   resident  block_table[r][id/page_size] >= 0: row = that block * page_size + id % page_size,
 *             read in place (wins over a stale hot copy);
 *   hit       the id sits in a hot slot: row = the slot's pool row; its stamp becomes `step`;
 *   miss      otherwise: the j-th miss in plan order takes the j-th smallest (stamp, slot) among
 *             slots whose stamp is < step and that were not hit in this call; exactly one row per
 *             layer of the group is copied from the pinned host pool
 *             (host_block_table[r][id/page_size]) into the slot, whose token becomes id and stamp
 *             `step`.
 * layer_begin and nl must be multiples of G = hot->layers_per_index.
 * Arguments (all device pointers):
 *   topk_ids         int32 [nl/G][R][P][K]; -1 = padding (row -1).
 *   block_table      int32 [R][max_pages]; < 0 = placeholder page (not resident).
 *   host_block_table int32 [R][max_pages]; < 0 = no host copy.
 *   ctx_len          int32 [R]; ids must be < ctx_len[r].
 *   out_rows         int32 [nl/G][R][P][K]; pool row per id (duplicates share the row; padding -1);
 *                    the same row id serves every layer of the group.
 *   out_stats        int32 [nl/G][R][4] = {status, resident, hits, misses}, counted over the plan.
 *   workspace        device scratch of >= hs_resolve_workspace_bytes_min(...) bytes (with
 *                    hs_resolve_workspace_bytes(...) the ordered miss layout is available), 16-byte
 *                    aligned; its contents need no initialisation and are garbage after the call.
 * A unit with a data error leaves its hot state and pool bytes unchanged, sets out_rows to -1 and
 * out_stats to {code, 0, 0, 0}; other units proceed.  Calling again with the same ids and step
 * returns the same rows with 0 misses (the replayable plan used by speculative decoding).
 * Launches two kernels on `stream` (resolve, then the miss copy of every layer), and one more small
 * kernel before them with the ordered miss layout.  Concurrent calls
 * that share hot state or workspace must be ordered by the caller. */
hs_status hs_resolve_topk(const hs_pool* pool, int32_t layer_begin, int32_t nl, int32_t R, int32_t P,
                          int32_t K, const int32_t* topk_ids, const int32_t* block_table,
                          const int32_t* host_block_table, const int32_t* ctx_len, int32_t max_pages,
                          const hs_hot_state* hot, int32_t step, int32_t* out_rows, int32_t* out_stats,
                          void* workspace, size_t workspace_bytes, hs_stream_t stream);

/* Resolve and gather in one call: the same results as hs_resolve_topk followed by a gather of
 * out_rows for every layer -- out_rows, out_stats, hot state and pool bytes identical, and
 * out[l][(r*P + p)*K + k] = layer layer_begin + l's row of topk_ids[l/G][r][p][k], for l < nl.  The miss copy is fused
 * into the gather: the resolver lists each missed id once with its host row and links the id's
 * repeated positions (other query positions of a multi-position plan), and the gather reads each
 * such row once from the pinned host pool and stores it into its hot slot and into every position
 * of the id, while resident and hit rows come from HBM in the same launch, so host-link and HBM
 * traffic overlap instead of running back to back.  The consumer then reads hot rows as ordinary pool rows
 * (Japanese article, section "仕組み": the sparse MLA kernel sees hot pages as normal pages).
 * Equivalent to hs_resolve_plan followed by hs_gather_planned on the same stream.
 *   out        device [nl][R*P*K][row_bytes] bytes, 16-byte aligned.
 *   workspace  as for hs_resolve_topk (hs_resolve_workspace_bytes covers every resolve call). */
hs_status hs_resolve_gather(const hs_pool* pool, int32_t layer_begin, int32_t nl, int32_t R, int32_t P,
                            int32_t K, const int32_t* topk_ids, const int32_t* block_table,
                            const int32_t* host_block_table, const int32_t* ctx_len, int32_t max_pages,
                            const hs_hot_state* hot, int32_t step, int32_t* out_rows, int32_t* out_stats,
                            void* out, void* workspace, size_t workspace_bytes, hs_stream_t stream);

/* First half of hs_resolve_gather (one launch; two with the ordered miss layout, whose counters a
 * small kernel clears first): everything hs_resolve_topk does except the miss copies.  Rows, stats and hot state are final; the victims' pool rows are NOT yet filled -- the
 * per-position host sources wait in `workspace` for hs_gather_planned, which must follow on the same
 * stream before anything reads those rows.  Same arguments as hs_resolve_topk. */
hs_status hs_resolve_plan(const hs_pool* pool, int32_t layer_begin, int32_t nl, int32_t R, int32_t P,
                          int32_t K, const int32_t* topk_ids, const int32_t* block_table,
                          const int32_t* host_block_table, const int32_t* ctx_len, int32_t max_pages,
                          const hs_hot_state* hot, int32_t step, int32_t* out_rows, int32_t* out_stats,
                          void* workspace, size_t workspace_bytes, hs_stream_t stream);

/* Second half of hs_resolve_gather (one launch): gathers all nl*R*P*K rows named by out_rows into
 * `out`, taking miss rows from the pinned host pool as recorded by hs_resolve_plan in `workspace`
 * and filling their hot slots in every layer.  nl, R, P, K, layer_begin, hot (only its capacity and
 * layers_per_index are read), out_rows, workspace and workspace_bytes must be those of the preceding
 * hs_resolve_plan call, and the pool's miss order (hs_pool_set_miss_order) must not change in between. */
hs_status hs_gather_planned(const hs_pool* pool, int32_t layer_begin, int32_t nl, int32_t R, int32_t P,
                            int32_t K, const hs_hot_state* hot, const int32_t* out_rows, const void* workspace,
                            size_t workspace_bytes, void* out, hs_stream_t stream);

/* Single-stride gather: out[l][i] = row rows[l][i] of layer layer_begin + l, for l < nl, i < n.
 *   rows        device int32 [nl][n]; -1 gives row_bytes zero bytes.
 *   out         device [nl][n][row_bytes] bytes, 16-byte aligned.
 *   out_status  optional device int32 (may be NULL): set to HS_ERR_ID_RANGE when a row id is
 *               outside [-1, num_gpu_blocks*page_size) (that output row is zero-filled); never
 *               written otherwise, so the caller zeroes it. */
hs_status hs_gather_rows(const hs_pool* pool, int32_t layer_begin, int32_t nl, const int32_t* rows,
                         int64_t n, void* out, int32_t* out_status, hs_stream_t stream);

/* Post-forward proactive offload, one launch for all layers: for every pair i < n and every layer
 * l, host page host_blocks[i] of layer l := GPU page gpu_blocks[i] of layer l (page_size*row_bytes
 * bytes).  The GPU block may be reused by later work on the same stream as soon as this call
 * returns; the host copy is complete when the stream reaches this point.
 *   gpu_blocks, host_blocks  device int32 [n].
 *   out_status  optional device int32: set to HS_ERR_TABLE_RANGE if a pair is out of range (that
 *               pair is skipped). */
hs_status hs_offload_pages(const hs_pool* pool, const int32_t* gpu_blocks, const int32_t* host_blocks,
                           int32_t n, int32_t* out_status, hs_stream_t stream);

/* hs_resolve_topk for callers that cannot allocate device memory (a plug-in inside an engine that has
 * reserved nearly all device memory, a decode loop that must not let cudaMalloc synchronise the
 * device, a C caller without a device allocator).  The pages have no counterpart: this is a library
 * convenience.  Same arguments and results as hs_resolve_topk, minus the workspace: the scratch is a
 * static __device__ array of HS_STATIC_SCRATCH_BYTES inside the library, held by every GPU that loads
 * the library until the process exits.  No call allocates anything.
 *   - Returns HS_ERR_INVALID_ARG when hs_resolve_workspace_bytes_min(nl / G, R, P, K, capacity)
 *     exceeds HS_STATIC_SCRATCH_BYTES, with G = hot->layers_per_index (the resolver's units are
 *     index groups; G = 1 without IndexShare): about 340 units of the MTP3 shape P*K = 8192,
 *     C = 4096, or about 800 units of K = 2048, C = 4096.  The ordered miss layout is used only where
 *     it fits too.
 *   - Returns HS_ERR_INVALID_ARG when the current device is not the pool's device.
 *   - The first call in each CUDA context looks up the array's device address (cudaGetSymbolAddress,
 *     with the pool's device current) and caches it for that context; make that first call before
 *     any stream capture.  A context created anew (after cudaDeviceReset, or after the primary
 *     context was released) is a new context: its first call looks the address up again, so it too
 *     should come before any capture.
 *   - Every call shares the one array and it keeps the last call's contents (nothing in it needs to
 *     start at zero).  Calls whose executions overlap on the GPU -- on different streams, or from
 *     different threads without ordering -- race on it; order them on one stream. */
#define HS_STATIC_SCRATCH_BYTES (32u << 20)
hs_status hs_resolve_topk_noalloc(const hs_pool* pool, int32_t layer_begin, int32_t nl, int32_t R, int32_t P,
                                  int32_t K, const int32_t* topk_ids, const int32_t* block_table,
                                  const int32_t* host_block_table, const int32_t* ctx_len, int32_t max_pages,
                                  const hs_hot_state* hot, int32_t step, int32_t* out_rows, int32_t* out_stats,
                                  hs_stream_t stream);

/* Static description of a status code. */
const char* hs_status_str(hs_status s);

/* Number of kernels the library has launched since load (a host-side counter). */
int64_t hs_launch_count(void);

/* Bounds-checked build of the library (compiled with HS_CHECKED=1; sparse_mla_kv_gb300/libhs_checked.so)
 * only -- a debugging aid with no counterpart in the pages.  In that build every address a kernel
 * derives from data it read (a table entry, a slot index, a miss-list entry, a repeat-chain link, an
 * output position) is checked against the extent of its buffer before the access, and a violation
 * skips the access and is recorded.  Synchronises the current device, then returns the site of the
 * first violation recorded since the previous call and clears it:
 *   0 none; 1 table page; 2 hot-state slot; 3 miss-list index; 4 GPU pool row; 5 host pool row;
 *   6 output position; 7 repeat-chain link; -2 the device or the record could not be read.
 * Returns -1 in the normal build, which compiles these checks away (its data errors are reported
 * through the status words described above). */
int32_t hs_check_status(void);

#ifdef __cplusplus
}
#endif

#endif /* HS_H_ */
