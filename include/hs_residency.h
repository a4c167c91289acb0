/*
 * hs_residency.h -- C ABI of the host-side residency manager that prepares the resolver's tables.
 *
 * Host code only (no device memory, no CUDA calls).  It decides which pages of each request are on
 * the GPU, which exist in the pinned host pool, and which GPU blocks serve as each request's hot
 * buffer; hs_resolve_topk / hs_resolve_gather (hs.h) then read the tables it exports.
 *
 * Passages it implements:
 *   - Japanese article (news.ainew.jp), the section before "仕組み" (the A/B example): under KV
 *     pressure each request frees its least recently used (cold) pages in place, and the freed blocks
 *     are reused as new tail pages and hot pages, so that every request keeps decoding.
 *   - "仕組み" (How it works): residency is tracked per page; the tail never leaves the GPU; hot pages
 *     are ordinary KV blocks leased from the same pool as resident pages when a request first needs
 *     them and returned when it no longer does; a block freed by one request can serve as another
 *     request's hot capacity; a completed prefix page's CPU copy is queued while the GPU keeps
 *     serving it, so the page can later give up its block without another copy, and the block may
 *     be reused once the copy has been queued (stream order).
 *
 * Policy (fixed where the pages are silent; every result is unique):
 *   - GPU and host blocks are handed out lowest free id first.
 *   - A request's tail is its last page.  A page is complete when it lies below ctx_len / page_size.
 *   - A page may be released when it is resident, complete, not the tail, has a host copy, and its
 *     offload has been collected (hs_res_collect).  The request that needs a block releases its own
 *     page with the smallest (last use, page) first, else the page with the smallest
 *     (last use, request, page) of any other request.  Last use is the last step hs_res_touch saw
 *     the page selected (-1: never).
 *   - A request leases its hot buffer (hot_blocks_per_request blocks, taken one by one like any
 *     other block) when it first has a placeholder page: at admission with a reused host prefix, or
 *     when its first page is released.  It keeps it until hs_res_finish.  A request is listed by
 *     hs_res_take_resets when it leases, so the caller empties its slots (hs_hot_reset_requests).
 *   - Host blocks are reference-counted: pages of requests (a reused prefix may be shared) and the
 *     caller's holds (hs_res_hold_host, e.g. a prefix cache).  A block is free at zero references.
 *   - A call that cannot find a block returns HS_ERR_CAPACITY: a failed admission leaves the request
 *     not admitted, a failed append leaves the context unchanged (blocks taken for its new pages are
 *     returned); releases made before the failure stay (each leaves a valid state).
 *
 * Typical decode step: hs_res_append_all (or hs_res_append per request) for the new tokens;
 * hs_res_take_fills (the model writes those blocks); hs_res_tables and hs_res_take_resets (copied to the
 * device: tables, and hs_hot_reset_requests for the listed requests); the resolver and gather;
 * hs_res_touch_all (or hs_res_touch per request) with the step's top-K; after the forward pass
 * hs_res_collect and one hs_offload_pages launch with the pairs.
 *
 * Not thread-safe: one caller at a time per manager.
 */
#ifndef HS_RESIDENCY_H_
#define HS_RESIDENCY_H_

#include <stdint.h>

#include "hs.h"

#ifdef __cplusplus
extern "C" {
#endif

typedef struct hs_residency hs_residency; /* opaque */

/* A manager for GPU blocks [0, num_gpu_blocks) and host blocks [0, num_host_blocks), all free,
 * request slots [0, max_requests) of at most max_pages pages each.  HS_ERR_INVALID_ARG on a bad
 * size (*out = NULL). */
hs_status hs_res_create(int32_t num_gpu_blocks, int32_t num_host_blocks, int32_t page_size, int32_t max_requests,
                        int32_t max_pages, int32_t hot_blocks_per_request, hs_residency** out);
void hs_res_destroy(hs_residency* m);

/* Admits request slot r (inactive) with ctx_len tokens.  Its first n_prefix pages are a reused
 * prefix that exists only in host memory, at prefix_host_blocks[0..n_prefix) (one reference each);
 * n_prefix <= (ctx_len - 1) / page_size, since the prompt's last token is always computed.  The other
 * pages get GPU blocks (listed by hs_res_take_fills: the prefill writes them); those complete get a
 * host block and a queued offload.  A prefix makes the request lease its hot buffer first. */
hs_status hs_res_admit(hs_residency* m, int32_t r, int32_t ctx_len, const int32_t* prefix_host_blocks,
                       int32_t n_prefix);

/* n_tokens >= 0 tokens appended to active request r: each page that starts gets a GPU block (a fill),
 * each page that completes gets a host block and a queued offload. */
hs_status hs_res_append(hs_residency* m, int32_t r, int32_t n_tokens);

/* hs_res_append for every request r with n_tokens[r] != 0, in request order (n_tokens is a host array
 * [max_requests]; zero entries, e.g. of inactive requests, are skipped).  One call per decode step
 * instead of one per request.  Stops at the first failing request and returns its status: the
 * requests before it keep their appends, it is left as a failed hs_res_append leaves it, and the
 * requests after it are not appended. */
hs_status hs_res_append_all(hs_residency* m, const int32_t* n_tokens);

/* The indexer selected ids[0..n) of request r at decode step `step` (non-decreasing across calls):
 * their pages' last use becomes `step`.  Ids outside [0, ctx_len) are ignored. */
hs_status hs_res_touch(hs_residency* m, int32_t r, const int32_t* ids, int64_t n, int32_t step);

/* hs_res_touch for every active request at once: ids is a host array [max_requests][n_per_request]
 * (row r holds request r's ids; entries outside [0, ctx_len) -- e.g. -1 padding -- are ignored, and the
 * rows of inactive requests are skipped).  One call per decode step instead of one per request. */
hs_status hs_res_touch_all(hs_residency* m, const int32_t* ids, int32_t n_per_request, int32_t step);

/* Request r leaves: its GPU blocks (pages and hot buffer) return to the pool, its host references are
 * dropped, and its queued offloads and fills are discarded. */
hs_status hs_res_finish(hs_residency* m, int32_t r);

/* The caller takes / drops one reference on each of blocks[0..n) of the host pool.  Dropping a
 * reference the caller does not hold is HS_ERR_INVALID_ARG (nothing changes). */
hs_status hs_res_hold_host(hs_residency* m, const int32_t* blocks, int32_t n);
hs_status hs_res_drop_host(hs_residency* m, const int32_t* blocks, int32_t n);

/* Numbers of queued offloads, pending hot resets and pending fills (sizes for the calls below). */
void hs_res_counts(const hs_residency* m, int32_t* queued, int32_t* resets, int32_t* fills);
int32_t hs_res_free_gpu_blocks(const hs_residency* m);

/* Moves the queued offloads, in queue order, to gpu_blocks / host_blocks (host arrays of at least
 * `capacity` entries) -- the pairs for the post-forward hs_offload_pages launch -- and empties the
 * queue; *n_out = their number.  HS_ERR_INVALID_ARG (nothing moved) if capacity is too small. */
hs_status hs_res_collect(hs_residency* m, int32_t* gpu_blocks, int32_t* host_blocks, int32_t capacity,
                         int32_t* n_out);

/* Moves the requests that leased a hot buffer since the last call (in lease order). */
hs_status hs_res_take_resets(hs_residency* m, int32_t* requests, int32_t capacity, int32_t* n_out);

/* Moves the (block, request, page) triples whose GPU block was assigned to a page since the last
 * call, in assignment order: the caller writes those pages' rows before the next forward pass. */
hs_status hs_res_take_fills(hs_residency* m, int32_t* blocks, int32_t* requests, int32_t* pages, int32_t capacity,
                            int32_t* n_out);

/* Writes the resolver's tables to host arrays: block_table and host_block_table
 * [max_requests][max_pages] (-1: placeholder / no host copy), hot_blocks
 * [max_requests][hot_blocks_per_request] (-1 until a buffer is leased), ctx_len [max_requests]
 * (0 for an inactive slot).  Any pointer may be NULL to skip that table. */
hs_status hs_res_tables(const hs_residency* m, int32_t* block_table, int32_t* host_block_table, int32_t* hot_blocks,
                        int32_t* ctx_len);

#ifdef __cplusplus
}
#endif

#endif /* HS_RESIDENCY_H_ */
