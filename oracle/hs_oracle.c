/*
 * Oracle for the Hybrid HiSparse top-K resolver: a plain, slow, sequential-per-unit CPU
 * implementation of resolve / gather / offload.
 *
 * TEST INFRASTRUCTURE ONLY.  Only the tests, the smoke check and the bench's CPU-baseline leg may
 * load it.  It shares no code, header, table or helper with the CUDA library and must never be used
 * as a fallback for it.
 *
 * What it follows (steps in the order the pages describe them):
 *   - "vLLM GLM 5.3 Optimizations: Hybrid HiSparse Offloading", "Technical Implementation of Hybrid
 *     HiSparse", item 2: resident tokens are read in place, hot tokens are read and their LRU entry
 *     refreshed, a miss copies a single row from pinned host memory into an LRU slot.
 *   - Japanese article, "仕組み" (How it works), figure caption: a miss copies one row into a hot
 *     page, a hit reuses it without a copy; the block table holds real blocks and null
 *     placeholders; rows are handed back as pool row ids and gathered with one stride.
 *   - Same section: a completed prefix page's CPU copy is queued while the GPU keeps serving it;
 *     all sparse-MLA layers are copied in a single launch after the forward pass.
 *   - "vLLM の他の部分との統合" (Integration): speculative decoding works through a per-step
 *     replayable resolver plan that shares the request's hot state.
 *   - "必要な時にスパーシティを活用する" (Using sparsity when it is needed): under GLM 5.3's IndexShare
 *     one indexer layer serves four sparse-MLA layers, so those layers select the same top-K.  Read
 *     here as: an index group of G consecutive layers has one top-K list and one LRU state per
 *     request; its decisions are made once, and each miss copies the token's row of every layer of
 *     the group (G = 1 is the plain per-layer case).
 * The LRU details the pages leave open are fixed as: hits are refreshed before victims are chosen;
 * victims are the smallest (last-used step, slot) among slots not used in this step; misses take
 * them in plan order (first occurrence, position-major then top-K order).
 *
 * Each unit (index group, request) is processed by hso_resolve_unit, one plain pass per step of the
 * method; library qsort is the only primitive.  Units are independent, so hso_resolve runs them on
 * an OpenMP loop (the order of independent units does not change any result).
 */
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

enum {
  ST_OK = 0,
  ST_INVALID_ARG = 1,
  ST_ID_RANGE = 2,
  ST_MISSING_ROW = 3,
  ST_CAPACITY = 4,
  ST_STEP_ORDER = 5,
  ST_TABLE_RANGE = 8
};

enum { CLS_NONE = 0, CLS_RESIDENT = 1, CLS_HIT = 2, CLS_MISS = 3 };

typedef struct { int32_t key; int32_t idx; } pair_t;

static int cmp_pair(const void* a, const void* b) {
  const pair_t* x = (const pair_t*)a;
  const pair_t* y = (const pair_t*)b;
  if (x->key != y->key) return x->key < y->key ? -1 : 1;
  if (x->idx != y->idx) return x->idx < y->idx ? -1 : 1;
  return 0;
}

/* Binary search in pairs sorted by (key, idx): index of the first pair with this key, or -1. */
static int32_t find_first(const pair_t* v, int32_t n, int32_t key) {
  int32_t lo = 0, hi = n;
  while (lo < hi) {
    int32_t mid = lo + (hi - lo) / 2;
    if (v[mid].key < key) lo = mid + 1; else hi = mid;
  }
  return (lo < n && v[lo].key == key) ? lo : -1;
}

static int64_t hot_row(const int32_t* hot_blocks_r, int32_t S, int32_t slot) {
  return (int64_t)hot_blocks_r[slot / S] * S + slot % S;
}

/*
 * One unit.  ids: [n] (n = P*K, position-major).  bt/hbt: this request's rows of the tables.
 * tok/stamp: this unit's C slots (updated in place unless an error is found).  pools/hosts: the
 * byte arrays of the G layers of this unit's index group, or NULL to skip byte work.
 * out_rows: [n]; out_stats: [4].  Returns the status (also written to out_stats[0]).
 */
int32_t hso_resolve_unit(int32_t S, int32_t B, int32_t num_gpu_blocks, int32_t num_host_blocks, int32_t G,
                         uint8_t* const* pools, uint8_t* const* hosts, int32_t n, const int32_t* ids,
                         const int32_t* bt, const int32_t* hbt, int32_t ctx_len, int32_t max_pages,
                         int32_t C, const int32_t* hot_blocks_r, int32_t* tok, int32_t* stamp,
                         int32_t step, int32_t* out_rows, int32_t* out_stats) {
  int32_t i, j, s;
  int err_step = 0, err_id = 0, err_table = 0, err_missing = 0, err_capacity = 0, hot_bad = 0;

  /* Step 1: validate what needs no classification. */
  for (s = 0; s < C; s++)
    if (stamp[s] > step) err_step = 1;
  for (i = 0; i < n; i++) {
    int32_t id = ids[i];
    if (id == -1) continue;
    if (id < -1 || id >= ctx_len || id / S >= max_pages) err_id = 1;
  }
  /* hot blocks are dereferenced only by hits and misses; checked after classification */
  for (j = 0; j < C / S; j++)
    if (hot_blocks_r[j] < 0 || hot_blocks_r[j] >= num_gpu_blocks) hot_bad = 1;

  pair_t* by_id = (pair_t*)malloc(sizeof(pair_t) * (size_t)(n > 0 ? n : 1));
  pair_t* by_tok = (pair_t*)malloc(sizeof(pair_t) * (size_t)(C > 0 ? C : 1));
  int32_t* first = (int32_t*)malloc(sizeof(int32_t) * (size_t)(n > 0 ? n : 1));
  int32_t* cls = (int32_t*)calloc((size_t)(n > 0 ? n : 1), sizeof(int32_t));
  int64_t* row = (int64_t*)malloc(sizeof(int64_t) * (size_t)(n > 0 ? n : 1));
  int32_t* slot_of = (int32_t*)malloc(sizeof(int32_t) * (size_t)(n > 0 ? n : 1));
  int64_t* src = (int64_t*)malloc(sizeof(int64_t) * (size_t)(n > 0 ? n : 1));
  int32_t* hit_slot = (int32_t*)calloc((size_t)(C > 0 ? C : 1), sizeof(int32_t));
  pair_t* cand = (pair_t*)malloc(sizeof(pair_t) * (size_t)(C > 0 ? C : 1));
  int32_t nres = 0, nhit = 0, nmiss = 0, ncand = 0;

  if (!err_step && !err_id) {
    /* Step 2: the plan -- distinct non-padding ids in first-occurrence order.  first[i] is the
     * index of the first occurrence of ids[i]; position i is in the plan iff first[i] == i. */
    int32_t m = 0;
    for (i = 0; i < n; i++)
      if (ids[i] >= 0) { by_id[m].key = ids[i]; by_id[m].idx = i; m++; }
    qsort(by_id, (size_t)m, sizeof(pair_t), cmp_pair);
    for (i = 0; i < n; i++) first[i] = -1;
    int32_t group_first = -1;
    for (j = 0; j < m; j++) {
      /* sorted by (id, position): the first pair of each id group holds its smallest position */
      if (j == 0 || by_id[j].key != by_id[j - 1].key) group_first = by_id[j].idx;
      first[by_id[j].idx] = group_first;
    }

    /* token -> lowest slot holding it */
    int32_t nt = 0;
    for (s = 0; s < C; s++)
      if (tok[s] >= 0) { by_tok[nt].key = tok[s]; by_tok[nt].idx = s; nt++; }
    qsort(by_tok, (size_t)nt, sizeof(pair_t), cmp_pair);

    /* Step 3: classify each plan entry (in plan order = increasing position). */
    for (i = 0; i < n; i++) {
      if (ids[i] < 0 || first[i] != i) continue;
      int32_t id = ids[i];
      int32_t page = id / S, off = id % S;
      if (bt[page] >= 0) {
        if (bt[page] >= num_gpu_blocks) err_table = 1;
        cls[i] = CLS_RESIDENT;
        row[i] = (int64_t)bt[page] * S + off;
        nres++;
      } else {
        int32_t f = find_first(by_tok, nt, id);
        if (f >= 0) {
          cls[i] = CLS_HIT;
          slot_of[i] = by_tok[f].idx;
          hit_slot[by_tok[f].idx] = 1;
          nhit++;
        } else {
          cls[i] = CLS_MISS;
          if (hbt[page] < 0) err_missing = 1;
          else if (hbt[page] >= num_host_blocks) err_table = 1;
          else src[i] = (int64_t)hbt[page] * S + off;
          nmiss++;
        }
      }
    }

    /* A unit with a hit or a miss reads or writes its hot blocks: they must lie in the pool. */
    if (hot_bad && nhit + nmiss > 0) err_table = 1;

    /* Step 4: capacity -- evictable slots are those not used in this step (stamp < step) and
     * not hit now. */
    for (s = 0; s < C; s++)
      if (stamp[s] < step && !hit_slot[s]) { cand[ncand].key = stamp[s]; cand[ncand].idx = s; ncand++; }
    if (nmiss > ncand) err_capacity = 1;
  }

  int32_t status = err_step ? ST_STEP_ORDER
                 : err_id ? ST_ID_RANGE
                 : err_table ? ST_TABLE_RANGE
                 : err_missing ? ST_MISSING_ROW
                 : err_capacity ? ST_CAPACITY
                 : ST_OK;

  if (status != ST_OK) {
    for (i = 0; i < n; i++) out_rows[i] = -1;
    out_stats[0] = status; out_stats[1] = 0; out_stats[2] = 0; out_stats[3] = 0;
  } else {
    /* Step 5: refresh the hits. */
    for (i = 0; i < n; i++)
      if (cls[i] == CLS_HIT) {
        stamp[slot_of[i]] = step;
        row[i] = hot_row(hot_blocks_r, S, slot_of[i]);
      }
    /* Step 6: victims in ascending (stamp, slot); the j-th miss in plan order takes the j-th. */
    qsort(cand, (size_t)ncand, sizeof(pair_t), cmp_pair);
    j = 0;
    for (i = 0; i < n; i++) {
      if (cls[i] != CLS_MISS) continue;
      int32_t v = cand[j++].idx;
      tok[v] = ids[i];
      stamp[v] = step;
      row[i] = hot_row(hot_blocks_r, S, v);
      if (pools && hosts) {
        for (int32_t g = 0; g < G; g++) {  /* the same row of every layer of the index group */
          uint8_t* pool = pools[g];
          const uint8_t* host = hosts[g];
          memcpy(pool + row[i] * (int64_t)B, host + src[i] * (int64_t)B, (size_t)B);
        }
      }
    }
    /* Step 7: emit a row for every position (duplicates share their first occurrence's row). */
    for (i = 0; i < n; i++)
      out_rows[i] = ids[i] < 0 ? -1 : (int32_t)row[first[i]];
    out_stats[0] = ST_OK; out_stats[1] = nres; out_stats[2] = nhit; out_stats[3] = nmiss;
  }

  free(by_id); free(by_tok); free(first); free(cls); free(row); free(slot_of); free(src);
  free(hit_slot); free(cand);
  return status;
}

/*
 * All units of one call: layers [layer_begin, layer_begin+nl) x R requests, in index groups of G
 * consecutive layers (layer_begin and nl multiples of G).  With ng = nl/G:
 * topk/out_rows: [ng][R][n]; out_stats: [ng][R][4]; tok/stamp: [num_layers/G][R][C];
 * bt/hbt: [R][max_pages]; hot_blocks: [R][C/S]; pools/hosts: [num_layers] byte arrays or NULL.
 */
void hso_resolve(int32_t S, int32_t B, int32_t num_gpu_blocks, int32_t num_host_blocks,
                 uint8_t** pools, uint8_t** hosts, int32_t G, int32_t layer_begin, int32_t nl, int32_t R,
                 int32_t n, const int32_t* topk, const int32_t* bt, const int32_t* hbt,
                 const int32_t* ctx_len, int32_t max_pages, int32_t C, const int32_t* hot_blocks,
                 int32_t* tok, int32_t* stamp, int32_t step, int32_t* out_rows, int32_t* out_stats,
                 int32_t threads) {
  int64_t u;
  int64_t units = (int64_t)(nl / G) * R;
#pragma omp parallel for schedule(dynamic, 1) num_threads(threads > 0 ? threads : 1)
  for (u = 0; u < units; u++) {
    int32_t gr = (int32_t)(u / R), r = (int32_t)(u % R);
    int32_t grp = layer_begin / G + gr;   /* index group; its layers are grp*G .. grp*G + G-1 */
    hso_resolve_unit(S, B, num_gpu_blocks, num_host_blocks, G, pools ? pools + (int64_t)grp * G : NULL,
                     hosts ? hosts + (int64_t)grp * G : NULL, n, topk + u * n, bt + (int64_t)r * max_pages,
                     hbt + (int64_t)r * max_pages, ctx_len[r], max_pages, C,
                     hot_blocks + (int64_t)r * (C / S), tok + ((int64_t)grp * R + r) * C,
                     stamp + ((int64_t)grp * R + r) * C, step, out_rows + u * n, out_stats + u * 4);
  }
}

/* Gather: out[l][i] = row rows[l][i] of pools[layer_begin + l]; -1 -> zeros; a row outside
 * [-1, num_rows) -> zeros and the return value is ST_ID_RANGE. */
int32_t hso_gather(int32_t B, int64_t num_rows, uint8_t** pools, int32_t layer_begin, int32_t nl,
                   const int32_t* rows, int64_t n, uint8_t* out, int32_t threads) {
  int32_t status = ST_OK;
  int64_t k;
#pragma omp parallel for schedule(static) num_threads(threads > 0 ? threads : 1)
  for (k = 0; k < (int64_t)nl * n; k++) {
    int32_t l = (int32_t)(k / n);
    int32_t r = rows[k];
    uint8_t* dst = out + k * (int64_t)B;
    if (r >= 0 && (int64_t)r < num_rows) {
      memcpy(dst, pools[layer_begin + l] + (int64_t)r * B, (size_t)B);
    } else {
      memset(dst, 0, (size_t)B);
      if (r != -1) {
#pragma omp atomic write
        status = ST_ID_RANGE;
      }
    }
  }
  return status;
}

/* Offload: for every pair i and layer l, host page hb[i] of layer l := GPU page gb[i] of layer l.
 * A pair out of range is skipped and the return value is ST_TABLE_RANGE. */
int32_t hso_offload(int32_t S, int32_t B, int32_t num_layers, int32_t num_gpu_blocks,
                    int32_t num_host_blocks, uint8_t** pools, uint8_t** hosts, const int32_t* gb,
                    const int32_t* hb, int32_t n) {
  int32_t status = ST_OK;
  int64_t page = (int64_t)S * B;
  for (int32_t i = 0; i < n; i++) {
    if (gb[i] < 0 || gb[i] >= num_gpu_blocks || hb[i] < 0 || hb[i] >= num_host_blocks) {
      status = ST_TABLE_RANGE;
      continue;
    }
    for (int32_t l = 0; l < num_layers; l++)
      memcpy(hosts[l] + (int64_t)hb[i] * page, pools[l] + (int64_t)gb[i] * page, (size_t)page);
  }
  return status;
}
