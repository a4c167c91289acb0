// Host-side residency manager (see hs_residency.h for the policy and the passages it follows).
//
// Data structures: the free GPU blocks and the free host blocks are min-heaps (lowest id first; a
// host entry is valid only while its block has no reference, so stale entries are skipped lazily).
// Each request keeps, besides its page tables, its releasable pages in a doubly-linked list sorted by
// (last use, page); a page's membership is recomputed whenever one of its conditions changes, so
// choosing a victim reads one list head per request.  A touch moves pages to the newest step, which
// sorts after every other key: they are unlinked and appended in page order, O(1) each (a page
// entering the list for another reason is placed by a walk from the tail, where recent keys are).
#include <algorithm>
#include <cstdint>
#include <functional>
#include <new>
#include <queue>
#include <utility>
#include <vector>

#include "hs_residency.h"

namespace {

struct Capacity {};  // thrown inside the manager when no block can be found; never crosses the ABI

struct Request {
  bool active = false;
  int32_t ctx = 0;
  std::vector<int32_t> bt, hbt, lu;
  std::vector<char> pending;       // offload queued, not yet collected
  std::vector<char> in_set;        // page is in the releasable list
  bool leased = false;             // hot buffer leased (possibly in progress)
  std::vector<int32_t> hot;
  // releasable pages, ascending (last use, page): head = the coldest; -1 ends the list
  std::vector<int32_t> nxt, prv;
  int32_t head = -1, tail = -1;

  bool before(int32_t a, int32_t b) const { return lu[a] < lu[b] || (lu[a] == lu[b] && a < b); }
  void unlink(int32_t p) {
    const int32_t a = prv[p], b = nxt[p];
    (a >= 0 ? nxt[a] : head) = b;
    (b >= 0 ? prv[b] : tail) = a;
  }
  // links p at its place, searching from the tail (its key must not be in the list yet)
  void link_sorted(int32_t p) {
    int32_t q = tail;
    while (q >= 0 && before(p, q)) q = prv[q];
    const int32_t b = q >= 0 ? nxt[q] : head;
    prv[p] = q;
    nxt[p] = b;
    (q >= 0 ? nxt[q] : head) = p;
    (b >= 0 ? prv[b] : tail) = p;
  }
};

struct QueuedCopy {
  int32_t gpu, host, r, p;
};

struct Fill {
  int32_t block, r, p;
};

}  // namespace

struct hs_residency {
  int32_t S, max_pages, Hc;
  int32_t S_shift;  // log2(S) when S is a power of two, else -1
  std::priority_queue<int32_t, std::vector<int32_t>, std::greater<int32_t>> free_gpu;
  std::priority_queue<int32_t, std::vector<int32_t>, std::greater<int32_t>> free_host;  // lazy
  std::vector<int32_t> host_ref, host_held;
  int32_t host_free_count = 0;
  std::vector<Request> req;
  std::vector<int32_t> moved;   // touch's scratch (kept between calls)
  std::vector<uint64_t> seen;   // touch's page bits
  std::vector<QueuedCopy> queue;
  std::vector<int32_t> resets;
  std::vector<Fill> fills;

  // ------------------------------------------------------------------ pools
  void host_unref(int32_t h) {
    if (--host_ref[h] == 0) {
      free_host.push(h);
      ++host_free_count;
    }
  }
  void host_ref_add(int32_t h) {
    if (host_ref[h]++ == 0) --host_free_count;  // its heap entry goes stale
  }
  int32_t alloc_host() {
    while (!free_host.empty()) {
      const int32_t h = free_host.top();
      free_host.pop();
      if (host_ref[h] == 0) {
        host_ref[h] = 1;
        --host_free_count;
        return h;
      }
    }
    throw Capacity{};
  }

  // ------------------------------------------------------------------ releasable pages
  bool releasable_now(const Request& x, int32_t p) const {
    const int32_t last = (x.ctx + S - 1) / S - 1;
    return p < last && p < x.ctx / S && x.bt[p] >= 0 && x.hbt[p] >= 0 && !x.pending[p];
  }
  void refresh(Request& x, int32_t p) {
    if (p < 0 || p >= max_pages) return;
    const bool want = releasable_now(x, p);
    if (want == (bool)x.in_set[p]) return;
    if (want) x.link_sorted(p);
    else x.unlink(p);
    x.in_set[p] = want;
  }
  void set_ctx(Request& x, int32_t ctx) {
    const int32_t old_last = (x.ctx + S - 1) / S - 1;
    x.ctx = ctx;
    refresh(x, old_last);  // the old tail may have become releasable
  }

  // ------------------------------------------------------------------ allocation under pressure
  bool pick_cold(int32_t r, int32_t* q_out, int32_t* p_out) const {
    const Request& own = req[r];
    if (own.head >= 0) {
      *q_out = r;
      *p_out = own.head;
      return true;
    }
    bool found = false;
    int32_t best_lu = 0, best_q = 0, best_p = 0;
    for (int32_t q = 0; q < (int32_t)req.size(); ++q) {
      const Request& x = req[q];
      if (q == r || !x.active || x.head < 0) continue;
      const int32_t lu = x.lu[x.head];
      if (!found || lu < best_lu) {  // ties on last use: the lower request index (scanned first)
        found = true;
        best_lu = lu;
        best_q = q;
        best_p = x.head;
      }
    }
    *q_out = best_q;
    *p_out = best_p;
    return found;
  }
  void release(int32_t q, int32_t p) {
    Request& x = req[q];
    const int32_t b = x.bt[p];
    x.bt[p] = -1;
    refresh(x, p);
    free_gpu.push(b);
    if (!x.leased) lease_hot(q);
  }
  void lease_hot(int32_t q) {
    Request& x = req[q];
    x.leased = true;
    x.hot.clear();
    const bool added = std::find(resets.begin(), resets.end(), q) == resets.end();
    if (added) resets.push_back(q);
    try {
      for (int32_t k = 0; k < Hc; ++k) x.hot.push_back(alloc_gpu(q));
    } catch (const Capacity&) {  // all or nothing: the next release tries again
      for (int32_t b : x.hot) free_gpu.push(b);
      x.hot.clear();
      x.leased = false;
      if (added) resets.erase(std::find(resets.begin(), resets.end(), q));
      throw;
    }
  }
  int32_t alloc_gpu(int32_t r) {
    while (free_gpu.empty()) {
      int32_t q, p;
      if (!pick_cold(r, &q, &p)) throw Capacity{};
      release(q, p);
    }
    const int32_t b = free_gpu.top();
    free_gpu.pop();
    return b;
  }
  void complete(int32_t r, int32_t p) {
    Request& x = req[r];
    const int32_t h = alloc_host();
    x.hbt[p] = h;
    x.pending[p] = 1;
    refresh(x, p);
    queue.push_back({x.bt[p], h, r, p});
  }

  // ------------------------------------------------------------------ operations
  void finish(int32_t r) {
    Request& x = req[r];
    queue.erase(std::remove_if(queue.begin(), queue.end(), [r](const QueuedCopy& c) { return c.r == r; }),
                queue.end());
    for (int32_t p = 0; p < max_pages; ++p) {
      if (x.bt[p] >= 0) free_gpu.push(x.bt[p]);
      if (x.hbt[p] >= 0) host_unref(x.hbt[p]);
    }
    for (int32_t b : x.hot) free_gpu.push(b);
    x = Request{};
    resets.erase(std::remove(resets.begin(), resets.end(), r), resets.end());
    fills.erase(std::remove_if(fills.begin(), fills.end(), [r](const Fill& f) { return f.r == r; }), fills.end());
  }

  // The pages of ids[0..n) were used at `step` (not older than any last use).  A releasable page whose
  // last use changes is unlinked, and all of them are linked again in page order: with the new key
  // (step, page) each lands at the tail, behind any page touched earlier in this step with a lower id.
  void touch(int32_t r, const int32_t* ids, int64_t n, int32_t step) {
    Request& x = req[r];
    moved.clear();
    // pass 1: the pages of the valid ids, as bits, in four interleaved bitmaps (the ids of one request
    // fall on few words, and four independent read-modify-write chains run about 3x faster than one);
    // pass 2: each page once, in page order
    const uint32_t ctx = (uint32_t)x.ctx;  // one unsigned compare rejects negative ids too
    const int32_t words = (max_pages + 63) / 64;
    const size_t stride = (size_t)words + 1;  // word `words` of each bitmap absorbs the invalid ids
    seen.assign(4 * stride, 0);
    uint64_t* const bm = seen.data();
    const uint32_t sink = (uint32_t)words * 64;
    auto page = [&](uint32_t t) -> uint32_t {
      return t < ctx ? (S_shift >= 0 ? t >> S_shift : t / (uint32_t)S) : sink;
    };
    int64_t i = 0;
    for (; i + 4 <= n; i += 4) {
      const uint32_t p0 = page((uint32_t)ids[i]), p1 = page((uint32_t)ids[i + 1]);
      const uint32_t p2 = page((uint32_t)ids[i + 2]), p3 = page((uint32_t)ids[i + 3]);
      bm[p0 >> 6] |= uint64_t(1) << (p0 & 63);
      bm[stride + (p1 >> 6)] |= uint64_t(1) << (p1 & 63);
      bm[2 * stride + (p2 >> 6)] |= uint64_t(1) << (p2 & 63);
      bm[3 * stride + (p3 >> 6)] |= uint64_t(1) << (p3 & 63);
    }
    for (; i < n; ++i) {
      const uint32_t p0 = page((uint32_t)ids[i]);
      bm[p0 >> 6] |= uint64_t(1) << (p0 & 63);
    }
    int32_t* lu = x.lu.data();
    for (int32_t w = 0; w < words; ++w) {
      for (uint64_t b = bm[w] | bm[stride + w] | bm[2 * stride + w] | bm[3 * stride + w]; b; b &= b - 1) {
        const int32_t p = w * 64 + __builtin_ctzll(b);
        if (lu[p] == step) continue;
        if (x.in_set[p]) {
          x.unlink(p);
          moved.push_back(p);
        }
        lu[p] = step;
      }
    }
    for (const int32_t p : moved) x.link_sorted(p);
    moved.clear();
  }

  void init_request(int32_t r, int32_t ctx) {
    Request& x = req[r];
    x = Request{};
    x.active = true;
    x.ctx = ctx;
    x.bt.assign(max_pages, -1);
    x.hbt.assign(max_pages, -1);
    x.lu.assign(max_pages, -1);
    x.pending.assign(max_pages, 0);
    x.in_set.assign(max_pages, 0);
    x.nxt.assign(max_pages, -1);
    x.prv.assign(max_pages, -1);
    x.head = x.tail = -1;
  }
};

extern "C" {

hs_status hs_res_create(int32_t num_gpu_blocks, int32_t num_host_blocks, int32_t page_size, int32_t max_requests,
                        int32_t max_pages, int32_t hot_blocks_per_request, hs_residency** out) {
  if (!out) return HS_ERR_INVALID_ARG;
  *out = nullptr;
  if (num_gpu_blocks < 0 || num_host_blocks < 0 || page_size < 1 || max_requests < 0 || max_pages < 1 ||
      hot_blocks_per_request < 0 || (int64_t)max_pages * page_size > INT32_MAX)
    return HS_ERR_INVALID_ARG;
  hs_residency* m = new (std::nothrow) hs_residency;
  if (!m) return HS_ERR_INVALID_ARG;
  try {
    m->S = page_size;
    m->S_shift = -1;
    for (int32_t k = 0; k < 31; ++k)
      if ((int32_t(1) << k) == page_size) m->S_shift = k;
    m->max_pages = max_pages;
    m->Hc = hot_blocks_per_request;
    std::vector<int32_t> g(num_gpu_blocks), h(num_host_blocks);
    for (int32_t i = 0; i < num_gpu_blocks; ++i) g[i] = i;
    for (int32_t i = 0; i < num_host_blocks; ++i) h[i] = i;
    m->free_gpu = decltype(m->free_gpu)(std::greater<int32_t>(), std::move(g));
    m->free_host = decltype(m->free_host)(std::greater<int32_t>(), std::move(h));
    m->host_ref.assign(num_host_blocks, 0);
    m->host_held.assign(num_host_blocks, 0);
    m->host_free_count = num_host_blocks;
    m->req.resize(max_requests);
  } catch (...) {
    delete m;
    return HS_ERR_INVALID_ARG;
  }
  *out = m;
  return HS_OK;
}

void hs_res_destroy(hs_residency* m) { delete m; }

hs_status hs_res_admit(hs_residency* m, int32_t r, int32_t ctx_len, const int32_t* prefix_host_blocks,
                       int32_t n_prefix) {
  if (!m || r < 0 || r >= (int32_t)m->req.size() || m->req[r].active) return HS_ERR_INVALID_ARG;
  const int32_t S = m->S;
  if (ctx_len < 1 || (ctx_len + S - 1) / S > m->max_pages || n_prefix < 0 || n_prefix > (ctx_len - 1) / S)
    return HS_ERR_INVALID_ARG;
  if (n_prefix > 0 && !prefix_host_blocks) return HS_ERR_INVALID_ARG;
  for (int32_t i = 0; i < n_prefix; ++i)
    if (prefix_host_blocks[i] < 0 || prefix_host_blocks[i] >= (int32_t)m->host_ref.size()) return HS_ERR_INVALID_ARG;
  m->init_request(r, ctx_len);
  Request& x = m->req[r];
  for (int32_t p = 0; p < n_prefix; ++p) {
    x.hbt[p] = prefix_host_blocks[p];
    m->host_ref_add(prefix_host_blocks[p]);
  }
  try {
    if (n_prefix > 0) m->lease_hot(r);
    const int32_t npages = (ctx_len + S - 1) / S;
    for (int32_t p = n_prefix; p < npages; ++p) {
      const int32_t b = m->alloc_gpu(r);
      x.bt[p] = b;
      m->fills.push_back({b, r, p});
      if (p < ctx_len / S) m->complete(r, p);
      else m->refresh(x, p);
    }
  } catch (const Capacity&) {
    m->finish(r);
    return HS_ERR_CAPACITY;
  }
  return HS_OK;
}

hs_status hs_res_append(hs_residency* m, int32_t r, int32_t n_tokens) {
  if (!m || r < 0 || r >= (int32_t)m->req.size() || !m->req[r].active || n_tokens < 0) return HS_ERR_INVALID_ARG;
  Request& x = m->req[r];
  const int32_t S = m->S;
  const int64_t old = x.ctx, nw = (int64_t)x.ctx + n_tokens;
  if ((nw + S - 1) / S > m->max_pages) return HS_ERR_INVALID_ARG;
  std::vector<int32_t> started;
  try {
    for (int32_t p = (int32_t)((old + S - 1) / S); p < (int32_t)((nw + S - 1) / S); ++p) {
      const int32_t b = m->alloc_gpu(r);
      x.bt[p] = b;
      started.push_back(p);
      m->fills.push_back({b, r, p});
    }
    if (nw / S - old / S > m->host_free_count) throw Capacity{};
  } catch (const Capacity&) {
    for (int32_t p : started) {
      for (size_t i = 0; i < m->fills.size(); ++i) {
        const Fill& f = m->fills[i];
        if (f.block == x.bt[p] && f.r == r && f.p == p) {
          m->fills.erase(m->fills.begin() + (ptrdiff_t)i);
          break;
        }
      }
      m->free_gpu.push(x.bt[p]);
      x.bt[p] = -1;
    }
    return HS_ERR_CAPACITY;
  }
  m->set_ctx(x, (int32_t)nw);
  for (int32_t p = (int32_t)(old / S); p < (int32_t)(nw / S); ++p) m->complete(r, p);
  return HS_OK;
}

hs_status hs_res_append_all(hs_residency* m, const int32_t* n_tokens) {
  if (!m || !n_tokens) return HS_ERR_INVALID_ARG;
  for (int32_t r = 0; r < (int32_t)m->req.size(); ++r) {
    if (n_tokens[r] == 0) continue;
    const hs_status st = hs_res_append(m, r, n_tokens[r]);
    if (st != HS_OK) return st;
  }
  return HS_OK;
}

hs_status hs_res_touch(hs_residency* m, int32_t r, const int32_t* ids, int64_t n, int32_t step) {
  if (!m || r < 0 || r >= (int32_t)m->req.size() || !m->req[r].active || n < 0) return HS_ERR_INVALID_ARG;
  if (n > 0 && !ids) return HS_ERR_INVALID_ARG;
  m->touch(r, ids, n, step);
  return HS_OK;
}

hs_status hs_res_touch_all(hs_residency* m, const int32_t* ids, int32_t n_per_request, int32_t step) {
  if (!m || n_per_request < 0 || (n_per_request > 0 && !ids)) return HS_ERR_INVALID_ARG;
  for (int32_t r = 0; r < (int32_t)m->req.size(); ++r)
    if (m->req[r].active) m->touch(r, ids + (int64_t)r * n_per_request, n_per_request, step);
  return HS_OK;
}

hs_status hs_res_finish(hs_residency* m, int32_t r) {
  if (!m || r < 0 || r >= (int32_t)m->req.size() || !m->req[r].active) return HS_ERR_INVALID_ARG;
  m->finish(r);
  return HS_OK;
}

hs_status hs_res_hold_host(hs_residency* m, const int32_t* blocks, int32_t n) {
  if (!m || n < 0 || (n > 0 && !blocks)) return HS_ERR_INVALID_ARG;
  for (int32_t i = 0; i < n; ++i)
    if (blocks[i] < 0 || blocks[i] >= (int32_t)m->host_ref.size()) return HS_ERR_INVALID_ARG;
  for (int32_t i = 0; i < n; ++i) {
    m->host_ref_add(blocks[i]);
    ++m->host_held[blocks[i]];
  }
  return HS_OK;
}

hs_status hs_res_drop_host(hs_residency* m, const int32_t* blocks, int32_t n) {
  if (!m || n < 0 || (n > 0 && !blocks)) return HS_ERR_INVALID_ARG;
  for (int32_t i = 0; i < n; ++i) {
    const int32_t h = blocks[i];
    if (h < 0 || h >= (int32_t)m->host_ref.size()) return HS_ERR_INVALID_ARG;
    int32_t times = 0;
    for (int32_t j = 0; j < n; ++j) times += blocks[j] == h;
    if (m->host_held[h] < times) return HS_ERR_INVALID_ARG;
  }
  for (int32_t i = 0; i < n; ++i) {
    --m->host_held[blocks[i]];
    m->host_unref(blocks[i]);
  }
  return HS_OK;
}

void hs_res_counts(const hs_residency* m, int32_t* queued, int32_t* resets, int32_t* fills) {
  if (queued) *queued = m ? (int32_t)m->queue.size() : 0;
  if (resets) *resets = m ? (int32_t)m->resets.size() : 0;
  if (fills) *fills = m ? (int32_t)m->fills.size() : 0;
}

int32_t hs_res_free_gpu_blocks(const hs_residency* m) { return m ? (int32_t)m->free_gpu.size() : 0; }

hs_status hs_res_collect(hs_residency* m, int32_t* gpu_blocks, int32_t* host_blocks, int32_t capacity,
                         int32_t* n_out) {
  if (!m || !n_out || capacity < (int32_t)m->queue.size()) return HS_ERR_INVALID_ARG;
  if (!m->queue.empty() && (!gpu_blocks || !host_blocks)) return HS_ERR_INVALID_ARG;
  int32_t k = 0;
  for (const QueuedCopy& c : m->queue) {
    gpu_blocks[k] = c.gpu;
    host_blocks[k] = c.host;
    ++k;
  }
  for (const QueuedCopy& c : m->queue) {
    Request& x = m->req[c.r];
    x.pending[c.p] = 0;
    m->refresh(x, c.p);
  }
  m->queue.clear();
  *n_out = k;
  return HS_OK;
}

hs_status hs_res_take_resets(hs_residency* m, int32_t* requests, int32_t capacity, int32_t* n_out) {
  if (!m || !n_out || capacity < (int32_t)m->resets.size()) return HS_ERR_INVALID_ARG;
  if (!m->resets.empty() && !requests) return HS_ERR_INVALID_ARG;
  std::copy(m->resets.begin(), m->resets.end(), requests);
  *n_out = (int32_t)m->resets.size();
  m->resets.clear();
  return HS_OK;
}

hs_status hs_res_take_fills(hs_residency* m, int32_t* blocks, int32_t* requests, int32_t* pages, int32_t capacity,
                            int32_t* n_out) {
  if (!m || !n_out || capacity < (int32_t)m->fills.size()) return HS_ERR_INVALID_ARG;
  if (!m->fills.empty() && (!blocks || !requests || !pages)) return HS_ERR_INVALID_ARG;
  int32_t k = 0;
  for (const Fill& f : m->fills) {
    blocks[k] = f.block;
    requests[k] = f.r;
    pages[k] = f.p;
    ++k;
  }
  *n_out = k;
  m->fills.clear();
  return HS_OK;
}

hs_status hs_res_tables(const hs_residency* m, int32_t* block_table, int32_t* host_block_table, int32_t* hot_blocks,
                        int32_t* ctx_len) {
  if (!m) return HS_ERR_INVALID_ARG;
  const int64_t P = m->max_pages, H = m->Hc;
  for (int64_t r = 0; r < (int64_t)m->req.size(); ++r) {  // whole rows: plain copies or fills
    const Request& x = m->req[r];
    if (block_table) {
      if (x.active) std::copy(x.bt.begin(), x.bt.end(), block_table + r * P);
      else std::fill(block_table + r * P, block_table + (r + 1) * P, -1);
    }
    if (host_block_table) {
      if (x.active) std::copy(x.hbt.begin(), x.hbt.end(), host_block_table + r * P);
      else std::fill(host_block_table + r * P, host_block_table + (r + 1) * P, -1);
    }
    if (hot_blocks) {
      if (x.active && x.leased && (int64_t)x.hot.size() == H) std::copy(x.hot.begin(), x.hot.end(), hot_blocks + r * H);
      else std::fill(hot_blocks + r * H, hot_blocks + (r + 1) * H, -1);
    }
    if (ctx_len) ctx_len[r] = x.active ? x.ctx : 0;
  }
  return HS_OK;
}

}  // extern "C"
