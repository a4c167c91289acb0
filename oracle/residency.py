"""Oracle for the host-side residency manager: page-level residency, cold-page release under
pressure, hot-buffer lease/return from the shared block pool, proactive offload queueing.

TEST INFRASTRUCTURE ONLY.  Only tests/ may import it.  Plain Python lists and linear scans; it
shares nothing with the native manager (sparse_mla_kv_gb300/csrc/residency.cpp).

What it follows:
  - Japanese article (news.ainew.jp), the section before "仕組み" (the A/B example): under KV
    pressure each request frees its least recently used (cold) pages in place, and the freed blocks
    are reused as new tail pages and hot pages, so both requests keep decoding.
  - "仕組み" (How it works): residency is tracked per page; the tail never leaves the GPU; hot pages
    are ordinary KV blocks leased from the same pool as resident pages when a request first needs
    them and returned when it no longer does; a block freed by one request can become another
    request's hot capacity; when a cacheable prefix page completes, its CPU copy is queued while the
    GPU keeps serving it, so the page can later give up its GPU block without another copy, and the
    block is reusable once the copy has been queued.
  - "vLLM の他の部分との統合": the hot buffer holds 2 x top-K rows per request by default.

Readings where the pages are silent (the same in the native manager):
  - blocks are handed out lowest id first (GPU and host pools alike);
  - "the tail" is the request's last page; complete pages are those below ctx // page_size;
  - a reused host prefix covers complete pages before the last token (the prompt's last token is
    always computed), so an admitted request always has its tail page on the GPU;
  - a page may be released when it is resident, complete, not the last page, has a host copy, and
    its offload is not waiting in the queue (the copy is queued when the caller collects the queue
    for the post-forward offload launch);
  - cold order is ascending (last step the indexer selected the page, page); never-selected pages
    (-1) go first.  The request that needs a block releases its own cold pages first, then the
    coldest page of any other request, ascending (last use, request, page);
  - a request leases its hot buffer (capacity / page_size blocks, taken one by one through the same
    allocation) when it first has a placeholder page: at admission with a host-only prefix, or when
    its first page is released; it returns the buffer when it finishes.  A lease that cannot be
    completed returns the blocks it took and is tried again at the request's next release;
  - host blocks are reference-counted (a prefix may be shared by several requests) and return to
    the free pool at zero;
  - when no block can be found the call fails with CAPACITY: a failed admission leaves the request
    not admitted (its blocks and host references are returned), a failed append leaves the context
    unchanged (blocks taken for its new pages are returned); releases made before the failure stay,
    each leaves a valid state.
"""
from __future__ import annotations

OK, INVALID_ARG, CAPACITY = 0, 1, 4


class ResidencyError(Exception):
    def __init__(self, code: int, what: str):
        super().__init__(f"{what} (status {code})")
        self.code = code


class _Req:
    def __init__(self, max_pages: int):
        self.ctx = 0
        self.bt = [-1] * max_pages        # GPU block per page, -1 placeholder
        self.hbt = [-1] * max_pages       # host block per page, -1 none
        self.lu = [-1] * max_pages        # last step the page was selected
        self.hot = None                   # leased hot blocks, None before the first lease
        self.pending = set()              # pages whose offload waits in the queue


class Residency:
    def __init__(self, num_gpu_blocks: int, num_host_blocks: int, page_size: int, max_requests: int,
                 max_pages: int, hot_blocks: int):
        self.S = page_size
        self.max_pages = max_pages
        self.Hc = hot_blocks
        self.free_gpu = list(range(num_gpu_blocks))      # kept sorted
        self.host_ref = [0] * num_host_blocks
        self.host_held = [0] * num_host_blocks             # references held by the caller
        self.reqs = [None] * max_requests
        self.queue = []                                  # (gpu block, host block, request, page)
        self.resets = []                                 # requests whose hot buffer was (re)leased
        self.fills = []                                  # (gpu block, request, page) to be written

    # ------------------------------------------------------------------ pools
    def _alloc_host(self) -> int:
        for h, c in enumerate(self.host_ref):
            if c == 0:
                self.host_ref[h] = 1
                return h
        raise ResidencyError(CAPACITY, "host pool exhausted")

    def _free_gpu_block(self, b: int) -> None:
        self.free_gpu.append(b)
        self.free_gpu.sort()

    def _eligible(self, x: _Req):
        last = (x.ctx + self.S - 1) // self.S - 1
        return [p for p in range(min(last, x.ctx // self.S))
                if x.bt[p] >= 0 and x.hbt[p] >= 0 and p not in x.pending]

    def _pick_cold(self, r: int):
        own = self._eligible(self.reqs[r])
        if own:
            x = self.reqs[r]
            p = min(own, key=lambda p: (x.lu[p], p))
            return r, p
        best = None
        for q, x in enumerate(self.reqs):
            if x is None or q == r:
                continue
            for p in self._eligible(x):
                key = (x.lu[p], q, p)
                if best is None or key < best[0]:
                    best = (key, q, p)
        return None if best is None else (best[1], best[2])

    def _release(self, q: int, p: int) -> None:
        x = self.reqs[q]
        b = x.bt[p]
        x.bt[p] = -1
        self._free_gpu_block(b)
        if x.hot is None:
            self._lease_hot(q)

    def _lease_hot(self, q: int) -> None:
        x = self.reqs[q]
        x.hot = []
        added = q not in self.resets
        if added:
            self.resets.append(q)
        try:
            for _ in range(self.Hc):
                x.hot.append(self._alloc_gpu(q))
        except ResidencyError:        # a lease is all or nothing: the next release tries again
            for b in x.hot:
                self._free_gpu_block(b)
            x.hot = None
            if added:
                self.resets.remove(q)
            raise

    def _alloc_gpu(self, r: int) -> int:
        while not self.free_gpu:
            pick = self._pick_cold(r)
            if pick is None:
                raise ResidencyError(CAPACITY, "no GPU block can be freed")
            self._release(*pick)
        return self.free_gpu.pop(0)

    def _complete(self, r: int, p: int) -> None:
        x = self.reqs[r]
        h = self._alloc_host()
        x.hbt[p] = h
        x.pending.add(p)
        self.queue.append((x.bt[p], h, r, p))

    # ------------------------------------------------------------------ operations
    def _check_req(self, r: int, active: bool) -> None:
        if not 0 <= r < len(self.reqs) or (self.reqs[r] is not None) != active:
            raise ResidencyError(INVALID_ARG, "bad request index or state")

    def admit(self, r: int, ctx: int, prefix_host_blocks=()) -> None:
        """A request with `ctx` tokens; its first len(prefix_host_blocks) pages exist only in host
        memory (reused prefix), the rest are written by prefill into fresh GPU blocks."""
        self._check_req(r, False)
        n_pref = len(prefix_host_blocks)
        if ctx < 1 or (ctx + self.S - 1) // self.S > self.max_pages or n_pref > (ctx - 1) // self.S:
            raise ResidencyError(INVALID_ARG, "bad context or prefix length")
        if any(not 0 <= h < len(self.host_ref) for h in prefix_host_blocks):
            raise ResidencyError(INVALID_ARG, "prefix host block out of range")
        x = self.reqs[r] = _Req(self.max_pages)
        x.ctx = ctx
        for p, h in enumerate(prefix_host_blocks):
            x.hbt[p] = h
            self.host_ref[h] += 1
        try:
            if n_pref:
                self._lease_hot(r)
            for p in range(n_pref, (ctx + self.S - 1) // self.S):
                b = self._alloc_gpu(r)
                x.bt[p] = b
                self.fills.append((b, r, p))
                if p < ctx // self.S:
                    self._complete(r, p)
        except ResidencyError:
            self.finish(r)
            raise

    def append(self, r: int, n: int) -> None:
        """n decoded (or prompt) tokens appended: pages that start get a GPU block, pages that
        complete get a host block and a queued offload."""
        self._check_req(r, True)
        x = self.reqs[r]
        old, new = x.ctx, x.ctx + n
        if n < 0 or (new + self.S - 1) // self.S > self.max_pages:
            raise ResidencyError(INVALID_ARG, "bad token count")
        started = []
        try:
            for p in range((old + self.S - 1) // self.S, (new + self.S - 1) // self.S):
                b = self._alloc_gpu(r)
                x.bt[p] = b
                started.append(p)
                self.fills.append((b, r, p))
            n_host_free = sum(1 for c in self.host_ref if c == 0)
            if new // self.S - old // self.S > n_host_free:
                raise ResidencyError(CAPACITY, "host pool exhausted")
        except ResidencyError:
            for p in started:
                self.fills.remove((x.bt[p], r, p))
                self._free_gpu_block(x.bt[p])
                x.bt[p] = -1
            raise
        x.ctx = new
        for p in range(old // self.S, new // self.S):
            self._complete(r, p)

    def append_all(self, n_tokens) -> None:
        """append() for every request with a non-zero entry of n_tokens [max_requests], in request order;
        the first failure stops the call (earlier appends stay)."""
        for r, n in enumerate(n_tokens):
            if int(n) != 0:
                self.append(r, int(n))

    def touch(self, r: int, ids, step: int) -> None:
        """The pages of the indexer's selected ids were used at `step` (non-decreasing)."""
        self._check_req(r, True)
        x = self.reqs[r]
        for t in ids:
            if 0 <= t < x.ctx:
                x.lu[t // self.S] = step

    def touch_all(self, ids, step: int) -> None:
        """touch() for every active request: ids [max_requests][n], row r for request r."""
        for r, x in enumerate(self.reqs):
            if x is not None:
                self.touch(r, ids[r], step)

    def collect(self):
        """Queued offloads (gpu block, host block) in queue order; the queue is emptied (the caller
        enqueues them in the post-forward offload launch)."""
        out = [(g, h) for g, h, _, _ in self.queue]
        for _, _, r, p in self.queue:
            self.reqs[r].pending.discard(p)
        self.queue = []
        return out

    def finish(self, r: int) -> None:
        self._check_req(r, True)
        x = self.reqs[r]
        self.queue = [e for e in self.queue if e[2] != r]
        for p in range(self.max_pages):
            if x.bt[p] >= 0:
                self._free_gpu_block(x.bt[p])
            if x.hbt[p] >= 0:
                self.host_ref[x.hbt[p]] -= 1
        for b in x.hot or []:
            self._free_gpu_block(b)
        self.reqs[r] = None
        self.resets = [q for q in self.resets if q != r]
        self.fills = [f for f in self.fills if f[1] != r]

    def hold_host(self, blocks) -> None:
        """The caller (a prefix cache) keeps these host blocks: one reference each."""
        if any(not 0 <= h < len(self.host_ref) for h in blocks):
            raise ResidencyError(INVALID_ARG, "host block out of range")
        for h in blocks:
            self.host_ref[h] += 1
            self.host_held[h] += 1

    def drop_host(self, blocks) -> None:
        """Drop references taken by hold_host."""
        if any(not 0 <= h < len(self.host_ref) or self.host_held[h] < blocks.count(h) for h in blocks):
            raise ResidencyError(INVALID_ARG, "host block not held")
        for h in blocks:
            self.host_ref[h] -= 1
            self.host_held[h] -= 1

    # ------------------------------------------------------------------ views
    def tables(self):
        """(block_table, host_block_table, hot_blocks, ctx_len) as lists of lists / list."""
        R = len(self.reqs)
        bt = [[-1] * self.max_pages for _ in range(R)]
        hbt = [[-1] * self.max_pages for _ in range(R)]
        hot = [[-1] * self.Hc for _ in range(R)]
        ctx = [0] * R
        for r, x in enumerate(self.reqs):
            if x is None:
                continue
            bt[r], hbt[r], ctx[r] = list(x.bt), list(x.hbt), x.ctx
            if x.hot is not None:
                hot[r] = list(x.hot)
        return bt, hbt, hot, ctx

    def take_resets(self):
        out, self.resets = self.resets, []
        return out

    def take_fills(self):
        out, self.fills = self.fills, []
        return out

    def free_gpu_blocks(self) -> int:
        return len(self.free_gpu)
