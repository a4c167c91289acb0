"""Seeded synthetic decode workloads shaped like the pages' workload.

This module only makes inputs: geometry, block tables (real blocks and null placeholders), host
block tables, leased hot blocks, per-step top-K id lists, context lengths and the pages to offload
after each step.  It holds none of the resolver's arithmetic.  The GPU path and the oracle are
both fed from here and from synth.content (row bytes).

Randomness: numpy PCG64 streams derived from SeedSequence([0x48535041, config, seed]); one
stream per (layer, request) unit so that a unit's top-K history does not depend on the others.
Block ids (GPU and host) are handed out through seeded permutations so rows are scattered.

Top-K laws (the indexer itself needs model weights, so its output is simulated):
  uniform   ids drawn without replacement, uniformly over [0, ctx).
  recency   P(id) proportional to the integral of x^-0.7 over the cell x in [ctx-id, ctx-id+1),
            i.e. "probability proportional to recency^-0.7"; distinct ids by rejection.
  keep f    a step keeps a uniform random subset of floor(f*K) ids of the previous list and
            draws the rest (excluding only the kept ones); the list is then shuffled, since an
            indexer's top-K order is arbitrary.
"""
from __future__ import annotations

from dataclasses import dataclass, field
from typing import Iterator, List, Optional

import numpy as np

SEED_TAG = 0x48535041  # "HSPA"


@dataclass
class Step:
    index: int
    topk: np.ndarray                 # int32 [L/G][R][P][K] (one list per index group of G layers)
    ctx_len: np.ndarray              # int32 [R]
    # table edits applied before this step's resolve: arrays of (r, page, value)
    bt_edits: np.ndarray = field(default_factory=lambda: np.zeros((0, 3), np.int32))
    hbt_edits: np.ndarray = field(default_factory=lambda: np.zeros((0, 3), np.int32))
    # GPU blocks whose content is (re)written before this step: (block, r, page) -> rows H(page)
    fills: np.ndarray = field(default_factory=lambda: np.zeros((0, 3), np.int64))
    # pages offloaded after this step's gather, all layers: parallel int32 arrays
    off_gpu: np.ndarray = field(default_factory=lambda: np.zeros(0, np.int32))
    off_host: np.ndarray = field(default_factory=lambda: np.zeros(0, np.int32))
    off_src: np.ndarray = field(default_factory=lambda: np.zeros((0, 2), np.int64))  # (r, page)


@dataclass
class Workload:
    name: str
    cfg: int
    seed: int
    L: int
    R: int
    P: int
    K: int
    C: int
    S: int
    B: int
    max_pages: int
    num_gpu_blocks: int
    num_host_blocks: int
    block_table: np.ndarray        # int32 [R][max_pages], state before step 0
    host_block_table: np.ndarray   # int32 [R][max_pages], state before step 0
    content_page: np.ndarray       # int64 [R][max_pages]: content id of each logical page
    hot_blocks: np.ndarray         # int32 [R][C/S]
    ctx_len: np.ndarray            # int32 [R], before step 0
    steps: int
    host_resident_init: np.ndarray  # int64 [n][2] (r, page) whose host copy exists at start
    gpu_resident_init: np.ndarray   # int64 [n][2] (r, page) resident at start
    content_seed: int = 0
    G: int = 1                      # layers per indexer (IndexShare); top-K lists are per group
    _gen: object = None             # step generator factory
    notes: str = ""

    @property
    def rows_per_step(self) -> int:
        return self.L * self.R * self.P * self.K

    def iter_steps(self, n: Optional[int] = None) -> Iterator[Step]:
        """Yield the first n steps (default: self.steps).  Deterministic for a given seed."""
        return self._gen(self, self.steps if n is None else n)

    # Pool contents at the start: GPU block -> (r, page) and host block -> (r, page).
    def gpu_block_owner(self) -> np.ndarray:
        """int64 [num_gpu_blocks][2] = (r, page) whose rows the block holds at start, (-1,-1) if none."""
        own = np.full((self.num_gpu_blocks, 2), -1, np.int64)
        rp = self.gpu_resident_init
        own[self.block_table[rp[:, 0], rp[:, 1]]] = rp
        return own

    def host_block_owner(self) -> np.ndarray:
        own = np.full((self.num_host_blocks, 2), -1, np.int64)
        rp = self.host_resident_init
        own[self.host_block_table[rp[:, 0], rp[:, 1]]] = rp
        return own


def _rngs(cfg: int, seed: int, n: int) -> List[np.random.Generator]:
    ss = np.random.SeedSequence([SEED_TAG, cfg, seed])
    return [np.random.Generator(np.random.PCG64(s)) for s in ss.spawn(n)]


def _layout_rng(cfg: int, seed: int) -> np.random.Generator:
    return np.random.Generator(np.random.PCG64(np.random.SeedSequence([SEED_TAG, cfg, seed, 1])))


def draw_distinct(rng: np.random.Generator, ctx: int, n: int, law: str, exclude: Optional[np.ndarray] = None,
                  alpha: float = 0.7) -> np.ndarray:
    """n distinct ids in [0, ctx), none in `exclude`, by the given law, in draw order."""
    if n <= 0:
        return np.zeros(0, np.int32)
    taken = np.zeros(ctx, bool)
    if exclude is not None and len(exclude):
        taken[exclude] = True
    avail = ctx - int(taken.sum())
    if n > avail:
        raise ValueError(f"cannot draw {n} distinct ids from {avail} available")
    out = []
    got = 0
    top = float(ctx + 1) ** (1.0 - alpha) - 1.0
    while got < n:
        m = 2 * (n - got) + 32
        if law == "uniform":
            cand = rng.integers(0, ctx, size=m)
        elif law == "recency":
            u = rng.random(m)
            x = np.floor((1.0 + u * top) ** (1.0 / (1.0 - alpha))).astype(np.int64)
            cand = np.clip(ctx - x, 0, ctx - 1)
        else:
            raise ValueError(law)
        _, first = np.unique(cand, return_index=True)
        cand = cand[np.sort(first)]
        cand = cand[~taken[cand]]
        cand = cand[: n - got]
        taken[cand] = True
        out.append(cand)
        got += len(cand)
    return np.concatenate(out).astype(np.int32)


def next_topk(rng: np.random.Generator, prev: Optional[np.ndarray], ctx: int, K: int, keep_frac: float,
              law: str) -> np.ndarray:
    """One top-K list: keep floor(keep_frac*K) of prev (if any), draw the rest, shuffle."""
    K = min(K, ctx)
    if prev is None or keep_frac <= 0:
        ids = draw_distinct(rng, ctx, K, law)
    else:
        nk = int(np.floor(keep_frac * K))
        prev = prev[prev >= 0]
        nk = min(nk, len(prev))
        kept = rng.choice(prev, size=nk, replace=False) if nk else np.zeros(0, np.int32)
        new = draw_distinct(rng, ctx, K - nk, law, exclude=kept)
        ids = np.concatenate([kept.astype(np.int32), new])
    return rng.permutation(ids).astype(np.int32)


# --------------------------------------------------------------------------- shared layout helpers
def _place(R: int, max_pages: int, resident: np.ndarray, hot_blocks_per_req: int, rng: np.random.Generator,
           extra_gpu_blocks: int = 0):
    """Assign scattered GPU blocks to resident (r, page) pairs and to hot buffers.

    resident: bool [R][max_pages].  Returns (block_table, hot_blocks, num_gpu_blocks)."""
    n_res = int(resident.sum())
    n = n_res + R * hot_blocks_per_req + extra_gpu_blocks
    perm = rng.permutation(n).astype(np.int32)
    bt = np.full((R, max_pages), -1, np.int32)
    rr, pp = np.nonzero(resident)
    bt[rr, pp] = perm[:n_res]
    hot = perm[n_res:n_res + R * hot_blocks_per_req].reshape(R, hot_blocks_per_req)
    return bt, hot, n


def _host_place(R: int, max_pages: int, has_host: np.ndarray, rng: np.random.Generator):
    n = int(has_host.sum())
    perm = rng.permutation(n).astype(np.int32)
    hbt = np.full((R, max_pages), -1, np.int32)
    rr, pp = np.nonzero(has_host)
    hbt[rr, pp] = perm
    return hbt, n


def _pairs(mask: np.ndarray) -> np.ndarray:
    rr, pp = np.nonzero(mask)
    return np.stack([rr, pp], 1).astype(np.int64)


# --------------------------------------------------------------------------- fixed-context configs
def _fixed_ctx_gen(law0: str, law: str, keep: float):
    def gen(w: Workload, n: int) -> Iterator[Step]:
        rngs = _rngs(w.cfg, w.seed, w.L * w.R)
        prev = [None] * (w.L * w.R)
        for s in range(n):
            topk = np.empty((w.L, w.R, w.P, w.K), np.int32)
            for l in range(w.L):
                for r in range(w.R):
                    u = l * w.R + r
                    if prev[u] is None:
                        ids = next_topk(rngs[u], None, int(w.ctx_len[r]), w.K, 0.0, law0)
                    else:
                        ids = next_topk(rngs[u], prev[u], int(w.ctx_len[r]), w.K, keep, law)
                    prev[u] = ids
                    topk[l, r, 0] = ids
            yield Step(index=s, topk=topk, ctx_len=w.ctx_len.copy())
    return gen


def config1(seed: int = 0, steps: int = 8) -> Workload:
    """Tiny decode: 1 layer, 4 requests, ctx 4096, page 64, 656-B rows; last 1024 tokens resident,
    older pages host-only, full host copy; K=256, hot buffer 512 rows; keep 50% per step; uniform."""
    L, R, P, K, C, S, B = 1, 4, 1, 256, 512, 64, 656
    ctx = 4096
    max_pages = ctx // S
    lr = _layout_rng(1, seed)
    resident = np.zeros((R, max_pages), bool)
    resident[:, max_pages - 16:] = True
    bt, hot, ngb = _place(R, max_pages, resident, C // S, lr)
    has_host = np.ones((R, max_pages), bool)
    hbt, nhb = _host_place(R, max_pages, has_host, lr)
    content = (np.arange(R)[:, None] * max_pages + np.arange(max_pages)[None, :]).astype(np.int64)
    return Workload("tiny-decode", 1, seed, L, R, P, K, C, S, B, max_pages, ngb, nhb, bt, hbt, content, hot,
                    np.full(R, ctx, np.int32), steps, _pairs(has_host), _pairs(resident),
                    content_seed=seed, _gen=_fixed_ctx_gen("uniform", "uniform", 0.5))


def config2(seed: int = 0, steps: int = 64, R: int = 64, resident_tokens: int = 16384) -> Workload:
    """Mixed-residency decode batch: 1 layer, 64 requests, ctx 131072; tail 16384 tokens resident,
    rest host-only, full host copy; K=2048, hot 4096; keep 80%, recency^-0.7 draws.
    resident_tokens = 131072 gives the same batch with full residency (no KV pressure)."""
    L, P, K, C, S, B = 1, 1, 2048, 4096, 64, 656
    ctx = 131072
    max_pages = ctx // S
    lr = _layout_rng(2, seed)
    resident = np.zeros((R, max_pages), bool)
    resident[:, max_pages - resident_tokens // S:] = True
    bt, hot, ngb = _place(R, max_pages, resident, C // S, lr)
    has_host = np.ones((R, max_pages), bool)
    hbt, nhb = _host_place(R, max_pages, has_host, lr)
    content = (np.arange(R)[:, None] * max_pages + np.arange(max_pages)[None, :]).astype(np.int64)
    return Workload("mixed-residency-decode", 2, seed, L, R, P, K, C, S, B, max_pages, ngb, nhb, bt, hbt,
                    content, hot, np.full(R, ctx, np.int32), steps, _pairs(has_host), _pairs(resident),
                    content_seed=seed, _gen=_fixed_ctx_gen("recency", "recency", 0.8))


def config4(seed: int = 0, steps: int = 32, R: int = 16) -> Workload:
    """No-residency cold start: 16 requests reuse a 1,048,576-token prefix that exists only in
    pinned host memory (all requests' host tables point at the same host blocks); each request's
    last page is its resident tail; hot buffer starts empty (4096 rows, K=2048); fresh uniform
    top-K every step."""
    L, P, K, C, S, B = 1, 1, 2048, 4096, 64, 656
    ctx = 1 << 20
    max_pages = ctx // S
    lr = _layout_rng(4, seed)
    resident = np.zeros((R, max_pages), bool)
    resident[:, max_pages - 1] = True
    bt, hot, ngb = _place(R, max_pages, resident, C // S, lr)
    nhb = max_pages - 1
    perm = lr.permutation(nhb).astype(np.int32)
    hbt = np.full((R, max_pages), -1, np.int32)
    hbt[:, : max_pages - 1] = perm[None, :]
    content = np.broadcast_to(np.arange(max_pages, dtype=np.int64)[None, :], (R, max_pages)).copy()
    host_init = np.stack([np.zeros(nhb, np.int64), np.arange(nhb, dtype=np.int64)], 1)  # owner: request 0
    return Workload("cold-start-prefix-reuse", 4, seed, L, R, P, K, C, S, B, max_pages, ngb, nhb, bt, hbt,
                    content, hot, np.full(R, ctx, np.int32), steps, host_init, _pairs(resident),
                    content_seed=seed, _gen=_fixed_ctx_gen("uniform", "uniform", 0.0))


# --------------------------------------------------------------------------- max batch with MTP3
def _mtp_lists(rng, prev0, ctx, K, P, keep0, keep_pos, law="recency"):
    """Position 0 keeps keep0 of its previous list (or draws K afresh); positions 1..P-1 keep
    floor(keep_pos*K) of position 0 and draw the rest.  Returns int32 [P][K]."""
    out = np.empty((P, K), np.int32)
    p0 = next_topk(rng, prev0, ctx, K, keep0 if prev0 is not None else 0.0, law)
    out[0] = p0
    for q in range(1, P):
        out[q] = next_topk(rng, p0, ctx, K, keep_pos, law)
    return out


def config5(seed: int = 0, steps: int = 128, R: int = 256, L: int = 4, layers_per_index: int = 1,
            capacity: int = 4096) -> Workload:
    """Max-batch mixed load with speculative decode (MTP3): 4 layers, 256 requests, contexts
    log-uniform in [8192, 1,048,576]; each non-tail page resident with a per-request probability
    f ~ U[0,1] (tail always resident); P=4 positions per request share one plan, position 0 keeps 80%
    of its previous list, positions 1..3 keep 90% of position 0; K=2048, hot 4096.  Each step appends
    U{1..4} tokens (the accepted MTP length) and ends with one offload launch of the pages completed
    in that step (all layers).  Host copies exist for the host-only pages; a page completed during the
    run gets a fresh host block when it is offloaded.  layers_per_index = G > 1 draws one top-K per
    index group of G layers (IndexShare) instead of one per layer.  capacity sets the hot rows per
    request: 4096 = 2K by default; (num_spec + 2) * K = 10240 is the pages' MTP sizing."""
    P, K, C, S, B = 4, 2048, capacity, 64, 656
    assert L % layers_per_index == 0
    lr = _layout_rng(5, seed)
    ctx0 = np.floor(np.exp(lr.uniform(np.log(8192), np.log(1 << 20), size=R))).astype(np.int64)
    frac = lr.uniform(0.0, 1.0, size=R)
    grow = lr.integers(1, 5, size=(steps, R)).astype(np.int64)          # accepted tokens per step
    ctx_final = ctx0 + grow.sum(axis=0)
    max_pages = int(((ctx_final + S - 1) // S).max())
    tail0 = (ctx0 - 1) // S
    pages_final = (ctx_final + S - 1) // S
    pidx = np.arange(max_pages)[None, :]
    u = lr.random((R, max_pages))
    resident = (pidx < tail0[:, None]) & (u < frac[:, None])
    resident |= (pidx >= tail0[:, None]) & (pidx < pages_final[:, None])   # tail and future pages
    bt, hot, ngb = _place(R, max_pages, resident, C // S, lr)
    complete0 = pidx < (ctx0 // S)[:, None]
    has_host = complete0 & ~resident
    hbt, nhb_init = _host_place(R, max_pages, has_host, lr)
    n_new = int((pages_final - ctx0 // S).sum()) + R
    content = (np.arange(R)[:, None] * max_pages + pidx).astype(np.int64)
    w = Workload("max-batch-mtp3", 5, seed, L, R, P, K, C, S, B, max_pages, ngb, nhb_init + n_new, bt, hbt, content,
                 hot, ctx0.astype(np.int32), steps, _pairs(has_host), _pairs(resident), content_seed=seed,
                 G=layers_per_index, notes="GPU blocks of future tail pages are assigned and filled up front")
    w._grow = grow
    w._nhb_init = nhb_init

    def gen(w: Workload, n: int) -> Iterator[Step]:
        ng = w.L // w.G
        rngs = _rngs(w.cfg, w.seed, ng * w.R)
        prev = [None] * (ng * w.R)
        ctx = w.ctx_len.astype(np.int64).copy()
        next_host = w._nhb_init
        pending_hbt = np.zeros((0, 3), np.int32)
        for s in range(n):
            topk = np.empty((ng, w.R, w.P, w.K), np.int32)
            for l in range(ng):
                for r in range(w.R):
                    uid = l * w.R + r
                    lists = _mtp_lists(rngs[uid], prev[uid], int(ctx[r]), w.K, w.P, 0.8, 0.9)
                    prev[uid] = lists[0]
                    topk[l, r] = lists
            g = w._grow[s % w._grow.shape[0]]
            new_ctx = ctx + g
            og, oh, src = [], [], []
            for r in range(w.R):
                for pg in range(int(ctx[r] // w.S), int(new_ctx[r] // w.S)):
                    og.append(int(w.block_table[r, pg]))
                    oh.append(next_host)
                    src.append((r, pg))
                    next_host += 1
            st = Step(index=s, topk=topk, ctx_len=ctx.astype(np.int32), hbt_edits=pending_hbt,
                      off_gpu=np.array(og, np.int32), off_host=np.array(oh, np.int32),
                      off_src=np.array(src, np.int64).reshape(-1, 2))
            pending_hbt = np.array([(r, pg, h) for (r, pg), h in zip(src, oh)], np.int32).reshape(-1, 3)
            ctx = new_ctx
            yield st
    w._gen = gen
    return w


# --------------------------------------------------------------------------- multi-turn agentic
def config3(seed: int = 0, turns: int = 13, decode_per_turn: int = 220, R: int = 32, L: int = 16,
            first_turn: int = 74160, prompt_per_turn: int = 753, resident_frac: float = 0.4,
            layers_per_index: int = 1) -> Workload:
    """Multi-turn agentic shape: 16 layers, 32 requests in lock-step, 13 turns (74,160-token first
    turn, then +753 prompt tokens and 220 decode tokens per turn); K=2048, hot 4096, top-K locality
    as in the mixed batch.  Residency stand-in: each request keeps its newest round(resident_frac *
    final pages) pages on the GPU (tail included); when a new page needs a block, the oldest resident
    page is released (its host copy already exists) and its block is reused for the new page, whose
    rows the model would write (an untimed fill here).  Every completed page is offloaded (all layers,
    one launch) after the step in which it completes, to a fresh host block; pages completed before
    the first step have host copies from the start.  layers_per_index = G > 1 draws one top-K per
    index group of G layers (IndexShare: one indexer per four sparse-MLA layers in GLM 5.3)."""
    K, C, S, B, P = 2048, 4096, 64, 656, 1
    assert L % layers_per_index == 0
    ctx_final = first_turn + (turns - 1) * (decode_per_turn + prompt_per_turn) + decode_per_turn
    max_pages = (ctx_final + S - 1) // S
    budget = int(round(resident_frac * max_pages))
    lr = _layout_rng(3, seed)
    ctx0 = first_turn
    n0 = (ctx0 + S - 1) // S
    resident = np.zeros((R, max_pages), bool)
    resident[:, max(0, n0 - budget):n0] = True
    bt, hot, ngb = _place(R, max_pages, resident, C // S, lr)
    complete0 = np.zeros((R, max_pages), bool)
    complete0[:, : ctx0 // S] = True
    hbt, nhb_init = _host_place(R, max_pages, complete0, lr)
    content = (np.arange(R)[:, None] * max_pages + np.arange(max_pages)[None, :]).astype(np.int64)
    steps = turns * decode_per_turn
    w = Workload("multi-turn-agentic", 3, seed, L, R, P, K, C, S, B, max_pages, ngb,
                 nhb_init + R * (max_pages - ctx0 // S) + R, bt, hbt, content, hot, np.full(R, ctx0, np.int32),
                 steps, _pairs(complete0), _pairs(resident), content_seed=seed, G=layers_per_index,
                 notes=f"resident budget {budget} pages per request")
    w._budget = budget
    w._nhb_init = nhb_init
    w._turn = (decode_per_turn, prompt_per_turn)

    def gen(w: Workload, n: int) -> Iterator[Step]:
        ng = w.L // w.G
        rngs = _rngs(w.cfg, w.seed, ng * w.R)
        prev = [None] * (ng * w.R)
        bt = w.block_table.copy()
        ctx = int(w.ctx_len[0])
        res_pages = [sorted(np.nonzero(bt[r] >= 0)[0].tolist()) for r in range(w.R)]
        next_host = w._nhb_init
        pending_hbt = np.zeros((0, 3), np.int32)
        dpt, ppt = w._turn
        done_pages = int(w.ctx_len[0]) // w.S      # pages whose host copy exists or is queued
        for s in range(n):
            # tokens written before this step: one decoded token per step, plus the next turn's prompt
            # at a turn boundary (except before the first step)
            bt_edits, fills = [], []
            if s > 0:
                add = 1 + (ppt if s % dpt == 0 else 0)
                new_ctx = ctx + add
                for pg in range((ctx + w.S - 1) // w.S, (new_ctx + w.S - 1) // w.S):   # pages that start
                    for r in range(w.R):
                        if len(res_pages[r]) >= w._budget:
                            old = res_pages[r].pop(0)
                            blk = int(bt[r, old])
                            bt[r, old] = -1
                            bt_edits.append((r, old, -1))
                        else:
                            raise RuntimeError("no block to reuse")
                        bt[r, pg] = blk
                        res_pages[r].append(pg)
                        bt_edits.append((r, pg, blk))
                        fills.append((blk, r, pg))
                ctx = new_ctx
            topk = np.empty((ng, w.R, 1, w.K), np.int32)
            for l in range(ng):
                for r in range(w.R):
                    uid = l * w.R + r
                    ids = next_topk(rngs[uid], prev[uid], ctx, w.K, 0.8 if prev[uid] is not None else 0.0, "recency")
                    prev[uid] = ids
                    topk[l, r, 0] = ids
            # pages completed by the tokens this step's context includes but the last offload did not
            og, oh, src = [], [], []
            for pg in range(done_pages, ctx // w.S):
                for r in range(w.R):
                    og.append(int(bt[r, pg]))
                    oh.append(next_host)
                    src.append((r, pg))
                    next_host += 1
            done_pages = ctx // w.S
            st = Step(index=s, topk=topk, ctx_len=np.full(w.R, ctx, np.int32),
                      bt_edits=np.array(bt_edits, np.int32).reshape(-1, 3),
                      hbt_edits=pending_hbt, fills=np.array(fills, np.int64).reshape(-1, 3),
                      off_gpu=np.array(og, np.int32), off_host=np.array(oh, np.int32),
                      off_src=np.array(src, np.int64).reshape(-1, 2))
            pending_hbt = np.array([(r, pg, h) for (r, pg), h in zip(src, oh)], np.int32).reshape(-1, 3)
            yield st
    w._gen = gen
    return w


CONFIGS = {1: config1, 2: config2, 3: config3, 4: config4, 5: config5}


def make(cfg: int, **kw) -> Workload:
    return CONFIGS[cfg](**kw)
