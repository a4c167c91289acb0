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
    topk: np.ndarray                 # int32 [L][R][P][K]
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
        for r, p in self.gpu_resident_init:
            own[self.block_table[r, p]] = (r, p)
        return own

    def host_block_owner(self) -> np.ndarray:
        own = np.full((self.num_host_blocks, 2), -1, np.int64)
        for r, p in self.host_resident_init:
            own[self.host_block_table[r, p]] = (r, p)
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


def config2(seed: int = 0, steps: int = 64, R: int = 64) -> Workload:
    """Mixed-residency decode batch: 1 layer, 64 requests, ctx 131072; tail 16384 tokens resident,
    rest host-only, full host copy; K=2048, hot 4096; keep 80%, recency^-0.7 draws."""
    L, P, K, C, S, B = 1, 1, 2048, 4096, 64, 656
    ctx = 131072
    max_pages = ctx // S
    lr = _layout_rng(2, seed)
    resident = np.zeros((R, max_pages), bool)
    resident[:, max_pages - 16384 // S:] = True
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


CONFIGS = {1: config1, 2: config2, 4: config4}


def make(cfg: int, **kw) -> Workload:
    return CONFIGS[cfg](**kw)
