"""Small hand-made resolver cases for the oracle tests: one pool layer, per-request tables,
hot state, and a helper to run one step through the oracle (with byte pools)."""
from __future__ import annotations

import numpy as np

import oracle
from synth import content


class Case:
    def __init__(self, *, R, S, B, C, max_pages, ctx, resident, host, hot_blocks, num_gpu_blocks, num_host_blocks,
                 bt, hbt, L=1, seed=7, content_page=None):
        self.R, self.S, self.B, self.C, self.L = R, S, B, C, L
        self.max_pages = max_pages
        self.ctx = np.asarray(ctx, np.int32)
        self.bt = np.asarray(bt, np.int32)
        self.hbt = np.asarray(hbt, np.int32)
        self.hot_blocks = np.asarray(hot_blocks, np.int32)
        self.ngb, self.nhb = num_gpu_blocks, num_host_blocks
        self.tok = np.full((L, R, C), -1, np.int32)
        self.stamp = np.full((L, R, C), -1, np.int32)
        self.seed = seed
        self.content_page = (np.arange(R)[:, None] * max_pages + np.arange(max_pages)[None, :]
                             if content_page is None else np.asarray(content_page))
        # byte pools filled from the closed-form row contents; hot blocks start zeroed
        self.pools = [np.zeros(num_gpu_blocks * S * B, np.uint8) for _ in range(L)]
        self.hosts = [np.zeros(max(num_host_blocks, 1) * S * B, np.uint8) for _ in range(L)]
        for l in range(L):
            for r in range(R):
                for p in range(max_pages):
                    rows = content.page_np(seed, l, int(self.content_page[r, p]), S, B).reshape(-1)
                    if self.bt[r, p] >= 0 and resident:
                        g = self.bt[r, p]
                        self.pools[l][g * S * B:(g + 1) * S * B] = rows
                    if self.hbt[r, p] >= 0 and host:
                        h = self.hbt[r, p]
                        self.hosts[l][h * S * B:(h + 1) * S * B] = rows

    def expected_row_bytes(self, l, r, token):
        return content.rows_np(self.seed, l, int(self.content_page[r, token // self.S]), token % self.S, self.B)

    def step(self, ids, step, bytes_=True, layer_begin=0):
        ids = np.asarray(ids, np.int32)
        if ids.ndim == 3:          # [R][P][K] -> one layer
            ids = ids[None]
        return oracle.resolve(S=self.S, B=self.B, num_gpu_blocks=self.ngb, num_host_blocks=self.nhb, topk=ids,
                              block_table=self.bt, host_block_table=self.hbt, ctx_len=self.ctx,
                              max_pages=self.max_pages, C=self.C, hot_blocks=self.hot_blocks, slot_token=self.tok,
                              slot_stamp=self.stamp, step=step, layer_begin=layer_begin,
                              pools=self.pools if bytes_ else None, hosts=self.hosts if bytes_ else None, threads=2)

    def gather(self, rows, layer_begin=0):
        rows = np.asarray(rows, np.int32).reshape(rows.shape[0], -1)
        return oracle.gather(B=self.B, num_rows=self.ngb * self.S, pools=self.pools, rows=rows,
                             layer_begin=layer_begin, threads=2)

    def hot_row(self, r, v):
        return int(self.hot_blocks[r][v // self.S]) * self.S + v % self.S


def host_only_case(*, R=1, S=4, B=16, C=8, pages=16, seed=3):
    """All pages are placeholders with a host copy; hot blocks are GPU blocks 0..R*C/S-1."""
    nb = C // S
    hot = np.arange(R * nb, dtype=np.int32).reshape(R, nb)
    bt = np.full((R, pages), -1, np.int32)
    hbt = (np.arange(R * pages, dtype=np.int32).reshape(R, pages))
    return Case(R=R, S=S, B=B, C=C, max_pages=pages, ctx=[pages * S] * R, resident=True, host=True, hot_blocks=hot,
                num_gpu_blocks=R * nb, num_host_blocks=R * pages, bt=bt, hbt=hbt, seed=seed)
