"""Drive one synthetic workload through the CUDA library and the oracle side by side.

Inputs come from synth (tables, top-K, closed-form row bytes); expected values come from the oracle
(rows, stats, slot state, and pool bytes when `oracle_bytes`) and from the closed-form row contents
(gathered bytes, hot-slot bytes).  Nothing expected is ever read back from the CUDA path."""
from __future__ import annotations

import numpy as np
import torch

import oracle
import sparse_mla_kv_gb300 as hs
from synth import content, device as sdev


class Rig:
    def __init__(self, w, *, oracle_bytes: bool = False, device: str = "cuda", check_hot_bytes: bool = True,
                 mode: str = "split", graph: bool = False, miss_sm_div: int = 0, prefetch: int = 0,
                 planes: tuple = ()):
        # "split" / "fused": the library's default miss layout for the pool (ordered only for large host
        # pools); a "+order" suffix forces the address-ordered layout on any pool, "+ranges" its range
        # schedule with the fused gather's default SM partition, "+ranges1" / "+ranges2" with one or two
        # miss warps in every fused-gather CTA; "+part" keeps the default layout and asks for the SM
        # partition (per-unit lists on small pools)
        base, _, opt = mode.partition("+")
        assert base in ("split", "fused") and opt in ("", "order", "ranges", "ranges1", "ranges2", "part")
        self.mode = base
        self.force_order = opt not in ("", "part")
        self.order_mode = hs.MISS_ORDER_ON if opt == "order" else (hs.MISS_ORDER_RANGES if self.force_order else None)
        self.miss_warps = {"ranges1": 1, "ranges2": 2, "ranges": 0, "part": 0}.get(opt, -1)
        self.graph = graph
        self.prep = None
        self.w = w
        self.dev = torch.device(device)
        self.oracle_bytes = oracle_bytes
        self.check_hot_bytes = check_hot_bytes
        L, R, C, S, B = w.L, w.R, w.C, w.S, w.B
        self.gpu = [torch.empty((w.num_gpu_blocks, S, B), dtype=torch.uint8, device=self.dev) for _ in range(L)]
        nhb = max(1, w.num_host_blocks)
        self.host = [sdev.pinned_empty((nhb, S, B)) for _ in range(L)]
        if oracle_bytes:
            for h in self.host:
                h.zero_()
        for l in range(L):
            sdev.fill_gpu_pool(w, l, self.gpu[l])
            if w.num_host_blocks:
                sdev.fill_host_pool(w, l, self.host[l], self.dev)
        self.pool = hs.Pool(self.gpu, self.host if w.num_host_blocks else None)
        if prefetch:
            self.pool.set_miss_prefetch(prefetch)
        self.planes = tuple(planes)
        if self.planes:
            self.pool.set_gather_planes(self.planes)
        if self.force_order:
            self.pool.set_miss_order(self.order_mode)
        self.pool.set_miss_warps(self.miss_warps)
        self.pool.set_miss_sm_divisor(miss_sm_div)
        self.bt_np = w.block_table.copy()
        self.hbt_np = w.host_block_table.copy()
        self.bt = torch.from_numpy(self.bt_np).to(self.dev)
        self.hbt = torch.from_numpy(self.hbt_np).to(self.dev)
        self.hot_blocks = torch.from_numpy(w.hot_blocks.astype(np.int32)).to(self.dev)
        self.G = G = w.G
        self.hot = hs.HotState.allocate(L, self.hot_blocks, C, layers_per_index=G)
        hs.hot_reset(self.pool, self.hot)
        self.ws = hs.alloc_workspace(L // G, R, w.P, w.K, C, self.dev)
        self.ordered = hs.miss_order_used(self.pool, self.hot, L, R, w.P, w.K, self.ws.numel())
        assert self.ordered or not (self.force_order and w.num_host_blocks)
        self.o_tok = np.full((L // G, R, C), -1, np.int32)
        self.o_stamp = np.full((L // G, R, C), -1, np.int32)
        self.o_pools = self.o_hosts = None
        if oracle_bytes:
            self.o_pools = [np.zeros(w.num_gpu_blocks * S * B, np.uint8) for _ in range(L)]
            self.o_hosts = [np.zeros(nhb * S * B, np.uint8) for _ in range(L)]
            own_g, own_h = w.gpu_block_owner(), w.host_block_owner()
            for l in range(L):
                for blk in np.nonzero(own_g[:, 0] >= 0)[0]:
                    r, p = own_g[blk]
                    self.o_pools[l][blk * S * B:(blk + 1) * S * B] = content.page_np(
                        w.content_seed, l, int(w.content_page[r, p]), S, B).reshape(-1)
                for blk in np.nonzero(own_h[:, 0] >= 0)[0]:
                    r, p = own_h[blk]
                    self.o_hosts[l][blk * S * B:(blk + 1) * S * B] = content.page_np(
                        w.content_seed, l, int(w.content_page[r, p]), S, B).reshape(-1)
        torch.cuda.synchronize()

    # ------------------------------------------------------------------ one step on both sides
    def apply_edits(self, st) -> None:
        w = self.w
        for r, p, v in st.bt_edits:
            self.bt_np[r, p] = v
        for r, p, v in st.hbt_edits:
            self.hbt_np[r, p] = v
        if len(st.bt_edits):
            self.bt.copy_(torch.from_numpy(self.bt_np))
        if len(st.hbt_edits):
            self.hbt.copy_(torch.from_numpy(self.hbt_np))
        if len(st.fills):
            blocks = st.fills[:, 0].astype(np.int64)
            owners = st.fills[:, 1:].astype(np.int64)
            for l in range(w.L):
                sdev.fill_blocks(w, l, self.gpu[l], blocks, owners, self.dev)
                if self.o_pools is not None:
                    for b, (r, p) in zip(blocks, owners):
                        self.o_pools[l][b * w.S * w.B:(b + 1) * w.S * w.B] = content.page_np(
                            w.content_seed, l, int(w.content_page[r, p]), w.S, w.B).reshape(-1)

    def step(self, st, *, check: bool = True):
        w = self.w
        self.apply_edits(st)
        topk = torch.from_numpy(st.topk).to(self.dev)
        ctx = torch.from_numpy(st.ctx_len.astype(np.int32)).to(self.dev)
        if self.graph:
            rows, stats, out = self._graph_step(st, topk, ctx)
        elif self.mode == "fused":
            rows, stats, out = hs.resolve_gather(self.pool, topk, self.bt, self.hbt, ctx, self.hot, st.index,
                                                 workspace=self.ws)
        else:
            rows, stats = hs.resolve_topk(self.pool, topk, self.bt, self.hbt, ctx, self.hot, st.index,
                                          workspace=self.ws)
            if self.G == 1:
                out = hs.gather_rows(self.pool, rows.reshape(w.L, -1))
            else:   # each layer of an index group gathers the group's rows
                out = torch.empty((w.L, w.R * w.P * w.K, w.B), dtype=torch.uint8, device=self.dev)
                for l in range(w.L):
                    hs.gather_rows(self.pool, rows[l // self.G].reshape(-1), layer_begin=l, out=out[l])
        if len(st.off_gpu) and not self.graph:
            hs.offload_pages(self.pool, torch.from_numpy(st.off_gpu).to(self.dev),
                             torch.from_numpy(st.off_host).to(self.dev))
        torch.cuda.synchronize()
        o_rows, o_stats = oracle.resolve(S=w.S, B=w.B, num_gpu_blocks=w.num_gpu_blocks,
                                         num_host_blocks=w.num_host_blocks, topk=st.topk, block_table=self.bt_np,
                                         host_block_table=self.hbt_np, ctx_len=st.ctx_len, max_pages=w.max_pages,
                                         C=w.C, hot_blocks=w.hot_blocks, slot_token=self.o_tok,
                                         slot_stamp=self.o_stamp, step=st.index, pools=self.o_pools,
                                         hosts=self.o_hosts, layers_per_index=self.G)
        if len(st.off_gpu) and self.o_pools is not None:
            oracle.offload(S=w.S, B=w.B, num_gpu_blocks=w.num_gpu_blocks, num_host_blocks=w.num_host_blocks,
                           pools=self.o_pools, hosts=self.o_hosts, gpu_blocks=st.off_gpu, host_blocks=st.off_host)
        if check:
            self.compare(st, rows, stats, out, o_rows, o_stats)
            self.check_offload(st)
        return rows, stats, out, o_rows, o_stats

    def check_offload(self, st) -> None:
        """Every page offloaded after this step holds, in every layer, the closed-form rows of its page."""
        w = self.w
        for (r, pg), h in zip(st.off_src, st.off_host):
            for l in range(w.L):
                exp = content.page_np(w.content_seed, l, int(w.content_page[r, pg]), w.S, w.B)
                assert np.array_equal(self.host[l][int(h)].numpy(), exp), f"offloaded page ({r},{pg}) layer {l}"

    def _graph_step(self, st, topk, ctx):
        """The whole step (resolve + gather, and the step's offload) captured into one CUDA graph, then
        replayed once."""
        w = self.w
        if self.prep is None:
            self.ctx_dev = torch.empty(w.R, dtype=torch.int32, device=self.dev)
            self.g_rows = torch.empty((w.L // self.G, w.R, w.P, w.K), dtype=torch.int32, device=self.dev)
            self.g_stats = torch.empty((w.L // self.G, w.R, 4), dtype=torch.int32, device=self.dev)
            self.g_out = torch.empty((w.L, w.R * w.P * w.K, w.B), dtype=torch.uint8, device=self.dev)
            self.prep = hs.PreparedStep(self.pool, self.hot, self.bt, self.hbt, self.ctx_dev, self.g_rows,
                                        self.g_stats, self.ws, self.g_out)
        self.ctx_dev.copy_(ctx)
        gb = torch.from_numpy(st.off_gpu).to(self.dev)
        hb = torch.from_numpy(st.off_host).to(self.dev)
        torch.cuda.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            if self.mode == "fused":
                self.prep.resolve_gather(topk, st.index)
            else:
                self.prep.resolve(topk, st.index)
                self.prep.gather()
            self.prep.offload(gb, hb, len(st.off_gpu))
        g.replay()
        torch.cuda.synchronize()
        return self.g_rows, self.g_stats, self.g_out.reshape(w.L, -1, w.B)

    def compare(self, st, rows, stats, out, o_rows, o_stats) -> None:
        w = self.w
        if self.planes:   # back to rows: each plane is a column range of the rows
            views = hs.plane_views(out, self.planes)
            out = torch.cat(views, dim=-1)
        g_rows = rows.cpu().numpy()
        g_stats = stats.cpu().numpy()
        assert np.array_equal(g_stats, o_stats), f"stats differ at step {st.index}"
        assert np.array_equal(g_rows, o_rows), f"rows differ at step {st.index}"
        assert np.array_equal(self.hot.slot_token.cpu().numpy(), self.o_tok), f"slot_token differs at step {st.index}"
        assert np.array_equal(self.hot.slot_stamp.cpu().numpy(), self.o_stamp), f"slot_stamp differs at step {st.index}"
        # gathered bytes == closed-form bytes of each logical token (zero for padding / failed units)
        ids = torch.from_numpy(st.topk).to(self.dev)
        ok = torch.from_numpy(o_stats[..., 0] == 0).to(self.dev)
        for l in range(w.L):
            idl = ids[l // self.G].reshape(w.R, -1).long()
            idl = torch.where(ok[l // self.G][:, None], idl, torch.full_like(idl, -1))
            r_idx = torch.arange(w.R, device=self.dev)[:, None].expand_as(idl).reshape(-1)
            flat = idl.reshape(-1)
            for c0 in range(0, flat.numel(), 1 << 18):
                exp = sdev.expected_rows(w, l, r_idx[c0:c0 + (1 << 18)], flat[c0:c0 + (1 << 18)])
                assert torch.equal(out[l][c0:c0 + (1 << 18)], exp), f"gathered bytes differ at step {st.index} layer {l}"
        if self.o_pools is not None:
            for l in range(w.L):
                assert np.array_equal(self.gpu[l].cpu().numpy().reshape(-1), self.o_pools[l]), \
                    f"pool bytes differ at step {st.index} layer {l}"
                if w.num_host_blocks:
                    assert np.array_equal(self.host[l].numpy().reshape(-1), self.o_hosts[l]), \
                        f"host pool differs at step {st.index} layer {l}"
        elif self.check_hot_bytes:
            self.check_hot_rows()

    def check_hot_rows(self) -> None:
        """Every filled hot slot's pool row holds the closed-form bytes of its token."""
        w = self.w
        tok = self.hot.slot_token
        for l in range(w.L):
            t = tok[l // self.G].long()
            r_idx = torch.arange(w.R, device=self.dev)[:, None].expand_as(t)
            v = torch.arange(w.C, device=self.dev)[None, :].expand_as(t)
            prow = self.hot_blocks.long()[r_idx, v // w.S] * w.S + v % w.S
            m = t >= 0
            rows_m, r_m, t_m = prow[m], r_idx[m], t[m]
            for c0 in range(0, rows_m.numel(), 1 << 18):
                sl = slice(c0, c0 + (1 << 18))
                got = self.gpu[l].reshape(-1, w.B)[rows_m[sl]]
                exp = sdev.expected_rows(w, l, r_m[sl], t_m[sl])
                assert torch.equal(got, exp), f"hot rows differ from their tokens' bytes (layer {l})"
