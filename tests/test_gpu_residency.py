"""End to end on the GPU with the native residency manager deciding residency (no precomputed
tables): requests decode under KV pressure, so pages are released once their host copy is queued,
hot buffers are leased from the same pool, and released pages come back through the resolver's miss
path from the host copies that the post-forward offload launches wrote.

Checked every step: resolver rows, stats and hot state against the oracle run on the same tables;
every gathered row and every filled hot slot against the closed-form bytes of its logical token;
every offloaded host page against the closed-form bytes of its page."""
from types import SimpleNamespace

import numpy as np
import pytest
import torch

import oracle
import sparse_mla_kv_gb300 as hs
from synth import content, device as sdev, workloads

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from sparse_mla_kv_gb300 import _build
    _build.build()
    hs.lib()


@pytest.mark.parametrize("mode", ["fused", "split"])
def test_managed_decode_under_pressure(mode):
    from sparse_mla_kv_gb300.residency import Residency

    dev = torch.device("cuda")
    L, R, S, B, K, C = 2, 6, 64, 656, 256, 512
    Hc, max_pages, G, H = C // S, 64, 190, 2048
    rng = np.random.default_rng(11)
    # content ids: request r's own page p -> r * max_pages + p; a shared host prefix -> 10**6 + p
    w = SimpleNamespace(S=S, B=B, content_seed=77,
                        content_page=(np.arange(R)[:, None] * max_pages + np.arange(max_pages)[None, :]).astype(np.int64))
    prefix_pages = 10
    prefix_host = list(range(H - prefix_pages, H))
    w.content_page[R - 1, :prefix_pages] = 10 ** 6 + np.arange(prefix_pages)

    gpu = [torch.zeros((G, S, B), dtype=torch.uint8, device=dev) for _ in range(L)]
    host = [sdev.pinned_empty((H, S, B)) for _ in range(L)]
    for l in range(L):   # the shared prefix exists only in host memory (written by DMA)
        sdev.fill_blocks(w, l, host[l], np.array(prefix_host), np.stack([np.full(prefix_pages, R - 1),
                                                                        np.arange(prefix_pages)], 1), dev)
    pool = hs.Pool(gpu, host)
    m = Residency(G, H, S, R, max_pages, Hc)
    m.hold_host(prefix_host)                 # a prefix cache keeps these host blocks

    hot_dev = torch.full((R, Hc), -1, dtype=torch.int32, device=dev)
    hot = hs.HotState.allocate(L, hot_dev, C)
    hs.hot_reset(pool, hot)
    o_tok = np.full((L, R, C), -1, np.int32)
    o_stamp = np.full((L, R, C), -1, np.int32)
    ws = hs.alloc_workspace(L, R, 1, K, C, dev)

    def apply_fills():
        f = m.take_fills()
        if f:
            blocks = np.array([x[0] for x in f])
            owners = np.array([(x[1], x[2]) for x in f])
            for l in range(L):
                sdev.fill_blocks(w, l, gpu[l], blocks, owners, dev)

    def offload_collected():
        pairs = m.collect()
        if not pairs:
            return 0
        gb = torch.tensor([p[0] for p in pairs], dtype=torch.int32, device=dev)
        hb = torch.tensor([p[1] for p in pairs], dtype=torch.int32, device=dev)
        hs.offload_pages(pool, gb, hb)
        torch.cuda.synchronize()
        _, hbt, _, _ = m.tables()
        for g_, h_ in pairs:
            r_, p_ = (int(v[0]) for v in np.nonzero(hbt == h_))
            for l in range(L):
                exp = content.page_np(w.content_seed, l, int(w.content_page[r_, p_]), S, B)
                assert np.array_equal(host[l][h_].numpy(), exp), (r_, p_, l)
        return len(pairs)

    for r in range(R - 1):                   # prefill: 21 pages each, copies queued and launched
        m.admit(r, 20 * S + 5)
        apply_fills()
        offload_collected()
    m.admit(R - 1, prefix_pages * S + 100, prefix_host)   # prefix reuse: placeholders + hot page
    apply_fills()
    offload_collected()

    prev = [[None] * R for _ in range(L)]
    released_seen = misses = offloads = 0
    for step in range(40):
        for r in range(R):
            m.append(r, int(rng.integers(8, 48)))
        apply_fills()
        bt_np, hbt_np, hot_np, ctx_np = m.tables()
        resets = m.take_resets()
        hot_dev.copy_(torch.from_numpy(hot_np))
        if resets:
            hs.hot_reset_requests(pool, hot, torch.tensor(resets, dtype=torch.int32, device=dev))
            o_tok[:, resets] = -1
            o_stamp[:, resets] = -1
        topk = np.empty((L, R, 1, K), np.int32)
        for l in range(L):
            for r in range(R):
                ids = workloads.next_topk(rng, prev[l][r], int(ctx_np[r]), K, 0.8 if prev[l][r] is not None else 0.0,
                                          "recency")
                prev[l][r] = ids
                topk[l, r, 0] = ids
        bt, hbt = torch.from_numpy(bt_np).to(dev), torch.from_numpy(hbt_np).to(dev)
        ctx = torch.from_numpy(ctx_np).to(dev)
        topk_d = torch.from_numpy(topk).to(dev)
        if mode == "fused":
            rows, stats, out = hs.resolve_gather(pool, topk_d, bt, hbt, ctx, hot, step, workspace=ws)
        else:
            rows, stats = hs.resolve_topk(pool, topk_d, bt, hbt, ctx, hot, step, workspace=ws)
            out = hs.gather_rows(pool, rows.reshape(L, -1))
        torch.cuda.synchronize()
        o_rows, o_stats = oracle.resolve(S=S, B=B, num_gpu_blocks=G, num_host_blocks=H, topk=topk, block_table=bt_np,
                                         host_block_table=hbt_np, ctx_len=ctx_np, max_pages=max_pages, C=C,
                                         hot_blocks=hot_np, slot_token=o_tok, slot_stamp=o_stamp, step=step)
        assert (o_stats[..., 0] == 0).all(), o_stats[..., 0]
        assert np.array_equal(stats.cpu().numpy(), o_stats), step
        assert np.array_equal(rows.cpu().numpy(), o_rows), step
        assert np.array_equal(hot.slot_token.cpu().numpy(), o_tok), step
        assert np.array_equal(hot.slot_stamp.cpu().numpy(), o_stamp), step
        misses += int(o_stats[..., 3].sum())
        r_idx = torch.arange(R, device=dev)[:, None].expand(R, K).reshape(-1)
        for l in range(L):
            exp = sdev.expected_rows(w, l, r_idx, topk_d[l].reshape(-1).long())
            assert torch.equal(out.reshape(L, -1, B)[l], exp), (step, l)
            t = hot.slot_token[l].long()
            filled = t >= 0
            if filled.any():
                rr = torch.arange(R, device=dev)[:, None].expand_as(t)[filled]
                v = torch.arange(C, device=dev)[None, :].expand_as(t)[filled]
                prow = hot_dev.long()[rr, v // S] * S + v % S
                assert torch.equal(gpu[l].reshape(-1, B)[prow], sdev.expected_rows(w, l, rr, t[filled])), (step, l)
        for r in range(R):
            m.touch(r, topk[0, r, 0], step)
        offloads += offload_collected()
        released_seen = max(released_seen, int(((bt_np < 0) & (hbt_np >= 0)).sum()) - prefix_pages)
    assert released_seen > 0 and misses > 0 and offloads > 0
    assert all(h[0] >= 0 for h in m.tables()[2])   # every request ended up with a hot buffer
    pool.close()
