"""hs_resolve_topk_noalloc: the resolver for callers that cannot allocate device memory.

Some callers cannot call cudaMalloc: a plug-in inside a serving engine that has already reserved
nearly all device memory for its KV cache, a decode loop that must not let cudaMalloc synchronise
the device, or a C caller with no device allocator.  This entry point takes no workspace; its scratch
is a fixed-size array compiled into the library.  The test calls it through the C ABI (ctypes on
libhs.so) and checks, on two calls in a row, that its rows, stats, hot state and pool bytes equal
those of hs_resolve_topk given a caller-allocated workspace (tolerance 0: integer and byte work),
with and without IndexShare (several layers reading one top-K list, whose units are index groups).
This file is collected last on purpose, so a run that stops at the first failure has already run
every other test; it also passes on its own in a fresh process.
"""
import ctypes

import numpy as np
import pytest
import torch

pytestmark = pytest.mark.gpu

HS_STATIC_SCRATCH_BYTES = 32 << 20


@pytest.fixture(scope="module")
def lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from sparse_mla_kv_gb300 import _build
    _build.build()
    import sparse_mla_kv_gb300 as hs
    L = hs.lib()
    p, i32 = ctypes.c_void_p, ctypes.c_int32
    L.hs_resolve_topk_noalloc.restype = i32
    L.hs_resolve_topk_noalloc.argtypes = [p, i32, i32, i32, i32, i32, p, p, p, p, i32, ctypes.POINTER(hs.HotStateC), i32,
                                          p, p, p]
    return L


def _twin(w, dev):
    """One workload's pool + hot state, built twice with identical bytes (the GPU pools are separate
    because misses write into them; the pinned host pool is only read and is shared)."""
    import sparse_mla_kv_gb300 as hs
    from synth import device as sdev
    host = [torch.empty((w.num_host_blocks, w.S, w.B), dtype=torch.uint8, pin_memory=True)]
    sdev.fill_host_pool(w, 0, host[0], dev)
    sides = []
    for _ in range(2):
        gpu = [torch.empty((w.num_gpu_blocks, w.S, w.B), dtype=torch.uint8, device=dev)]
        sdev.fill_gpu_pool(w, 0, gpu[0])
        pool = hs.Pool(gpu, host)
        hot = hs.HotState.allocate(1, torch.from_numpy(w.hot_blocks).to(dev), w.C)
        hs.hot_reset(pool, hot)
        sides.append((pool, gpu, hot))
    return sides


@pytest.mark.parametrize("cfg", [1, 4])
def test_noalloc_matches_workspace_entry_point_twice(lib, cfg):
    import sparse_mla_kv_gb300 as hs
    from synth import workloads
    dev = torch.device("cuda")
    w = workloads.config1(seed=11, steps=2) if cfg == 1 else workloads.config4(seed=11, steps=2, R=4)
    (pool_a, gpu_a, hot_a), (pool_b, gpu_b, hot_b) = _twin(w, dev)
    bt = torch.from_numpy(w.block_table).to(dev)
    hbt = torch.from_numpy(w.host_block_table).to(dev)
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    assert hs.resolve_workspace_bytes_min(w.L, w.R, w.P, w.K, w.C) <= HS_STATIC_SCRATCH_BYTES
    for st in w.iter_steps():   # two calls in a row
        topk = torch.from_numpy(st.topk).to(dev)
        ctx = torch.from_numpy(st.ctx_len).to(dev)
        rows_a, stats_a = hs.resolve_topk(pool_a, topk, bt, hbt, ctx, hot_a, st.index)
        rows_b = torch.empty_like(topk)
        stats_b = torch.empty((w.L, w.R, 4), dtype=torch.int32, device=dev)
        code = lib.hs_resolve_topk_noalloc(pool_b.handle, 0, w.L, w.R, w.P, w.K, ctypes.c_void_p(topk.data_ptr()),
                                           ctypes.c_void_p(bt.data_ptr()), ctypes.c_void_p(hbt.data_ptr()),
                                           ctypes.c_void_p(ctx.data_ptr()), w.max_pages, ctypes.byref(hot_b.c),
                                           st.index, ctypes.c_void_p(rows_b.data_ptr()),
                                           ctypes.c_void_p(stats_b.data_ptr()), stream)
        assert code == 0, hs.status_str(code)
        torch.cuda.synchronize()
        assert (stats_a[..., 0] == 0).all() and int(stats_a[..., 3].sum()) > 0
        assert torch.equal(stats_a, stats_b)
        assert torch.equal(rows_a, rows_b)
        assert torch.equal(hot_a.slot_token, hot_b.slot_token)
        assert torch.equal(hot_a.slot_stamp, hot_b.slot_stamp)
        assert torch.equal(gpu_a[0], gpu_b[0])
    pool_a.close()
    pool_b.close()


def _group_inputs(rng, R, ctx, K, ng, prev=None):
    """[ng][R][1][K] distinct ids per (group, request); half of each list kept from prev."""
    out = np.empty((ng, R, 1, K), np.int32)
    for g in range(ng):
        for r in range(R):
            if prev is None:
                out[g, r, 0] = rng.choice(ctx, size=K, replace=False)
            else:
                keep = rng.choice(prev[g, r, 0], size=K // 2, replace=False)
                rest = np.setdiff1d(np.arange(ctx), keep)
                out[g, r, 0] = rng.permutation(np.concatenate([keep, rng.choice(rest, size=K - K // 2, replace=False)]))
    return out


@pytest.mark.parametrize("G,R", [(2, 16), (4, 256)])
def test_noalloc_index_share_matches_workspace_entry_point_twice(lib, G, R):
    """IndexShare (G layers per index group): the scratch bound counts index groups, so a shape with
    4 layers x 256 requests (1024 per-layer units, beyond the built-in array) is accepted with G = 4
    (256 units); rows, stats, hot state and the pool bytes of every layer equal those of
    hs_resolve_topk given a caller workspace, on two calls in a row."""
    import sparse_mla_kv_gb300 as hs
    dev = torch.device("cuda")
    rng = np.random.default_rng(G * 1000 + R)
    L, S, B, K, C, P = 4, 64, 16, 2048, 4096, 1
    pages, tail = 128, 16
    ctx = pages * S
    ng = L // G
    assert hs.resolve_workspace_bytes_min(ng, R, P, K, C) <= HS_STATIC_SCRATCH_BYTES
    if R == 256:   # the per-layer count alone would not fit
        assert hs.resolve_workspace_bytes_min(L, R, P, K, C) > HS_STATIC_SCRATCH_BYTES
    n_res = R * tail
    perm = rng.permutation(n_res + R * (C // S)).astype(np.int32)
    bt = np.full((R, pages), -1, np.int32)
    bt[:, pages - tail:] = perm[:n_res].reshape(R, tail)
    hot_blocks = perm[n_res:].reshape(R, C // S)
    hbt = rng.permutation(R * pages).astype(np.int32).reshape(R, pages)
    ngb = n_res + R * (C // S)
    host = [torch.randint(0, 256, (R * pages, S, B), dtype=torch.uint8).pin_memory() for _ in range(L)]
    base = [torch.randint(0, 256, (ngb, S, B), dtype=torch.uint8, device=dev) for _ in range(L)]
    sides = []
    for _ in range(2):
        gpu = [b.clone() for b in base]
        pool = hs.Pool(gpu, host)
        hot = hs.HotState.allocate(L, torch.from_numpy(hot_blocks).to(dev), C, layers_per_index=G)
        hs.hot_reset(pool, hot)
        sides.append((pool, gpu, hot))
    (pool_a, gpu_a, hot_a), (pool_b, gpu_b, hot_b) = sides
    bt_d, hbt_d = torch.from_numpy(bt).to(dev), torch.from_numpy(hbt).to(dev)
    ctx_d = torch.full((R,), ctx, dtype=torch.int32, device=dev)
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    ids = None
    for step in (5, 6):   # two calls in a row
        ids = _group_inputs(rng, R, ctx, K, ng, ids)
        topk = torch.from_numpy(ids).to(dev)
        rows_a, stats_a = hs.resolve_topk(pool_a, topk, bt_d, hbt_d, ctx_d, hot_a, step)
        rows_b = torch.empty_like(topk)
        stats_b = torch.empty((ng, R, 4), dtype=torch.int32, device=dev)
        code = lib.hs_resolve_topk_noalloc(pool_b.handle, 0, L, R, P, K, ctypes.c_void_p(topk.data_ptr()),
                                           ctypes.c_void_p(bt_d.data_ptr()), ctypes.c_void_p(hbt_d.data_ptr()),
                                           ctypes.c_void_p(ctx_d.data_ptr()), pages, ctypes.byref(hot_b.c), step,
                                           ctypes.c_void_p(rows_b.data_ptr()), ctypes.c_void_p(stats_b.data_ptr()),
                                           stream)
        assert code == 0, hs.status_str(code)
        torch.cuda.synchronize()
        assert (stats_a[..., 0] == 0).all() and int(stats_a[..., 3].sum()) > 0
        assert torch.equal(stats_a, stats_b)
        assert torch.equal(rows_a, rows_b)
        assert torch.equal(hot_a.slot_token, hot_b.slot_token)
        assert torch.equal(hot_a.slot_stamp, hot_b.slot_stamp)
        for l in range(L):
            assert torch.equal(gpu_a[l], gpu_b[l]), f"layer {l}"
    pool_a.close()
    pool_b.close()


def test_noalloc_refuses_shapes_beyond_its_scratch(lib):
    import sparse_mla_kv_gb300 as hs
    dev = torch.device("cuda")
    S, C = 64, 4096
    gpu = [torch.zeros((C // S, S, 16), dtype=torch.uint8, device=dev)]
    pool = hs.Pool(gpu, None)
    hot = hs.HotState.allocate(1, torch.arange(C // S, dtype=torch.int32, device=dev)[None], C)
    R, P, K = 400, 4, 2048     # 400 units x 96 KB of scratch > the built-in 32 MiB
    assert hs.resolve_workspace_bytes_min(1, R, P, K, C) > HS_STATIC_SCRATCH_BYTES
    dummy = torch.zeros(16, dtype=torch.int32, device=dev)
    d = ctypes.c_void_p(dummy.data_ptr())
    code = lib.hs_resolve_topk_noalloc(pool.handle, 0, 1, R, P, K, d, d, d, d, 1, ctypes.byref(hot.c), 0, d, d,
                                       ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert code == 1    # HS_ERR_INVALID_ARG, nothing launched
    pool.close()
