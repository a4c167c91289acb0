"""GPU parity: the CUDA library (through its C ABI) against the oracle, bit for bit.

Compared on every step: out_rows, out_stats, slot_token, slot_stamp (oracle), gathered bytes
(closed-form row contents), and pool bytes (oracle with byte pools) or hot-slot bytes (closed form).
Tolerance is zero everywhere: this is integer and byte work."""
import ctypes

import numpy as np
import pytest
import torch

import oracle
import sparse_mla_kv_gb300 as hs
from synth import workloads
from tests.casekit import Case
from tests.test_bruteforce_vs_oracle import _ids, _random_case

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from sparse_mla_kv_gb300 import _build
    _build.build()
    hs.lib()


def _rig(w, **kw):
    from tests.gpukit import Rig
    return Rig(w, **kw)


MODES = ["split", "fused"]
# the same, plus both paths with the address-ordered miss layout forced on (small pools default to
# per-unit lists)
MODES_ORDER = MODES + ["split+order", "fused+order", "split+ranges", "fused+ranges", "fused+ranges1",
                       "fused+ranges2", "fused+part"]


def _base(mode):
    return mode.partition("+")[0]


def _set_order(pool, mode):
    """+order: the address-ordered miss layout on any pool (its spread schedule on small pools);
    +ranges: its range schedule with the fused gather's default SM partition; +ranges1 / +ranges2: with one
    or two miss warps in every fused-gather CTA; +part: the default layout with the SM partition."""
    opt = mode.partition("+")[2]
    if opt == "part":
        pool.set_miss_warps(0)
    elif opt == "order":
        pool.set_miss_order(hs.MISS_ORDER_ON)
    elif opt.startswith("ranges"):
        pool.set_miss_order(hs.MISS_ORDER_RANGES)
        pool.set_miss_warps({"ranges1": 1, "ranges2": 2}.get(opt, 0))


@pytest.mark.parametrize("mode", MODES_ORDER)
def test_tiny_decode_all_bytes(mode):
    w = workloads.config1(seed=0, steps=8)
    rig = _rig(w, oracle_bytes=True, mode=mode)
    misses = 0
    for st in w.iter_steps():
        _, stats, _, _, _ = rig.step(st)
        misses += int(stats[..., 3].sum())
    assert misses > 0


@pytest.mark.parametrize("mode", ["split", "fused", "split+order", "fused+order", "fused+ranges"])
def test_miss_prefetch_same_results(mode):
    """With the resolver's miss prefetch on, every path and miss layout gives the oracle's rows, stats,
    hot state and bytes (tiny decode, all bytes compared) and the closed-form bytes on an IndexShare MTP3
    batch (two layers per index group: each miss is prefetched in both layers)."""
    w = workloads.config1(seed=6, steps=6)
    rig = _rig(w, oracle_bytes=True, mode=mode, prefetch=hs.MISS_PREFETCH_ON)
    misses = 0
    for st in w.iter_steps():
        _, stats, _, _, _ = rig.step(st)
        misses += int(stats[..., 3].sum())
    assert misses > 0
    w = workloads.config5(seed=7, R=6, L=4, layers_per_index=2, steps=4)
    rig = _rig(w, mode=mode, prefetch=hs.MISS_PREFETCH_ON)
    for st in w.iter_steps():
        rig.step(st)


@pytest.mark.parametrize("div", [2, 3, 32, -1])
def test_sm_partition_divisors(div):
    """The fused gather's SM partition gives the oracle's bytes whatever share of the SMs copies the
    misses (every second, third or 32nd SM), and with no miss SM at all (-1: every CTA streams its HBM
    rows, then drains the misses -- the path of a launch whose CTAs land on no miss SM), on the tiny
    decode and on a small MTP3 batch."""
    w = workloads.config1(seed=4, steps=6)
    rig = _rig(w, oracle_bytes=True, mode="fused+ranges", miss_sm_div=div)
    misses = 0
    for st in w.iter_steps():
        _, stats, _, _, _ = rig.step(st)
        misses += int(stats[..., 3].sum())
    assert misses > 0
    w = workloads.config5(seed=5, R=6, L=2, steps=4)
    rig = _rig(w, mode="fused+ranges", miss_sm_div=div)
    for st in w.iter_steps():
        rig.step(st)


@pytest.mark.parametrize("div", [0, -1])
def test_partition_phase_timestamps(div):
    """hs_pool_set_phase_timestamps: every SM-partition launch records its start, the end of its HBM rows,
    the end of its misses and its own end, in order, without changing any result (small MTP3 batch with
    the range schedule; the default share of miss SMs and no miss SM)."""
    w = workloads.config5(seed=11, R=6, L=2, steps=4)
    rig = _rig(w, mode="fused+ranges", miss_sm_div=div)
    ts = torch.zeros(4, dtype=torch.int64, device="cuda")
    rig.pool.set_phase_timestamps(ts)
    for st in w.iter_steps():
        ts.zero_()
        ts[0] = -1
        _, stats, *_ = rig.step(st)
        t = ts.cpu().tolist()
        assert t[0] > 0 and t[3] >= t[1] >= t[0] and t[1] > 0, t
        if int(stats[..., 3].sum()):
            assert t[3] >= t[2] >= t[0] and t[2] > 0, t
    rig.pool.set_phase_timestamps(None)
    assert hs.lib().hs_pool_set_phase_timestamps(rig.pool.handle, ctypes.c_void_p(ts.data_ptr() + 8)) == 1


@pytest.mark.parametrize("mode", MODES)
def test_tiny_decode_other_seeds_and_replay(mode):
    for seed in (1, 2):
        w = workloads.config1(seed=seed, steps=6)
        rig = _rig(w, oracle_bytes=True, mode=mode)
        for st in w.iter_steps():
            rows, stats, *_ = rig.step(st)
            # replay the same step: same rows, no misses, state unchanged
            tok = rig.hot.slot_token.clone()
            rows2, stats2, *_ = rig.step(st)
            assert torch.equal(rows, rows2)
            assert int(stats2[..., 3].sum()) == 0
            assert torch.equal(tok, rig.hot.slot_token)


def _case_to_gpu(case, dev):
    S, B = case.S, case.B
    gpu = [torch.from_numpy(case.pools[0].reshape(case.ngb, S, B).copy()).to(dev)]
    host = [torch.from_numpy(case.hosts[0].reshape(-1, S, B).copy()).pin_memory()]
    pool = hs.Pool(gpu, host)
    hot_blocks = torch.from_numpy(case.hot_blocks).to(dev)
    hot = hs.HotState.allocate(1, hot_blocks, case.C)
    hs.hot_reset(pool, hot)
    return pool, gpu, host, hot


@pytest.mark.parametrize("mode", MODES_ORDER)
def test_random_small_cases_vs_oracle(mode):
    """Random small shapes (page sizes 1/2/4, several positions, duplicates, padding, replays,
    invalid ids, steps going backwards) through the library and the oracle with byte pools."""
    rng = np.random.default_rng(777)
    dev = torch.device("cuda")
    seen = set()
    for ci in range(150):
        case, P, K = _random_case(rng)
        pool, gpu, host, hot = _case_to_gpu(case, dev)
        _set_order(pool, mode)
        bt, hbt = torch.from_numpy(case.bt).to(dev), torch.from_numpy(case.hbt).to(dev)
        ctx = torch.from_numpy(case.ctx).to(dev)
        t = 0
        for si in range(int(rng.integers(1, 10))):
            u = rng.random()
            t = t if u < 0.1 else (max(0, t - 2) if u < 0.13 else t + int(rng.integers(1, 3)))
            ids = _ids(rng, case, P, K)
            if _base(mode) == "fused":
                rows, stats, g = hs.resolve_gather(pool, torch.from_numpy(ids[None]).to(dev), bt, hbt, ctx, hot, t)
            else:
                rows, stats = hs.resolve_topk(pool, torch.from_numpy(ids[None]).to(dev), bt, hbt, ctx, hot, t)
                g = hs.gather_rows(pool, rows.reshape(1, -1))
            o_rows, o_stats = case.step(ids, t)
            torch.cuda.synchronize()
            seen.update(o_stats[0, :, 0].tolist())
            msg = f"case {ci} step {si}"
            assert np.array_equal(stats.cpu().numpy(), o_stats), msg
            assert np.array_equal(rows.cpu().numpy(), o_rows), msg
            assert np.array_equal(hot.slot_token.cpu().numpy(), case.tok), msg
            assert np.array_equal(hot.slot_stamp.cpu().numpy(), case.stamp), msg
            assert np.array_equal(gpu[0].cpu().numpy().reshape(-1), case.pools[0]), msg
            o_out, _ = case.gather(o_rows.reshape(1, -1))
            assert np.array_equal(g.cpu().numpy(), o_out), msg
        pool.close()
    assert {0, 2, 5}.issubset(seen)


def _group_case_to_gpu(case, dev, G):
    S, B = case.S, case.B
    gpu = [torch.from_numpy(p.reshape(case.ngb, S, B).copy()).to(dev) for p in case.pools]
    host = [torch.from_numpy(h.reshape(-1, S, B).copy()).pin_memory() for h in case.hosts]
    pool = hs.Pool(gpu, host)
    hot = hs.HotState.allocate(case.L, torch.from_numpy(case.hot_blocks).to(dev), case.C, layers_per_index=G)
    hs.hot_reset(pool, hot)
    return pool, gpu, host, hot


@pytest.mark.parametrize("mode", MODES_ORDER)
def test_index_share_random_small_cases_vs_oracle(mode):
    """IndexShare: G in {2, 4} layers read one top-K list and share one hot state per request; calls
    cover a window of index groups.  Rows, stats, the group states, every layer's pool bytes and the
    gathered bytes of every layer equal the oracle's."""
    rng = np.random.default_rng(4242)
    dev = torch.device("cuda")
    for ci in range(60):
        case0, P, K = _random_case(rng)
        G = int(rng.choice([2, 4]))
        ng_total = int(rng.integers(1, 3))
        case = Case(R=case0.R, S=case0.S, B=case0.B, C=case0.C, max_pages=case0.max_pages, ctx=case0.ctx,
                    resident=True, host=True, hot_blocks=case0.hot_blocks, num_gpu_blocks=case0.ngb,
                    num_host_blocks=case0.nhb, bt=case0.bt, hbt=case0.hbt, L=G * ng_total, seed=case0.seed)
        case.tok = np.full((ng_total, case.R, case.C), -1, np.int32)
        case.stamp = np.full((ng_total, case.R, case.C), -1, np.int32)
        pool, gpu, host, hot = _group_case_to_gpu(case, dev, G)
        _set_order(pool, mode)
        bt, hbt = torch.from_numpy(case.bt).to(dev), torch.from_numpy(case.hbt).to(dev)
        ctx = torch.from_numpy(case.ctx).to(dev)
        g0 = int(rng.integers(0, ng_total))
        ng = int(rng.integers(1, ng_total - g0 + 1))
        lb = g0 * G
        t = 0
        for si in range(int(rng.integers(1, 8))):
            t += int(rng.integers(0, 3))
            ids = np.stack([_ids(rng, case, P, K) for _ in range(ng)])
            ids_d = torch.from_numpy(ids).to(dev)
            if _base(mode) == "fused":
                rows, stats, g = hs.resolve_gather(pool, ids_d, bt, hbt, ctx, hot, t, layer_begin=lb)
            else:
                rows, stats = hs.resolve_topk(pool, ids_d, bt, hbt, ctx, hot, t, layer_begin=lb)
                g = torch.stack([hs.gather_rows(pool, rows[l // G].reshape(-1), layer_begin=lb + l)
                                 for l in range(ng * G)])
            o_rows, o_stats = oracle.resolve(
                S=case.S, B=case.B, num_gpu_blocks=case.ngb, num_host_blocks=case.nhb, topk=ids,
                block_table=case.bt, host_block_table=case.hbt, ctx_len=case.ctx, max_pages=case.max_pages,
                C=case.C, hot_blocks=case.hot_blocks, slot_token=case.tok, slot_stamp=case.stamp, step=t,
                layer_begin=lb, pools=case.pools, hosts=case.hosts, threads=2, layers_per_index=G)
            torch.cuda.synchronize()
            msg = f"case {ci} step {si} G={G}"
            assert np.array_equal(stats.cpu().numpy(), o_stats), msg
            assert np.array_equal(rows.cpu().numpy(), o_rows), msg
            assert np.array_equal(hot.slot_token.cpu().numpy(), case.tok), msg
            assert np.array_equal(hot.slot_stamp.cpu().numpy(), case.stamp), msg
            for l in range(case.L):
                assert np.array_equal(gpu[l].cpu().numpy().reshape(-1), case.pools[l]), f"{msg} layer {l}"
            o_out, _ = case.gather(np.repeat(o_rows.reshape(ng, -1), G, axis=0), layer_begin=lb)
            assert np.array_equal(g.cpu().numpy().reshape(o_out.shape), o_out), msg
        pool.close()


@pytest.mark.parametrize("mode", MODES)
def test_index_share_multi_turn_agentic(mode):
    """IndexShare on the agentic shape: 8 layers in 2 index groups of 4 (one indexer per four
    sparse-MLA layers), 32 requests at 74,160+ tokens, compressed turns so that turn boundaries,
    block reuse and all-layer offloads fall inside 14 steps."""
    w = workloads.config3(seed=5, decode_per_turn=6, L=8, layers_per_index=4)
    rig = _rig(w, mode=mode)
    misses = 0
    for st in w.iter_steps(14):
        _, stats, *_ = rig.step(st)
        misses += int(stats[..., 3].sum())
    assert misses > 0


@pytest.mark.parametrize("mode", MODES_ORDER)
def test_index_share_graph_capture(mode):
    """IndexShare steps captured into CUDA graphs (resolve, the per-layer or fused gather, offload)."""
    w = workloads.config3(seed=6, decode_per_turn=6, L=4, R=8, layers_per_index=2)
    rig = _rig(w, mode=mode, graph=True)
    for st in w.iter_steps(13):
        rig.step(st)


@pytest.mark.parametrize("mode", ["fused", "split+order", "fused+order"])
def test_index_share_mtp3_64_requests(mode):
    """IndexShare with MTP3 plans: 4 layers in one index group, 64 requests, P=4 positions."""
    w = workloads.config5(seed=2, steps=3, R=64, layers_per_index=4)
    rig = _rig(w, mode=mode)
    for st in w.iter_steps(3):
        rig.step(st)


@pytest.mark.parametrize("mode", MODES)
def test_mixed_residency_decode_full_size(mode):
    """The 64-request, 131072-token, K=2048 mixed-residency batch (the benchmarked workload) for all
    of its 64 steps."""
    w = workloads.config2(seed=0, steps=64)
    rig = _rig(w, mode=mode)
    tot = np.zeros(3, np.int64)
    for st in w.iter_steps():
        _, stats, *_ = rig.step(st)
        tot += stats[..., 1:].sum(axis=(0, 1)).cpu().numpy()
    assert tot[1] > 0 and tot[2] > 0   # both hits and misses happened


@pytest.mark.parametrize("mode", MODES)
def test_full_residency_batch(mode):
    """The mixed batch with every page resident (no KV pressure): every id is read in place, there is
    no hit and no miss, and the hot state stays empty -- the resolver's full-residency path."""
    w = workloads.config2(seed=1, steps=4, R=16, resident_tokens=131072)
    rig = _rig(w, mode=mode)
    for st in w.iter_steps():
        _, stats, *_ = rig.step(st)
        s = stats.cpu().numpy()
        assert (s[..., 0] == 0).all() and (s[..., 2:] == 0).all() and (s[..., 1] > 0).all()
    assert (rig.hot.slot_token.cpu().numpy() == -1).all()


@pytest.mark.parametrize("mode", MODES_ORDER)
def test_cold_start_prefix_reuse_full_size(mode):
    """16 requests reusing a 1,048,576-token host-only prefix, empty hot buffers, 32 steps."""
    w = workloads.config4(seed=0, steps=32)
    rig = _rig(w, mode=mode)
    for st in w.iter_steps():
        _, stats, *_ = rig.step(st)
    assert int(stats[..., 3].sum()) > 0


@pytest.mark.parametrize("mode", MODES_ORDER)
def test_whole_step_captured_in_a_cuda_graph(mode):
    """Each decode step -- resolve + gather and the step's single offload launch -- captured into one
    CUDA graph and replayed (no host decision anywhere on the path): results identical to the oracle.
    Uses the agentic workload with compressed turns so steps with offloads and table edits occur."""
    w = workloads.config3(seed=4, decode_per_turn=6, L=2, R=8)
    rig = _rig(w, mode=mode, graph=True)
    for st in w.iter_steps(13):
        rig.step(st)
    w1 = workloads.config1(seed=6, steps=6)
    rig1 = _rig(w1, mode=mode, graph=True, oracle_bytes=True)
    for st in w1.iter_steps():
        rig1.step(st)


def test_max_batch_mtp3_full_size():
    """4 layers x 256 requests, contexts log-uniform to 1,048,576 tokens, per-page residency, P=4 query
    positions sharing one plan per step, contexts growing by the accepted MTP length, and one offload
    launch of the completed pages (all layers) after every step -- the full-size configuration,
    fused path, first 6 steps."""
    w = workloads.config5(seed=0, steps=6)
    rig = _rig(w, mode="fused")
    assert rig.ordered   # a host pool of tens of GB: misses are filed in address order by default
    offloaded = 0
    for st in w.iter_steps(6):
        _, stats, *_ = rig.step(st)
        offloaded += len(st.off_gpu)
    assert offloaded > 0


@pytest.mark.parametrize("mode", MODES_ORDER)
def test_mtp3_hot_sizing_and_verify_replays(mode):
    """The pages' MTP hot-buffer sizing, (num_spec + 2) * K = 10240 rows per request with P = 4 positions
    sharing one plan, 64 requests.  Every step is resolved a second time with the same ids (a verify
    iteration replaying the plan): identical rows, no miss, hot state unchanged."""
    w = workloads.config5(seed=3, steps=4, R=64, capacity=10240)
    rig = _rig(w, mode=mode)
    for st in w.iter_steps(4):
        rows, stats, *_ = rig.step(st)
        rows, stats = rows.clone(), stats.clone()
        tok, stamp = rig.hot.slot_token.clone(), rig.hot.slot_stamp.clone()
        rows2, stats2, *_ = rig.step(st)
        assert torch.equal(rows, rows2)
        assert int(stats2[..., 3].sum()) == 0
        assert torch.equal(stats[..., 1].add(stats[..., 3]).add(stats[..., 2]),
                           stats2[..., 1].add(stats2[..., 2]))
        assert torch.equal(tok, rig.hot.slot_token) and torch.equal(stamp, rig.hot.slot_stamp)


@pytest.mark.parametrize("mode", ["split", "split+order"])
def test_max_batch_mtp3_split_path_64_requests(mode):
    w = workloads.config5(seed=1, steps=4, R=64)
    rig = _rig(w, mode=mode)
    for st in w.iter_steps(4):
        rig.step(st)


def test_multi_turn_agentic_full_geometry():
    """16 layers x 32 requests at the first turn's 74,160-token context with a 40% resident budget:
    24 steps cover the first completed page (offloaded for all 16 layers in one launch) and the
    release of each request's oldest resident page whose block is reused for the new page."""
    w = workloads.config3(seed=0)
    rig = _rig(w, mode="fused")
    saw_edit = saw_off = False
    for st in w.iter_steps(24):
        rig.step(st)
        saw_edit |= len(st.bt_edits) > 0
        saw_off |= len(st.off_gpu) > 0
    assert saw_edit and saw_off


@pytest.mark.parametrize("mode", MODES_ORDER)
def test_multi_turn_agentic_turn_boundaries(mode):
    """Same geometry with 6 decode steps per turn, so two turn boundaries (753 prompt tokens: a dozen
    pages complete and start at once) fall inside 14 steps."""
    w = workloads.config3(seed=2, decode_per_turn=6, L=4)
    rig = _rig(w, mode=mode)
    for st in w.iter_steps(14):
        rig.step(st)


@pytest.mark.parametrize("mode", MODES_ORDER)
def test_data_errors_are_isolated_per_unit(mode):
    w = workloads.config1(seed=3, steps=3)
    rig = _rig(w, oracle_bytes=True, mode=mode)
    steps = list(w.iter_steps())
    rig.step(steps[0])
    st = steps[1]
    st.topk[0, 1, 0, 5] = 5000          # out of range for request 1
    st.topk[0, 2, 0, 7] = -7            # invalid id for request 2
    rows, stats, *_ = rig.step(st)
    s = stats.cpu().numpy()[0]
    assert s[1, 0] == 2 and s[2, 0] == 2 and s[0, 0] == 0 and s[3, 0] == 0
    st2 = steps[2]
    st2.index = 0   # older than the stamps of requests 0 and 3 (step 1); requests 1 and 2 failed at
    rows, stats, *_ = rig.step(st2)   # step 1, so their newest stamp is still 0 and step 0 replays
    assert stats.cpu().numpy()[0, :, 0].tolist() == [5, 0, 0, 5]


def test_empty_and_degenerate_shapes():
    dev = torch.device("cuda")
    case = Case(R=2, S=4, B=16, C=8, max_pages=4, ctx=[16, 16], resident=True, host=True,
                hot_blocks=[[0, 1], [2, 3]], num_gpu_blocks=6, num_host_blocks=8, bt=[[-1, -1, -1, 4], [-1, -1, -1, 5]],
                hbt=[[0, 1, 2, 3], [4, 5, 6, 7]])
    pool, gpu, host, hot = _case_to_gpu(case, dev)
    bt, hbt = torch.from_numpy(case.bt).to(dev), torch.from_numpy(case.hbt).to(dev)
    ctx = torch.from_numpy(case.ctx).to(dev)
    # K = 0: an empty plan; stats OK with zero counts
    rows, stats = hs.resolve_topk(pool, torch.zeros((1, 2, 1, 0), dtype=torch.int32, device=dev), bt, hbt, ctx, hot, 0)
    assert stats.cpu().tolist() == [[[0, 0, 0, 0], [0, 0, 0, 0]]]
    # all padding
    ids = torch.full((1, 2, 2, 3), -1, dtype=torch.int32, device=dev)
    rows, stats = hs.resolve_topk(pool, ids, bt, hbt, ctx, hot, 1)
    assert (rows == -1).all() and stats.cpu().tolist() == [[[0, 0, 0, 0], [0, 0, 0, 0]]]
    # zero requests / zero layers: no-op
    hs.resolve_topk(pool, torch.zeros((0, 2, 1, 4), dtype=torch.int32, device=dev), bt, hbt, ctx, hot, 1)
    out = hs.gather_rows(pool, torch.zeros((1, 0), dtype=torch.int32, device=dev))
    assert out.numel() == 0
    # every slot used in one step: capacity exactly C
    ids = torch.tensor([[[[0, 1, 2, 3, 4, 5, 6, 7]], [[8, 9, 10, 11, 0, 1, 2, 3]]]], dtype=torch.int32, device=dev)
    rows, stats = hs.resolve_topk(pool, ids, bt, hbt, ctx, hot, 2)
    o_rows, o_stats = case.step(ids.cpu().numpy()[0], 2)
    assert np.array_equal(stats.cpu().numpy(), o_stats) and np.array_equal(rows.cpu().numpy(), o_rows)
    assert o_stats[0, :, 3].tolist() == [8, 8]
    pool.close()


@pytest.mark.parametrize("mode", ["fused", "fused+part", "fused+ranges", "fused+ranges1", "fused+order"])
def test_degenerate_shapes_through_the_fused_layouts(mode):
    """The fused gathers on degenerate steps: an empty plan (K = 0), an all-padding step (rows -1, zero
    bytes), and a step that uses every hot slot (capacity exactly C): rows, stats and every gathered byte
    equal the oracle's, in every miss layout (per-unit lists, SM partition, mixed range layout, spread)."""
    dev = torch.device("cuda")
    case = Case(R=2, S=4, B=16, C=8, max_pages=4, ctx=[16, 16], resident=True, host=True,
                hot_blocks=[[0, 1], [2, 3]], num_gpu_blocks=6, num_host_blocks=8, bt=[[-1, -1, -1, 4], [-1, -1, -1, 5]],
                hbt=[[0, 1, 2, 3], [4, 5, 6, 7]])
    pool, gpu, host, hot = _case_to_gpu(case, dev)
    _set_order(pool, mode)
    bt, hbt = torch.from_numpy(case.bt).to(dev), torch.from_numpy(case.hbt).to(dev)
    ctx = torch.from_numpy(case.ctx).to(dev)
    rows, stats, out = hs.resolve_gather(pool, torch.zeros((1, 2, 1, 0), dtype=torch.int32, device=dev), bt, hbt,
                                         ctx, hot, 0)
    assert stats.cpu().tolist() == [[[0, 0, 0, 0], [0, 0, 0, 0]]] and out.numel() == 0
    ids = torch.full((1, 2, 2, 3), -1, dtype=torch.int32, device=dev)
    rows, stats, out = hs.resolve_gather(pool, ids, bt, hbt, ctx, hot, 1)
    assert (rows == -1).all() and stats.cpu().tolist() == [[[0, 0, 0, 0], [0, 0, 0, 0]]]
    assert int(out.count_nonzero()) == 0
    ids = torch.tensor([[[[0, 1, 2, 3, 4, 5, 6, 7]], [[8, 9, 10, 11, 0, 1, 2, 3]]]], dtype=torch.int32, device=dev)
    rows, stats, out = hs.resolve_gather(pool, ids, bt, hbt, ctx, hot, 2)
    o_rows, o_stats = case.step(ids.cpu().numpy()[0], 2)
    assert np.array_equal(stats.cpu().numpy(), o_stats) and np.array_equal(rows.cpu().numpy(), o_rows)
    assert o_stats[0, :, 3].tolist() == [8, 8]
    o_out, _ = case.gather(o_rows.reshape(1, -1))
    assert np.array_equal(out.cpu().numpy().reshape(o_out.shape), o_out)
    pool.close()


def test_largest_shapes_and_shape_limits():
    """P*K = 8192 ids with C = 4096 (the MTP3 shape) and with C = 10240 (the pages' MTP sizing
    (num_spec + 2) * K), C = 8192 and the largest capacity C = 16384: parity over three steps; a shape
    whose plan does not fit in one CTA's shared memory is rejected on the host."""
    dev = torch.device("cuda")
    rng = np.random.default_rng(5)
    for P, K, C in ((4, 2048, 4096), (4, 2048, 10240), (1, 1024, 8192), (1, 4096, 8192), (1, 1024, 16384)):
        S, B, R, pages = 64, 32, 3, 512
        ctx = pages * S
        nb = C // S
        ngb = R * nb + R * 16
        perm = rng.permutation(ngb).astype(np.int32)
        hot_blocks = perm[:R * nb].reshape(R, nb)
        bt = np.full((R, pages), -1, np.int32)
        bt[:, pages - 16:] = perm[R * nb:].reshape(R, 16)
        hbt = rng.permutation(R * pages).astype(np.int32).reshape(R, pages)
        case = Case(R=R, S=S, B=B, C=C, max_pages=pages, ctx=[ctx] * R, resident=True, host=True,
                    hot_blocks=hot_blocks, num_gpu_blocks=ngb, num_host_blocks=R * pages, bt=bt, hbt=hbt)
        pool, gpu, host, hot = _case_to_gpu(case, dev)
        bt_t, hbt_t, ctx_t = (torch.from_numpy(x).to(dev) for x in (case.bt, case.hbt, case.ctx))
        for t in range(3):
            base = [rng.choice(ctx, K, replace=False) for _ in range(R)]
            ids = np.stack([np.stack([np.where(rng.random(K) < 0.9, b, rng.integers(0, ctx, K)) for _ in range(P)])
                            for b in base]).astype(np.int32)
            rows, stats = hs.resolve_topk(pool, torch.from_numpy(ids[None]).to(dev), bt_t, hbt_t, ctx_t, hot, t)
            o_rows, o_stats = case.step(ids, t)
            torch.cuda.synchronize()
            assert np.array_equal(stats.cpu().numpy(), o_stats), (P, K, C, t)
            assert np.array_equal(rows.cpu().numpy(), o_rows), (P, K, C, t)
            assert np.array_equal(hot.slot_token.cpu().numpy(), case.tok)
            assert np.array_equal(hot.slot_stamp.cpu().numpy(), case.stamp)
            assert np.array_equal(gpu[0].cpu().numpy().reshape(-1), case.pools[0])
        pool.close()
    big = hs.resolve_smem_bytes(1, 8192, 16384, 64)
    assert big > 227 * 1024
    S, C = 64, 16384
    gpu = [torch.zeros((C // S + 1, S, 16), dtype=torch.uint8, device=dev)]
    pool = hs.Pool(gpu, [torch.zeros((4, S, 16), dtype=torch.uint8).pin_memory()])
    hot = hs.HotState.allocate(1, torch.arange(C // S, dtype=torch.int32, device=dev)[None], C)
    bt = torch.full((1, 4), -1, dtype=torch.int32, device=dev)
    with pytest.raises(hs.HSError) as e:
        hs.resolve_topk(pool, torch.zeros((1, 1, 1, 8192), dtype=torch.int32, device=dev), bt, bt,
                        torch.tensor([256], dtype=torch.int32, device=dev), hot, 0)
    assert e.value.code == 1
    pool.close()


@pytest.mark.parametrize("mode", MODES_ORDER)
def test_snapshot_restore_continues_identically(mode):
    """Checkpoint/resume: the hot state and pool bytes copied out mid-run and copied back give the same
    continuation (rows, stats, state, gathered bytes), with a fresh workspace full of garbage -- the
    library keeps nothing between calls and needs nothing from the workspace's previous contents."""
    w = workloads.config1(seed=5, steps=8)
    rig = _rig(w, mode=mode, oracle_bytes=True)
    steps = list(w.iter_steps())
    for st in steps[:4]:
        rig.step(st)
    snap = (rig.hot.slot_token.clone(), rig.hot.slot_stamp.clone(), [g.clone() for g in rig.gpu],
            rig.o_tok.copy(), rig.o_stamp.copy(), [p.copy() for p in rig.o_pools])
    first = []
    for st in steps[4:]:
        rows, stats, out, *_ = rig.step(st)
        first.append((rows.clone(), stats.clone(), out.clone()))
    rig.hot.slot_token.copy_(snap[0])
    rig.hot.slot_stamp.copy_(snap[1])
    for g, s_ in zip(rig.gpu, snap[2]):
        g.copy_(s_)
    rig.o_tok[...], rig.o_stamp[...] = snap[3], snap[4]
    for dst, src in zip(rig.o_pools, snap[5]):
        dst[...] = src
    rig.ws.fill_(0xA5)
    for st, (r0, s0, o0) in zip(steps[4:], first):
        rows, stats, out, *_ = rig.step(st)
        assert torch.equal(rows, r0) and torch.equal(stats, s0) and torch.equal(out, o0)


def test_miss_order_decision():
    """hs_resolve_miss_order: the default (AUTO) keeps per-unit lists for a small host pool; ON files
    misses in address order when the workspace has room for it (hs_resolve_workspace_bytes) and not
    with the minimal workspace; OFF never; an unknown mode is refused."""
    dev = torch.device("cuda")
    S, C, R, P, K = 4, 8, 3, 1, 8
    gpu = [torch.zeros((32, S, 16), dtype=torch.uint8, device=dev) for _ in range(2)]
    host = [torch.zeros((16, S, 16), dtype=torch.uint8).pin_memory() for _ in range(2)]
    pool = hs.Pool(gpu, host)
    hot = hs.HotState.allocate(2, torch.zeros((R, C // S), dtype=torch.int32, device=dev), C)
    full, small = hs.resolve_workspace_bytes(2, R, P, K, C), hs.resolve_workspace_bytes_min(2, R, P, K, C)
    assert full > small
    assert not hs.miss_order_used(pool, hot, 2, R, P, K, full)
    pool.set_miss_order(hs.MISS_ORDER_ON)
    assert hs.miss_order_used(pool, hot, 2, R, P, K, full)
    assert hs.miss_order_used(pool, hot, 1, R, P, K, full, layer_begin=1)
    assert not hs.miss_order_used(pool, hot, 2, R, P, K, small)
    for mode in (hs.MISS_ORDER_RANGES, hs.MISS_ORDER_SPREAD):
        pool.set_miss_order(mode)
        assert hs.miss_order_used(pool, hot, 2, R, P, K, full)
        assert not hs.miss_order_used(pool, hot, 2, R, P, K, small)
    pool.set_miss_order(hs.MISS_ORDER_OFF)
    assert not hs.miss_order_used(pool, hot, 2, R, P, K, full)
    with pytest.raises(hs.HSError):
        pool.set_miss_order(5)
    with pytest.raises(hs.HSError):
        pool.set_miss_warps(3)
    with pytest.raises(hs.HSError):
        pool.set_miss_warps(-2)
    pool.set_miss_warps(-1)
    for bad in (-2, 1, 33):
        with pytest.raises(hs.HSError):
            pool.set_miss_sm_divisor(bad)
    for ok in (0, 2, 32, -1):
        pool.set_miss_sm_divisor(ok)
    for bad in (-1, 2):
        with pytest.raises(hs.HSError):
            pool.set_miss_prefetch(bad)
    pool.set_miss_prefetch(hs.MISS_PREFETCH_ON)
    pool.set_miss_prefetch(hs.MISS_PREFETCH_OFF)
    no_host = hs.Pool(gpu)
    no_host.set_miss_order(hs.MISS_ORDER_ON)
    assert not hs.miss_order_used(no_host, hot, 2, R, P, K, full)
    pool.close()
    no_host.close()


def test_hot_reset_of_listed_requests_only():
    """hs_hot_reset_requests empties the slots of the listed requests in every index group and leaves
    the others (and entries outside [0, R)) alone."""
    dev = torch.device("cuda")
    S, C, R, L, G = 4, 8, 5, 4, 2
    gpu = [torch.zeros((64, S, 16), dtype=torch.uint8, device=dev) for _ in range(L)]
    pool = hs.Pool(gpu)
    hot = hs.HotState.allocate(L, torch.arange(R * (C // S), dtype=torch.int32, device=dev).reshape(R, -1), C,
                               layers_per_index=G)
    tok = torch.arange(L // G * R * C, dtype=torch.int32, device=dev).reshape(L // G, R, C)
    hot.slot_token.copy_(tok)
    hot.slot_stamp.copy_(tok + 7)
    hs.hot_reset_requests(pool, hot, torch.tensor([3, 0, 9, -1], dtype=torch.int32, device=dev))
    torch.cuda.synchronize()
    exp_t, exp_s = tok.clone(), tok + 7
    exp_t[:, [0, 3]] = -1
    exp_s[:, [0, 3]] = -1
    assert torch.equal(hot.slot_token, exp_t) and torch.equal(hot.slot_stamp, exp_s)
    pool.close()


def test_gather_standalone_multilayer_and_status():
    dev = torch.device("cuda")
    L, S, B, ngb = 3, 8, 656, 40
    gpu = [torch.randint(0, 256, (ngb, S, B), dtype=torch.uint8, device=dev) for _ in range(L)]
    pool = hs.Pool(gpu, None)
    rng = np.random.default_rng(1)
    n = 5003  # ragged tail
    rows = rng.integers(-1, ngb * S, size=(L, n)).astype(np.int32)
    out = hs.gather_rows(pool, torch.from_numpy(rows).to(dev))
    pools_np = [g.cpu().numpy().reshape(-1) for g in gpu]
    o_out, st = oracle.gather(B=B, num_rows=ngb * S, pools=pools_np, rows=rows)
    assert st == 0 and np.array_equal(out.cpu().numpy(), o_out)
    bad = rows.copy()
    bad[1, 17] = ngb * S
    bad[2, 4000] = -9
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    out = hs.gather_rows(pool, torch.from_numpy(bad).to(dev), status=status)
    o_out, st = oracle.gather(B=B, num_rows=ngb * S, pools=pools_np, rows=bad)
    assert int(status.item()) == st == 2 and np.array_equal(out.cpu().numpy(), o_out)
    # a layer window
    out = hs.gather_rows(pool, torch.from_numpy(rows[:2]).to(dev), layer_begin=1)
    o_out, _ = oracle.gather(B=B, num_rows=ngb * S, pools=pools_np, rows=rows[:2], layer_begin=1)
    assert np.array_equal(out.cpu().numpy(), o_out)
    pool.close()


@pytest.mark.parametrize("planes", [(512, 16, 128), (656,), (16, 640), (128, 128, 128, 272)])
def test_gather_planes_standalone(planes):
    """hs_gather_rows with the plane layout: each plane holds, for every position, its column range of
    the oracle's gathered rows (ragged tail, -1 rows, several layers); the bulk copy mode falls back to
    loads with planes set."""
    dev = torch.device("cuda")
    L, S, B, ngb = 3, 8, 656, 40
    gpu = [torch.randint(0, 256, (ngb, S, B), dtype=torch.uint8, device=dev) for _ in range(L)]
    pool = hs.Pool(gpu, None)
    pool.set_gather_planes(planes)
    rng = np.random.default_rng(2)
    n = 4099
    rows = rng.integers(-1, ngb * S, size=(L, n)).astype(np.int32)
    pools_np = [g.cpu().numpy().reshape(-1) for g in gpu]
    o_out, st = oracle.gather(B=B, num_rows=ngb * S, pools=pools_np, rows=rows)
    assert st == 0
    # the layout written out: per layer, plane p = every position's bytes [c_p, c_p + planes[p]) in turn
    cuts = np.cumsum((0,) + tuple(planes))
    expect = np.stack([np.concatenate([o_out[l][:, cuts[p]:cuts[p + 1]].reshape(-1) for p in range(len(planes))])
                       for l in range(L)])
    for copy in (hs.GATHER_COPY_LOADS, hs.GATHER_COPY_BULK):
        pool.set_gather_copy(copy)
        out = hs.gather_rows(pool, torch.from_numpy(rows).to(dev))
        assert np.array_equal(out.cpu().numpy().reshape(L, -1), expect), f"planes {planes} copy mode {copy}"
        back = torch.cat(hs.plane_views(out, planes), dim=-1)
        assert np.array_equal(back.cpu().numpy(), o_out)
    # back to rows
    pool.set_gather_planes(())
    out = hs.gather_rows(pool, torch.from_numpy(rows).to(dev))
    assert np.array_equal(out.cpu().numpy(), o_out)
    for bad in ((512, 16), (512, 16, 120, 8), (0, 656), (16,) * 5):
        with pytest.raises(hs.HSError):
            pool.set_gather_planes(bad)
    pool.close()


@pytest.mark.parametrize("mode", ["split", "fused", "fused+order", "fused+ranges", "fused+ranges1", "fused+part"])
def test_planes_through_the_resolver(mode):
    """The fused gathers (per-unit lists, spread schedule, SM partition, mixed range layout) and the
    split path write the plane layout {512, 16, 128}: converted back to rows, every gathered byte, pool
    byte and slot equals the oracle's (tiny decode) and the closed form (small MTP3 batch with IndexShare)."""
    w = workloads.config1(seed=8, steps=6)
    rig = _rig(w, oracle_bytes=True, mode=mode, planes=(512, 16, 128))
    for st in w.iter_steps():
        rig.step(st)
    w = workloads.config5(seed=9, R=6, L=4, layers_per_index=2, steps=4)
    rig = _rig(w, mode=mode, planes=(512, 16, 128))
    for st in w.iter_steps():
        rig.step(st)


@pytest.mark.parametrize("mode", ["split+order", "fused+order", "split+ranges", "fused+ranges", "fused+ranges1",
                                  "fused+ranges2"])
@pytest.mark.parametrize("P", [1, 4])
def test_ordered_misses_overflowing_their_bucket(mode, P):
    """Every page's host copy lies in the first two host blocks (one host-row range), so with the
    address-ordered layout forced on almost all misses overflow their bucket into the overflow list:
    rows, stats, slot state, pool bytes and gathered bytes must still equal the oracle's, with repeats
    of missed ids across positions (P = 4)."""
    rng = np.random.default_rng(40 + P)
    dev = torch.device("cuda")
    R, S, B, pages, C = 8, 64, 656, 64, 1024
    K = 256 if P == 1 else 128
    nb = C // S
    perm = rng.permutation(R + R * nb).astype(np.int32)
    bt = np.full((R, pages), -1, np.int32)
    bt[:, pages - 1] = perm[:R]
    hot = perm[R:].reshape(R, nb)
    hbt = (np.arange(pages, dtype=np.int32)[None, :] % 2).repeat(R, 0)
    case = Case(R=R, S=S, B=B, C=C, max_pages=pages, ctx=[pages * S] * R, resident=True, host=True, hot_blocks=hot,
                num_gpu_blocks=R + R * nb, num_host_blocks=512, bt=bt, hbt=hbt, seed=9)
    pool, gpu, host, hot_t = _case_to_gpu(case, dev)
    _set_order(pool, mode)
    bt_d, hbt_d, ctx = torch.from_numpy(case.bt).to(dev), torch.from_numpy(case.hbt).to(dev), torch.from_numpy(case.ctx).to(dev)
    prev = None
    for t in range(3):
        ids = np.empty((R, P, K), np.int32)
        for r in range(R):
            base = rng.choice(pages * S, size=K, replace=False) if prev is None else np.concatenate(
                [rng.choice(prev[r, 0], size=K // 2, replace=False),
                 rng.choice(np.setdiff1d(np.arange(pages * S), prev[r, 0]), size=K - K // 2, replace=False)])
            ids[r, 0] = rng.permutation(base)
            for q in range(1, P):
                ids[r, q] = rng.permutation(np.concatenate([ids[r, 0][:int(0.9 * K)],
                                                            rng.choice(pages * S, size=K - int(0.9 * K))]))
        prev = ids
        topk = torch.from_numpy(ids[None]).to(dev)
        if _base(mode) == "fused":
            rows, stats, g = hs.resolve_gather(pool, topk, bt_d, hbt_d, ctx, hot_t, t)
        else:
            rows, stats = hs.resolve_topk(pool, topk, bt_d, hbt_d, ctx, hot_t, t)
            g = hs.gather_rows(pool, rows.reshape(1, -1))
        o_rows, o_stats = case.step(ids, t)
        torch.cuda.synchronize()
        assert (o_stats[..., 0] == 0).all() and int(o_stats[..., 3].sum()) > 500
        assert np.array_equal(stats.cpu().numpy(), o_stats), t
        assert np.array_equal(rows.cpu().numpy(), o_rows), t
        assert np.array_equal(hot_t.slot_token.cpu().numpy(), case.tok), t
        assert np.array_equal(hot_t.slot_stamp.cpu().numpy(), case.stamp), t
        assert np.array_equal(gpu[0].cpu().numpy().reshape(-1), case.pools[0]), t
        o_out, _ = case.gather(o_rows.reshape(1, -1))
        assert np.array_equal(g.cpu().numpy(), o_out), t
    pool.close()


@pytest.mark.parametrize("B", [656, 32])
def test_gather_bulk_copies_equal_the_oracle(B):
    """hs_pool_set_gather_copy(BULK): whole rows through shared-memory stages with bulk copies.  The
    same bytes as the oracle's gather for ragged sizes (fewer rows than warps, rows not a multiple of
    the stages), padding rows, rows outside the pool (zero-filled, ID_RANGE status), several layers
    and a layer window; repeated calls reuse the stages."""
    dev = torch.device("cuda")
    L, S, ngb = 3, 8, 40
    gpu = [torch.randint(0, 256, (ngb, S, B), dtype=torch.uint8, device=dev) for _ in range(L)]
    pool = hs.Pool(gpu, None)
    pool.set_gather_copy(hs.GATHER_COPY_BULK)
    pools_np = [g.cpu().numpy().reshape(-1) for g in gpu]
    rng = np.random.default_rng(B)
    for n in (1, 5, 127, 128, 129, 5003, 300001):
        rows = rng.integers(-1, ngb * S, size=(L, n)).astype(np.int32)
        status = torch.zeros(1, dtype=torch.int32, device=dev)
        for _ in range(2):
            out = hs.gather_rows(pool, torch.from_numpy(rows).to(dev), status=status)
            o_out, st = oracle.gather(B=B, num_rows=ngb * S, pools=pools_np, rows=rows)
            assert st == 0 and int(status.item()) == 0 and np.array_equal(out.cpu().numpy(), o_out), n
    bad = rng.integers(-1, ngb * S, size=(L, 5003)).astype(np.int32)
    bad[1, 17] = ngb * S
    bad[2, 4000] = -9
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    out = hs.gather_rows(pool, torch.from_numpy(bad).to(dev), status=status)
    o_out, st = oracle.gather(B=B, num_rows=ngb * S, pools=pools_np, rows=bad)
    assert int(status.item()) == st == 2 and np.array_equal(out.cpu().numpy(), o_out)
    out = hs.gather_rows(pool, torch.from_numpy(bad[:2]).to(dev), layer_begin=1)
    o_out, _ = oracle.gather(B=B, num_rows=ngb * S, pools=pools_np, rows=bad[:2], layer_begin=1)
    assert np.array_equal(out.cpu().numpy(), o_out)
    with pytest.raises(hs.HSError):
        pool.set_gather_copy(7)
    pool.close()


def test_offload_standalone_all_layers_one_launch():
    dev = torch.device("cuda")
    L, S, B, ngb, nhb = 4, 64, 656, 30, 50
    gpu = [torch.randint(0, 256, (ngb, S, B), dtype=torch.uint8, device=dev) for _ in range(L)]
    host = [torch.zeros((nhb, S, B), dtype=torch.uint8).pin_memory() for _ in range(L)]
    pool = hs.Pool(gpu, host)
    gb = np.array([3, 17, 0, 29, 8], np.int32)
    hb = np.array([49, 0, 7, 21, 22], np.int32)
    n0 = hs.launch_count()
    hs.offload_pages(pool, torch.from_numpy(gb).to(dev), torch.from_numpy(hb).to(dev))
    assert hs.launch_count() - n0 == 1
    torch.cuda.synchronize()
    pools_np = [g.cpu().numpy().reshape(-1) for g in gpu]
    hosts_np = [np.zeros(nhb * S * B, np.uint8) for _ in range(L)]
    oracle.offload(S=S, B=B, num_gpu_blocks=ngb, num_host_blocks=nhb, pools=pools_np, hosts=hosts_np, gpu_blocks=gb,
                   host_blocks=hb)
    for l in range(L):
        assert np.array_equal(host[l].numpy().reshape(-1), hosts_np[l])
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    hs.offload_pages(pool, torch.tensor([ngb], dtype=torch.int32, device=dev),
                     torch.tensor([0], dtype=torch.int32, device=dev), status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 8
    for l in range(L):
        assert np.array_equal(host[l].numpy().reshape(-1), hosts_np[l])
    pool.close()


def test_host_argument_errors():
    dev = torch.device("cuda")
    gpu = [torch.zeros((4, 4, 16), dtype=torch.uint8, device=dev)]
    with pytest.raises(TypeError):
        hs.Pool(gpu, [torch.zeros((4, 4, 16), dtype=torch.uint8)])      # host memory not pinned
    pool = hs.Pool(gpu, [torch.zeros((4, 4, 16), dtype=torch.uint8).pin_memory()])
    hot = hs.HotState.allocate(1, torch.tensor([[0, 1]], dtype=torch.int32, device=dev), 8)
    bt = torch.full((1, 4), -1, dtype=torch.int32, device=dev)
    ctx = torch.tensor([16], dtype=torch.int32, device=dev)
    ids = torch.zeros((1, 1, 1, 2), dtype=torch.int32, device=dev)
    with pytest.raises(hs.HSError) as e:
        hs.resolve_topk(pool, ids, bt, bt, ctx, hot, -1)             # negative step
    assert e.value.code == 1
    with pytest.raises(hs.HSError):
        hs.resolve_topk(pool, ids, bt, bt, ctx, hot, 0, layer_begin=1)  # layer window outside the pool
    small_ws = torch.empty(16, dtype=torch.uint8, device=dev)
    with pytest.raises(hs.HSError):
        hs.resolve_topk(pool, ids, bt, bt, ctx, hot, 0, workspace=small_ws)
    bad_cap = hs.HotState.allocate(1, torch.tensor([[0, 1]], dtype=torch.int32, device=dev), 6)  # not a page multiple
    with pytest.raises(hs.HSError):
        hs.resolve_topk(pool, ids, bt, bt, ctx, bad_cap, 0)
    pool.close()
