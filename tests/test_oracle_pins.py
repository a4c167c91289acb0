"""Pins for the oracle: checks against facts that do not come from the oracle itself.

  - the worked example of the figure (three residency states), expected values derived by hand;
  - Mattson's stack-distance theorem for LRU (K=1, one access per step): an access hits iff its
    stack distance is <= capacity;
  - closed forms: full residency; unbounded capacity (misses = first-ever touches); an empty buffer
    hands slots out in order; the closed-form row contents for gathered and offloaded bytes;
  - hand-computed duplicate/padding/MTP-plan cases, every data-error code, the error precedence,
    replay idempotence, and invariants on the tiny-decode workload.
"""
import os

import numpy as np
import pytest

import oracle
from synth import content, workloads
from tests.casekit import Case, host_only_case

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "figure_three_residency_states.txt")


def _parse_golden():
    geo, hot, panels, cur = {}, None, [], None
    for line in open(GOLDEN):
        line = line.split("#")[0].strip()
        if not line:
            continue
        t = line.split()
        if t[0] == "geometry":
            geo = {k: int(v) for k, v in (x.split("=") for x in t[1:])}
        elif t[0] == "hot_blocks":
            hot = [int(x) for x in t[1:]]
        elif t[0] == "panel":
            cur = {"name": t[1], "steps": []}
            panels.append(cur)
        elif t[0] in ("block_table", "host_table"):
            cur[t[0]] = [int(x) for x in t[1:]]
        elif t[0] == "step":
            i = t.index("ids"), t.index("rows"), t.index("stats"), t.index("copies")
            cur["steps"].append(dict(
                t=int(t[1]), ids=[int(x) for x in t[i[0] + 1:i[1]]], rows=[int(x) for x in t[i[1] + 1:i[2]]],
                stats=[int(x) for x in t[i[2] + 1:i[3]]],
                copies=[tuple(int(y) for y in x.split(":")) for x in t[i[3] + 1:]]))
    return geo, hot, panels


@pytest.mark.parametrize("panel", ["full", "mixed", "none"])
def test_figure_three_residency_states(panel):
    geo, hot, panels = _parse_golden()
    p = [x for x in panels if x["name"] == panel][0]
    S, C = geo["page_size"], geo["capacity"]
    pages = len(p["block_table"])
    B = 32
    case = Case(R=1, S=S, B=B, C=C, max_pages=pages, ctx=[geo["ctx"]], resident=True, host=True,
                hot_blocks=[hot], num_gpu_blocks=geo["gpu_blocks"], num_host_blocks=geo["host_blocks"],
                bt=[p["block_table"]], hbt=[p["host_table"]])
    for st in p["steps"]:
        before = case.pools[0].copy()
        rows, stats = case.step(np.array(st["ids"], np.int32).reshape(1, 1, -1), st["t"])
        assert rows.reshape(-1).tolist() == st["rows"]
        assert stats.reshape(-1).tolist() == st["stats"]
        # exactly the listed rows were copied, from the listed host rows
        changed = {i // B for i in np.nonzero(before != case.pools[0])[0]}
        assert changed <= {dst for _, dst in st["copies"]}
        for src, dst in st["copies"]:
            assert (case.pools[0][dst * B:(dst + 1) * B] == case.hosts[0][src * B:(src + 1) * B]).all()
        assert stats[0, 0, 3] == len(st["copies"])


def _mattson_hits(seq, C):
    """Hit/miss of each access under LRU of capacity C via stack distances (Mattson et al., 1970)."""
    stack, out = [], []
    for x in seq:
        d = stack.index(x) + 1 if x in stack else None
        out.append(d is not None and d <= C)
        if d is not None:
            stack.pop(d - 1)
        stack.insert(0, x)
    return out


@pytest.mark.parametrize("C,S,seed", [(4, 1, 0), (8, 2, 1), (8, 4, 2), (16, 4, 3), (12, 4, 4)])
def test_lru_k1_matches_stack_distance(C, S, seed):
    rng = np.random.default_rng(seed)
    pages = 12
    case = host_only_case(S=S, C=C, pages=pages, B=16, seed=seed)
    ctx = pages * S
    # skewed reuse so that both hits and misses occur at every stack depth
    seq = [int(min(ctx - 1, rng.geometric(0.08))) if rng.random() < 0.5 else int(rng.integers(0, ctx))
           for _ in range(300)]
    expect = _mattson_hits(seq, C)
    for t, x in enumerate(seq):
        rows, stats = case.step(np.array([[[x]]], np.int32), t, bytes_=False)
        hit = stats[0, 0, 2] == 1
        assert stats[0, 0, 0] == 0
        assert hit == expect[t], f"access {t} of token {x}"
        assert stats[0, 0, 2] + stats[0, 0, 3] == 1


def test_full_residency_closed_form():
    """All pages resident: row = block*S + offset, no hits, no misses, hot state untouched."""
    w = workloads.config1(seed=5, steps=3)
    bt = np.arange(w.R * w.max_pages, dtype=np.int32).reshape(w.R, w.max_pages)
    ngb = w.R * w.max_pages + w.R * (w.C // w.S)
    hot = (w.R * w.max_pages + np.arange(w.R * (w.C // w.S), dtype=np.int32)).reshape(w.R, -1)
    case = Case(R=w.R, S=w.S, B=16, C=w.C, max_pages=w.max_pages, ctx=w.ctx_len, resident=False, host=False,
                hot_blocks=hot, num_gpu_blocks=ngb, num_host_blocks=0, bt=bt, hbt=np.full_like(bt, -1))
    for st in w.iter_steps():
        tok0, stamp0 = case.tok.copy(), case.stamp.copy()
        rows, stats = case.step(st.topk, st.index, bytes_=False)
        ids = st.topk[0, :, 0, :]
        expect = bt[np.arange(w.R)[:, None], ids // w.S] * w.S + ids % w.S
        assert (rows[0, :, 0, :] == expect).all()
        assert (stats[0, :, 0] == 0).all() and (stats[0, :, 2:] == 0).all()
        assert (stats[0, :, 1] == w.K).all()
        assert (case.tok == tok0).all() and (case.stamp == stamp0).all()


def test_unbounded_capacity_misses_are_first_touches():
    rng = np.random.default_rng(11)
    pages, S = 16, 4
    case = host_only_case(S=S, C=pages * S, pages=pages, B=16)
    # make pages 12..15 resident tail
    seen = set()
    for t in range(40):
        ids = rng.choice(pages * S, size=6, replace=False).astype(np.int32)
        rows, stats = case.step(ids.reshape(1, 1, -1), t, bytes_=False)
        expect_miss = sum(1 for x in ids if x not in seen)
        seen.update(int(x) for x in ids)
        assert stats[0, 0, 3] == expect_miss
        assert stats[0, 0, 2] == len(ids) - expect_miss


def test_empty_buffer_hands_out_slots_in_order():
    case = host_only_case(R=2, S=4, C=16, pages=16, B=16)
    ids = np.array([[[40, 3, 17, 62, 5, 33]], [[1, 2, 3, 60, 61, 59]]], np.int32)
    rows, stats = case.step(ids, 0)
    for r in range(2):
        assert rows[0, r, 0].tolist() == [case.hot_row(r, j) for j in range(6)]
        assert case.tok[0, r, :6].tolist() == ids[r, 0].tolist()
        assert (case.tok[0, r, 6:] == -1).all()
        assert case.stamp[0, r, :6].tolist() == [0] * 6


def test_victims_in_stamp_then_slot_order_after_hits_refresh():
    """Hand-worked: C=4, S=2.  Step 0 fills slots 0..3 with 10,11,12,13 (stamp 0).  Step 1 touches
    11 and 13 (hits -> stamp 1) and misses 20: eligible slots are 0 and 2 (stamp 0), the smallest
    (stamp, slot) is slot 0.  Step 2 misses 21, 22, 23 while hitting 20: eligible are slots 1, 2, 3
    with stamps 1, 0, 1 -> order slot 2, slot 1, slot 3."""
    case = host_only_case(S=2, C=4, pages=16, B=16)
    case.step(np.array([[[10, 11, 12, 13]]], np.int32), 0)
    rows, stats = case.step(np.array([[[11, 20, 13]]], np.int32), 1)
    assert stats[0, 0].tolist() == [0, 0, 2, 1]
    assert rows[0, 0, 0].tolist() == [case.hot_row(0, 1), case.hot_row(0, 0), case.hot_row(0, 3)]
    rows, stats = case.step(np.array([[[21, 20, 22, 23]]], np.int32), 2)
    assert stats[0, 0].tolist() == [0, 0, 1, 3]
    assert rows[0, 0, 0].tolist() == [case.hot_row(0, 2), case.hot_row(0, 0), case.hot_row(0, 1), case.hot_row(0, 3)]
    assert case.tok[0, 0].tolist() == [20, 22, 21, 23]
    assert case.stamp[0, 0].tolist() == [2, 2, 2, 2]


def test_plan_dedup_padding_and_positions():
    """P=2 positions sharing one plan: first occurrence is position-major; duplicates and repeats
    across positions share one row; -1 is padding.  Hand-worked on an empty buffer."""
    case = host_only_case(S=4, C=8, pages=16, B=16)
    ids = np.array([[[9, -1, 4, 9], [7, 4, 30, -1]]], np.int32)  # [R=1][P=2][K=4]
    rows, stats = case.step(ids, 0)
    h = [case.hot_row(0, v) for v in range(8)]
    # plan: 9, 4, 7, 30 -> slots 0, 1, 2, 3
    assert rows[0, 0].tolist() == [[h[0], -1, h[1], h[0]], [h[2], h[1], h[3], -1]]
    assert stats[0, 0].tolist() == [0, 0, 0, 4]
    # replay of the step (same ids, same step): identical rows, all hits, state unchanged
    tok, stamp = case.tok.copy(), case.stamp.copy()
    rows2, stats2 = case.step(ids, 0)
    assert (rows2 == rows).all() and stats2[0, 0].tolist() == [0, 0, 4, 0]
    assert (case.tok == tok).all() and (case.stamp == stamp).all()


def test_resident_wins_over_stale_hot_copy():
    """A token whose page became resident is read in place even though a hot slot still holds it;
    that slot is not refreshed (it ages out)."""
    case = host_only_case(S=4, C=8, pages=4, B=16)      # hot blocks 0, 1
    case.step(np.array([[[5]]], np.int32), 0)          # token 5 -> slot 0
    case.ngb = 3                                        # page 1 becomes resident in a new block 2
    case.pools = [np.zeros(3 * 4 * 16, np.uint8)]
    case.bt[0, 1] = 2
    rows, stats = case.step(np.array([[[5]]], np.int32), 1)
    assert rows.reshape(-1).tolist() == [2 * 4 + 1]
    assert stats[0, 0].tolist() == [0, 1, 0, 0]
    assert case.stamp[0, 0, 0] == 0


def test_no_eviction_of_rows_used_in_the_same_step():
    """capacity == distinct non-resident ids of the step suffices; one less is HS_ERR_CAPACITY."""
    case = host_only_case(S=2, C=4, pages=8, B=16)
    case.step(np.array([[[0, 1, 2, 3]]], np.int32), 0)
    rows, stats = case.step(np.array([[[0, 1, 4, 5]]], np.int32), 1)   # 2 hits + 2 misses into slots 2,3
    assert stats[0, 0].tolist() == [0, 0, 2, 2]
    tok, stamp = case.tok.copy(), case.stamp.copy()
    rows, stats = case.step(np.array([[[0, 1, 4, 5, 6]]], np.int32), 2)  # 4 hits + 1 miss, 0 evictable
    assert stats[0, 0].tolist() == [4, 0, 0, 0]
    assert (rows == -1).all() and (case.tok == tok).all() and (case.stamp == stamp).all()


def test_rows_filled_earlier_in_the_same_step_are_not_evicted():
    """Two calls at the same step (a plan extended within one step): the second call may not evict
    the row the first call filled, so with C=4 and 3 evictable slots, 4 new misses overflow."""
    case = host_only_case(S=2, C=4, pages=16, B=16)
    case.step(np.array([[[10, 11, 12, 13]]], np.int32), 0)
    rows, stats = case.step(np.array([[[20]]], np.int32), 1)          # evicts slot 0
    assert stats[0, 0].tolist() == [0, 0, 0, 1] and rows.reshape(-1).tolist() == [case.hot_row(0, 0)]
    tok, stamp = case.tok.copy(), case.stamp.copy()
    rows, stats = case.step(np.array([[[21, 22, 23, 24]]], np.int32), 1)
    assert stats[0, 0].tolist() == [4, 0, 0, 0]
    assert (case.tok == tok).all() and (case.stamp == stamp).all()
    rows, stats = case.step(np.array([[[21, 22, 20]]], np.int32), 1)   # 2 misses fit; 20 is a hit
    assert stats[0, 0].tolist() == [0, 0, 1, 2]
    assert rows.reshape(-1).tolist() == [case.hot_row(0, 1), case.hot_row(0, 2), case.hot_row(0, 0)]


def test_error_codes_and_precedence_leave_state_untouched():
    def fresh():
        c = host_only_case(R=2, S=4, C=8, pages=8, B=16)
        c.step(np.array([[[1, 2]], [[1, 2]]], np.int32), 3)
        return c

    cases = {
        "id_range_high": ([[[1, 32]], [[1, 2]]], 4, 2),
        "id_range_neg": ([[[-2, 1]], [[1, 2]]], 4, 2),
        "step_order": ([[[1, 5]], [[1, 2]]], 2, 5),
    }
    for name, (ids, t, code) in cases.items():
        c = fresh()
        tok, stamp, pool = c.tok.copy(), c.stamp.copy(), c.pools[0].copy()
        rows, stats = c.step(np.array(ids, np.int32), t)
        assert stats[0, 0, 0] == code, name
        assert (rows[0, 0] == -1).all() and stats[0, 0, 1:].tolist() == [0, 0, 0]
        assert stats[0, 1, 0] == (5 if code == 5 else 0)   # the other request is independent
        assert (c.tok[0, 0] == tok[0, 0]).all() and (c.stamp[0, 0] == stamp[0, 0]).all()
    # missing host copy
    c = fresh()
    c.hbt[0, 3] = -1
    tok, stamp, pool = c.tok.copy(), c.stamp.copy(), c.pools[0].copy()
    rows, stats = c.step(np.array([[[13, 1]], [[13, 2]]], np.int32), 4)
    assert stats[0, 0, 0] == 3 and stats[0, 1, 0] == 0
    assert (c.tok[0, 0] == tok[0, 0]).all() and (c.pools[0].reshape(-1, 16)[:2] == pool.reshape(-1, 16)[:2]).all()
    # table range: a host block past the host pool, a resident block past the GPU pool, a bad hot block
    for what in ("host", "gpu", "hot"):
        c = fresh()
        if what == "host":
            c.hbt[0, 3] = c.nhb
        elif what == "gpu":
            c.bt[0, 3] = c.ngb
        else:
            c.hot_blocks[0, 1] = -4
        rows, stats = c.step(np.array([[[13, 1]], [[13, 2]]], np.int32), 4)
        assert stats[0, 0, 0] == 8, what
    # precedence: STEP_ORDER > ID_RANGE > TABLE_RANGE > MISSING_ROW > CAPACITY
    c = fresh()
    c.hbt[0, 3] = -1
    c.hot_blocks[0, 1] = c.ngb
    rows, stats = c.step(np.array([[[13, 99]], [[1, 2]]], np.int32), 1)
    assert stats[0, 0, 0] == 5
    rows, stats = c.step(np.array([[[13, 99]], [[1, 2]]], np.int32), 4)
    assert stats[0, 0, 0] == 2
    rows, stats = c.step(np.array([[[13, 9]], [[1, 2]]], np.int32), 4)
    assert stats[0, 0, 0] == 8
    c.hot_blocks[0, 1] = 1
    rows, stats = c.step(np.array([[[13, 9]], [[1, 2]]], np.int32), 4)
    assert stats[0, 0, 0] == 3
    c.hbt[0, 3] = 3                                  # 9 misses, 8 evictable slots
    rows, stats = c.step(np.array([[[13, 9, 20, 21, 22, 23, 24, 25, 26]],
                                   [[1, 2, -1, -1, -1, -1, -1, -1, -1]]], np.int32), 4)
    assert stats[0, 0, 0] == 4


def test_fully_resident_unit_needs_no_hot_buffer():
    """Full residency (Japanese article, "仕組み": all sparse-MLA KV on the GPU) reads every id in place,
    so a request that holds no hot blocks (entries -1) resolves normally; as soon as one of its ids is a
    hit or a miss, the unusable hot blocks give HS_ERR_TABLE_RANGE and nothing changes."""
    S, C, pages, B = 4, 8, 6, 16
    bt = np.array([[0, 1, 2, -1, -1, 3]], np.int32)
    hbt = np.array([[-1, -1, -1, 0, 1, -1]], np.int32)
    c = Case(R=1, S=S, B=B, C=C, max_pages=pages, ctx=[pages * S], resident=True, host=True,
             hot_blocks=[[-1, -1]], num_gpu_blocks=4, num_host_blocks=2, bt=bt, hbt=hbt)
    rows, stats = c.step(np.array([[[0, 5, 9, 21, 5]]], np.int32), 0)
    assert stats[0, 0].tolist() == [0, 4, 0, 0]
    assert rows.reshape(-1).tolist() == [0, 5, 9, 3 * S + 1, 5]
    pool = c.pools[0].copy()
    rows, stats = c.step(np.array([[[0, 13]]], np.int32), 1)          # 13 sits on a host-only page
    assert stats[0, 0].tolist() == [8, 0, 0, 0] and (rows == -1).all()
    assert (c.tok == -1).all() and (c.stamp == -1).all() and (c.pools[0] == pool).all()


def test_tiny_decode_bytes_and_invariants():
    """Tiny-decode workload, 8 steps, with byte pools: every gathered row equals the closed-form row
    of its logical token; resident bytes never change; only victim rows change, one per miss; no
    token sits in two slots; at most C valid slots."""
    w = workloads.config1(seed=0, steps=8)
    owner = w.gpu_block_owner()
    case = Case(R=w.R, S=w.S, B=w.B, C=w.C, max_pages=w.max_pages, ctx=w.ctx_len, resident=True, host=True,
                hot_blocks=w.hot_blocks, num_gpu_blocks=w.num_gpu_blocks, num_host_blocks=w.num_host_blocks,
                bt=w.block_table, hbt=w.host_block_table, seed=w.content_seed, content_page=w.content_page)
    resident_blocks = np.nonzero(owner[:, 0] >= 0)[0]
    res_bytes = case.pools[0].reshape(w.num_gpu_blocks, -1)[resident_blocks].copy()
    for st in w.iter_steps():
        before = case.pools[0].reshape(-1, w.B).copy()
        rows, stats = case.step(st.topk, st.index)
        assert (stats[0, :, 0] == 0).all()
        out, gst = case.gather(rows.reshape(1, -1))
        assert gst == 0
        ids = st.topk[0, :, 0, :]
        r_idx = np.repeat(np.arange(w.R), w.K)
        expect = content.rows_np(w.content_seed, 0, w.content_page[r_idx, ids.reshape(-1) // w.S],
                                 ids.reshape(-1) % w.S, w.B)
        assert (out[0] == expect).all()
        after = case.pools[0].reshape(-1, w.B)
        changed = np.nonzero((before != after).any(1))[0]
        assert len(changed) <= stats[0, :, 3].sum()
        assert (case.pools[0].reshape(w.num_gpu_blocks, -1)[resident_blocks] == res_bytes).all()
        for r in range(w.R):
            valid = case.tok[0, r][case.tok[0, r] >= 0]
            assert len(valid) == len(set(valid.tolist())) <= w.C
            assert stats[0, r, 1] + stats[0, r, 2] + stats[0, r, 3] == len(set(ids[r].tolist()))


def test_offload_copies_pages_for_all_layers():
    L, S, B = 3, 4, 32
    ngb, nhb = 5, 6
    rng = np.random.default_rng(0)
    pools = [rng.integers(0, 256, ngb * S * B, dtype=np.uint8) for _ in range(L)]
    hosts = [np.zeros(nhb * S * B, np.uint8) for _ in range(L)]
    gb = np.array([4, 0, 2], np.int32)
    hb = np.array([1, 5, 0], np.int32)
    st = oracle.offload(S=S, B=B, num_gpu_blocks=ngb, num_host_blocks=nhb, pools=pools, hosts=hosts,
                        gpu_blocks=gb, host_blocks=hb)
    assert st == 0
    P = S * B
    for l in range(L):
        for g, h in zip(gb, hb):
            assert (hosts[l][h * P:(h + 1) * P] == pools[l][g * P:(g + 1) * P]).all()
        untouched = [h for h in range(nhb) if h not in hb]
        for h in untouched:
            assert (hosts[l][h * P:(h + 1) * P] == 0).all()
    st = oracle.offload(S=S, B=B, num_gpu_blocks=ngb, num_host_blocks=nhb, pools=pools, hosts=hosts,
                        gpu_blocks=np.array([5], np.int32), host_blocks=np.array([0], np.int32))
    assert st == 8


def test_gather_zero_rows_and_range():
    S, B, ngb = 4, 16, 2
    pools = [np.arange(ngb * S * B, dtype=np.uint8)]
    out, st = oracle.gather(B=B, num_rows=ngb * S, pools=pools, rows=np.array([[7, -1, 0]], np.int32))
    assert st == 0
    assert (out[0, 0] == pools[0][7 * B:8 * B]).all() and (out[0, 1] == 0).all()
    out, st = oracle.gather(B=B, num_rows=ngb * S, pools=pools, rows=np.array([[8, -3]], np.int32))
    assert st == 2 and (out == 0).all()


@pytest.mark.parametrize("G,layer_begin,nl", [(4, 4, 4), (2, 2, 4), (4, 0, 8)])
def test_index_share_equals_layers_given_the_same_topk(G, layer_begin, nl):
    """IndexShare (one indexer per group of G layers): a group resolved once with one shared state
    must give what G independent layers give when each is handed the group's top-K -- the same rows
    and stats for every layer, per-layer states equal to the group's, and every layer's pool holding
    its own copy of each miss row.  Layers outside [layer_begin, layer_begin + nl) stay untouched."""
    L, R, S, B, C, K, pages = 8, 3, 4, 16, 8, 4, 12
    rng = np.random.default_rng(100 + G + layer_begin)
    nb = C // S
    hot = np.arange(R * nb, dtype=np.int32).reshape(R, nb)
    res = rng.random((R, pages)) < 0.3
    res[:, -1] = True
    bt = np.full((R, pages), -1, np.int32)
    bt[res] = R * nb + np.arange(int(res.sum()), dtype=np.int32)
    hbt = np.arange(R * pages, dtype=np.int32).reshape(R, pages)
    geo = dict(R=R, S=S, B=B, C=C, max_pages=pages, ctx=[pages * S] * R, resident=True, host=True, hot_blocks=hot,
               num_gpu_blocks=R * nb + int(res.sum()), num_host_blocks=R * pages, bt=bt, hbt=hbt, L=L, seed=5)
    per_layer, shared = Case(**geo), Case(**geo)
    shared.tok = np.full((L // G, R, C), -1, np.int32)
    shared.stamp = np.full((L // G, R, C), -1, np.int32)
    untouched = [p.copy() for p in per_layer.pools]
    kw = dict(S=S, B=B, num_gpu_blocks=geo["num_gpu_blocks"], num_host_blocks=R * pages, block_table=bt,
              host_block_table=hbt, ctx_len=per_layer.ctx, max_pages=pages, C=C, hot_blocks=hot,
              layer_begin=layer_begin, threads=2)
    misses = 0
    for t in range(10):
        ids = rng.integers(-1, pages * S, size=(nl // G, R, 1, K)).astype(np.int32)
        if t == 6:
            ids[0, 1, 0, 0] = pages * S           # one failing unit: ID_RANGE, no mutation there
        s_rows, s_stats = oracle.resolve(topk=ids, slot_token=shared.tok, slot_stamp=shared.stamp, step=t,
                                         pools=shared.pools, hosts=shared.hosts, layers_per_index=G, **kw)
        p_rows, p_stats = oracle.resolve(topk=np.repeat(ids, G, axis=0), slot_token=per_layer.tok,
                                         slot_stamp=per_layer.stamp, step=t, pools=per_layer.pools,
                                         hosts=per_layer.hosts, **kw)
        assert np.array_equal(p_rows, np.repeat(s_rows, G, axis=0)), t
        assert np.array_equal(p_stats, np.repeat(s_stats, G, axis=0)), t
        if t == 6:
            assert s_stats[0, 1, 0] == 2
        misses += int(s_stats[..., 3].sum())
        for l in range(L):
            assert np.array_equal(per_layer.tok[l], shared.tok[l // G]), (t, l)
            assert np.array_equal(per_layer.stamp[l], shared.stamp[l // G]), (t, l)
            assert np.array_equal(per_layer.pools[l], shared.pools[l]), (t, l)
    assert misses > 0
    for l in list(range(layer_begin)) + list(range(layer_begin + nl, L)):
        assert np.array_equal(shared.pools[l], untouched[l]), l
        assert (shared.tok[l // G] == -1).all()
    # every filled slot of every layer of a called group holds its token's closed-form bytes
    for l in range(layer_begin, layer_begin + nl):
        for r in range(R):
            for v in range(C):
                tok = int(shared.tok[l // G, r, v])
                if tok >= 0:
                    row = shared.hot_row(r, v)
                    assert np.array_equal(shared.pools[l][row * B:(row + 1) * B],
                                          shared.expected_row_bytes(l, r, tok)), (l, r, v)


def test_snapshot_and_restore_continue_identically():
    """Invariant: the resolver's state is the slot tokens, stamps and pool bytes, nothing hidden -- a
    snapshot taken mid-run and restored into a fresh case continues exactly like the original."""
    w = workloads.config1(seed=4, steps=8)
    geo = dict(R=w.R, S=w.S, B=w.B, C=w.C, max_pages=w.max_pages, ctx=w.ctx_len, resident=True, host=True,
               hot_blocks=w.hot_blocks, num_gpu_blocks=w.num_gpu_blocks, num_host_blocks=w.num_host_blocks,
               bt=w.block_table, hbt=w.host_block_table, seed=w.content_seed, content_page=w.content_page)
    a = Case(**geo)
    steps = list(w.iter_steps())
    for st in steps[:4]:
        a.step(st.topk, st.index)
    snap = (a.tok.copy(), a.stamp.copy(), [p.copy() for p in a.pools])
    out_a = [a.step(st.topk, st.index) for st in steps[4:]]
    b = Case(**geo)
    b.tok[...], b.stamp[...] = snap[0], snap[1]
    for dst, src in zip(b.pools, snap[2]):
        dst[...] = src
    out_b = [b.step(st.topk, st.index) for st in steps[4:]]
    for (ra, sa), (rb, sb) in zip(out_a, out_b):
        assert np.array_equal(ra, rb) and np.array_equal(sa, sb)
    assert np.array_equal(a.tok, b.tok) and np.array_equal(a.stamp, b.stamp)
    assert all(np.array_equal(x, y) for x, y in zip(a.pools, b.pools))
    assert sum(int(s[..., 3].sum()) for _, s in out_a) > 0
