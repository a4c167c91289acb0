"""Pins for the residency-manager oracle (oracle/residency.py): facts fixed by the pages or by the
definition, checked without the native manager.

  - the A/B example (Japanese article, the section before "仕組み"): with a pool too small for both
    requests, both keep decoding -- each frees its cold pages and the freed blocks become tail and
    hot pages;
  - closed forms: without pressure blocks are handed out in order and nothing is released;
  - LRU order of cold pages; a page whose offload is still queued is not released; the tail stays;
  - hot buffers are leased once, when the first placeholder appears, and returned at finish; a block
    freed by one request serves another;
  - invariants after every operation of random sequences: every GPU block is free, a resident page of
    exactly one request, or a hot block of exactly one request; every complete page is resident or
    has a host copy; the last page is resident; host reference counts match the references.
"""
import numpy as np
import pytest

from oracle.residency import CAPACITY, INVALID_ARG, Residency, ResidencyError


def check_invariants(m: Residency, num_gpu_blocks: int) -> None:
    owner = {}
    for b in m.free_gpu:
        assert b not in owner, f"block {b} free twice"
        owner[b] = "free"
    bt, hbt, hot, ctx = m.tables()
    refs = list(m.host_held)
    for r, x in enumerate(m.reqs):
        if x is None:
            assert all(v == -1 for v in bt[r]) and ctx[r] == 0
            continue
        npages = (x.ctx + m.S - 1) // m.S
        assert x.bt[npages - 1] >= 0, "the last page left the GPU"
        for p in range(m.max_pages):
            if x.bt[p] >= 0:
                assert p < npages
                assert x.bt[p] not in owner, f"block {x.bt[p]} owned twice"
                owner[x.bt[p]] = ("page", r, p)
            if x.hbt[p] >= 0:
                refs[x.hbt[p]] += 1
            if p < x.ctx // m.S:
                assert x.bt[p] >= 0 or x.hbt[p] >= 0, "a complete page has neither copy"
        for b in x.hot or []:
            assert b not in owner, f"hot block {b} owned twice"
            owner[b] = ("hot", r)
        for p in x.pending:
            assert any(e[2] == r and e[3] == p and e[0] == x.bt[p] for e in m.queue)
    assert sorted(owner) == list(range(num_gpu_blocks)), "a GPU block is lost"
    assert refs == m.host_ref, "host reference counts"


def test_no_pressure_blocks_in_order_and_nothing_released():
    m = Residency(64, 64, 4, 3, 16, 2)
    m.admit(0, 10)                    # pages 0..2 (0, 1 complete)
    m.admit(1, 4)                     # page 0 (complete)
    assert m.take_fills() == [(0, 0, 0), (1, 0, 1), (2, 0, 2), (3, 1, 0)]
    assert m.collect() == [(0, 0), (1, 1), (3, 2)]
    m.append(0, 3)                    # ctx 13: page 2 completes, page 3 starts
    assert m.take_fills() == [(4, 0, 3)]
    assert m.collect() == [(2, 3)]
    bt, hbt, hot, ctx = m.tables()
    assert bt[0][:4] == [0, 1, 2, 4] and hbt[0][:4] == [0, 1, 3, -1] and ctx[:2] == [13, 4]
    assert hot[0] == [-1, -1] and m.take_resets() == []
    check_invariants(m, 64)


def test_ab_example_both_requests_keep_decoding():
    """Pool of 40 blocks; A and B each reach 24 pages, so both cannot be fully resident.  Every step
    both decode one page of tokens; neither ever fails, both end with placeholders and hot buffers,
    and each stays within the pool."""
    S, G = 4, 40
    m = Residency(G, 1000, S, 2, 64, 4)
    m.admit(0, 16 * S)
    m.collect()
    m.admit(1, 16 * S)
    m.collect()
    step = 0
    for _ in range(8):
        for r in (0, 1):
            m.append(r, S)
            m.touch(r, [m.reqs[r].ctx - 1], step)   # the indexer reads the newest page
            step += 1
        m.take_fills()
        m.collect()
        check_invariants(m, G)
    bt, hbt, hot, ctx = m.tables()
    for r in (0, 1):
        assert ctx[r] == 24 * S
        assert -1 in bt[r][:24], "no page was released"
        assert hot[r] != [-1] * 4, "no hot buffer was leased"
        assert bt[r][23] >= 0


def test_cold_pages_leave_in_lru_order_and_the_tail_stays():
    S = 2
    m = Residency(8, 64, S, 1, 16, 1)
    m.admit(0, 5 * S)                 # pages 0..4 complete, blocks 0..4
    m.collect()
    m.append(0, 3 * S)                # pages 5, 6, 7: blocks 5..7, the pool is full
    assert -1 not in m.tables()[0][0][:8]
    m.collect()
    # last use: page 0 at 3, 1 at 1, 2 at 2, 3 never, 4 at 5, 5 at 6, 6 at 7, 7 (tail) at 8
    for page, step in ((1, 1), (2, 2), (0, 3), (4, 5), (5, 6), (6, 7), (7, 8)):
        m.touch(0, [page * S + 1], step)
    m.append(0, S)                    # page 8 starts: page 3 (never used) goes, then the hot lease
                                      # takes page 1 (used at step 1)
    bt, hbt, hot, ctx = m.tables()
    bt = bt[0]
    assert [p for p in range(9) if bt[p] < 0] == [1, 3]
    assert hot[0] == [3] and bt[8] == 1   # the lease takes the block page 3 freed (lowest first)
    m.collect()
    m.append(0, 2 * S)                # pages 9, 10: page 2 (step 2), then page 0 (step 3)
    bt = m.tables()[0][0]
    assert [p for p in range(11) if bt[p] < 0] == [0, 1, 2, 3]
    assert bt[7] >= 0                 # the old tail (complete, used at 8) is still resident
    check_invariants(m, 8)


def test_a_page_whose_offload_is_queued_is_not_released():
    S = 2
    m = Residency(2, 64, S, 1, 16, 1)
    m.admit(0, 2 * S)                 # pages 0, 1 complete; their offloads are queued
    with pytest.raises(ResidencyError) as e:
        m.append(0, 1)                # page 2 starts: no free block, pages 0/1 still queued
    assert e.value.code == CAPACITY
    m2 = Residency(4, 64, S, 1, 16, 1)
    m2.admit(0, 2 * S)
    m2.collect()                      # copies enqueued: pages may now give up their blocks
    m2.append(0, 1)                   # page 2 takes block 2
    m2.collect()
    m2.append(0, 2 * S)               # pages 3, 4: block 3; then page 0 goes to the hot lease and
                                      # page 1's block to page 4
    bt, hbt, hot, _ = m2.tables()
    bt = bt[0]
    assert bt[:5] == [-1, -1, 2, 3, 1] and hot[0] == [0]
    check_invariants(m2, 4)


def test_hot_buffer_leased_once_and_returned_to_other_requests():
    S = 2
    m = Residency(10, 64, S, 2, 32, 2)
    m.admit(0, 6 * S)                 # 6 pages
    m.collect()
    m.admit(1, 2 * S)                 # 2 pages: 8 blocks used, 2 free
    m.collect()
    m.append(1, 3 * S)                # pages 2, 3 use the free blocks; page 4: pressure.  Request 1
                                      # releases its page 0 and leases its buffer, which takes a page
                                      # of request 0, which then needs a buffer of its own
    assert m.take_resets() == [1, 0]
    bt, hbt, hot, _ = m.tables()
    assert hot[1] == [6, 2] and hot[0] == [0, 1]
    assert bt[0][:6] == [-1, -1, -1, -1, 4, 5] and bt[1][:5] == [-1, 7, 8, 9, 3]
    check_invariants(m, 10)
    m.collect()
    m.append(1, 2 * S)
    assert m.take_resets() == []      # leased once
    check_invariants(m, 10)
    free_before = m.free_gpu_blocks()
    n_blocks_r1 = sum(1 for b in m.tables()[0][1] if b >= 0) + 2
    m.finish(1)
    assert m.free_gpu_blocks() == free_before + n_blocks_r1
    placeholders0 = sum(1 for b in m.tables()[0][0] if b < 0)
    m.append(0, 2 * S)                # request 0 grows into the returned blocks without releasing
    assert sum(1 for b in m.tables()[0][0] if b < 0) == placeholders0 - 2
    assert m.take_resets() == []
    check_invariants(m, 10)


def test_prefix_reuse_admission_starts_with_placeholders_and_a_hot_page():
    """No residency (Japanese article, "仕組み"): a request reusing a host-only prefix starts with
    placeholders and a hot page; the host prefix is shared (reference counts)."""
    S = 4
    m = Residency(16, 16, S, 2, 8, 1)
    m.hold_host([5, 6])                        # a prefix cache holds host blocks 5, 6
    m.admit(0, 2 * S + 3, prefix_host_blocks=[5, 6])
    m.admit(1, 2 * S + 1, prefix_host_blocks=[5, 6])
    bt, hbt, hot, ctx = m.tables()
    assert bt[0][:3] == [-1, -1, 1] and hbt[0][:2] == [5, 6]
    assert hot[0] == [0] and hot[1] == [2] and bt[1][:3] == [-1, -1, 3]
    assert m.host_ref[5] == 3 and m.take_resets() == [0, 1]
    m.finish(0)
    assert m.host_ref[5] == 2
    check_invariants(m, 16)
    m.finish(1)
    m.drop_host([5, 6])
    assert m.host_ref[5] == 0 and m.free_gpu_blocks() == 16
    check_invariants(m, 16)


def test_argument_errors():
    m = Residency(4, 4, 2, 2, 4, 1)
    for f in (lambda: m.append(0, 1), lambda: m.admit(2, 1), lambda: m.admit(0, 9), lambda: m.admit(0, 0),
              lambda: m.admit(0, 4, prefix_host_blocks=[0, 1]), lambda: m.admit(0, 4, prefix_host_blocks=[7])):
        with pytest.raises(ResidencyError) as e:
            f()
        assert e.value.code == INVALID_ARG


def random_ops(seed: int, n_ops: int):
    """A seeded random sequence of manager operations (shared with the native parity test)."""
    rng = np.random.default_rng(seed)
    S = int(rng.choice([1, 2, 4]))
    R = int(rng.integers(1, 5))
    max_pages = int(rng.integers(4, 24))
    Hc = int(rng.integers(1, 4))
    G = int(rng.integers(R + Hc, R * (max_pages // 2 + Hc) + 2))
    H = int(rng.integers(R * max_pages // 2, R * max_pages * 2 + 2))
    ops = []
    step = 0
    for _ in range(n_ops):
        u = rng.random()
        r = int(rng.integers(0, R))
        if u < 0.15:
            ctx = int(rng.integers(1, max_pages * S // 2 + 2))
            npref = int(rng.integers(0, (ctx - 1) // S + 2)) if rng.random() < 0.4 else 0   # may overshoot
            pref = [int(x) for x in rng.integers(0, H, npref)]
            ops.append(("admit", r, ctx, pref))
        elif u < 0.55:
            if rng.random() < 0.15:   # every request at once (zero for some; inactive ones fail the call)
                counts = [int(x) if rng.random() < 0.7 else 0 for x in rng.integers(0, 2 * S + 1, R)]
                ops.append(("append_all", counts))
            else:
                ops.append(("append", r, int(rng.integers(0, 2 * S + 1))))
        elif u < 0.75:
            if rng.random() < 0.3:
                ops.append(("touch_all", [[int(x) for x in rng.integers(-1, max_pages * S, 4)] for _ in range(R)], step))
            else:
                ops.append(("touch", r, [int(x) for x in rng.integers(-1, max_pages * S, 4)], step))
            step += int(rng.integers(0, 2))
        elif u < 0.90:
            ops.append(("collect",))
        elif u < 0.93:
            ops.append(("hold" if rng.random() < 0.6 else "drop", [int(x) for x in rng.integers(0, H, 2)]))
        else:
            ops.append(("finish", r))
    return (G, H, S, R, max_pages, Hc), ops


def apply_op(m, op):
    """Apply one op to a manager (oracle or native: same method names); returns the op's result
    or ('error', code)."""
    try:
        kind = op[0]
        if kind == "admit":
            return m.admit(op[1], op[2], op[3])
        if kind == "append":
            return m.append(op[1], op[2])
        if kind == "touch":
            return m.touch(op[1], op[2], op[3])
        if kind == "append_all":
            return m.append_all(op[1])
        if kind == "touch_all":
            return m.touch_all(np.array(op[1], np.int32), op[2])
        if kind == "collect":
            return m.collect()
        if kind == "hold":
            return m.hold_host(op[1])
        if kind == "drop":
            return m.drop_host(op[1])
        return m.finish(op[1])
    except Exception as e:     # both sides raise an error carrying .code
        return ("error", getattr(e, "code", None))


@pytest.mark.parametrize("seed", range(40))
def test_invariants_hold_on_random_operation_sequences(seed):
    (G, H, S, R, max_pages, Hc), ops = random_ops(seed, 120)
    m = Residency(G, H, S, R, max_pages, Hc)
    n_err = 0
    for op in ops:
        res = apply_op(m, op)
        if isinstance(res, tuple) and res and res[0] == "error":
            n_err += 1
            assert res[1] in (INVALID_ARG, CAPACITY)
        check_invariants(m, G)
    assert n_err < len(ops)
