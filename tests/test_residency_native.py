"""Parity of the native residency manager (libhs.so, host code) with its oracle: the same random
operation sequences through both, compared after every operation -- return values and error codes,
the exported tables, free block counts, the offload queue, hot-buffer resets and fills.  Host-only
calls: runs without a GPU."""
import numpy as np
import pytest

import oracle.residency as ores
from tests.test_residency_pins import apply_op, check_invariants, random_ops


@pytest.fixture(scope="module")
def native():
    from sparse_mla_kv_gb300 import _build
    _build.build()
    from sparse_mla_kv_gb300.residency import Residency
    return Residency


def _same_tables(o, n):
    ob, oh, ohot, octx = o.tables()
    nb, nh, nhot, nctx = n.tables()
    assert np.array_equal(np.array(ob, np.int32), nb)
    assert np.array_equal(np.array(oh, np.int32), nh)
    assert np.array_equal(np.array(ohot, np.int32).reshape(nhot.shape), nhot)
    assert np.array_equal(np.array(octx, np.int32), nctx)


@pytest.mark.parametrize("seed", range(200))
def test_native_manager_equals_oracle_on_random_sequences(native, seed):
    (G, H, S, R, max_pages, Hc), ops = random_ops(1000 + seed, 150)
    o = ores.Residency(G, H, S, R, max_pages, Hc)
    n = native(G, H, S, R, max_pages, Hc)
    rng = np.random.default_rng(seed)
    for i, op in enumerate(ops):
        ro, rn = apply_op(o, op), apply_op(n, op)
        assert ro == rn, (i, op, ro, rn)
        _same_tables(o, n)
        assert o.free_gpu_blocks() == n.free_gpu_blocks(), (i, op)
        if rng.random() < 0.3:
            assert o.take_resets() == n.take_resets(), (i, op)
            assert o.take_fills() == n.take_fills(), (i, op)
        check_invariants(o, G)
    assert o.collect() == n.collect()
    n.close()


def test_native_manager_on_a_pressure_scenario(native):
    """Four requests decoding in lock-step over a pool that holds about half of their pages, with
    the indexer touching a sliding set of pages: both sides agree on every release, lease and copy."""
    G, H, S, R, P, Hc = 96, 4096, 4, 4, 64, 4
    o = ores.Residency(G, H, S, R, P, Hc)
    n = native(G, H, S, R, P, Hc)
    rng = np.random.default_rng(3)
    for r in range(R):
        for m in (o, n):
            m.admit(r, 20 * S + 1)
        assert o.collect() == n.collect()
    for step in range(60):
        for r in range(R):
            for m in (o, n):
                m.append(r, 1)
        ids = np.stack([rng.integers(-1, o.reqs[r].ctx + 3, 8) for r in range(R)]).astype(np.int32)
        if step % 2:
            for m in (o, n):
                m.touch_all(ids, step)
        else:
            for r in range(R):
                for m in (o, n):
                    m.touch(r, ids[r].tolist(), step)
        assert o.take_fills() == n.take_fills()
        assert o.take_resets() == n.take_resets()
        assert o.collect() == n.collect()
        _same_tables(o, n)
        check_invariants(o, G)
    released = sum(1 for r in range(R) for p in range(P) if o.reqs[r].bt[p] < 0 and o.reqs[r].hbt[p] >= 0)
    assert released > 0
    n.close()


def test_native_manager_on_a_larger_decode_loop(native):
    """16 requests with growing contexts over a pool of about 60% of their demand, 512 top-K ids each per
    step (batched appends and touches, as a serving loop calls them): the native manager and the oracle
    agree on every export after every step, and pages are released and leased along the way."""
    from synth import workloads
    R, S, K, Hc, P = 16, 16, 512, 8, 256
    rng = np.random.default_rng(21)
    ctx = [40 * S] * R
    G = int(0.6 * R * (ctx[0] // S + 30 + Hc))
    o = ores.Residency(G, 1 << 16, S, R, P, Hc)
    n = native(G, 1 << 16, S, R, P, Hc)
    for r in range(R):
        for m in (o, n):
            m.admit(r, ctx[r])
    assert o.collect() == n.collect()
    assert o.take_fills() == n.take_fills()
    prev = [None] * R
    for step in range(30):
        grow = rng.integers(1, 2 * S, R).astype(np.int32)
        for m in (o, n):
            m.append_all(grow)
        ids = np.empty((R, K), np.int32)
        for r in range(R):
            ctx[r] += int(grow[r])
            ids[r] = workloads.next_topk(rng, prev[r], ctx[r], K, 0.8 if prev[r] is not None else 0.0, "recency")
            prev[r] = ids[r]
        assert o.take_fills() == n.take_fills()
        assert o.take_resets() == n.take_resets()
        for m in (o, n):
            m.touch_all(ids, step)
        assert o.collect() == n.collect()
        _same_tables(o, n)
        assert o.free_gpu_blocks() == n.free_gpu_blocks()
        check_invariants(o, G)
    released = sum(1 for r in range(R) for p in range(P) if o.reqs[r].bt[p] < 0 and o.reqs[r].hbt[p] >= 0)
    assert released > 0
    n.close()
