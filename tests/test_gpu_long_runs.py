"""GPU parity for long runs: the victim sort at large step indices, and a 300-step LRU sequence.

The resolver orders eviction candidates by (last-used step, slot) with an LSD radix sort over 8-bit
digits of (stamp - smallest live stamp); it takes one pass per byte of the live stamps' span.  A
server's step counter keeps growing, so after a few hundred steps the span needs two passes, after
65,536 steps three, and against never-used slots (stamp -1) near the top of the int32 range four.
These tests write hot states whose live stamps span 9, 17 and 31 bits (never-used slots, ties, the
smallest and the largest stamp below the step), and 32 bits with a few stamps far below -1 (a state
the library never writes, which both sides must still order), into both the library and the oracle,
resolve several steps from there, and compare rows, stats, slot tokens, slot stamps and pool bytes
exactly.

The last test replays a 300-step single-token access sequence through the GPU and checks each
access's hit or miss against Mattson's stack-distance rule for LRU (an access hits iff its stack
distance is at most the capacity; Mattson et al., 1970), which needs no implementation of the
resolver at all, and the final hot state against the oracle.

Source of the rule: "vLLM GLM 5.3 Optimizations: Hybrid HiSparse Offloading", "Technical
Implementation of Hybrid HiSparse", item 2 (a miss is copied into an LRU slot); the order of victims
is the deterministic (stamp, slot) reading used throughout."""
import numpy as np
import pytest
import torch

import sparse_mla_kv_gb300 as hs
from synth import content
from tests.casekit import Case, host_only_case

pytestmark = pytest.mark.gpu

MODES_ORDER = ["split", "fused", "split+order", "fused+order", "split+ranges", "fused+ranges", "fused+ranges1",
               "fused+ranges2", "fused+part"]
INT32_MAX = 2**31 - 1


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from sparse_mla_kv_gb300 import _build
    _build.build()
    hs.lib()


def _long_case(rng, *, S, B, R, pages, C, tail_pages):
    """Host copies of every page; the last tail_pages pages of each request resident."""
    nb = C // S
    resident = np.zeros((R, pages), bool)
    resident[:, pages - tail_pages:] = True
    n_res = int(resident.sum())
    perm = rng.permutation(n_res + R * nb).astype(np.int32)
    bt = np.full((R, pages), -1, np.int32)
    rr, pp = np.nonzero(resident)
    bt[rr, pp] = perm[:n_res]
    hot = perm[n_res:].reshape(R, nb)
    hbt = rng.permutation(R * pages).astype(np.int32).reshape(R, pages)
    return Case(R=R, S=S, B=B, C=C, max_pages=pages, ctx=[pages * S] * R, resident=True, host=True,
                hot_blocks=hot, num_gpu_blocks=n_res + R * nb, num_host_blocks=R * pages, bt=bt, hbt=hbt,
                seed=int(rng.integers(1 << 30)))


def _inject_state(rng, case, t, below=None):
    """Fill every unit's hot state with distinct tokens and stamps spanning [-1, t - 1]: about 12% of
    the slots never used, the rest tied in small groups on a few values that include 0 and t - 1 and
    random values in between.  `below`: a few filled slots get this stamp instead (a value under -1,
    which the library never writes; both sides must still order it first).  Each filled slot's pool
    row holds its token's bytes (both sides)."""
    S, B, C = case.S, case.B, case.C
    ctx = int(case.ctx[0])
    for r in range(case.R):
        toks = rng.choice(ctx, size=C, replace=False).astype(np.int32)
        empty = rng.random(C) < 0.12
        levels = np.concatenate([[0, 1, t // 2, t - 2, t - 1], rng.integers(0, t, size=40)]).astype(np.int64)
        stamps = levels[rng.integers(0, len(levels), size=C)].astype(np.int32)
        stamps[empty] = -1
        toks[empty] = -1
        if below is not None:
            stamps[rng.choice(np.nonzero(~empty)[0], size=3, replace=False)] = below
        case.tok[0, r] = toks
        case.stamp[0, r] = stamps
        for v in np.nonzero(~empty)[0]:
            row = case.hot_row(r, int(v))
            case.pools[0][row * B:(row + 1) * B] = case.expected_row_bytes(0, r, int(toks[v]))


def _step_ids(rng, case, P, K):
    """[R][P][K] ids: about 40% held in hot slots, 40% host-only misses, 20% resident; positions 1..P-1
    keep 90% of position 0 (repeats of missed ids across positions)."""
    S = case.S
    out = np.empty((case.R, P, K), np.int32)
    for r in range(case.R):
        held = case.tok[0, r][case.tok[0, r] >= 0]
        res = np.nonzero(case.bt[r] >= 0)[0]
        res_ids = (res[:, None] * S + np.arange(S)[None, :]).reshape(-1)
        nh, nr = int(0.4 * K), int(0.2 * K)
        a = rng.choice(held, size=min(nh, len(held)), replace=False)
        b = rng.choice(res_ids, size=nr, replace=False)
        taken = set(a.tolist()) | set(b.tolist())
        c = []
        while len(a) + len(b) + len(c) < K:
            x = int(rng.integers(0, int(case.ctx[r])))
            if x not in taken and case.bt[r, x // S] < 0:
                taken.add(x)
                c.append(x)
        p0 = rng.permutation(np.concatenate([a, b, np.array(c, np.int64)])).astype(np.int32)
        out[r, 0] = p0
        for q in range(1, P):
            keep = p0[rng.choice(K, size=int(0.9 * K), replace=False)]
            extra = []
            ks = set(keep.tolist())
            while len(keep) + len(extra) < K:
                x = int(rng.integers(0, int(case.ctx[r])))
                if x not in ks:
                    ks.add(x)
                    extra.append(x)
            out[r, q] = rng.permutation(np.concatenate([keep, np.array(extra, np.int64)])).astype(np.int32)
    return out


def _to_gpu(case, dev, mode):
    S, B = case.S, case.B
    gpu = [torch.from_numpy(case.pools[0].reshape(case.ngb, S, B).copy()).to(dev)]
    host = [torch.from_numpy(case.hosts[0].reshape(-1, S, B).copy()).pin_memory()]
    pool = hs.Pool(gpu, host)
    opt = mode.partition("+")[2]
    if opt == "part":
        pool.set_miss_warps(0)
    elif opt == "order":
        pool.set_miss_order(hs.MISS_ORDER_ON)
    elif opt:
        pool.set_miss_order(hs.MISS_ORDER_RANGES)
        pool.set_miss_warps({"ranges1": 1, "ranges2": 2}.get(opt, 0))
    hot = hs.HotState.allocate(1, torch.from_numpy(case.hot_blocks).to(dev), case.C)
    hot.slot_token.copy_(torch.from_numpy(case.tok))
    hot.slot_stamp.copy_(torch.from_numpy(case.stamp))
    return pool, gpu, hot


def _passes(case, t):
    """Radix passes the victim sort of this state takes at step t (from the oracle's own state):
    bytes of (largest - smallest) stamp below t."""
    live = case.stamp[case.stamp < t]
    span = int(live.max()) - int(live.min())
    return (span.bit_length() + 7) // 8


@pytest.mark.parametrize("mode", MODES_ORDER)
@pytest.mark.parametrize("t0,bits,below", [(300, 9, None), (70_000, 17, None), (INT32_MAX - 10, 31, None),
                                           (1000, 32, -2**31)])
@pytest.mark.parametrize("S,B,P", [(64, 656, 1), (4, 32, 4)])
def test_victim_sort_over_long_stamp_spans(mode, t0, bits, below, S, B, P):
    rng = np.random.default_rng([t0 % 1000, S, P, len(mode)])
    dev = torch.device("cuda")
    K = 256 if S == 64 else 64
    C = 2 * K
    pages = 64 if S == 64 else 256
    case = _long_case(rng, S=S, B=B, R=6, pages=pages, C=C, tail_pages=8 if S == 64 else 32)
    _inject_state(rng, case, t0, below)
    assert _passes(case, t0) == (bits + 7) // 8
    live = case.stamp[case.stamp < t0]
    assert (int(live.max()) - int(live.min())).bit_length() == bits
    pool, gpu, hot = _to_gpu(case, dev, mode)
    bt, hbt = torch.from_numpy(case.bt).to(dev), torch.from_numpy(case.hbt).to(dev)
    ctx = torch.from_numpy(case.ctx).to(dev)
    misses = 0
    for k in range(4):
        t = t0 + k
        ids = _step_ids(rng, case, P, K)
        topk = torch.from_numpy(ids[None]).to(dev)
        if mode.startswith("fused"):
            rows, stats, g = hs.resolve_gather(pool, topk, bt, hbt, ctx, hot, t)
        else:
            rows, stats = hs.resolve_topk(pool, topk, bt, hbt, ctx, hot, t)
            g = hs.gather_rows(pool, rows.reshape(1, -1))
        o_rows, o_stats = case.step(ids, t)
        torch.cuda.synchronize()
        msg = f"step {t}"
        assert (o_stats[..., 0] == 0).all(), msg
        assert np.array_equal(stats.cpu().numpy(), o_stats), msg
        assert np.array_equal(rows.cpu().numpy(), o_rows), msg
        assert np.array_equal(hot.slot_token.cpu().numpy(), case.tok), msg
        assert np.array_equal(hot.slot_stamp.cpu().numpy(), case.stamp), msg
        assert np.array_equal(gpu[0].cpu().numpy().reshape(-1), case.pools[0]), msg
        o_out, _ = case.gather(o_rows.reshape(1, -1))
        assert np.array_equal(g.cpu().numpy(), o_out), msg
        m = int(o_stats[..., 3].sum())
        misses += m
        # victims are a strict subset of the candidates, so their order decides the result
        assert 0 < m
    assert misses > 0
    pool.close()


@pytest.mark.parametrize("mode", ["split", "fused"])
@pytest.mark.parametrize("C,S,seed", [(4, 1, 0), (8, 4, 2), (12, 4, 4)])
def test_lru_300_steps_stack_distance_on_gpu(mode, C, S, seed):
    """K = 1, one access per step, every page host-only: the resolver is plain LRU of capacity C, so
    the j-th access hits iff its Mattson stack distance is <= C.  300 steps take the victim sort past
    one byte of stamp span."""
    from tests.test_oracle_pins import _mattson_hits
    rng = np.random.default_rng(seed)
    pages = 12
    dev = torch.device("cuda")
    case = host_only_case(S=S, C=C, pages=pages, B=16, seed=seed)
    ctx_n = pages * S
    seq = [int(min(ctx_n - 1, rng.geometric(0.08))) if rng.random() < 0.5 else int(rng.integers(0, ctx_n))
           for _ in range(300)]
    expect = _mattson_hits(seq, C)
    gpu = [torch.from_numpy(case.pools[0].reshape(case.ngb, S, 16).copy()).to(dev)]
    host = [torch.from_numpy(case.hosts[0].reshape(-1, S, 16).copy()).pin_memory()]
    pool = hs.Pool(gpu, host)
    hot = hs.HotState.allocate(1, torch.from_numpy(case.hot_blocks).to(dev), C)
    hs.hot_reset(pool, hot)
    bt, hbt = torch.from_numpy(case.bt).to(dev), torch.from_numpy(case.hbt).to(dev)
    ctx = torch.from_numpy(case.ctx).to(dev)
    stats_all, out_all = [], []
    for t, x in enumerate(seq):
        topk = torch.tensor([[[[x]]]], dtype=torch.int32, device=dev)
        if mode == "fused":
            rows, stats, g = hs.resolve_gather(pool, topk, bt, hbt, ctx, hot, t)
        else:
            rows, stats = hs.resolve_topk(pool, topk, bt, hbt, ctx, hot, t)
            g = hs.gather_rows(pool, rows.reshape(1, -1))
        stats_all.append(stats.clone())
        out_all.append(g.clone())
        case.step(np.array([[[x]]], np.int32), t, bytes_=False)
    torch.cuda.synchronize()
    st = torch.stack(stats_all).cpu().numpy().reshape(len(seq), 4)
    assert (st[:, 0] == 0).all()
    assert (st[:, 2] + st[:, 3] == 1).all()
    hits = st[:, 2] == 1
    assert hits.tolist() == expect
    assert 0 < hits.sum() < len(seq)
    assert np.array_equal(hot.slot_token.cpu().numpy(), case.tok)
    assert np.array_equal(hot.slot_stamp.cpu().numpy(), case.stamp)
    # every access gathered its token's bytes
    for t, x in enumerate(seq):
        exp = content.rows_np(case.seed, 0, int(case.content_page[0, x // S]), x % S, 16)
        assert np.array_equal(out_all[t].cpu().numpy().reshape(-1), exp), f"access {t}"
    pool.close()
