"""Cross-check: the C oracle against the independent pure-Python brute force (oracle/bruteforce.py)
on thousands of random tiny cases -- rows, stats, slot tokens, slot stamps and pool bytes after every
step.  Cases mix residency, missing host copies, duplicates, padding, several query positions,
replayed steps (same step number) and occasional invalid ids or steps going backwards."""
import os

import numpy as np
import pytest

from oracle import bruteforce
from tests.casekit import Case

N_CASES = int(os.environ.get("HS_BRUTE_CASES", "10000"))


def _random_case(rng):
    S = int(rng.choice([1, 2, 4]))
    R = int(rng.integers(1, 3))
    K = int(rng.integers(1, 9))
    P = int(rng.integers(1, 4))
    C = int(rng.integers(max(1, K), 3 * K + 1))
    C = max(S, (C + S - 1) // S * S)
    pages = int(rng.integers(2, 9))
    ctx = [int(rng.integers(S, pages * S + 1)) for _ in range(R)]
    nb_hot = C // S
    n_res = int(rng.integers(0, pages))
    ngb = R * nb_hot + R * pages
    perm = rng.permutation(ngb).astype(np.int32)
    hot = perm[:R * nb_hot].reshape(R, nb_hot)
    bt = np.full((R, pages), -1, np.int32)
    hbt = np.full((R, pages), -1, np.int32)
    k = R * nb_hot
    hperm = rng.permutation(R * pages).astype(np.int32)
    for r in range(R):
        res = rng.random(pages) < n_res / pages
        for p in range(pages):
            if res[p]:
                bt[r, p] = perm[k]
                k += 1
            if rng.random() < 0.95:
                hbt[r, p] = hperm[r * pages + p]
    if rng.random() < 0.05:          # a request without a usable hot buffer (fine while fully resident)
        hot[int(rng.integers(0, R)), int(rng.integers(0, nb_hot))] = int(rng.choice([-1, ngb]))
    case = Case(R=R, S=S, B=16, C=C, max_pages=pages, ctx=ctx, resident=True, host=True, hot_blocks=hot,
                num_gpu_blocks=ngb, num_host_blocks=R * pages, bt=bt, hbt=hbt, seed=int(rng.integers(1 << 30)))
    return case, P, K


def _ids(rng, case, P, K):
    out = np.full((case.R, P, K), -1, np.int32)
    for r in range(case.R):
        for p in range(P):
            for k in range(K):
                u = rng.random()
                if u < 0.1:
                    continue
                if u < 0.12:
                    out[r, p, k] = int(rng.integers(case.ctx[r], case.ctx[r] + 5))  # out of range
                else:
                    out[r, p, k] = int(rng.integers(0, case.ctx[r]))
    return out


def test_bruteforce_agrees_with_oracle():
    rng = np.random.default_rng(20240531)
    statuses = set()
    for ci in range(N_CASES):
        case, P, K = _random_case(rng)
        B, S = case.B, case.S
        slots = [[[-1, -1] for _ in range(case.C)] for _ in range(case.R)]
        pool = {}
        for row in range(case.ngb * S):
            pool[row] = case.pools[0][row * B:(row + 1) * B].tobytes()
        host = {row: case.hosts[0][row * B:(row + 1) * B].tobytes() for row in range(case.nhb * S)}
        t = 0
        for si in range(int(rng.integers(1, 12))):
            u = rng.random()
            if u < 0.1:
                pass                      # replay the same step number
            elif u < 0.13:
                t = max(0, t - 2)         # may go backwards -> STEP_ORDER
            else:
                t += int(rng.integers(1, 3))
            ids = _ids(rng, case, P, K)
            if rng.random() < 0.05 and case.R:
                ids = np.where(ids >= case.ctx[0], -1, ids)   # sometimes drop the invalid ids
            rows, stats = case.step(ids, t)
            for r in range(case.R):
                b_rows, b_stats = bruteforce.resolve_unit(
                    S=S, num_gpu_blocks=case.ngb, num_host_blocks=case.nhb, ids=ids[r].reshape(-1).tolist(),
                    bt=case.bt[r].tolist(), hbt=case.hbt[r].tolist(), ctx_len=int(case.ctx[r]),
                    max_pages=case.max_pages, C=case.C, hot_blocks_r=case.hot_blocks[r].tolist(), slots=slots[r],
                    step=t, pool=pool, host=host)
                statuses.add(b_stats[0])
                msg = f"case {ci} step {si} request {r}"
                assert rows[0, r].reshape(-1).tolist() == b_rows, msg
                assert stats[0, r].tolist() == b_stats, msg
                assert case.tok[0, r].tolist() == [s[0] for s in slots[r]], msg
                assert case.stamp[0, r].tolist() == [s[1] for s in slots[r]], msg
            got = case.pools[0]
            for row in range(case.ngb * S):
                assert got[row * B:(row + 1) * B].tobytes() == pool[row], f"case {ci} pool row {row}"
    # the random mix reaches success and every data-error class
    assert {0, 2, 3, 5, 8}.issubset(statuses), statuses


def test_bruteforce_agrees_with_oracle_index_share():
    """IndexShare: G consecutive layers read one top-K list and share one hot state per request; the
    brute force keeps one slot list per (group, request) and copies every miss into each layer."""
    import oracle

    rng = np.random.default_rng(20240601)
    for ci in range(max(1, N_CASES // 10)):
        case0, P, K = _random_case(rng)
        G = int(rng.choice([2, 4]))
        ng_total = int(rng.integers(1, 3))
        L = G * ng_total
        case = Case(R=case0.R, S=case0.S, B=case0.B, C=case0.C, max_pages=case0.max_pages, ctx=case0.ctx,
                    resident=True, host=True, hot_blocks=case0.hot_blocks, num_gpu_blocks=case0.ngb,
                    num_host_blocks=case0.nhb, bt=case0.bt, hbt=case0.hbt, L=L, seed=case0.seed)
        case.tok = np.full((ng_total, case.R, case.C), -1, np.int32)
        case.stamp = np.full((ng_total, case.R, case.C), -1, np.int32)
        B, S = case.B, case.S
        g0 = int(rng.integers(0, ng_total))            # first group of the calls
        ng = int(rng.integers(1, ng_total - g0 + 1))
        slots = [[[[-1, -1] for _ in range(case.C)] for _ in range(case.R)] for _ in range(ng_total)]
        pools = [{row: case.pools[l][row * B:(row + 1) * B].tobytes() for row in range(case.ngb * S)}
                 for l in range(L)]
        hosts = [{row: case.hosts[l][row * B:(row + 1) * B].tobytes() for row in range(case.nhb * S)}
                 for l in range(L)]
        t = 0
        for si in range(int(rng.integers(1, 8))):
            t += int(rng.integers(0, 3))
            ids = np.stack([_ids(rng, case, P, K) for _ in range(ng)])
            rows, stats = oracle.resolve(S=S, B=B, num_gpu_blocks=case.ngb, num_host_blocks=case.nhb, topk=ids,
                                         block_table=case.bt, host_block_table=case.hbt, ctx_len=case.ctx,
                                         max_pages=case.max_pages, C=case.C, hot_blocks=case.hot_blocks,
                                         slot_token=case.tok, slot_stamp=case.stamp, step=t, layer_begin=g0 * G,
                                         pools=case.pools, hosts=case.hosts, threads=2, layers_per_index=G)
            for gi in range(ng):
                grp = g0 + gi
                for r in range(case.R):
                    b_rows, b_stats = bruteforce.resolve_unit(
                        S=S, num_gpu_blocks=case.ngb, num_host_blocks=case.nhb, ids=ids[gi, r].reshape(-1).tolist(),
                        bt=case.bt[r].tolist(), hbt=case.hbt[r].tolist(), ctx_len=int(case.ctx[r]),
                        max_pages=case.max_pages, C=case.C, hot_blocks_r=case.hot_blocks[r].tolist(),
                        slots=slots[grp][r], step=t, group_pools=pools[grp * G:(grp + 1) * G],
                        group_hosts=hosts[grp * G:(grp + 1) * G])
                    msg = f"case {ci} step {si} group {grp} request {r}"
                    assert rows[gi, r].reshape(-1).tolist() == b_rows, msg
                    assert stats[gi, r].tolist() == b_stats, msg
            for grp in range(ng_total):
                for r in range(case.R):
                    assert case.tok[grp, r].tolist() == [s[0] for s in slots[grp][r]], f"case {ci} tokens"
                    assert case.stamp[grp, r].tolist() == [s[1] for s in slots[grp][r]], f"case {ci} stamps"
            for l in range(L):
                got = case.pools[l]
                for row in range(case.ngb * S):
                    assert got[row * B:(row + 1) * B].tobytes() == pools[l][row], f"case {ci} layer {l} row {row}"
