"""Brute-force twin of the oracle for tiny inputs, written independently in plain Python.

TEST INFRASTRUCTURE ONLY (imported by tests).  It shares nothing with hs_oracle.c: no sorting,
no binary search.  The hot buffer is a Python list of [token, stamp] slots scanned linearly;
victims are taken one at a time by scanning for the smallest (stamp, slot) among the slots that
are still eligible (selection instead of a sort); the plan is built by scanning a list of ids
already seen.  Semantics follow the same passages as hs_oracle.c (resident in place, hit refresh,
miss copies exactly one row into an LRU slot; replayable per-step plan shared by all positions).
"""
from __future__ import annotations

OK, ID_RANGE, MISSING_ROW, CAPACITY, STEP_ORDER, TABLE_RANGE = 0, 2, 3, 4, 5, 8


def resolve_unit(*, S, num_gpu_blocks, num_host_blocks, ids, bt, hbt, ctx_len, max_pages, C, hot_blocks_r,
                 slots, step, pool=None, host=None, group_pools=None, group_hosts=None):
    """ids: flat list (positions then top-K); bt/hbt: lists over pages; slots: list of C [token, stamp]
    (mutated on success); pool/host: dict row -> bytes (pool mutated on success).  Under IndexShare
    (several layers read one indexer's top-K and share these slots) group_pools/group_hosts list one
    such dict per layer of the group, and every miss is copied in each of them.
    Returns (rows list, [status, resident, hits, misses])."""
    if pool is not None:
        group_pools, group_hosts = [pool], [host]
    errors = set()
    if any(st > step for _, st in slots):
        errors.add(STEP_ORDER)
    for x in ids:
        if x != -1 and (x < -1 or x >= ctx_len or x // S >= max_pages):
            errors.add(ID_RANGE)
    hot_ok = all(0 <= b < num_gpu_blocks for b in hot_blocks_r)

    def slot_row(v):
        return hot_blocks_r[v // S] * S + v % S

    plan = []                      # distinct ids in order of first appearance
    kind = {}                      # id -> ("res", row) | ("hit", slot) | ("miss", src_row)
    if STEP_ORDER not in errors and ID_RANGE not in errors:
        for x in ids:
            if x >= 0 and x not in plan:
                plan.append(x)
        for x in plan:
            page, off = x // S, x % S
            if bt[page] >= 0:
                if bt[page] >= num_gpu_blocks:
                    errors.add(TABLE_RANGE)
                kind[x] = ("res", bt[page] * S + off)
                continue
            holder = None
            for v in range(C):     # lowest slot holding the token
                if slots[v][0] == x:
                    holder = v
                    break
            if holder is not None:
                kind[x] = ("hit", holder)
            else:
                if hbt[page] < 0:
                    errors.add(MISSING_ROW)
                elif hbt[page] >= num_host_blocks:
                    errors.add(TABLE_RANGE)
                kind[x] = ("miss", hbt[page] * S + off)
        hit_slots = [kind[x][1] for x in plan if kind[x][0] == "hit"]
        n_miss = sum(1 for x in plan if kind[x][0] == "miss")
        if not hot_ok and (hit_slots or n_miss):      # only hits and misses touch the hot blocks
            errors.add(TABLE_RANGE)
        eligible = [v for v in range(C) if slots[v][1] < step and v not in hit_slots]
        if n_miss > len(eligible):
            errors.add(CAPACITY)

    for code in (STEP_ORDER, ID_RANGE, TABLE_RANGE, MISSING_ROW, CAPACITY):
        if code in errors:
            return [-1] * len(ids), [code, 0, 0, 0]

    row_of = {}
    for x in plan:
        if kind[x][0] == "res":
            row_of[x] = kind[x][1]
    for x in plan:
        if kind[x][0] == "hit":
            v = kind[x][1]
            slots[v][1] = step
            row_of[x] = slot_row(v)
    taken = set()
    for x in plan:
        if kind[x][0] != "miss":
            continue
        best = None
        for v in range(C):
            if v in taken or v in hit_slots or slots[v][1] >= step:
                continue
            if best is None or (slots[v][1], v) < (slots[best][1], best):
                best = v
        taken.add(best)
        slots[best][0] = x
        slots[best][1] = step
        row_of[x] = slot_row(best)
        for lp, lh in zip(group_pools or [], group_hosts or []):
            lp[row_of[x]] = lh[kind[x][1]]
    rows = [row_of[x] if x >= 0 else -1 for x in ids]
    counts = [sum(1 for x in plan if kind[x][0] == k) for k in ("res", "hit", "miss")]
    return rows, [OK] + counts
