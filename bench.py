#!/usr/bin/env python3
"""Benchmark of the Hybrid HiSparse decode hot path (resolve + gather, + offload of completed pages).

Default workload: the max batch with speculative decode (MTP3) at full size -- 4 sparse-MLA layers,
256 requests with contexts log-uniform in [8192, 1,048,576] tokens, each non-tail page resident with
a per-request probability f ~ U[0, 1] (the tail always resident, host copies of the host-only pages:
about 80 GB of GPU pool and 80 GB of pinned host pool), page 64, 656-byte rows, K = 2048, P = 4 query
positions sharing one plan (90% overlap), hot buffer 4096 rows per request; each step appends 1-4
tokens per request and ends with one offload launch of the pages it completed (all layers).
8,388,608 resolved rows per step.  Synthetic, seeded.  --config 1..4 select the other workloads
(tiny decode, the mixed-residency batch, multi-turn agentic decode, cold start with prefix reuse).

One step = the fused path (hs_resolve_plan + hs_gather_planned: the resolver, then one gather that
also carries the miss copies) or, with --path split, hs_resolve_topk + hs_gather_rows, over the
step's batch, then one hs_offload_pages launch for the pages the step completes (all layers).  Table
edits and the model's page writes of a step are applied before its timed events.  L2 is flushed (a
256 MB write) before every timed step, outside the timed events, and the host waits for each step
before enqueueing the next.  With --timing graph (or both) each timed step is also captured as one
CUDA graph and replayed once.

Prints one JSON line (rank 0).  `--impl reference` times the CPU oracle on the host cores instead.
The oracle legs (the reference arm and the cpu_baseline of the GPU line) run on the first requests
of the same workload, as many as keep the oracle's byte pools within a few GB (all of them for
configs 1, 2 and 4), with their block ids renumbered densely; rows/s adds over independent requests.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402
import torch  # noqa: E402

METRIC = "top-K rows resolved+gathered/s; achieved GB/s vs HBM / host-link roofline"
UNIT = "rows/s"
FALLBACK_HBM_GBS = 6800.0
L2_FLUSH_BYTES = 256 << 20


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--config", type=int, default=5, choices=[1, 2, 3, 4, 5])
    ap.add_argument("--requests", type=int, default=None, help="requests per rank (configs 2-5)")
    ap.add_argument("--layers", type=int, default=None, help="sparse-MLA layers (configs 3, 5)")
    ap.add_argument("--layers-per-index", type=int, default=1,
                    help="IndexShare: layers that read one indexer's top-K and share one hot state (configs 3, 5)")
    ap.add_argument("--capacity", type=int, default=None, help="hot rows per request (config 5)")
    ap.add_argument("--decode-per-turn", type=int, default=None, help="decode steps per turn (config 3)")
    ap.add_argument("--full-residency", action="store_true",
                    help="config 2 with every page resident (no KV pressure: no hit, no miss)")
    ap.add_argument("--seed", type=int, default=0)
    ap.add_argument("--cpu-seconds", type=float, default=12.0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--settle-seconds", type=float, default=60.0,
                    help="upper bound on the untimed passes over the timed steps that run until two in a row agree "
                         "within 5%% (at least two passes)")
    ap.add_argument("--soak-seconds", type=float, default=None,
                    help="seconds of repeated gathers before the timed steps (default 1.5; 5 for host pools of "
                         "16 GiB or more, whose first seconds of reads after pinning run unevenly)")
    ap.add_argument("--no-clocks", action="store_true", help="do not sample nvidia-smi during the timed steps")
    ap.add_argument("--passes", type=int, default=2, choices=[1, 2],
                    help="2: an untimed pass over the warm-up and timed steps precedes the timed pass")
    ap.add_argument("--no-prefault", action="store_true",
                    help="skip the one bulk read of the pinned host pool through the GPU before timing")
    ap.add_argument("--run-ahead", action="store_true",
                    help="enqueue all timed steps without waiting for each (default: wait for each step's end "
                         "before enqueueing the next; the L2 flush queued ahead of each step keeps the GPU busy "
                         "while the step is enqueued)")
    ap.add_argument("--residency", action="store_true",
                    help="time the host-side residency manager (native and its oracle) on a decode loop under "
                         "KV pressure instead of the GPU path; host only")
    ap.add_argument("--gather-ab", action="store_true",
                    help="after the timed passes, time the plain gather (hs_gather_rows) of the last step's "
                         "resolved rows with 16-byte loads and with bulk copies (hs_pool_set_gather_copy), "
                         "alternating, in this process")
    ap.add_argument("--miss-warps-ab", action="store_true",
                    help="after the timed passes, replay the last timed step's planned gather (hs_gather_planned) "
                         "with the SM partition and with 1 and 2 miss warps in every CTA (hs_pool_set_miss_warps), "
                         "alternating, in this process")
    ap.add_argument("--miss-sm-ab", type=str, default="",
                    help="comma-separated SM divisors (e.g. 4,5,6,8): after the timed passes, replay the last timed "
                         "step's planned gather with the SM partition at each divisor (hs_pool_set_miss_sm_divisor), "
                         "alternating, in this process")
    ap.add_argument("--prefetch-ab", type=int, default=0, metavar="ROUNDS",
                    help="after the timed passes, ROUNDS rounds of whole timed passes alternating the resolver's miss "
                         "prefetch off and on (hs_pool_set_miss_prefetch), in this process")
    ap.add_argument("--miss-prefetch", choices=["off", "on"], default="off",
                    help="the resolver's miss prefetch for the timed passes (hs_pool_set_miss_prefetch)")
    ap.add_argument("--gather-phases", action="store_true",
                    help="after the timed passes, replay the last timed step's planned gather with the SM partition's "
                         "device timestamps on (hs_pool_set_phase_timestamps): when its HBM rows and its misses end")
    ap.add_argument("--planes-ab", action="store_true",
                    help="after the timed passes, replay the last timed step's gather with the output in rows and in "
                         "the planes {512, 16, 128} (hs_pool_set_gather_planes), alternating, in this process")
    ap.add_argument("--miss-warps", type=int, default=-1, choices=[-1, 0, 1, 2],
                    help="fused gather: -1 = the library's default (SM partition with the range schedule, one miss "
                         "warp per CTA with per-unit lists), 0 = SM partition, 1 or 2 = that many miss warps in every "
                         "CTA (hs_pool_set_miss_warps)")
    ap.add_argument("--link-probe", action="store_true",
                    help="measure the miss path's host-link rate against the span of host memory it reads "
                         "(one layer, all-miss steps) instead of a workload")
    ap.add_argument("--probe-pool-gb", type=float, default=72.0, help="pinned host pool of the link probe")
    ap.add_argument("--probe-windows-gb", type=float, nargs="+", default=[1, 4, 10, 20, 40, 72],
                    help="spans of the host pool the link probe's misses read")
    ap.add_argument("--probe-base-pages", action="store_true",
                    help="link probe: register the host pool without huge pages (for comparison)")
    ap.add_argument("--probe-cpu-fill", action="store_true",
                    help="link probe: write the host pool with CPU stores instead of DMA (for comparison)")
    ap.add_argument("--schedule-ab", type=int, default=0, metavar="ROUNDS",
                    help="after the timed passes, ROUNDS rounds of two more timed passes over the same steps, one "
                         "with the range schedule and one with the spread schedule of the ordered miss layout "
                         "(hs_pool_set_miss_order), in this process")
    ap.add_argument("--miss-order", choices=["auto", "on", "off", "ranges", "spread"], default="auto",
                    help="miss layout handed to the copy warps: auto (the library's default: host-address order "
                         "for host pools of 16 GiB or more), on (always address order), off (per-unit lists), "
                         "ranges (address order with the range schedule on any pool)")
    ap.add_argument("--timing", choices=["auto", "eager", "graph", "both"], default="auto",
                    help="eager: the C-ABI calls of each timed step bracketed by events; graph: each timed step "
                         "captured as one CUDA graph and replayed once, the replay bracketed by events; both: "
                         "eager is the headline and the graph replay is reported beside it; auto: both for host "
                         "pools under 16 GiB, eager alone above")
    ap.add_argument("--oracle-pool-gb", type=float, default=8.0,
                    help="the oracle legs run on the first requests whose byte pools fit in this many GB")
    ap.add_argument("--path", choices=["fused", "split"], default="fused",
                    help="fused: hs_resolve_plan + hs_gather_planned (miss copies inside the gather); "
                         "split: hs_resolve_topk (resolver + miss-copy kernel) + hs_gather_rows")
    return ap.parse_args()


# ----------------------------------------------------------------------------- distributed plumbing
def dist_env():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


def dist_init(ws):
    if ws > 1:
        import torch.distributed as dist
        os.environ.setdefault("MASTER_ADDR", "127.0.0.1")
        backend = "nccl" if torch.cuda.is_available() else "gloo"
        dist.init_process_group(backend=backend)
        return dist
    return None


def rank_seed(seed: int, rank: int) -> int:
    """Each rank serves its own independent batch of requests (the path shards by request: every
    (layer, request) unit, table row, hot buffer and output slice is independent), so ranks draw
    different requests from the same generator: weak scaling, no data-path collective."""
    return seed + 1000003 * rank


def barrier(dist):
    if dist is not None:
        dist.barrier()


def max_over_ranks(dist, x: float, device) -> float:
    if dist is None:
        return x
    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


# ----------------------------------------------------------------------------- workload
def make_workload(args, seed: int, n_steps: int):
    from synth import workloads
    kw = {}
    if args.requests is not None and args.config != 1:
        kw["R"] = args.requests
    if args.config in (3, 5):
        if args.layers is not None:
            kw["L"] = args.layers
        kw["layers_per_index"] = args.layers_per_index
    if args.config == 5 and args.capacity is not None:
        kw["capacity"] = args.capacity
    if args.config == 3 and args.decode_per_turn is not None:
        kw["decode_per_turn"] = args.decode_per_turn
    if args.config == 2 and args.full_residency:
        kw["resident_tokens"] = 131072
    w = workloads.make(args.config, seed=seed, **kw)
    w.steps = max(w.steps, n_steps)
    steps = list(w.iter_steps(n_steps))
    return w, steps


class Tables:
    """The step's tables as the resolver sees them: the initial block tables edited step by step
    (page release and block reuse, new host copies), the step's contexts, and its offload pairs.
    restore() goes back to the state before the first step, so that passes replay identically."""

    def __init__(self, w, steps):
        self.w, self.steps = w, steps
        self.restore()

    def restore(self):
        self.bt = self.w.block_table.copy()
        self.hbt = self.w.host_block_table.copy()

    def edit(self, i) -> bool:
        """Apply step i's table edits; True if a table changed."""
        st = self.steps[i]
        for r, p_, v in st.bt_edits:
            self.bt[r, p_] = v
        for r, p_, v in st.hbt_edits:
            self.hbt[r, p_] = v
        return bool(len(st.bt_edits) or len(st.hbt_edits))


def subset_workload(w, steps, n_req: int):
    """The first n_req requests of a workload and of its steps, with the GPU and host blocks they use
    renumbered densely (0, 1, ... in their original order), so that byte pools for them stay small.
    Requests are independent units: their rows, hits, misses, copies and offloads are the same as in
    the whole batch, only at other block addresses.  Returns (workload, steps)."""
    import dataclasses
    from synth.workloads import Step
    if n_req >= w.R:
        return w, steps
    n = n_req
    g_used = [w.block_table[:n][w.block_table[:n] >= 0].ravel(), w.hot_blocks[:n].ravel()]
    h_used = [w.host_block_table[:n][w.host_block_table[:n] >= 0].ravel()]
    for st in steps:
        e = st.bt_edits[st.bt_edits[:, 0] < n]
        g_used.append(e[e[:, 2] >= 0, 2])
        e = st.hbt_edits[st.hbt_edits[:, 0] < n]
        h_used.append(e[e[:, 2] >= 0, 2])
        m = st.off_src[:, 0] < n if len(st.off_src) else np.zeros(0, bool)
        g_used.append(st.off_gpu[m])
        h_used.append(st.off_host[m])
        g_used.append(st.fills[st.fills[:, 1] < n, 0])
    gu = np.unique(np.concatenate([np.asarray(x, np.int64) for x in g_used]))
    hu = np.unique(np.concatenate([np.asarray(x, np.int64) for x in h_used]))
    gmap = np.full(w.num_gpu_blocks, -1, np.int64)
    gmap[gu] = np.arange(len(gu))
    hmap = np.full(max(1, w.num_host_blocks), -1, np.int64)
    hmap[hu] = np.arange(len(hu))

    def remap(a, m):
        a = np.asarray(a)
        out = a.astype(np.int64).copy()
        ok = a >= 0
        out[ok] = m[a[ok]]
        return out.astype(a.dtype)

    def remap_edits(e, m):
        e = e[e[:, 0] < n].copy()
        e[:, 2] = remap(e[:, 2], m)
        return e

    bt = remap(w.block_table[:n], gmap)
    hbt = remap(w.host_block_table[:n], hmap)
    keep_g = w.gpu_resident_init[w.gpu_resident_init[:, 0] < n]
    keep_h = w.host_resident_init[w.host_resident_init[:, 0] < n]
    sub = dataclasses.replace(w, R=n, block_table=bt, host_block_table=hbt, content_page=w.content_page[:n],
                              hot_blocks=remap(w.hot_blocks[:n], gmap), ctx_len=w.ctx_len[:n],
                              num_gpu_blocks=max(1, len(gu)), num_host_blocks=len(hu),
                              host_resident_init=keep_h, gpu_resident_init=keep_g)
    out = []
    for st in steps:
        m = st.off_src[:, 0] < n if len(st.off_src) else np.zeros(0, bool)
        fills = st.fills[st.fills[:, 1] < n].copy()
        fills[:, 0] = remap(fills[:, 0], gmap)
        out.append(Step(index=st.index, topk=np.ascontiguousarray(st.topk[:, :n]), ctx_len=st.ctx_len[:n].copy(),
                        bt_edits=remap_edits(st.bt_edits, gmap), hbt_edits=remap_edits(st.hbt_edits, hmap),
                        fills=fills, off_gpu=remap(st.off_gpu[m], gmap).astype(np.int32),
                        off_host=remap(st.off_host[m], hmap).astype(np.int32), off_src=st.off_src[m]))
    return sub, out


def oracle_requests(w, steps, pool_gb: float) -> int:
    """How many leading requests the oracle legs take: all of them when their byte pools (GPU mirror
    and host pool, every layer) fit in pool_gb, else proportionally fewer (at least one)."""
    total = w.L * (w.num_gpu_blocks + max(1, w.num_host_blocks)) * w.S * w.B
    if total <= pool_gb * 1e9:
        return w.R
    return max(1, min(w.R, int(w.R * pool_gb * 1e9 / total)))


def measured_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        d = json.load(open(p))
        return float(d["hbm_gbs"]), "measured"
    except Exception:
        return FALLBACK_HBM_GBS, "fallback"


def traffic_record(kernel: str, src: str, rows: int):
    """DRAM bytes per launch of `kernel` from a committed ncu summary, if it was taken on the current
    kernel source: as captured when the capture processed `rows` rows, else scaled by rows when the
    summary says its traffic grows in proportion to the rows (a smaller case of the same workload)."""
    p = os.path.join(ROOT, "profiles", "ncu_traffic.json")
    try:
        recs = json.load(open(p))[kernel]
    except Exception:
        return None
    sha = hashlib.sha256(open(os.path.join(ROOT, "sparse_mla_kv_gb300", "csrc", src), "rb").read()).hexdigest()
    recs = recs if isinstance(recs, list) else [recs]
    for d in recs:
        if d.get("source_sha256") != sha:
            continue
        if d.get("rows") == rows:
            return dict(d, source=d.get("capture", "ncu"))
    for d in recs:
        if d.get("source_sha256") == sha and d.get("scales_with_rows") and d.get("rows"):
            return dict(d, dram_bytes_per_launch=d["dram_bytes_per_launch"] * rows / d["rows"],
                        source=f"{d.get('capture', 'ncu')}, scaled by rows ({d['rows']} -> {rows})")
    return None


class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.path = os.path.join("/tmp", f"hs_clocks_{os.getpid()}.csv")
        try:
            self.f = open(self.path, "w")
            self.p = subprocess.Popen(["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                                       "-i", str(gpu_index), "-lms", "100"], stdout=self.f, stderr=subprocess.DEVNULL)
        except Exception:
            self.p = None

    def stop(self):
        if self.p is None:
            return None
        self.p.terminate()
        try:
            self.p.wait(timeout=5)
        except Exception:
            self.p.kill()
        self.f.close()
        rows = []
        for line in open(self.path):
            parts = [x.strip() for x in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                rows.append((float(parts[1]), float(parts[2]), parts[5:9]))
            except ValueError:
                continue
        os.unlink(self.path)
        if not rows:
            return None
        mx = max(r[1] for r in rows)
        loaded = [r for r in rows if r[0] > 0.5 * mx] or rows
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in loaded for i, v in enumerate(r[2]) if v.lower() == "active"})
        return {"sm_mhz": statistics.median(r[0] for r in loaded), "sm_max_mhz": mx, "reasons": reasons,
                "samples": len(rows), "window": "soak + timed steps"}


# ----------------------------------------------------------------------------- the CPU oracle leg
def oracle_step(o, w, tb, st, pools, hosts, tok, stamp, threads):
    """One step through the oracle: resolve with miss copies, gather, and the step's offload."""
    S, B = w.S, w.B
    rows, _ = o.resolve(S=S, B=B, num_gpu_blocks=w.num_gpu_blocks, num_host_blocks=w.num_host_blocks, topk=st.topk,
                        block_table=tb.bt, host_block_table=tb.hbt, ctx_len=st.ctx_len, max_pages=w.max_pages,
                        C=w.C, hot_blocks=w.hot_blocks, slot_token=tok, slot_stamp=stamp, step=st.index,
                        pools=pools, hosts=hosts, threads=threads, layers_per_index=w.G)
    o.gather(B=B, num_rows=w.num_gpu_blocks * S, pools=pools,
             rows=np.repeat(rows.reshape(w.L // w.G, -1), w.G, axis=0), threads=threads)
    if len(st.off_gpu):
        o.offload(S=S, B=B, num_gpu_blocks=w.num_gpu_blocks, num_host_blocks=w.num_host_blocks, pools=pools,
                  hosts=hosts, gpu_blocks=st.off_gpu, host_blocks=st.off_host)


def oracle_run(w, steps, seconds: float, threads=None):
    """Time the oracle (resolve with byte pools + gather + offload) over the workload's steps,
    restarting from an empty hot state and the initial tables until `seconds` have passed.  Pools hold
    a constant byte pattern (the bytes do not change the work).  Returns (rows/s, steps timed,
    threads)."""
    import oracle
    threads = threads or oracle.default_threads()
    S, B = w.S, w.B
    pools = [np.full(w.num_gpu_blocks * S * B, 7, np.uint8) for _ in range(w.L)]
    hosts = [np.full(max(1, w.num_host_blocks) * S * B, 9, np.uint8) for _ in range(w.L)]
    tb = Tables(w, steps)
    done = 0
    t_total = 0.0
    while t_total < seconds:
        tb.restore()
        tok = np.full((w.L // w.G, w.R, w.C), -1, np.int32)
        stamp = np.full((w.L // w.G, w.R, w.C), -1, np.int32)
        for i, st in enumerate(steps):
            tb.edit(i)
            t0 = time.perf_counter()
            oracle_step(oracle, w, tb, st, pools, hosts, tok, stamp, threads)
            t_total += time.perf_counter() - t0
            done += 1
            if t_total >= seconds:
                break
    return done * w.rows_per_step / t_total, done, threads


def run_reference(args, ws, rank):
    if rank != 0:
        return 0
    import oracle
    oracle.build()
    w_full, steps_full = make_workload(args, args.seed, args.warmup + args.steps)
    n_req = oracle_requests(w_full, steps_full, args.oracle_pool_gb)
    w, steps = subset_workload(w_full, steps_full, n_req)
    threads = oracle.default_threads()
    S, B = w.S, w.B
    pools = [np.full(w.num_gpu_blocks * S * B, 7, np.uint8) for _ in range(w.L)]
    hosts = [np.full(max(1, w.num_host_blocks) * S * B, 9, np.uint8) for _ in range(w.L)]
    tok = np.full((w.L // w.G, w.R, w.C), -1, np.int32)
    stamp = np.full((w.L // w.G, w.R, w.C), -1, np.int32)
    tb = Tables(w, steps)
    t_timed = 0.0
    for i, st in enumerate(steps):   # warm-up steps untimed, then exactly `steps` timed steps
        tb.edit(i)
        t0 = time.perf_counter()
        oracle_step(oracle, w, tb, st, pools, hosts, tok, stamp, threads)
        dt = time.perf_counter() - t0
        if i >= args.warmup:
            t_timed += dt
    value = args.steps * w.rows_per_step / t_timed
    part = "" if n_req == w_full.R else (f", on its first {n_req} of {w_full.R} requests (block ids renumbered; "
                                          f"{w.rows_per_step} of {w_full.rows_per_step} rows per step)")
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * t_timed / args.steps,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "u8", "data": "synthetic",
        "config": config_dict(w_full, args),
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": threads, "kind": "oracle",
                         "sample": f"{args.steps} timed steps of the workload (after {args.warmup} warm-up){part}; "
                                   "resolve with miss copies + gather + offload, host cores"},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


def config_dict(w, args):
    names = {1: "tiny decode", 2: "mixed-residency decode batch", 3: "multi-turn agentic decode",
             4: "no-residency cold start (prefix reuse)", 5: "max batch with MTP3"}
    share = f", IndexShare {w.G} layers per indexer" if w.G > 1 else ""
    if w.cfg == 2 and getattr(args, "full_residency", False):
        share += ", full residency"
    return {"workload": f"{names[w.cfg]}: {w.L} layer(s){share}, {w.R} requests, ctx {int(w.ctx_len[0])}, "
                        f"page {w.S}, row {w.B} B, K={w.K}, P={w.P}, hot {w.C} rows/request",
            "layers": w.L, "layers_per_index": w.G, "requests": w.R, "ctx": int(w.ctx_len[0]), "page": w.S,
            "row_bytes": w.B, "K": w.K, "P": w.P, "hot_rows": w.C, "rows_per_step": w.rows_per_step,
            "seed": args.seed, "index_dtype": "int32",
            "offload": "one hs_offload_pages launch per step for the pages it completes (all layers), timed",
            "l2": "flushed (256 MB write) before every timed step, outside the timing",
            "path": getattr(args, "path", "fused"), "timing": "eager C-ABI calls, CUDA events on the launch stream",
            "warmup_passes": getattr(args, "passes", 2)}


# ----------------------------------------------------------------------------- the GPU leg
def run_ours(args, ws, rank, local):
    dist = dist_init(ws)
    dev = torch.device(f"cuda:{local}")
    torch.cuda.set_device(dev)
    from sparse_mla_kv_gb300 import _build
    if rank == 0 or ws == 1:
        _build.build()
    barrier(dist)
    import sparse_mla_kv_gb300 as hs
    from synth import device as sdev

    W, K = args.warmup, args.steps
    w, steps = make_workload(args, rank_seed(args.seed, rank), W + K)
    L, G, R, P, Kk, C, S, B = w.L, w.G, w.R, w.P, w.K, w.C, w.S, w.B
    NG = L // G   # resolver units per request: index groups
    gpu = [torch.empty((w.num_gpu_blocks, S, B), dtype=torch.uint8, device=dev) for _ in range(L)]
    host = [sdev.pinned_empty((max(1, w.num_host_blocks), S, B)) for _ in range(L)]
    for l in range(L):
        sdev.fill_gpu_pool(w, l, gpu[l])
        sdev.fill_host_pool(w, l, host[l], dev)
    pool = hs.Pool(gpu, host)
    order_modes = {"auto": hs.MISS_ORDER_AUTO, "on": hs.MISS_ORDER_ON, "off": hs.MISS_ORDER_OFF,
                   "ranges": hs.MISS_ORDER_RANGES, "spread": hs.MISS_ORDER_SPREAD}
    pool.set_miss_order(order_modes[args.miss_order])
    pool.set_miss_warps(args.miss_warps)
    prefetch_mode = hs.MISS_PREFETCH_ON if args.miss_prefetch == "on" else hs.MISS_PREFETCH_OFF
    pool.set_miss_prefetch(prefetch_mode)
    from sparse_mla_kv_gb300.hostmem import huge_page_fraction
    huge_frac = [round(huge_page_fraction(h), 4) for h in host]
    tb = Tables(w, steps)
    bt = torch.from_numpy(tb.bt).to(dev)
    hbt = torch.from_numpy(tb.hbt).to(dev)
    # pinned staging for the tables' per-step uploads (a copy from pageable memory can go through the
    # device's translation of host memory, which the step's zero-copy misses depend on)
    bt_stage = torch.empty(tuple(bt.shape), dtype=torch.int32, pin_memory=True)
    hbt_stage = torch.empty(tuple(hbt.shape), dtype=torch.int32, pin_memory=True)
    ctx = torch.from_numpy(w.ctx_len.astype(np.int32)).to(dev)
    hot = hs.HotState.allocate(L, torch.from_numpy(w.hot_blocks).to(dev), C, layers_per_index=G)
    hs.hot_reset(pool, hot)
    topk_all = torch.from_numpy(np.stack([st.topk for st in steps])).to(dev)   # inputs resident in HBM
    ctx_all = torch.from_numpy(np.stack([st.ctx_len.astype(np.int32) for st in steps])).to(dev)
    off_g = [torch.from_numpy(st.off_gpu.astype(np.int32)).to(dev) for st in steps]
    off_h = [torch.from_numpy(st.off_host.astype(np.int32)).to(dev) for st in steps]
    # the step's results in one device buffer (rows, then stats), so a caller reads them back in one copy
    n_rows_dev = NG * R * P * Kk
    res_dev = torch.empty(n_rows_dev + NG * R * 4, dtype=torch.int32, device=dev)
    out_rows = res_dev[:n_rows_dev].view(NG, R, P, Kk)
    out_stats = res_dev[n_rows_dev:].view(NG, R, 4)
    ws_buf = hs.alloc_workspace(NG, R, P, Kk, C, dev)
    host_total = L * max(1, w.num_host_blocks) * S * B
    miss_order = ("per-unit lists" if not hs.miss_order_used(pool, hot, L, R, P, Kk, ws_buf.numel())
                  else "host-address buckets, " + ("range schedule" if args.miss_order == "ranges" or
                                                   (host_total >= (40 << 30) and args.miss_order != "spread")
                                                   else "spread schedule"))
    gout = torch.empty((L, R * P * Kk, B), dtype=torch.uint8, device=dev)
    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream()
    prep = hs.PreparedStep(pool, hot, bt, hbt, ctx, out_rows, out_stats, ws_buf, gout)

    # host-link bandwidth (bulk pinned copies, both directions) for the step roofline: measured after the
    # timed passes, the best of several trials, so that a host whose first reads of fresh pinned memory
    # are slow does not lower the peak
    def link_peaks():
        hbuf = torch.empty(256 << 20, dtype=torch.uint8, pin_memory=True)
        dbuf = torch.empty(256 << 20, dtype=torch.uint8, device=dev)

        def copy_rate(dst, src):
            best = 0.0
            for _ in range(5):
                dst.copy_(src, non_blocking=True)
                torch.cuda.synchronize()
                e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                e0.record()
                for _ in range(4):
                    dst.copy_(src, non_blocking=True)
                e1.record()
                e1.synchronize()
                best = max(best, 4 * (256 << 20) / (e0.elapsed_time(e1) * 1e-3) / 1e9)
            return best

        return copy_rate(dbuf, hbuf), copy_rate(hbuf, dbuf)

    fused = args.path == "fused"

    # One bulk DMA read of the whole pinned host pool through the GPU before anything is timed: the
    # first GPU accesses to freshly pinned host pages are slow (their GPU mappings are set up on
    # first use), which a long-running server pays once, not per step.
    if not args.no_prefault:
        scratch = torch.empty(64 << 20, dtype=torch.uint8, device=dev)
        for h in host:
            flat = h.view(-1)
            for o in range(0, flat.numel(), scratch.numel()):
                n_ = min(scratch.numel(), flat.numel() - o)
                scratch[:n_].copy_(flat[o:o + n_], non_blocking=True)
        torch.cuda.synchronize()
        del scratch

    def restore():
        """Back to the state before the first step: tables, contexts and empty hot buffers."""
        tb.restore()
        torch.cuda.current_stream().synchronize()
        np.copyto(bt_stage.numpy(), tb.bt)
        np.copyto(hbt_stage.numpy(), tb.hbt)
        bt.copy_(bt_stage, non_blocking=True)
        hbt.copy_(hbt_stage, non_blocking=True)
        hs.hot_reset(pool, hot)

    def before(i, upload_tables=True):
        """Step i's inputs that come from outside the hot path, applied before its timed events:
        table edits (released pages, reused blocks, new host copies), the model's writes of the pages
        that start, and the step's contexts."""
        st = steps[i]
        changed = tb.edit(i)
        if changed and upload_tables:
            torch.cuda.current_stream().synchronize()   # the staging buffers' previous upload has landed
            np.copyto(bt_stage.numpy(), tb.bt)
            np.copyto(hbt_stage.numpy(), tb.hbt)
            bt.copy_(bt_stage, non_blocking=True)
            hbt.copy_(hbt_stage, non_blocking=True)
        if len(st.fills):
            blocks = st.fills[:, 0].astype(np.int64)
            owners = st.fills[:, 1:].astype(np.int64)
            for l in range(L):
                sdev.fill_blocks(w, l, gpu[l], blocks, owners, dev)
        ctx.copy_(ctx_all[i])
        return changed

    def phase1(i):
        (prep.plan if fused else prep.resolve)(topk_all[i], steps[i].index)

    def phase2():
        (prep.gather_planned if fused else prep.gather)()

    def phase3(i):
        prep.offload(off_g[i], off_h[i], len(steps[i].off_gpu))

    # warm-up: one untimed pass over the warm-up AND the timed steps, then the state is restored and
    # the warm-up steps replayed, so the timed steps start from exactly the state they would have had.
    # The timed steps' host rows have then been read through the GPU once, as in a long-running
    # server; right after another process unpins a large amount of host memory, the first GPU reads
    # of pinned pages can stall for milliseconds for a few seconds (--passes 1 skips the first pass).
    for p_ in range(args.passes):
        restore()
        for i in range(W + (K if p_ + 1 < args.passes else 0)):
            before(i)
            phase1(i)
            phase2()
            phase3(i)
        torch.cuda.synchronize()
        st_w = out_stats.cpu().numpy()
        assert (st_w[..., 0] == 0).all(), "warm-up step reported a data error"

    # clock soak: the last warm-up step's gather again and again (it rewrites the same bytes, so the
    # workload state does not change), each after an L2 flush, so the HBM and the host link carry this
    # step's traffic while the clocks settle and the sampler sees the GPU under load
    sampler = ClockSampler(local) if rank == 0 and not args.no_clocks else None
    host_pool_bytes = L * max(1, w.num_host_blocks) * S * B
    soak = args.soak_seconds if args.soak_seconds is not None else (5.0 if host_pool_bytes >= 16 << 30 else 1.5)
    t_end = time.time() + soak
    while time.time() < t_end:
        for _ in range(20):
            flush.fill_(1)
            phase2()
        torch.cuda.synchronize()

    stats_all = torch.empty((K, NG, R, 4), dtype=torch.int32, device=dev)

    def timed_pass(split: bool):
        """The K timed steps, each behind an L2 flush and bracketed by CUDA events on the launch
        stream.  split=False: events around the whole step only, so the gather launch overlaps the
        resolver's tail (programmatic dependent launch); split=True: events between the calls too,
        which time each separately at the cost of that overlap."""
        ev = [[torch.cuda.Event(enable_timing=True) for _ in range(4)] for _ in range(K)]
        for k in range(K):
            i = W + k
            before(i)
            flush.fill_(k & 0xFF)
            ev[k][0].record(stream)
            phase1(i)
            if split:
                ev[k][1].record(stream)
            phase2()
            if split:
                ev[k][3].record(stream)
            phase3(i)
            ev[k][2].record(stream)
            stats_all[k].copy_(out_stats, non_blocking=True)   # after the step's events: not timed
            if not args.run_ahead:
                ev[k][2].synchronize()
        torch.cuda.synchronize()
        return ev

    def replay_warmup():
        restore()
        for i in range(W):
            before(i)
            phase1(i)
            phase2()
            phase3(i)
        torch.cuda.synchronize()

    # settle: untimed passes over the timed steps until two in a row agree within 5% (at most
    # --settle-seconds).  On host pools of tens of GB the first seconds after pinning read unevenly
    # on some machines; a long-running server sees the settled rate.
    settle_medians = []
    t_settle = time.time()
    while True:
        replay_warmup()
        ev_u = timed_pass(split=False)
        settle_medians.append(statistics.median(ev_u[k][0].elapsed_time(ev_u[k][2]) for k in range(K)))
        if len(settle_medians) >= 2 and abs(settle_medians[-1] - settle_medians[-2]) <= 0.05 * settle_medians[-2]:
            break
        if time.time() - t_settle > args.settle_seconds:
            break

    replay_warmup()
    barrier(dist)
    torch.cuda.synchronize()
    n_launch0 = hs.launch_count()
    wall0 = time.perf_counter()
    ev = timed_pass(split=False)
    wall = time.perf_counter() - wall0
    barrier(dist)
    # our kernels inside the timed region (the model's page writes are torch's, not ours)
    launches = hs.launch_count() - n_launch0
    clocks = sampler.stop() if sampler else None
    t_step = [ev[k][0].elapsed_time(ev[k][2]) * 1e-3 for k in range(K)]
    st_all = stats_all.cpu().numpy()
    assert (st_all[..., 0] == 0).all(), "a timed step reported a data error"

    # second pass over the same steps for the per-call split (roofline of the gather): the state is
    # restored and the warm-up steps replayed, so each timed step starts from the same state again
    restore()
    for i in range(W):
        before(i)
        phase1(i)
        phase2()
        phase3(i)
    torch.cuda.synchronize()
    ev_s = timed_pass(split=True)
    assert np.array_equal(stats_all.cpu().numpy(), st_all), "the split pass resolved differently"
    t_res = [ev_s[k][0].elapsed_time(ev_s[k][1]) * 1e-3 for k in range(K)]
    t_gat = [ev_s[k][1].elapsed_time(ev_s[k][3]) * 1e-3 for k in range(K)]
    t_off = [ev_s[k][3].elapsed_time(ev_s[k][2]) * 1e-3 for k in range(K)]
    t_step_split = [ev_s[k][0].elapsed_time(ev_s[k][2]) * 1e-3 for k in range(K)]

    # graph pass: the same timed steps, each captured as one CUDA graph (untimed; its kernels and
    # arguments fixed at capture, the tables read at replay) and replayed once behind an L2 flush, the
    # replay bracketed by events.  The host enqueues one graph instead of the step's C-ABI calls.
    timing = args.timing
    if timing == "auto":
        timing = "both" if host_pool_bytes < (16 << 30) else "eager"
    graph = None
    if timing in ("graph", "both"):
        replay_warmup()
        n0 = hs.launch_count()
        graphs = []
        for k in range(K):
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g):
                phase1(W + k)
                phase2()
                phase3(W + k)
            graphs.append(g)
        nodes = hs.launch_count() - n0
        stats_g = torch.empty_like(stats_all)
        ev_g = [[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in range(K)]
        for k in range(K):
            before(W + k)
            flush.fill_(k & 0xFF)
            ev_g[k][0].record(stream)
            graphs[k].replay()
            ev_g[k][1].record(stream)
            stats_g[k].copy_(out_stats, non_blocking=True)
            ev_g[k][1].synchronize()
        torch.cuda.synchronize()
        assert np.array_equal(stats_g.cpu().numpy(), st_all), "the graph replays resolved differently"
        t_graph = [ev_g[k][0].elapsed_time(ev_g[k][1]) * 1e-3 for k in range(K)]
        sum_g = max_over_ranks(dist, float(sum(t_graph)), dev)
        graph = {"value": ws * w.rows_per_step * K / sum_g, "unit": UNIT, "ms_per_step": 1e3 * sum_g / K,
                 "step_us_median": 1e6 * statistics.median(t_graph), "kernels_per_step": nodes / K,
                 "timing": "each timed step captured as one CUDA graph, replayed once behind an L2 flush; "
                           "events around the replay"}
        del graphs
    schedule_ab = None
    if args.schedule_ab and hs.miss_order_used(pool, hot, L, R, P, Kk, ws_buf.numel()):
        # whole timed passes over the same steps, alternating the two schedules of the ordered layout (each
        # pass plans and gathers in one mode), so both see the same machine state
        sums = {"ranges": [], "spread": []}
        steps_med = {"ranges": [], "spread": []}
        for rnd in range(args.schedule_ab):
            for name, mode in (("ranges", hs.MISS_ORDER_RANGES), ("spread", hs.MISS_ORDER_SPREAD)):
                pool.set_miss_order(mode)
                replay_warmup()
                ev_ab = timed_pass(split=False)
                ts = [ev_ab[k][0].elapsed_time(ev_ab[k][2]) * 1e-3 for k in range(K)]
                sums[name].append(1e3 * sum(ts) / K)
                steps_med[name].append(1e6 * statistics.median(ts))
        pool.set_miss_order(order_modes[args.miss_order])
        schedule_ab = {"rounds": args.schedule_ab,
                       "ms_per_step": {k: [round(x, 3) for x in v] for k, v in sums.items()},
                       "step_us_median": {k: [round(x, 1) for x in v] for k, v in steps_med.items()},
                       "how": "per round, one timed pass (the K timed steps after the warm-up replay) with each "
                              "schedule of the ordered miss layout; mean step time of each pass"}
    prefetch_ab = None
    if args.prefetch_ab:
        # whole timed passes over the same steps, alternating the resolver's miss prefetch off and on
        sums = {"off": [], "on": []}
        steps_med = {"off": [], "on": []}
        for rnd in range(args.prefetch_ab):
            for name, mode in (("off", hs.MISS_PREFETCH_OFF), ("on", hs.MISS_PREFETCH_ON)):
                pool.set_miss_prefetch(mode)
                replay_warmup()
                ev_ab = timed_pass(split=False)
                ts = [ev_ab[k][0].elapsed_time(ev_ab[k][2]) * 1e-3 for k in range(K)]
                sums[name].append(1e3 * sum(ts) / K)
                steps_med[name].append(1e6 * statistics.median(ts))
        pool.set_miss_prefetch(prefetch_mode)
        prefetch_ab = {"rounds": args.prefetch_ab, "miss_order": miss_order,
                       "ms_per_step": {k: [round(x, 4) for x in v] for k, v in sums.items()},
                       "step_us_median": {k: [round(x, 1) for x in v] for k, v in steps_med.items()},
                       "how": "per round, one timed pass (the K timed steps after the warm-up replay) with the "
                              "miss prefetch off, then on; mean and median step time of each pass"}
    miss_warps_ab = None
    if args.miss_warps_ab and fused:
        # the last timed step's plan stays in the workspace: replaying hs_gather_planned rewrites the same
        # bytes (hot slots and outputs), so each replay is the same gather with another miss-warp count
        reps = max(5, K)
        t_mw = {0: [], 1: [], 2: []}
        for rep in range(reps + 1):
            for mwc in (0, 1, 2):
                pool.set_miss_warps(mwc)
                flush.fill_(rep & 0xFF)
                e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                e0.record(stream)
                phase2()
                e1.record(stream)
                e1.synchronize()
                if rep:
                    t_mw[mwc].append(e0.elapsed_time(e1) * 1e-3)
        pool.set_miss_warps(args.miss_warps)
        miss_warps_ab = {"repeats": reps, "miss_order": miss_order,
                         "gather_us_median_partition": 1e6 * statistics.median(t_mw[0]),
                         "gather_us_median_1": 1e6 * statistics.median(t_mw[1]),
                         "gather_us_median_2": 1e6 * statistics.median(t_mw[2]),
                         "how": "hs_gather_planned of the last timed step replayed with the SM partition and with 1 "
                                "and 2 miss warps in every CTA (hs_pool_set_miss_warps 0, 1, 2), alternating behind "
                                "L2 flushes; medians"}
    miss_sm_ab = None
    if args.miss_sm_ab and fused:
        # the same replay as the miss-warp A/B, with the SM partition at each divisor
        divs = [int(x) for x in args.miss_sm_ab.split(",") if x.strip()]   # -1: no miss SM
        reps = max(5, K)
        t_div = {d: [] for d in divs}
        pool.set_miss_warps(0)
        for rep in range(reps + 1):
            for dv in divs:
                pool.set_miss_sm_divisor(dv)
                flush.fill_(rep & 0xFF)
                e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                e0.record(stream)
                phase2()
                e1.record(stream)
                e1.synchronize()
                if rep:
                    t_div[dv].append(e0.elapsed_time(e1) * 1e-3)
        pool.set_miss_sm_divisor(0)
        pool.set_miss_warps(args.miss_warps)
        miss_sm_ab = {"repeats": reps, "miss_order": miss_order,
                      "gather_us_median": {str(d): round(1e6 * statistics.median(t_div[d]), 1) for d in divs},
                      "how": "hs_gather_planned of the last timed step replayed with the SM partition, every divisor-th "
                             "SM copying misses (hs_pool_set_miss_sm_divisor), alternating behind L2 flushes; medians"}
    gather_phases = None
    if args.gather_phases and fused:
        # the last timed step's planned gather replayed in the SM partition with device timestamps: start,
        # the last HBM-row CTA's end, the last miss warp's end and the last CTA's end (globaltimer, ns)
        ts = torch.zeros(4, dtype=torch.int64, device=dev)
        pool.set_phase_timestamps(ts)
        pool.set_miss_warps(0)
        reps = max(5, K)
        rec = []
        for rep in range(reps + 1):
            ts.zero_()
            ts[0] = -1   # all ones: the atomic minimum of the CTAs' starts
            flush.fill_(rep & 0xFF)
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            phase2()
            e1.record(stream)
            e1.synchronize()
            t = ts.cpu().tolist()
            if rep and t[3] > 0:
                rec.append((e0.elapsed_time(e1) * 1e3, (t[1] - t[0]) / 1e3 if t[1] else None,
                            (t[2] - t[0]) / 1e3 if t[2] else None, (t[3] - t[0]) / 1e3))
        pool.set_phase_timestamps(None)
        pool.set_miss_warps(args.miss_warps)

        def med(j):
            v = [r[j] for r in rec if r[j] is not None]
            return round(statistics.median(v), 1) if v else None
        gather_phases = {"repeats": len(rec), "miss_order": miss_order, "event_us": med(0), "hbm_rows_done_us": med(1),
                         "misses_done_us": med(2), "kernel_us": med(3),
                         "how": "hs_gather_planned of the last timed step replayed in the SM partition with "
                                "hs_pool_set_phase_timestamps; medians of the device timestamps relative to the first "
                                "CTA's start, and of the events around the launch"}
    planes_ab = None
    if args.planes_ab and B == 656:
        # the last timed step's gather (planned gather when fused, plain gather of its rows otherwise)
        # replayed with each output layout; the bytes differ only in their order
        rows_p = out_rows.reshape(NG, -1)
        reps = max(5, K)
        t_pl = {"rows": [], "planes": []}
        for rep in range(reps + 1):
            for name, pl in (("rows", ()), ("planes", (512, 16, 128))):
                pool.set_gather_planes(pl)
                flush.fill_(rep & 0xFF)
                e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                e0.record(stream)
                if fused:
                    phase2()
                else:
                    for l in range(L):
                        hs.gather_rows(pool, rows_p[l // G], layer_begin=l, out=gout[l])
                e1.record(stream)
                e1.synchronize()
                if rep:
                    t_pl[name].append(e0.elapsed_time(e1) * 1e-3)
        pool.set_gather_planes(())
        planes_ab = {"repeats": reps, "path": args.path,
                     "gather_us_median": {k: round(1e6 * statistics.median(v), 1) for k, v in t_pl.items()},
                     "how": "the last timed step's gather replayed with the output in rows and in planes "
                            "{512, 16, 128} (hs_pool_set_gather_planes), alternating behind L2 flushes; medians"}
    gather_ab = None
    if args.gather_ab:
        # the plain gather of the last timed step's rows, every layer of each index group reading its
        # group's rows, with each copy mode in turn; the pool's misses are filled by then (stream order)
        rows_l = out_rows.reshape(NG, -1)
        reps = max(5, K)
        t_ab = {hs.GATHER_COPY_LOADS: [], hs.GATHER_COPY_BULK: []}
        for rep in range(reps + 1):
            for mode in (hs.GATHER_COPY_LOADS, hs.GATHER_COPY_BULK):
                pool.set_gather_copy(mode)
                flush.fill_(rep & 0xFF)
                e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                e0.record(stream)
                for l in range(L):
                    hs.gather_rows(pool, rows_l[l // G], layer_begin=l, out=gout[l])
                e1.record(stream)
                e1.synchronize()
                if rep:   # the first round is a warm-up
                    t_ab[mode].append(e0.elapsed_time(e1) * 1e-3)
        pool.set_gather_copy(hs.GATHER_COPY_LOADS)
        ab_bytes = L * R * P * Kk * (2 * B + 4)
        gather_ab = {"rows": L * R * P * Kk, "algorithmic_bytes": ab_bytes, "repeats": reps,
                     "loads_us_median": 1e6 * statistics.median(t_ab[hs.GATHER_COPY_LOADS]),
                     "bulk_us_median": 1e6 * statistics.median(t_ab[hs.GATHER_COPY_BULK]),
                     "loads_gbs": ab_bytes / statistics.median(t_ab[hs.GATHER_COPY_LOADS]) / 1e9,
                     "bulk_gbs": ab_bytes / statistics.median(t_ab[hs.GATHER_COPY_BULK]) / 1e9,
                     "how": "hs_gather_rows of the last timed step's rows, one call per layer, the two copy "
                            "modes alternating behind L2 flushes; medians"}
    h2d_gbs, d2h_gbs = link_peaks()

    sum_t = max_over_ranks(dist, float(sum(t_step)), dev)
    counts = st_all[..., 1:].sum(axis=(1, 2))           # [K][resident, hits, misses]
    hits_misses = counts.sum(axis=0)

    rows_per_step = w.rows_per_step
    value = ws * rows_per_step * K / sum_t
    ms_per_step = 1e3 * sum_t / K
    headline_timing = "eager C-ABI calls, CUDA events on the launch stream"
    t_head = t_step
    if timing == "graph":
        t_head = t_graph
        value, ms_per_step = graph["value"], graph["ms_per_step"]
        launches = int(round(graph["kernels_per_step"] * K))
        headline_timing = graph["timing"]

    # roofline of the dominant kernel (the gather; fused path: the gather that also carries the miss
    # copies): algorithmic HBM bytes per launch / mean launch time from the events around it.
    # Per gathered row: 656 B out + 4 B row id (+ 4 B host source when fused) + 656 B row read from
    # HBM -- or, for a miss in the fused path, 656 B read over the host link and 656 B into its slot.
    # Under IndexShare every layer of a group gathers, and copies, the group's rows.
    hbm_peak, peak_kind = measured_peaks()
    n_rows = L * R * P * Kk
    m_mean = float(counts[:, 2].mean())
    gather_bytes = n_rows * (2 * B + (8 if fused else 4))
    t_g = statistics.fmean(t_gat)
    # the fused gather's kernel: with the range schedule and the SM partition (the default for it) the
    # partition kernel, else the mixed kernel
    partition = fused and ((miss_order.endswith("range schedule") and args.miss_warps <= 0) or
                           (miss_order == "per-unit lists" and args.miss_warps == 0))
    gkernel = "gather_partition_kernel" if partition else ("gather_fused_kernel" if fused else "gather_kernel")
    tr = traffic_record(gkernel, "gather.cu", n_rows)
    # The fused gather moves its miss rows over the host link while it streams the other rows from HBM:
    # its roof is the slower of the two, each against its own peak -- HBM against the measured copy
    # peak, the host link against this run's bulk pinned host-to-device copy rate (MEASURED_PEAKS
    # holds no link figure)
    link_bytes = m_mean * G * B if fused else 0.0
    t_hbm_roof = gather_bytes / (hbm_peak * 1e9)
    t_link_roof = link_bytes / (h2d_gbs * 1e9)
    hbm_part = {"achieved": gather_bytes / t_g / 1e9, "peak": hbm_peak, "unit": "GB/s", "frac": t_hbm_roof / t_g,
                "peak_kind": peak_kind, "algorithmic_bytes_per_launch": gather_bytes}
    link_part = {"achieved": link_bytes / t_g / 1e9, "peak": h2d_gbs, "unit": "GB/s", "frac": t_link_roof / t_g,
                 "peak_kind": "measured in this run: bulk pinned host-to-device cudaMemcpyAsync, 256 MB, best of 5",
                 "algorithmic_bytes_per_launch": link_bytes}
    bound = "host_link" if t_link_roof > t_hbm_roof else "hbm"
    main = link_part if bound == "host_link" else hbm_part
    roofline = {"bound": bound, "kernel": gkernel,
                "achieved": main["achieved"], "peak": main["peak"], "unit": "GB/s", "frac": main["frac"],
                "peak_kind": main["peak_kind"], "algorithmic_bytes_per_launch": main["algorithmic_bytes_per_launch"],
                "timing": "mean launch time from the split pass (events between the calls)",
                "components": {"hbm": hbm_part, "host_link": link_part},
                "traffic": tr["dram_bytes_per_launch"] if tr else None,
                "traffic_source": tr.get("source") if tr else None}

    # whole-step roofline: max(HBM bytes / HBM peak, miss bytes / H2D rate, offload bytes / D2H rate),
    # step by step with each step's own miss and offload counts
    roofs, meas = [], []
    page_bytes = S * B
    for k in range(K):
        m = int(counts[k, 2]) * G
        n_off = len(steps[W + k].off_gpu) * L
        hbm_step = n_rows * (2 * B + 16) + NG * R * 8 * C + m * (B + 8) + n_off * page_bytes
        roofs.append(max(hbm_step / (hbm_peak * 1e9), m * B / (h2d_gbs * 1e9), n_off * page_bytes / (d2h_gbs * 1e9)))
        meas.append(t_head[k])
    # the post-forward offload (a9): its launches in the split pass, bytes moved over the link / time
    off_k = [k for k in range(K) if len(steps[W + k].off_gpu)]
    offload = None
    if off_k:
        off_bytes = sum(len(steps[W + k].off_gpu) * L * page_bytes for k in off_k)
        off_time = sum(t_off[k] for k in off_k)
        offload = {"launches": len(off_k), "pages_x_layers": sum(len(steps[W + k].off_gpu) * L for k in off_k),
                   "bytes": off_bytes, "achieved_gbs": off_bytes / off_time / 1e9, "d2h_peak_gbs": d2h_gbs,
                   "frac": off_bytes / off_time / 1e9 / d2h_gbs, "bound": "host link (D2H)",
                   "timing": "split pass, events around the hs_offload_pages launch"}
    step_roof = {"t_roof_us": 1e6 * statistics.fmean(roofs), "t_measured_us": 1e6 * statistics.fmean(meas),
                 "frac": sum(roofs) / sum(meas), "misses_per_step_mean": m_mean,
                 "offloaded_pages_per_step_mean": statistics.fmean(len(steps[W + k].off_gpu) for k in range(K)),
                 "h2d_gbs_measured_bulk_copy": h2d_gbs, "d2h_gbs_measured_bulk_copy": d2h_gbs, "path": args.path,
                 "step_us_median": 1e6 * statistics.median(t_head),
                 "split_pass": "phase times from a second pass over the same steps with events between the "
                               "calls (they stop the gather launch from overlapping the resolver)",
                 "phase1_us_mean": 1e6 * statistics.fmean(t_res), "phase2_us_mean": 1e6 * t_g,
                 "phase3_offload_us_mean": 1e6 * statistics.fmean(t_off),
                 "phase1_us_median": 1e6 * statistics.median(t_res), "phase2_us_median": 1e6 * statistics.median(t_gat),
                 "phase2_us_max": 1e6 * max(t_gat), "split_step_us_median": 1e6 * statistics.median(t_step_split),
                 "phase2_us_all": [round(1e6 * x, 1) for x in t_gat],
                 "step_us_all": [round(1e6 * x, 1) for x in t_head],
                 "phase1": "hs_resolve_plan" if fused else "hs_resolve_topk (resolver + miss copy)",
                 "phase2": "hs_gather_planned" if fused else "hs_gather_rows",
                 "phase3": "hs_offload_pages", "offload": offload}

    # end to end through the C ABI with host buffers: H2D of the step's top-K and contexts (one packed
    # copy) and (when the step edits them) block tables, D2H of its rows and stats (one packed copy),
    # inside the timed events
    e2e = None
    if not args.no_e2e:
        # per step, top-K ids then contexts, packed in one pinned buffer and one device buffer
        inp_host = torch.from_numpy(np.stack([np.concatenate([st.topk.reshape(-1), st.ctx_len.astype(np.int32)])
                                              for st in steps])).pin_memory()
        inp_dev = torch.empty(n_rows_dev + R, dtype=torch.int32, device=dev)
        topk_dev = inp_dev[:n_rows_dev].view(NG, R, P, Kk)
        ctx_e2e = inp_dev[n_rows_dev:]
        bt_host = torch.empty(tuple(bt.shape), dtype=torch.int32, pin_memory=True)
        hbt_host = torch.empty(tuple(hbt.shape), dtype=torch.int32, pin_memory=True)
        res_host = torch.empty(res_dev.numel(), dtype=torch.int32, pin_memory=True)
        stats_host = res_host[n_rows_dev:].view(NG, R, 4)
        prep2 = hs.PreparedStep(pool, hot, bt, hbt, ctx_e2e, out_rows, out_stats, ws_buf, gout, stream=stream)

        def e2e_step(i):
            if fused:
                prep2.resolve_gather(topk_dev, steps[i].index)
            else:
                prep2.resolve(topk_dev, steps[i].index)
                prep2.gather()
            prep2.offload(off_g[i], off_h[i], len(steps[i].off_gpu))

        restore()
        for i in range(W):
            before(i)
            inp_dev.copy_(inp_host[i], non_blocking=True)
            e2e_step(i)
        torch.cuda.synchronize()
        ev2 = [[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in range(K)]
        h2d_bytes = []
        barrier(dist)
        for k in range(K):
            i = W + k
            changed = before(i, upload_tables=False)
            if changed:
                bt_host.copy_(torch.from_numpy(tb.bt))
                hbt_host.copy_(torch.from_numpy(tb.hbt))
            flush.fill_(k & 0xFF)
            ev2[k][0].record(stream)
            inp_dev.copy_(inp_host[i], non_blocking=True)
            nb = inp_host[i].numel() * 4
            if changed:
                bt.copy_(bt_host, non_blocking=True)
                hbt.copy_(hbt_host, non_blocking=True)
                nb += 2 * bt_host.numel() * 4
            h2d_bytes.append(nb)
            e2e_step(i)
            res_host.copy_(res_dev, non_blocking=True)
            ev2[k][1].record(stream)
            ev2[k][1].synchronize()
            assert (stats_host.numpy()[..., 0] == 0).all()
        torch.cuda.synchronize()
        barrier(dist)
        t2 = max_over_ranks(dist, float(sum(ev2[k][0].elapsed_time(ev2[k][1]) * 1e-3 for k in range(K))), dev)
        e2e = {"value": ws * rows_per_step * K / t2, "unit": UNIT,
               "h2d_bytes_per_step": int(statistics.fmean(h2d_bytes)),
               "d2h_bytes_per_step": int(res_host.numel() * 4),
               "copies": "per step one H2D of top-K + contexts, one D2H of rows + stats (packed buffers)"}

    cpu = cpu1 = None
    if rank == 0 and ws == 1 and not args.no_cpu_baseline:
        import oracle
        oracle.build()
        n_req = oracle_requests(w, steps, args.oracle_pool_gb)
        w_o, steps_o = subset_workload(w, steps, n_req)
        part = "" if n_req == w.R else (f" on its first {n_req} of {w.R} requests (block ids renumbered; "
                                        f"{w_o.rows_per_step} rows per step)")
        v, n_done, thr = oracle_run(w_o, steps_o, args.cpu_seconds)
        cpu = {"value": v, "unit": UNIT, "cores": thr, "kind": "oracle",
               "sample": f"{n_done} steps of this workload{part}, restarting from an empty hot state after its "
                         f"{len(steps_o)} steps; resolve with miss copies + gather + offload, about "
                         f"{args.cpu_seconds:.0f} s of host time"}
        v1, n1, _ = oracle_run(w_o, steps_o, args.cpu_seconds / 4, threads=1)
        cpu1 = {"value": v1, "unit": UNIT, "cores": 1, "kind": "oracle",
                "sample": f"{n1} steps{part}, one host thread, about {args.cpu_seconds / 4:.0f} s"}

    if rank == 0:
        line = {
            "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": ws, "steps": K, "warmup": W,
            "ms_per_step": ms_per_step, "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "dtype": "u8", "data": "synthetic",
            "config": dict(config_dict(w, args), miss_order=miss_order, miss_prefetch=args.miss_prefetch,
                           timing=headline_timing,
                           host_pool_huge_page_fraction=huge_frac,
                           settle_passes=len(settle_medians),
                           settle_step_us_medians=[round(1e3 * m, 1) for m in settle_medians]),
            "gathered_gbs": value * B / 1e9, "roofline": roofline, "step_roofline": step_roof,
            "cpu_baseline": cpu, "cpu_baseline_1thread": cpu1, "e2e": e2e, "gpu_launches": int(launches),
            "graph_replay": graph, "gather_copy_ab": gather_ab, "miss_warps_ab": miss_warps_ab, "miss_sm_ab": miss_sm_ab, "planes_ab": planes_ab,
            "gather_phases": gather_phases,
            "schedule_ab": schedule_ab, "prefetch_ab": prefetch_ab,
            "clocks": clocks,
            "wall_s_timed_region": wall, "timed_counts": {"resident": int(hits_misses[0]),
                                                          "hits": int(hits_misses[1]),
                                                          "misses": int(hits_misses[2])},
        }
        print(json.dumps(line), flush=True)
    pool.close()
    if dist is not None:
        dist.destroy_process_group()
    return 0


def run_residency(args):
    """The residency manager's own step: R requests decode under KV pressure (the pool holds about 60%
    of what they grow to); each step appends each request's tokens, touches the pages of its top-K,
    collects the offload queue and takes the tables, fills and resets.  Timed through the native
    manager and through its oracle on the same operations."""
    import oracle.residency as ores
    from sparse_mla_kv_gb300 import _build
    _build.build()
    from sparse_mla_kv_gb300.residency import Residency
    from synth import workloads
    R, S, K, C, max_pages = args.requests or 64, 64, 2048, 4096, 1024
    ctx0, grow = 48 * S, 16
    G = int(0.6 * R * (ctx0 // S + args.steps * grow // S + C // S))
    rng = np.random.default_rng(args.seed)
    prev = [None] * R
    ops = []
    ctx = [ctx0] * R
    for t in range(args.warmup + args.steps):
        step = []
        for r in range(R):
            ctx[r] += int(rng.integers(1, 2 * grow))
            ids = workloads.next_topk(rng, prev[r], ctx[r], K, 0.8 if prev[r] is not None else 0.0, "recency")
            prev[r] = ids
            step.append((r, ctx[r], ids))
        ops.append(step)

    # the step's inputs, prepared before the timing (as the GPU leg's inputs are resident): tokens appended
    # per request and the top-K ids of all requests as one [R][K] array
    grows = []
    last = [ctx0] * R
    for step in ops:
        g = np.zeros(R, np.int32)
        for r, c, _ in step:
            g[r] = c - last[r]
            last[r] = c
        grows.append(g)
    ids_all = [np.stack([ids for _, _, ids in step]).astype(np.int32) for step in ops]

    def drive(m, native):
        for r in range(R):
            m.admit(r, ctx0)
        m.collect()
        m.take_fills()
        tab = None
        times = []
        for t in range(len(ops)):
            t0 = time.perf_counter()
            m.append_all(grows[t])
            m.take_fills()
            tab = m.tables(tab) if native else m.tables()
            m.take_resets()
            m.touch_all(ids_all[t], t)
            m.collect()
            if t >= args.warmup:
                times.append(time.perf_counter() - t0)
        return times

    t_native = drive(Residency(G, 1 << 20, S, R, max_pages, C // S), True)
    t_oracle = drive(ores.Residency(G, 1 << 20, S, R, max_pages, C // S), False)
    v = len(t_native) / sum(t_native)
    vo = len(t_oracle) / sum(t_oracle)
    print(json.dumps({
        "metric": "residency manager decode steps/s (host)", "value": v, "unit": "steps/s", "n_gpus": 0,
        "calls_per_step": "hs_res_append_all, take_fills, tables (into the previous step's arrays), take_resets, "
                          "touch_all, collect",
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 / v, "higher_is_better": True,
        "dtype": "int32", "data": "synthetic",
        "config": {"workload": f"{R} requests decoding under KV pressure, K={K} top-K touches, page {S}, "
                               f"hot {C} rows, GPU pool {G} blocks (about 60% of the demand)",
                   "requests": R, "K": K, "gpu_blocks": G},
        "cpu_baseline": {"value": vo, "unit": "steps/s", "cores": 1, "kind": "oracle",
                         "sample": "the same operations through oracle/residency.py"},
        "speedup_vs_oracle": v / vo}), flush=True)
    return 0


def run_link_probe(args):
    """Rate of the library's miss path against the span of pinned host memory its misses touch.

    One layer, 64 requests, K = 2048, hot buffers of 4096 rows, 656-byte rows, page 64.  The requests
    share one host prefix that fills a window of the pinned host pool (their host tables point at the
    same host blocks, in a seeded permutation); each request's last page is resident.  The pool has
    --probe-pool-gb of pinned, device-mapped, huge-page host memory, written by DMA from the device;
    only the window is read.  Every step empties the hot buffers first (untimed), so each of the step's
    R x K uniform top-K ids on a host page is a miss.  Per (window, miss order) the same steps are timed
    three ways with events: hs_resolve_topk (resolver + miss-copy kernel), hs_resolve_plan (the
    resolver alone) and hs_resolve_plan + hs_gather_planned (the fused gather, which carries the
    misses).  The miss copy's time is the first minus the second, step by step.  Host pools and the
    order of the reads, not the bytes, change between the rows of the table."""
    dev = torch.device("cuda:0")
    torch.cuda.set_device(dev)
    from sparse_mla_kv_gb300 import _build
    _build.build()
    import sparse_mla_kv_gb300 as hs
    from sparse_mla_kv_gb300.hostmem import pinned_host_pool
    S, B, K, C, R = 64, 656, 2048, 4096, args.requests or 64
    page = S * B
    pool_bytes = int(args.probe_pool_gb * 1e9) // page * page
    nhb = pool_bytes // page
    windows = sorted({min(nhb, int(g * 1e9) // page) for g in args.probe_windows_gb})
    host = pinned_host_pool((nhb, S, B), huge=not args.probe_base_pages)
    from sparse_mla_kv_gb300.hostmem import huge_page_fraction
    flat = host.view(-1)
    if args.probe_cpu_fill:
        # written by CPU stores (a served pool is written by DMA or GPU stores; this is the comparison)
        flat.numpy()[:] = 7
    else:
        # written by DMA from the device
        dbuf = torch.arange(1 << 30, dtype=torch.int64, device=dev).to(torch.uint8)
        for o in range(0, flat.numel(), dbuf.numel()):
            n_ = min(dbuf.numel(), flat.numel() - o)
            flat[o:o + n_].copy_(dbuf[:n_], non_blocking=True)
        torch.cuda.synchronize()
        del dbuf
    ngb = R * (C // S) + R
    gpu = torch.zeros((ngb, S, B), dtype=torch.uint8, device=dev)
    pool = hs.Pool([gpu], [host])
    hot_blocks = torch.arange(R * (C // S), dtype=torch.int32, device=dev).reshape(R, C // S)
    hot = hs.HotState.allocate(1, hot_blocks, C)
    ws_buf = hs.alloc_workspace(1, R, 1, K, C, dev)
    out_rows = torch.empty((1, R, 1, K), dtype=torch.int32, device=dev)
    out_stats = torch.empty((1, R, 4), dtype=torch.int32, device=dev)
    gout = torch.empty((1, R * K, B), dtype=torch.uint8, device=dev)
    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream()
    rng = np.random.default_rng(args.seed)
    n_steps = args.warmup + args.steps
    table = []
    for wb in windows:
        max_pages = wb + 1
        ctx_n = max_pages * S
        hrow = rng.permutation(wb).astype(np.int32)
        bt = torch.full((R, max_pages), -1, dtype=torch.int32, device=dev)
        bt[:, wb] = torch.arange(R * (C // S), R * (C // S) + R, dtype=torch.int32, device=dev)
        hbt = torch.full((R, max_pages), -1, dtype=torch.int32, device=dev)
        hbt[:, :wb] = torch.from_numpy(hrow).to(dev)[None, :]
        ctx = torch.full((R,), ctx_n, dtype=torch.int32, device=dev)
        topk = []
        for _ in range(n_steps):
            ids = np.empty((R, K), np.int32)
            for r in range(R):
                c = rng.integers(0, wb * S, size=3 * K)
                _, first = np.unique(c, return_index=True)
                ids[r] = c[np.sort(first)][:K]
            topk.append(torch.from_numpy(ids.reshape(1, R, 1, K)).to(dev))
        prep = hs.PreparedStep(pool, hot, bt, hbt, ctx, out_rows, out_stats, ws_buf, gout)
        for order, mode in (("per-unit lists", hs.MISS_ORDER_OFF), ("host-address buckets", hs.MISS_ORDER_ON)):
            pool.set_miss_order(mode)

            def timed(call):
                ts = []
                for i in range(n_steps):
                    hs.hot_reset(pool, hot)
                    flush.fill_(i & 0xFF)
                    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                    e0.record(stream)
                    call(i)
                    e1.record(stream)
                    e1.synchronize()
                    if i >= args.warmup:
                        ts.append(e0.elapsed_time(e1) * 1e3)
                return ts

            def split(i):
                prep.resolve(topk[i], 1)

            def plan(i):
                prep.plan(topk[i], 1)

            def fused(i):
                prep.plan(topk[i], 1)
                prep.gather_planned()

            med = []
            t0 = time.time()
            while True:   # settle: until two passes agree within 5% (reads of fresh pinned memory start slow)
                med.append(statistics.median(timed(split)))
                if len(med) >= 2 and abs(med[-1] - med[-2]) <= 0.05 * med[-2]:
                    break
                if time.time() - t0 > args.settle_seconds:
                    break
            t_split = timed(split)
            t_plan = timed(plan)
            t_fused = timed(fused)
            misses = int(out_stats[..., 3].sum())
            t_copy = statistics.median(a - b for a, b in zip(t_split, t_plan))
            t_fg = statistics.median(a - b for a, b in zip(t_fused, t_plan))
            table.append({"window_gb": round(wb * page / 1e9, 2), "miss_order": order, "misses_per_step": misses,
                          "resolver_us": round(statistics.median(t_plan), 1),
                          "miss_copy_us": round(t_copy, 1), "miss_copy_gbs": round(misses * B / t_copy / 1e3, 1),
                          "fused_gather_us": round(t_fg, 1), "fused_gather_miss_gbs": round(misses * B / t_fg / 1e3, 1),
                          "settle_passes": len(med)})
            print(json.dumps(table[-1]), file=sys.stderr, flush=True)
    pool.close()
    print(json.dumps({"metric": "miss-path host-link rate vs span of host memory read", "unit": "GB/s",
                      "pool_gb": round(pool_bytes / 1e9, 2), "requests": R, "K": K, "row_bytes": B,
                      "host_pages": "base pages" if args.probe_base_pages else "huge pages (madvise)",
                      "huge_page_fraction": round(huge_page_fraction(host), 4),
                      "host_fill": "CPU stores" if args.probe_cpu_fill else "DMA from the device",
                      "steps": args.steps, "warmup": args.warmup, "table": table,
                      "how": run_link_probe.__doc__.split("\n\n")[1].replace("\n", " ").strip()}), flush=True)
    return 0


def main():
    args = parse()
    ws, rank, local = dist_env()
    if args.residency:
        return run_residency(args) if rank == 0 else 0
    if args.link_probe:
        return run_link_probe(args) if rank == 0 else 0
    if args.impl == "reference":
        return run_reference(args, ws, rank)
    return run_ours(args, ws, rank, local)


if __name__ == "__main__":
    sys.exit(main())
