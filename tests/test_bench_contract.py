"""bench.py's host legs on CPU: the reference arm (the oracle timed on the host cores) prints one JSON line
with the keys the benchmark contract names, a rank-1 process of a two-rank launch exits without work, and the
residency-manager leg times the native manager and its oracle."""
import json
import os
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _run(args, env=None):
    e = dict(os.environ)
    e.update(env or {})
    return subprocess.run([sys.executable, os.path.join(ROOT, "bench.py")] + args, capture_output=True, text=True,
                          timeout=600, cwd=ROOT, env=e)


def test_reference_arm_prints_one_contract_line():
    # the default workload (the full-size MTP3 batch); the oracle takes its first requests within 1 GB
    p = _run(["--impl", "reference", "--steps", "2", "--warmup", "3", "--oracle-pool-gb", "1"])
    assert p.returncode == 0, p.stderr[-2000:]
    lines = [l for l in p.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1
    d = json.loads(lines[0])
    for key in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step", "higher_is_better", "scaling",
                "vs_baseline", "dtype", "data", "config", "cpu_baseline", "e2e"):
        assert key in d, key
    assert d["impl"] == "reference" and d["steps"] == 2 and d["warmup"] == 3 and d["n_gpus"] == 1
    assert d["value"] > 0 and d["unit"] == "rows/s" and d["higher_is_better"] is True
    assert d["cpu_baseline"]["kind"] == "oracle" and d["cpu_baseline"]["cores"] >= 1
    assert d["e2e"]["value"] == d["value"] and d["e2e"]["h2d_bytes_per_step"] == 0
    assert "workload" in d["config"] and d["config"]["requests"] == 256 and d["config"]["P"] == 4
    assert "first" in d["cpu_baseline"]["sample"]   # a stated subset of the requests


def test_reference_arm_small_config_takes_every_request():
    p = _run(["--impl", "reference", "--config", "1", "--steps", "2", "--warmup", "3"])
    assert p.returncode == 0, p.stderr[-2000:]
    d = json.loads([l for l in p.stdout.splitlines() if l.startswith("{")][0])
    assert d["config"]["requests"] == 4 and "first" not in d["cpu_baseline"]["sample"]


@pytest.mark.parametrize("cfg", [3, 5])
def test_request_subset_resolves_like_the_whole_batch(cfg):
    """The oracle legs time the first requests of a workload with their blocks renumbered.  Requests are
    independent, so the subset must resolve exactly as those requests do in the whole batch: the same
    stats, and rows that are the whole batch's rows with their blocks renumbered, on every step."""
    import numpy as np
    sys.path.insert(0, ROOT)
    import bench
    import oracle
    from synth import workloads
    oracle.build()
    if cfg == 3:
        w = workloads.config3(seed=3, R=6, L=2, turns=2, decode_per_turn=3)
    else:
        w = workloads.config5(seed=3, R=6, L=2, steps=4)
    steps = list(w.iter_steps(5 if cfg == 3 else 4))
    n = 3
    ws, sts = bench.subset_workload(w, steps, n)
    assert ws.R == n and ws.num_gpu_blocks < w.num_gpu_blocks and ws.rows_per_step * w.R == w.rows_per_step * n
    pairs = []   # (block in the whole batch, block in the subset) of every resolved row
    tb_f, tb_s = bench.Tables(w, steps), bench.Tables(ws, sts)
    tok_f = np.full((w.L // w.G, w.R, w.C), -1, np.int32)
    stamp_f = tok_f.copy()
    tok_s = np.full((ws.L // ws.G, n, ws.C), -1, np.int32)
    stamp_s = tok_s.copy()
    for i, (st, ss) in enumerate(zip(steps, sts)):
        tb_f.edit(i)
        tb_s.edit(i)
        kw = dict(S=w.S, B=w.B, max_pages=w.max_pages, C=w.C, step=st.index, threads=2, layers_per_index=w.G)
        rf, sf = oracle.resolve(num_gpu_blocks=w.num_gpu_blocks, num_host_blocks=w.num_host_blocks, topk=st.topk,
                                block_table=tb_f.bt, host_block_table=tb_f.hbt, ctx_len=st.ctx_len,
                                hot_blocks=w.hot_blocks, slot_token=tok_f, slot_stamp=stamp_f, **kw)
        rs, ss_ = oracle.resolve(num_gpu_blocks=ws.num_gpu_blocks, num_host_blocks=ws.num_host_blocks, topk=ss.topk,
                                 block_table=tb_s.bt, host_block_table=tb_s.hbt, ctx_len=ss.ctx_len,
                                 hot_blocks=ws.hot_blocks, slot_token=tok_s, slot_stamp=stamp_s, **kw)
        assert (sf[..., 0] == 0).all()
        assert np.array_equal(sf[:, :n], ss_), f"step {i}"
        assert np.array_equal(tok_f[:, :n], tok_s) and np.array_equal(stamp_f[:, :n], stamp_s)
        # rows: the same offsets, and one consistent renumbering of the blocks
        a, b = rf[:, :n].ravel(), rs.ravel()
        assert np.array_equal(a < 0, b < 0)
        a, b = a[a >= 0], b[b >= 0]
        assert np.array_equal(a % w.S, b % w.S)
        pairs.append(np.stack([a // w.S, b // w.S], 1))
        # offloads: the same pages
        m = st.off_src[:, 0] < n if len(st.off_src) else np.zeros(0, bool)
        assert np.array_equal(st.off_src[m], ss.off_src)
    # one renumbering for the whole run: each block maps to one block and back
    u = np.unique(np.concatenate(pairs), axis=0)
    assert len(np.unique(u[:, 0])) == len(u) == len(np.unique(u[:, 1]))


def test_reference_arm_other_ranks_exit_without_work():
    p = _run(["--impl", "reference", "--steps", "2", "--warmup", "3", "--gpus", "2"],
             env={"RANK": "1", "LOCAL_RANK": "1", "WORLD_SIZE": "2", "MASTER_ADDR": "127.0.0.1", "MASTER_PORT": "29555"})
    assert p.returncode == 0, p.stderr[-2000:]
    assert not [l for l in p.stdout.splitlines() if l.startswith("{")]


def test_residency_leg_times_native_and_oracle():
    p = _run(["--residency", "--steps", "3", "--warmup", "1", "--requests", "8"])
    assert p.returncode == 0, p.stderr[-2000:]
    lines = [l for l in p.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert d["unit"] == "steps/s" and d["value"] > 0 and d["steps"] == 3 and d["warmup"] == 1
    assert d["cpu_baseline"]["kind"] == "oracle" and d["cpu_baseline"]["value"] > 0
    assert d["config"]["requests"] == 8
