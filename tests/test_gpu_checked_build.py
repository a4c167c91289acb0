"""The bounds-checked build on the GPU.

libhs_checked.so is the library compiled with HS_CHECKED=1: every address a kernel derives from data
it read (table entries, slot indices, miss-list entries, repeat-chain links, output positions) is
checked against the extent of its buffer before the access, and a violation skips the access and is
recorded for hs_check_status.  This test builds it and runs GPU parity cases through it in a child
process: the tiny decode and the cold start with prefix reuse (configs 1 and 4, every mode), MTP3
plans with repeat chains, IndexShare groups, random small cases, output planes, the SM partition at
several divisors, and the data-error cases (bad ids,
steps, table entries -- inputs the normal build already turns into status words).  Each case must
give the oracle's results exactly, and no kernel may record a violation (checked after every test
by the fixture in conftest.py)."""
import os
import subprocess
import sys

import pytest
import torch

pytestmark = pytest.mark.gpu
ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_checked_build_gives_identical_results_and_no_violation():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from sparse_mla_kv_gb300 import _build
    _build.build()
    _build.build(variant="checked")
    env = dict(os.environ, HS_LIB_VARIANT="checked")
    probe = subprocess.run([sys.executable, "-c", "import sparse_mla_kv_gb300 as hs; print(hs.check_status())"],
                           cwd=ROOT, env=env, capture_output=True, text=True, timeout=300)
    assert probe.returncode == 0 and probe.stdout.strip() == "0", probe.stdout + probe.stderr   # not -1: checked
    sel = ("tiny_decode_all_bytes or cold_start_prefix_reuse or data_errors or random_small_cases or "
           "mtp3_hot_sizing or index_share_random or victim_sort_over_long_stamp_spans or "
           "planes_through_the_resolver or sm_partition_divisors")
    p = subprocess.run([sys.executable, "-m", "pytest", "-q", "-x", "-m", "gpu", "-k", sel, "-p", "no:cacheprovider",
                        "tests/test_gpu_parity.py", "tests/test_gpu_long_runs.py"],
                       cwd=ROOT, env=env, capture_output=True, text=True, timeout=1500)
    assert p.returncode == 0, p.stdout[-3000:] + p.stderr[-2000:]
    assert " passed" in p.stdout and "failed" not in p.stdout
