"""The C ABI without a GPU: the library builds for sm_103a, loads, exports every function that
the headers in include/ declare, and its host-side logic (argument checks that need no device, size queries,
status strings) behaves as documented.  No compute call is made here."""
import ctypes
import os
import re
import shutil
import subprocess

import pytest

import sparse_mla_kv_gb300 as hs

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADERS = sorted(os.path.join(ROOT, "include", f) for f in os.listdir(os.path.join(ROOT, "include"))
                 if f.endswith(".h"))


@pytest.fixture(scope="module")
def lib():
    if not os.path.exists(hs.LIB_PATH):
        if shutil.which("nvcc") is None and not os.path.exists("/usr/local/cuda/bin/nvcc"):
            pytest.skip("no nvcc to build the library")
        from sparse_mla_kv_gb300 import _build
        _build.build()
    return hs.lib()


def declared_functions():
    text = "".join(open(h).read() for h in HEADERS)
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(hs_[a-z0-9_]+)\s*\(", text)))


def test_header_declares_the_boundary():
    names = declared_functions()
    for must in ("hs_pool_create", "hs_pool_destroy", "hs_hot_reset", "hs_resolve_topk", "hs_gather_rows",
                 "hs_offload_pages", "hs_status_str", "hs_resolve_workspace_bytes", "hs_hot_reset_requests",
                 "hs_res_create", "hs_res_admit", "hs_res_append", "hs_res_collect", "hs_res_tables"):
        assert must in names


def test_library_exports_every_declared_symbol(lib):
    for name in declared_functions():
        assert hasattr(lib, name), name
    nm = shutil.which("nm")
    if nm:
        out = subprocess.run([nm, "-D", "--defined-only", hs.LIB_PATH], capture_output=True, text=True).stdout
        exported = set(re.findall(r"\b(hs_[a-z0-9_]+)\b", out))
        assert set(declared_functions()) <= exported


def test_status_strings(lib):
    for code in (0, 1, 2, 3, 4, 5, 6, 7, 8):
        s = hs.status_str(code)
        assert s and s != "unknown status"
    assert hs.status_str(99) == "unknown status"


NB = 1024   # buckets per index group of the address-ordered miss layout


def _ordered_extra(ng, R, P, K, C):
    # bucket counters (NB + 1 per index group, 16-byte aligned) and NB buckets per group of twice
    # the even share of the group's R * min(P*K, C) possible misses, 16 B per entry
    per_group = R * min(P * K, C)
    cap = -(-2 * per_group // NB)
    return -(-4 * ng * (NB + 1) // 16) * 16 + 16 * ng * NB * cap


def test_size_queries(lib):
    # workspace: 16-byte-aligned miss counts + (host row, pool row, position) per possible miss
    # (min(P*K, C) per unit, 16 B each) + one host source per position (16-byte aligned) + 256 B of
    # the fused gather's work counters
    assert hs.resolve_workspace_bytes_min(1, 64, 1, 2048, 4096) == 256 + 16 * 64 * 2048 + 4 * 64 * 2048 + 256
    assert hs.resolve_workspace_bytes_min(4, 256, 4, 2048, 4096) == 4096 + 16 * 1024 * 4096 + 4 * 1024 * 8192 + 256
    assert hs.resolve_workspace_bytes_min(1, 3, 1, 5, 4) == 16 + 16 * 3 * 4 + 64 + 256
    assert hs.resolve_workspace_bytes_min(1, 1, 0, 5, 4) == 0
    # the full size adds the address-ordered miss layout's room
    for shape in ((1, 64, 1, 2048, 4096), (4, 256, 4, 2048, 4096), (1, 3, 1, 5, 4), (16, 32, 1, 2048, 4096)):
        assert hs.resolve_workspace_bytes(*shape) == hs.resolve_workspace_bytes_min(*shape) + _ordered_extra(*shape)
    assert hs.resolve_workspace_bytes(1, 1, 0, 5, 4) == 0
    # the benchmarked shapes and the MTP3 sizing (num_spec + 2) * K = 10240 fit in one CTA's shared
    # memory; oversize plans report 0 or > 227 KB
    for P, K, C in ((1, 256, 512), (1, 2048, 4096), (4, 2048, 4096), (4, 2048, 10240), (1, 1024, 16384)):
        assert 0 < hs.resolve_smem_bytes(P, K, C, 64) <= 227 * 1024
    assert hs.resolve_smem_bytes(1, 8192, 16384, 64) > 227 * 1024
    assert hs.resolve_smem_bytes(1, 16385, 4096, 64) == 0
    assert hs.resolve_smem_bytes(1, 16, 16385, 1) == 0
    assert hs.resolve_smem_bytes(1, 16, 100, 64) == 0          # capacity not a multiple of the page


def test_pool_create_rejects_bad_descriptions_before_touching_a_device(lib):
    L = lib
    h = ctypes.c_void_p()
    assert L.hs_pool_create(None, ctypes.byref(h)) == 1
    buf = (ctypes.c_void_p * 1)(ctypes.c_void_p(16))
    bad = [
        hs.PoolDesc(0, 64, 656, 10, 0, ctypes.cast(buf, ctypes.POINTER(ctypes.c_void_p)), None),
        hs.PoolDesc(1, 64, 650, 10, 0, ctypes.cast(buf, ctypes.POINTER(ctypes.c_void_p)), None),
        hs.PoolDesc(1, 0, 656, 10, 0, ctypes.cast(buf, ctypes.POINTER(ctypes.c_void_p)), None),
        hs.PoolDesc(1, 64, 656, 1 << 26, 0, ctypes.cast(buf, ctypes.POINTER(ctypes.c_void_p)), None),
        hs.PoolDesc(1, 64, 656, 10, 5, ctypes.cast(buf, ctypes.POINTER(ctypes.c_void_p)), None),
        hs.PoolDesc(1, 64, 656, 10, 0, None, None),
        hs.PoolDesc(129, 64, 656, 10, 0, ctypes.cast(buf, ctypes.POINTER(ctypes.c_void_p)), None),
    ]
    for d in bad:
        assert L.hs_pool_create(ctypes.byref(d), ctypes.byref(h)) == 1
        assert not h.value
    mis = (ctypes.c_void_p * 1)(ctypes.c_void_p(24))   # not 16-byte aligned
    d = hs.PoolDesc(1, 64, 656, 10, 0, ctypes.cast(mis, ctypes.POINTER(ctypes.c_void_p)), None)
    assert L.hs_pool_create(ctypes.byref(d), ctypes.byref(h)) == 1


def test_calls_on_null_handles_are_rejected(lib):
    L = lib
    hot = hs.HotStateC(64, None, None, None)
    assert L.hs_resolve_topk(None, 0, 1, 1, 1, 1, None, None, None, None, 1, ctypes.byref(hot), 0, None, None, None,
                             0, None) == 1
    assert L.hs_gather_rows(None, 0, 1, None, 1, None, None, None) == 1
    assert L.hs_offload_pages(None, None, None, 1, None, None) == 1
    assert L.hs_hot_reset(None, ctypes.byref(hot), 1, None) == 1
    assert L.hs_pool_set_miss_order(None, hs.MISS_ORDER_ON) == 1
    assert L.hs_pool_set_gather_copy(None, hs.GATHER_COPY_BULK) == 1
    assert L.hs_pool_set_miss_warps(None, 1) == 1
    assert L.hs_pool_set_miss_sm_divisor(None, 6) == 1
    assert L.hs_pool_set_miss_prefetch(None, 1) == 1
    assert L.hs_pool_set_gather_planes(None, 0, None) == 1
    assert L.hs_pool_set_phase_timestamps(None, None) == 1
    assert L.hs_resolve_miss_order(None, 0, 1, 1, 1, 1, ctypes.byref(hot), 1 << 30) == -1
    assert L.hs_resolve_workspace_bytes_min(1, 1, 0, 5, 4) == 0
    assert L.hs_resolve_workspace_bytes_min(1, 1, 1, 16385, 4) == 0   # plan beyond HS_MAX_PLAN
    assert L.hs_launch_count() == 0
    assert L.hs_check_status() == -1   # the normal build has no bounds checks to report (no CUDA call)


def test_checked_build_exports_every_declared_symbol(lib):
    """The bounds-checked variant (HS_CHECKED=1) builds for sm_103a and exports the same boundary."""
    from sparse_mla_kv_gb300 import _build
    path = _build.build(variant="checked")
    nm = shutil.which("nm")
    if not nm:
        pytest.skip("no nm")
    out = subprocess.run([nm, "-D", "--defined-only", path], capture_output=True, text=True).stdout
    assert set(declared_functions()) <= set(re.findall(r"\b(hs_[a-z0-9_]+)\b", out))


def test_plane_views_split_rows_without_copying():
    """plane_views cuts a gather output written in planes into per-plane views: plane p of layer l is
    the positions' bytes [c_p, c_p + w_p) laid out one plane after the other (CPU tensors here)."""
    import torch
    nl, n, planes = 2, 5, (512, 16, 128)
    rows = torch.randint(0, 256, (nl, n, sum(planes)), dtype=torch.uint8)
    cuts = [0, 512, 528, 656]
    written = torch.cat([torch.cat([rows[l, :, cuts[p]:cuts[p + 1]].reshape(-1) for p in range(3)])
                         for l in range(nl)]).reshape(nl, n, sum(planes))
    views = hs.plane_views(written, planes)
    assert [tuple(v.shape) for v in views] == [(nl, n, 512), (nl, n, 16), (nl, n, 128)]
    assert torch.equal(torch.cat(views, dim=-1), rows)
    assert all(v.data_ptr() >= written.data_ptr() for v in views)   # views into the same storage
    one = hs.plane_views(written[0], planes)                         # a single layer
    assert torch.equal(torch.cat(one, dim=-1), rows[0])
    try:
        hs.plane_views(written, (512, 16))
        raise AssertionError("sizes that do not sum to the row were accepted")
    except ValueError:
        pass
