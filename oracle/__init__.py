"""Oracle: plain CPU implementation of the resolve / gather / offload semantics.

TEST INFRASTRUCTURE ONLY.  Only tests/, __graft_entry__.smoke() and bench.py's cpu_baseline and
reference legs may import this package.  The product library (sparse_mla_kv_gb300) never imports
it and has no fallback to it.

hs_oracle.c holds the arithmetic (see its header for the passages it follows); this module only
builds it with gcc and marshals numpy arrays.  bruteforce.py is a second, independent pure-Python
formulation used to cross-check it on tiny inputs.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
from typing import Optional, Sequence

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "hs_oracle.c")
_LIB = os.path.join(_HERE, "libhs_oracle.so")
_lib = None

STATUS = {0: "OK", 1: "INVALID_ARG", 2: "ID_RANGE", 3: "MISSING_ROW", 4: "CAPACITY", 5: "STEP_ORDER",
          8: "TABLE_RANGE"}


def build(force: bool = False) -> str:
    """Compile hs_oracle.c into libhs_oracle.so (OpenMP if the compiler has it)."""
    if not force and os.path.exists(_LIB) and os.path.getmtime(_LIB) >= os.path.getmtime(_SRC):
        return _LIB
    base = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", _SRC, "-o", _LIB]
    r = subprocess.run(base[:1] + ["-fopenmp"] + base[1:], capture_output=True, text=True)
    if r.returncode != 0:
        r2 = subprocess.run(base, capture_output=True, text=True)
        if r2.returncode != 0:
            raise RuntimeError("oracle build failed:\n" + r.stderr + r2.stderr)
    return _LIB


def lib():
    global _lib
    if _lib is None:
        build()
        _lib = load_library(_LIB)
    return _lib


def use_library(L) -> None:
    """Route the wrappers below through another build of the oracle (tests plant mistakes in
    copies of hs_oracle.c this way); None restores the default build."""
    global _lib
    _lib = L


def load_library(path: str):
    """Load a compiled hs_oracle.c and declare its signatures."""
    L = ctypes.CDLL(path)
    i32, i64, p = ctypes.c_int32, ctypes.c_int64, ctypes.c_void_p
    L.hso_resolve_unit.restype = i32
    L.hso_resolve_unit.argtypes = [i32, i32, i32, i32, i32, p, p, i32, p, p, p, i32, i32, i32, p, p, p, i32, p, p]
    L.hso_resolve.restype = None
    L.hso_resolve.argtypes = [i32, i32, i32, i32, p, p, i32, i32, i32, i32, i32, p, p, p, p, i32, i32, p, p, p,
                              i32, p, p, i32]
    L.hso_gather.restype = i32
    L.hso_gather.argtypes = [i32, i64, p, i32, i32, p, i64, p, i32]
    L.hso_offload.restype = i32
    L.hso_offload.argtypes = [i32, i32, i32, i32, i32, p, p, p, p, i32]
    return L


def _ptr(a: Optional[np.ndarray]):
    return None if a is None else ctypes.c_void_p(a.ctypes.data)


def _c32(a) -> np.ndarray:
    a = np.ascontiguousarray(a, dtype=np.int32)
    return a


def _ptr_array(arrs: Optional[Sequence[np.ndarray]]):
    if arrs is None:
        return None, None
    for a in arrs:
        assert a.dtype == np.uint8 and a.flags.c_contiguous
    arr = (ctypes.c_void_p * len(arrs))(*[a.ctypes.data for a in arrs])
    return ctypes.cast(arr, ctypes.c_void_p), arr


def default_threads() -> int:
    return len(os.sched_getaffinity(0)) if hasattr(os, "sched_getaffinity") else (os.cpu_count() or 1)


def resolve(*, S: int, B: int, num_gpu_blocks: int, num_host_blocks: int, topk: np.ndarray, block_table,
            host_block_table, ctx_len, max_pages: int, C: int, hot_blocks, slot_token: np.ndarray,
            slot_stamp: np.ndarray, step: int, layer_begin: int = 0, pools=None, hosts=None,
            threads: Optional[int] = None, layers_per_index: int = 1):
    """Resolve all units of topk [ng][R][P][K] at `step`: ng index groups of G = layers_per_index
    consecutive layers from layer `layer_begin` (a multiple of G; G = 1: one group per layer).

    slot_token/slot_stamp int32 [num_layers/G][R][C] are updated in place; pools/hosts (per-layer
    uint8 arrays [blocks*S*B], all layers) get the miss copies when given.  Returns (out_rows,
    out_stats)."""
    G = max(1, int(layers_per_index))
    assert layer_begin % G == 0
    topk = _c32(topk)
    nl, R = topk.shape[0] * G, topk.shape[1]
    n = int(np.prod(topk.shape[2:]))
    assert slot_token.dtype == np.int32 and slot_token.flags.c_contiguous
    assert slot_stamp.dtype == np.int32 and slot_stamp.flags.c_contiguous
    bt, hbt, cl, hb = _c32(block_table), _c32(host_block_table), _c32(ctx_len), _c32(hot_blocks)
    out_rows = np.empty(topk.shape, np.int32)
    out_stats = np.empty((nl // G, R, 4), np.int32)
    pp, _k1 = _ptr_array(pools)
    hp, _k2 = _ptr_array(hosts)
    lib().hso_resolve(S, B, num_gpu_blocks, num_host_blocks, pp, hp, G, layer_begin, nl, R, n, _ptr(topk), _ptr(bt),
                      _ptr(hbt), _ptr(cl), max_pages, C, _ptr(hb), _ptr(slot_token), _ptr(slot_stamp), step,
                      _ptr(out_rows), _ptr(out_stats), threads or default_threads())
    return out_rows, out_stats


def gather(*, B: int, num_rows: int, pools, rows: np.ndarray, layer_begin: int = 0,
           threads: Optional[int] = None):
    """rows int32 [nl][n] -> (uint8 [nl][n][B], status)."""
    rows = _c32(rows)
    nl, n = rows.shape
    out = np.empty((nl, n, B), np.uint8)
    pp, _k = _ptr_array(pools)
    st = lib().hso_gather(B, num_rows, pp, layer_begin, nl, _ptr(rows), n, _ptr(out), threads or default_threads())
    return out, st


def offload(*, S: int, B: int, num_gpu_blocks: int, num_host_blocks: int, pools, hosts, gpu_blocks, host_blocks):
    gb, hb = _c32(gpu_blocks), _c32(host_blocks)
    pp, _k1 = _ptr_array(pools)
    hp, _k2 = _ptr_array(hosts)
    return lib().hso_offload(S, B, len(pools), num_gpu_blocks, num_host_blocks, pp, hp, _ptr(gb), _ptr(hb), len(gb))
