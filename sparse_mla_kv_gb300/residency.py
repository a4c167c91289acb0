"""Python binding of the host-side residency manager (include/hs_residency.h): argument marshalling
only; every decision is made by the native library."""
from __future__ import annotations

import ctypes
from typing import List, Sequence, Tuple

import numpy as np

from . import HSError, lib

_declared = False


def _lib():
    global _declared
    L = lib()
    if not _declared:
        i32, i64, p = ctypes.c_int32, ctypes.c_int64, ctypes.c_void_p
        P32 = ctypes.POINTER(ctypes.c_int32)
        L.hs_res_create.restype = i32
        L.hs_res_create.argtypes = [i32, i32, i32, i32, i32, i32, ctypes.POINTER(p)]
        L.hs_res_destroy.restype = None
        L.hs_res_destroy.argtypes = [p]
        L.hs_res_admit.restype = i32
        L.hs_res_admit.argtypes = [p, i32, i32, P32, i32]
        L.hs_res_append.restype = i32
        L.hs_res_append.argtypes = [p, i32, i32]
        L.hs_res_append_all.restype = i32
        L.hs_res_append_all.argtypes = [p, P32]
        L.hs_res_touch.restype = i32
        L.hs_res_touch.argtypes = [p, i32, P32, i64, i32]
        L.hs_res_touch_all.restype = i32
        L.hs_res_touch_all.argtypes = [p, P32, i32, i32]
        L.hs_res_finish.restype = i32
        L.hs_res_finish.argtypes = [p, i32]
        L.hs_res_hold_host.restype = i32
        L.hs_res_hold_host.argtypes = [p, P32, i32]
        L.hs_res_drop_host.restype = i32
        L.hs_res_drop_host.argtypes = [p, P32, i32]
        L.hs_res_counts.restype = None
        L.hs_res_counts.argtypes = [p, P32, P32, P32]
        L.hs_res_free_gpu_blocks.restype = i32
        L.hs_res_free_gpu_blocks.argtypes = [p]
        L.hs_res_collect.restype = i32
        L.hs_res_collect.argtypes = [p, P32, P32, i32, P32]
        L.hs_res_take_resets.restype = i32
        L.hs_res_take_resets.argtypes = [p, P32, i32, P32]
        L.hs_res_take_fills.restype = i32
        L.hs_res_take_fills.argtypes = [p, P32, P32, P32, i32, P32]
        L.hs_res_tables.restype = i32
        L.hs_res_tables.argtypes = [p, P32, P32, P32, P32]
        _declared = True
    return L


def _i32(a) -> Tuple[np.ndarray, object]:
    arr = np.ascontiguousarray(np.asarray(a, dtype=np.int32).reshape(-1))
    return arr, arr.ctypes.data_as(ctypes.POINTER(ctypes.c_int32))


def _check(code: int, what: str) -> None:
    if code != 0:
        raise HSError(code, what)


class Residency:
    """Page residency of up to max_requests requests over a GPU block pool and a host block pool (see
    include/hs_residency.h).  Tables come back as numpy int32 arrays ready to copy to the device."""

    def __init__(self, num_gpu_blocks: int, num_host_blocks: int, page_size: int, max_requests: int,
                 max_pages: int, hot_blocks: int):
        self.R, self.max_pages, self.Hc = int(max_requests), int(max_pages), int(hot_blocks)
        h = ctypes.c_void_p()
        _check(_lib().hs_res_create(num_gpu_blocks, num_host_blocks, page_size, max_requests, max_pages, hot_blocks,
                                    ctypes.byref(h)), "hs_res_create")
        self.h = h

    def close(self) -> None:
        if getattr(self, "h", None) is not None and self.h.value:
            _lib().hs_res_destroy(self.h)
            self.h = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    def admit(self, r: int, ctx: int, prefix_host_blocks: Sequence[int] = ()) -> None:
        arr, ptr = _i32(prefix_host_blocks)
        _check(_lib().hs_res_admit(self.h, r, ctx, ptr, arr.size), "hs_res_admit")

    def append(self, r: int, n: int) -> None:
        _check(_lib().hs_res_append(self.h, r, n), "hs_res_append")

    def append_all(self, n_tokens) -> None:
        """n_tokens [max_requests]: append() for every request with a non-zero entry, in request order,
        in one call."""
        arr = np.ascontiguousarray(np.asarray(n_tokens, dtype=np.int32).reshape(-1))
        if arr.size != self.R:
            raise ValueError("n_tokens must have max_requests entries")
        _check(_lib().hs_res_append_all(self.h, arr.ctypes.data_as(ctypes.POINTER(ctypes.c_int32))),
               "hs_res_append_all")

    def touch(self, r: int, ids, step: int) -> None:
        arr, ptr = _i32(ids)
        _check(_lib().hs_res_touch(self.h, r, ptr, arr.size, step), "hs_res_touch")

    def touch_all(self, ids, step: int) -> None:
        """ids [max_requests][n]: every active request's selected ids in one call (rows of inactive
        requests are ignored)."""
        arr = np.ascontiguousarray(np.asarray(ids, dtype=np.int32))
        if arr.ndim != 2 or arr.shape[0] != self.R:
            raise ValueError("ids must be [max_requests][n]")
        _check(_lib().hs_res_touch_all(self.h, arr.ctypes.data_as(ctypes.POINTER(ctypes.c_int32)), arr.shape[1],
                                       step), "hs_res_touch_all")

    def finish(self, r: int) -> None:
        _check(_lib().hs_res_finish(self.h, r), "hs_res_finish")

    def hold_host(self, blocks: Sequence[int]) -> None:
        arr, ptr = _i32(blocks)
        _check(_lib().hs_res_hold_host(self.h, ptr, arr.size), "hs_res_hold_host")

    def drop_host(self, blocks: Sequence[int]) -> None:
        arr, ptr = _i32(blocks)
        _check(_lib().hs_res_drop_host(self.h, ptr, arr.size), "hs_res_drop_host")

    def counts(self) -> Tuple[int, int, int]:
        q, rs, f = ctypes.c_int32(), ctypes.c_int32(), ctypes.c_int32()
        _lib().hs_res_counts(self.h, ctypes.byref(q), ctypes.byref(rs), ctypes.byref(f))
        return q.value, rs.value, f.value

    def free_gpu_blocks(self) -> int:
        return int(_lib().hs_res_free_gpu_blocks(self.h))

    def collect(self) -> List[Tuple[int, int]]:
        n_q = self.counts()[0]
        if n_q == 0:
            return []
        g, gp = _i32(np.zeros(max(1, n_q)))
        hb, hp = _i32(np.zeros(max(1, n_q)))
        n = ctypes.c_int32()
        _check(_lib().hs_res_collect(self.h, gp, hp, g.size, ctypes.byref(n)), "hs_res_collect")
        return [(int(g[i]), int(hb[i])) for i in range(n.value)]

    def collect_arrays(self) -> Tuple[np.ndarray, np.ndarray]:
        pairs = self.collect()
        a = np.array(pairs, np.int32).reshape(-1, 2)
        return a[:, 0].copy(), a[:, 1].copy()

    def take_resets(self) -> List[int]:
        n_r = self.counts()[1]
        if n_r == 0:
            return []
        a, ap = _i32(np.zeros(max(1, n_r)))
        n = ctypes.c_int32()
        _check(_lib().hs_res_take_resets(self.h, ap, a.size, ctypes.byref(n)), "hs_res_take_resets")
        return [int(x) for x in a[:n.value]]

    def take_fills(self) -> List[Tuple[int, int, int]]:
        n_f = self.counts()[2]
        if n_f == 0:
            return []
        b, bp = _i32(np.zeros(max(1, n_f)))
        r, rp = _i32(np.zeros(max(1, n_f)))
        p, pp = _i32(np.zeros(max(1, n_f)))
        n = ctypes.c_int32()
        _check(_lib().hs_res_take_fills(self.h, bp, rp, pp, b.size, ctypes.byref(n)), "hs_res_take_fills")
        return [(int(b[i]), int(r[i]), int(p[i])) for i in range(n.value)]

    def tables(self, out=None):
        """(block_table [R][max_pages], host_block_table [R][max_pages], hot_blocks [R][Hc], ctx_len [R]).
        out: a tuple returned by an earlier call, refilled in place (no new arrays; e.g. pinned buffers
        that are then copied to the device)."""
        if out is None:
            bt = np.empty((self.R, self.max_pages), np.int32)
            hbt = np.empty((self.R, self.max_pages), np.int32)
            hot = np.empty((self.R, max(1, self.Hc)), np.int32)
            ctx = np.empty(self.R, np.int32)
        else:
            bt, hbt, hot, ctx = out
            hot = hot.base if hot.base is not None and hot.shape[1] != max(1, self.Hc) else hot
            for a, shape in ((bt, (self.R, self.max_pages)), (hbt, (self.R, self.max_pages)),
                             (hot, (self.R, max(1, self.Hc))), (ctx, (self.R,))):
                if a.dtype != np.int32 or a.shape != shape or not a.flags.c_contiguous:
                    raise ValueError("out must be the arrays of an earlier tables() call")
        P = ctypes.POINTER(ctypes.c_int32)
        _check(_lib().hs_res_tables(self.h, bt.ctypes.data_as(P), hbt.ctypes.data_as(P), hot.ctypes.data_as(P),
                                    ctx.ctypes.data_as(P)), "hs_res_tables")
        return bt, hbt, hot[:, :self.Hc], ctx
