"""Hybrid HiSparse top-K resolver for sparse-MLA decode, GB300-native (sm_103a).

Thin Python binding over the C ABI in include/hs.h (libhs.so, built in-tree by _build.py).  This
module only marshals arguments: torch tensors are passed as raw pointers and the current torch
CUDA stream as the launch stream.  Every step of the path runs in the library's CUDA kernels; there
is no CPU fallback, and every call raises if the library is missing or returns an error.

Operations (the passages that define them are cited in include/hs.h):
  resolve_topk   fused per-step top-K resolver (resident / hot hit / one-row miss copy)
  gather_rows    single-stride gather of resolved pool rows
  offload_pages  post-forward proactive copy of completed pages, all layers in one launch
  hot_reset      empty the hot buffers
"""
from __future__ import annotations

import ctypes
import os
from typing import Optional, Sequence

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
# HS_LIB_VARIANT=checked loads the bounds-checked build (libhs_checked.so, see hs_check_status)
LIB_VARIANT = os.environ.get("HS_LIB_VARIANT", "")
LIB_PATH = os.path.join(_HERE, f"libhs_{LIB_VARIANT}.so" if LIB_VARIANT else "libhs.so")

HS_OK = 0
MISS_ORDER_AUTO, MISS_ORDER_OFF, MISS_ORDER_ON, MISS_ORDER_RANGES, MISS_ORDER_SPREAD = 0, 1, 2, 3, 4
GATHER_COPY_LOADS, GATHER_COPY_BULK = 0, 1
MISS_PREFETCH_OFF, MISS_PREFETCH_ON = 0, 1
MAX_PLANES = 4
STATUS_NAMES = {0: "OK", 1: "INVALID_ARG", 2: "ID_RANGE", 3: "MISSING_ROW", 4: "CAPACITY", 5: "STEP_ORDER",
                6: "CUDA", 7: "TIMEOUT", 8: "TABLE_RANGE"}
MAX_LAYERS = 128


class HSError(RuntimeError):
    def __init__(self, code: int, what: str):
        super().__init__(f"{what}: {STATUS_NAMES.get(code, code)} ({status_str(code)})")
        self.code = code


class PoolDesc(ctypes.Structure):
    _fields_ = [("num_layers", ctypes.c_int32), ("page_size", ctypes.c_int32), ("row_bytes", ctypes.c_int32),
                ("num_gpu_blocks", ctypes.c_int32), ("num_host_blocks", ctypes.c_int32),
                ("gpu_layer_base", ctypes.POINTER(ctypes.c_void_p)),
                ("host_layer_base", ctypes.POINTER(ctypes.c_void_p))]


class HotStateC(ctypes.Structure):
    _fields_ = [("capacity", ctypes.c_int32), ("hot_blocks", ctypes.c_void_p), ("slot_token", ctypes.c_void_p),
                ("slot_stamp", ctypes.c_void_p), ("layers_per_index", ctypes.c_int32)]


_lib = None


def lib():
    """The loaded libhs.so (raises if it has not been built)."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(f"{LIB_PATH} is missing: build it with sparse_mla_kv_gb300._build.build("
                               f"variant={LIB_VARIANT!r}) (there is no fallback implementation)")
        L = ctypes.CDLL(LIB_PATH)
        i32, i64, sz, p = ctypes.c_int32, ctypes.c_int64, ctypes.c_size_t, ctypes.c_void_p
        L.hs_status_str.restype = ctypes.c_char_p
        L.hs_status_str.argtypes = [i32]
        L.hs_launch_count.restype = i64
        L.hs_launch_count.argtypes = []
        L.hs_check_status.restype = i32
        L.hs_check_status.argtypes = []
        L.hs_pool_create.restype = i32
        L.hs_pool_create.argtypes = [ctypes.POINTER(PoolDesc), ctypes.POINTER(p)]
        L.hs_pool_destroy.restype = None
        L.hs_pool_destroy.argtypes = [p]
        L.hs_hot_reset.restype = i32
        L.hs_hot_reset.argtypes = [p, ctypes.POINTER(HotStateC), i32, p]
        L.hs_hot_reset_requests.restype = i32
        L.hs_hot_reset_requests.argtypes = [p, ctypes.POINTER(HotStateC), i32, p, i32, p]
        L.hs_resolve_workspace_bytes.restype = sz
        L.hs_resolve_workspace_bytes.argtypes = [i32, i32, i32, i32, i32]
        L.hs_resolve_workspace_bytes_min.restype = sz
        L.hs_resolve_workspace_bytes_min.argtypes = [i32, i32, i32, i32, i32]
        L.hs_pool_set_miss_order.restype = i32
        L.hs_pool_set_miss_order.argtypes = [p, i32]
        L.hs_pool_set_gather_copy.restype = i32
        L.hs_pool_set_gather_copy.argtypes = [p, i32]
        L.hs_pool_set_miss_warps.restype = i32
        L.hs_pool_set_miss_warps.argtypes = [p, i32]
        L.hs_pool_set_miss_sm_divisor.restype = i32
        L.hs_pool_set_miss_sm_divisor.argtypes = [p, i32]
        L.hs_pool_set_miss_prefetch.restype = i32
        L.hs_pool_set_miss_prefetch.argtypes = [p, i32]
        L.hs_pool_set_phase_timestamps.restype = i32
        L.hs_pool_set_phase_timestamps.argtypes = [p, ctypes.c_void_p]
        L.hs_pool_set_gather_planes.restype = i32
        L.hs_pool_set_gather_planes.argtypes = [p, i32, ctypes.POINTER(i32)]
        L.hs_resolve_miss_order.restype = i32
        L.hs_resolve_miss_order.argtypes = [p, i32, i32, i32, i32, i32, ctypes.POINTER(HotStateC), sz]
        L.hs_resolve_smem_bytes.restype = sz
        L.hs_resolve_smem_bytes.argtypes = [i32, i32, i32, i32]
        L.hs_resolve_topk.restype = i32
        L.hs_resolve_topk.argtypes = [p, i32, i32, i32, i32, i32, p, p, p, p, i32, ctypes.POINTER(HotStateC), i32, p, p,
                                      p, sz, p]
        L.hs_resolve_gather.restype = i32
        L.hs_resolve_gather.argtypes = [p, i32, i32, i32, i32, i32, p, p, p, p, i32, ctypes.POINTER(HotStateC), i32, p,
                                        p, p, p, sz, p]
        L.hs_resolve_plan.restype = i32
        L.hs_resolve_plan.argtypes = L.hs_resolve_topk.argtypes
        L.hs_gather_planned.restype = i32
        L.hs_gather_planned.argtypes = [p, i32, i32, i32, i32, i32, ctypes.POINTER(HotStateC), p, p, sz, p, p]
        L.hs_gather_rows.restype = i32
        L.hs_gather_rows.argtypes = [p, i32, i32, p, i64, p, p, p]
        L.hs_offload_pages.restype = i32
        L.hs_offload_pages.argtypes = [p, p, p, i32, p, p]
        _lib = L
    return _lib


def status_str(code: int) -> str:
    try:
        return lib().hs_status_str(int(code)).decode()
    except RuntimeError:
        return STATUS_NAMES.get(code, str(code))


def check_status() -> int:
    """Bounds-checked build: the first bounds violation recorded since the last call (0 = none); -1 in
    the normal build.  Synchronises the device."""
    return int(lib().hs_check_status())


def launch_count() -> int:
    """Kernels the library has launched in this process."""
    return int(lib().hs_launch_count())


def _check(code: int, what: str) -> None:
    if code != HS_OK:
        raise HSError(code, what)


def _stream(stream) -> ctypes.c_void_p:
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream)


def _dev_i32(t: torch.Tensor, name: str) -> ctypes.c_void_p:
    if not isinstance(t, torch.Tensor) or t.dtype != torch.int32 or not t.is_cuda or not t.is_contiguous():
        raise TypeError(f"{name} must be a contiguous int32 CUDA tensor")
    return ctypes.c_void_p(t.data_ptr())


def _opt(t: Optional[torch.Tensor], name: str) -> Optional[ctypes.c_void_p]:
    return None if t is None else _dev_i32(t, name)


class Pool:
    """Geometry and base pointers of the paged KV pool: per layer one GPU tensor
    [num_gpu_blocks, page_size, row_bytes] (resident pages and leased hot blocks share it) and one
    pinned host tensor [num_host_blocks, page_size, row_bytes].  The tensors stay owned by the caller;
    this object keeps references so they outlive the handle."""

    def __init__(self, gpu_layers: Sequence[torch.Tensor], host_layers: Optional[Sequence[torch.Tensor]] = None):
        if not gpu_layers or len(gpu_layers) > MAX_LAYERS:
            raise ValueError("need 1..128 layers")
        g0 = gpu_layers[0]
        if g0.dim() != 3:
            raise ValueError("GPU layer tensors must be [num_gpu_blocks, page_size, row_bytes]")
        self.num_gpu_blocks, self.page_size, self.row_bytes = (int(x) for x in g0.shape)
        self.num_layers = len(gpu_layers)
        for t in gpu_layers:
            if t.dtype != torch.uint8 or not t.is_cuda or not t.is_contiguous() or tuple(t.shape) != tuple(g0.shape):
                raise TypeError("GPU layer tensors must be contiguous uint8 CUDA tensors of one shape")
        host_layers = list(host_layers or [])
        self.num_host_blocks = int(host_layers[0].shape[0]) if host_layers else 0
        if host_layers:
            if len(host_layers) != self.num_layers:
                raise ValueError("one host tensor per layer")
            for t in host_layers:
                if (t.dtype != torch.uint8 or t.is_cuda or not t.is_pinned() or not t.is_contiguous()
                        or tuple(t.shape) != (self.num_host_blocks, self.page_size, self.row_bytes)):
                    raise TypeError("host layer tensors must be contiguous pinned uint8 CPU tensors "
                                    "[num_host_blocks, page_size, row_bytes]")
        self.gpu_layers = list(gpu_layers)
        self.host_layers = host_layers
        gp = (ctypes.c_void_p * self.num_layers)(*[t.data_ptr() for t in gpu_layers])
        hp = (ctypes.c_void_p * self.num_layers)(*[t.data_ptr() for t in host_layers]) if host_layers else None
        desc = PoolDesc(self.num_layers, self.page_size, self.row_bytes, self.num_gpu_blocks, self.num_host_blocks,
                        ctypes.cast(gp, ctypes.POINTER(ctypes.c_void_p)),
                        ctypes.cast(hp, ctypes.POINTER(ctypes.c_void_p)) if hp is not None else None)
        h = ctypes.c_void_p()
        with torch.cuda.device(g0.device):
            _check(lib().hs_pool_create(ctypes.byref(desc), ctypes.byref(h)), "hs_pool_create")
        self.handle = h
        self.planes = ()

    def set_miss_order(self, mode: int) -> None:
        """MISS_ORDER_AUTO (default), MISS_ORDER_OFF, MISS_ORDER_ON, MISS_ORDER_RANGES or MISS_ORDER_SPREAD:
        see hs_pool_set_miss_order."""
        _check(lib().hs_pool_set_miss_order(self.handle, int(mode)), "hs_pool_set_miss_order")

    def set_gather_copy(self, mode: int) -> None:
        """GATHER_COPY_LOADS (default) or GATHER_COPY_BULK: see hs_pool_set_gather_copy."""
        _check(lib().hs_pool_set_gather_copy(self.handle, int(mode)), "hs_pool_set_gather_copy")

    def set_miss_warps(self, warps: int) -> None:
        """Fused gather: -1 = default, 0 = SM partition, 1 or 2 = that many miss warps in every CTA; see
        hs_pool_set_miss_warps."""
        _check(lib().hs_pool_set_miss_warps(self.handle, int(warps)), "hs_pool_set_miss_warps")

    def set_phase_timestamps(self, ts: Optional[torch.Tensor]) -> None:
        """ts: int64 CUDA tensor of 4 (or None to stop): the SM-partition gather's device timestamps; see
        hs_pool_set_phase_timestamps."""
        if ts is not None and (ts.dtype != torch.int64 or not ts.is_cuda or ts.numel() < 4 or not ts.is_contiguous()):
            raise TypeError("ts must be a contiguous int64 CUDA tensor of at least 4 elements")
        _check(lib().hs_pool_set_phase_timestamps(self.handle, ctypes.c_void_p(ts.data_ptr()) if ts is not None else None),
               "hs_pool_set_phase_timestamps")
        self._phase_ts = ts

    def set_gather_planes(self, plane_bytes=()) -> None:
        """Output layout of the gathers: () = rows; else the row cut into planes of these byte sizes
        (multiples of 16 summing to row_bytes, at most MAX_PLANES), each layer's output holding the planes
        one after the other; see hs_pool_set_gather_planes and plane_views."""
        pb = [int(x) for x in plane_bytes]
        arr = (ctypes.c_int32 * max(1, len(pb)))(*pb)
        _check(lib().hs_pool_set_gather_planes(self.handle, len(pb), arr), "hs_pool_set_gather_planes")
        self.planes = tuple(pb)

    def set_miss_prefetch(self, mode: int) -> None:
        """MISS_PREFETCH_ON: the resolver prefetches each miss's host row into L2 when it classifies it;
        see hs_pool_set_miss_prefetch."""
        _check(lib().hs_pool_set_miss_prefetch(self.handle, int(mode)), "hs_pool_set_miss_prefetch")

    def set_miss_sm_divisor(self, divisor: int) -> None:
        """SM partition: every divisor-th SM copies the misses (2..32, 0 = default, -1 = none: HBM rows
        first, then misses on every SM); see hs_pool_set_miss_sm_divisor."""
        _check(lib().hs_pool_set_miss_sm_divisor(self.handle, int(divisor)), "hs_pool_set_miss_sm_divisor")

    def close(self) -> None:
        if getattr(self, "handle", None) is not None and self.handle.value:
            lib().hs_pool_destroy(self.handle)
            self.handle = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


class HotState:
    """Per-request hot buffers: leased block ids [R][C/page_size] (shared by all layers) and the
    per-(index group, request) slot token/stamp arrays [num_layers/G][R][C] (-1 = empty / never used).
    G = layers_per_index: 1 when every layer has its own top-K; G > 1 under IndexShare, where G
    consecutive layers read one indexer's top-K and share one state."""

    def __init__(self, capacity: int, hot_blocks: torch.Tensor, slot_token: torch.Tensor, slot_stamp: torch.Tensor,
                 layers_per_index: int = 1):
        self.capacity = int(capacity)
        self.G = max(1, int(layers_per_index))
        self.hot_blocks, self.slot_token, self.slot_stamp = hot_blocks, slot_token, slot_stamp
        self.c = HotStateC(self.capacity, _dev_i32(hot_blocks, "hot_blocks"), _dev_i32(slot_token, "slot_token"),
                           _dev_i32(slot_stamp, "slot_stamp"), self.G)

    @classmethod
    def allocate(cls, num_layers: int, hot_blocks: torch.Tensor, capacity: int,
                 layers_per_index: int = 1) -> "HotState":
        G = max(1, int(layers_per_index))
        if num_layers % G:
            raise ValueError("num_layers must be a multiple of layers_per_index")
        R = int(hot_blocks.shape[0])
        dev = hot_blocks.device
        tok = torch.empty((num_layers // G, R, capacity), dtype=torch.int32, device=dev)
        st = torch.empty((num_layers // G, R, capacity), dtype=torch.int32, device=dev)
        return cls(capacity, hot_blocks, tok, st, G)

    @property
    def R(self) -> int:
        return int(self.hot_blocks.shape[0])


def hot_reset(pool: Pool, hot: HotState, stream=None) -> None:
    _check(lib().hs_hot_reset(pool.handle, ctypes.byref(hot.c), hot.R, _stream(stream)), "hs_hot_reset")


def hot_reset_requests(pool: Pool, hot: HotState, requests: torch.Tensor, stream=None) -> None:
    """Empty the hot slots of the listed requests (device int32 [n]) in every index group."""
    n = int(requests.numel())
    if n:
        _check(lib().hs_hot_reset_requests(pool.handle, ctypes.byref(hot.c), hot.R, _dev_i32(requests, "requests"),
                                           n, _stream(stream)), "hs_hot_reset_requests")


def resolve_workspace_bytes(nl: int, R: int, P: int, K: int, capacity: int) -> int:
    return int(lib().hs_resolve_workspace_bytes(nl, R, P, K, capacity))


def resolve_workspace_bytes_min(nl: int, R: int, P: int, K: int, capacity: int) -> int:
    return int(lib().hs_resolve_workspace_bytes_min(nl, R, P, K, capacity))


def miss_order_used(pool: Pool, hot: HotState, nl: int, R: int, P: int, K: int, workspace_bytes: int,
                    layer_begin: int = 0) -> bool:
    """Whether a resolve call of this shape files its misses in host address order."""
    v = int(lib().hs_resolve_miss_order(pool.handle, layer_begin, nl, R, P, K, ctypes.byref(hot.c),
                                        int(workspace_bytes)))
    if v < 0:
        raise ValueError("bad arguments to hs_resolve_miss_order")
    return bool(v)


def resolve_smem_bytes(P: int, K: int, capacity: int, page_size: int = 64) -> int:
    return int(lib().hs_resolve_smem_bytes(P, K, capacity, page_size))


def alloc_workspace(nl: int, R: int, P: int, K: int, capacity: int, device) -> torch.Tensor:
    nbytes = resolve_workspace_bytes(nl, R, P, K, capacity)
    return torch.empty(max(16, nbytes), dtype=torch.uint8, device=device)


def resolve_topk(pool: Pool, topk: torch.Tensor, block_table: torch.Tensor, host_block_table: torch.Tensor,
                 ctx_len: torch.Tensor, hot: HotState, step: int, *, layer_begin: int = 0,
                 out_rows: Optional[torch.Tensor] = None, out_stats: Optional[torch.Tensor] = None,
                 workspace: Optional[torch.Tensor] = None, stream=None):
    """topk int32 [ng][R][P][K] -> (out_rows int32 [ng][R][P][K], out_stats int32 [ng][R][4]), for the
    ng index groups of G = hot.G layers starting at layer_begin (ng = layers when G = 1)."""
    if topk.dim() != 4:
        raise ValueError("topk must be [ng][R][P][K]")
    ng, R, P, K = (int(x) for x in topk.shape)
    nl = ng * hot.G
    if block_table.dim() != 2 or block_table.shape[0] != R or tuple(host_block_table.shape) != tuple(block_table.shape):
        raise ValueError("block tables must both be [R][max_pages]")
    if hot.R != R:
        raise ValueError("hot state has a different number of requests")
    dev = topk.device
    if out_rows is None:
        out_rows = torch.empty_like(topk)
    if out_stats is None:
        out_stats = torch.empty((ng, R, 4), dtype=torch.int32, device=dev)
    if workspace is None:
        workspace = alloc_workspace(ng, R, P, K, hot.capacity, dev)
    if workspace.dtype != torch.uint8 or not workspace.is_cuda:
        raise TypeError("workspace must be a uint8 CUDA tensor")
    code = lib().hs_resolve_topk(pool.handle, layer_begin, nl, R, P, K, _dev_i32(topk, "topk"),
                                 _dev_i32(block_table, "block_table"), _dev_i32(host_block_table, "host_block_table"),
                                 _dev_i32(ctx_len, "ctx_len"), int(block_table.shape[1]), ctypes.byref(hot.c),
                                 int(step), _dev_i32(out_rows, "out_rows"), _dev_i32(out_stats, "out_stats"),
                                 ctypes.c_void_p(workspace.data_ptr()), workspace.numel(), _stream(stream))
    _check(code, "hs_resolve_topk")
    return out_rows, out_stats


def resolve_gather(pool: Pool, topk: torch.Tensor, block_table: torch.Tensor, host_block_table: torch.Tensor,
                   ctx_len: torch.Tensor, hot: HotState, step: int, *, layer_begin: int = 0,
                   out_rows: Optional[torch.Tensor] = None, out_stats: Optional[torch.Tensor] = None,
                   out: Optional[torch.Tensor] = None, workspace: Optional[torch.Tensor] = None, stream=None):
    """Resolve and gather in one call (miss copies fused into the gather).  topk [ng][R][P][K] for ng
    index groups of G = hot.G layers (nl = ng * G layers).
    Returns (out_rows [ng][R][P][K], out_stats [ng][R][4], out uint8 [nl][R*P*K][row_bytes])."""
    if topk.dim() != 4:
        raise ValueError("topk must be [ng][R][P][K]")
    ng, R, P, K = (int(x) for x in topk.shape)
    nl = ng * hot.G
    if block_table.dim() != 2 or block_table.shape[0] != R or tuple(host_block_table.shape) != tuple(block_table.shape):
        raise ValueError("block tables must both be [R][max_pages]")
    if hot.R != R:
        raise ValueError("hot state has a different number of requests")
    dev = topk.device
    out_rows = torch.empty_like(topk) if out_rows is None else out_rows
    out_stats = torch.empty((ng, R, 4), dtype=torch.int32, device=dev) if out_stats is None else out_stats
    workspace = alloc_workspace(ng, R, P, K, hot.capacity, dev) if workspace is None else workspace
    if out is None:
        out = torch.empty((nl, R * P * K, pool.row_bytes), dtype=torch.uint8, device=dev)
    if out.dtype != torch.uint8 or not out.is_cuda or not out.is_contiguous() or out.numel() != nl * R * P * K * pool.row_bytes:
        raise TypeError("out must be a contiguous uint8 CUDA tensor of nl*R*P*K*row_bytes bytes")
    code = lib().hs_resolve_gather(pool.handle, layer_begin, nl, R, P, K, _dev_i32(topk, "topk"),
                                   _dev_i32(block_table, "block_table"),
                                   _dev_i32(host_block_table, "host_block_table"), _dev_i32(ctx_len, "ctx_len"),
                                   int(block_table.shape[1]), ctypes.byref(hot.c), int(step),
                                   _dev_i32(out_rows, "out_rows"), _dev_i32(out_stats, "out_stats"),
                                   ctypes.c_void_p(out.data_ptr()), ctypes.c_void_p(workspace.data_ptr()),
                                   workspace.numel(), _stream(stream))
    _check(code, "hs_resolve_gather")
    return out_rows, out_stats, out


def gather_rows(pool: Pool, rows: torch.Tensor, *, layer_begin: int = 0, out: Optional[torch.Tensor] = None,
                status: Optional[torch.Tensor] = None, stream=None) -> torch.Tensor:
    """rows int32 [nl][n] (or [n] for one layer) -> uint8 [nl][n][row_bytes] (or [n][row_bytes]), each
    layer's bytes in the pool's output layout (rows, or planes: see plane_views)."""
    squeeze = rows.dim() == 1
    r2 = rows.reshape(1, -1) if squeeze else rows.reshape(rows.shape[0], -1)
    nl, n = int(r2.shape[0]), int(r2.shape[1])
    if out is None:
        out = torch.empty((nl, n, pool.row_bytes), dtype=torch.uint8, device=rows.device)
    if out.dtype != torch.uint8 or not out.is_cuda or not out.is_contiguous() or out.numel() != nl * n * pool.row_bytes:
        raise TypeError("out must be a contiguous uint8 CUDA tensor of nl*n*row_bytes bytes")
    code = lib().hs_gather_rows(pool.handle, layer_begin, nl, _dev_i32(r2, "rows"), n, ctypes.c_void_p(out.data_ptr()),
                                _opt(status, "status"), _stream(stream))
    _check(code, "hs_gather_rows")
    return out.reshape(n, pool.row_bytes) if squeeze else out


def plane_views(out: torch.Tensor, plane_bytes) -> list:
    """Views of a gather output written in a plane layout (Pool.set_gather_planes): out uint8
    [nl][n][row_bytes] (or [n][row_bytes]) -> one uint8 tensor per plane, [nl][n][plane_bytes[p]] (or
    [n][plane_bytes[p]]).  No copy."""
    squeeze = out.dim() == 2
    o = out.reshape(1, out.shape[0], out.shape[1]) if squeeze else out
    nl, n, rb = int(o.shape[0]), int(o.shape[1]), int(o.shape[2])
    if sum(plane_bytes) != rb:
        raise ValueError("plane sizes must sum to the row size")
    flat = o.reshape(nl, n * rb)
    views, off = [], 0
    for w in plane_bytes:
        v = flat[:, off:off + n * w].reshape(nl, n, w)
        views.append(v[0] if squeeze else v)
        off += n * w
    return views


def offload_pages(pool: Pool, gpu_blocks: torch.Tensor, host_blocks: torch.Tensor, *,
                  status: Optional[torch.Tensor] = None, stream=None) -> None:
    n = int(gpu_blocks.numel())
    if int(host_blocks.numel()) != n:
        raise ValueError("gpu_blocks and host_blocks differ in length")
    if n == 0:
        return
    code = lib().hs_offload_pages(pool.handle, _dev_i32(gpu_blocks, "gpu_blocks"), _dev_i32(host_blocks, "host_blocks"),
                                  n, _opt(status, "status"), _stream(stream))
    _check(code, "hs_offload_pages")


class PreparedStep:
    """Pre-marshalled resolve / gather / offload calls over one fixed set of device buffers, for a
    decode loop: per call only the top-K pointer and the step number change.  Still just the C ABI;
    this only avoids rebuilding ctypes arguments every step."""

    def __init__(self, pool: Pool, hot: HotState, block_table: torch.Tensor, host_block_table: torch.Tensor,
                 ctx_len: torch.Tensor, out_rows: torch.Tensor, out_stats: torch.Tensor, workspace: torch.Tensor,
                 gather_out: torch.Tensor, *, layer_begin: int = 0, gather_status: Optional[torch.Tensor] = None,
                 stream=None):
        ng, R, P, K = (int(x) for x in out_rows.shape)
        self.shape = (ng, R, P, K)
        self.G = hot.G
        self.nl = nl = ng * hot.G
        self.pool, self.hot = pool, hot
        self._keep = (block_table, host_block_table, ctx_len, out_rows, out_stats, workspace, gather_out, gather_status)
        self.L = lib()
        # stream=None: launch on whatever torch stream is current at each call (so the calls can be
        # captured into a CUDA graph); otherwise always on the given stream
        self._fixed_stream = None if stream is None else _stream(stream)
        self.lb = int(layer_begin)
        self.max_pages = int(block_table.shape[1])
        self.args_bt = (_dev_i32(block_table, "block_table"), _dev_i32(host_block_table, "host_block_table"),
                        _dev_i32(ctx_len, "ctx_len"))
        self.rows = _dev_i32(out_rows, "out_rows")
        self.stats = _dev_i32(out_stats, "out_stats")
        self.ws = ctypes.c_void_p(workspace.data_ptr())
        self.ws_n = workspace.numel()
        self.gout = ctypes.c_void_p(gather_out.data_ptr())
        self.gstatus = _opt(gather_status, "gather_status")
        self.n_per_layer = R * P * K
        if gather_out.numel() != nl * self.n_per_layer * pool.row_bytes:
            raise ValueError("gather_out must hold nl*R*P*K rows")

    @property
    def stream(self) -> ctypes.c_void_p:
        return self._fixed_stream if self._fixed_stream is not None else _stream(None)

    def resolve(self, topk: torch.Tensor, step: int) -> None:
        nl, (_, R, P, K) = self.nl, self.shape
        if tuple(topk.shape) != self.shape:
            raise ValueError("topk shape differs from the prepared shape")
        _check(self.L.hs_resolve_topk(self.pool.handle, self.lb, nl, R, P, K, _dev_i32(topk, "topk"), *self.args_bt,
                                      self.max_pages, ctypes.byref(self.hot.c), int(step), self.rows, self.stats,
                                      self.ws, self.ws_n, self.stream), "hs_resolve_topk")

    def plan(self, topk: torch.Tensor, step: int) -> None:
        nl, (_, R, P, K) = self.nl, self.shape
        if tuple(topk.shape) != self.shape:
            raise ValueError("topk shape differs from the prepared shape")
        _check(self.L.hs_resolve_plan(self.pool.handle, self.lb, nl, R, P, K, _dev_i32(topk, "topk"), *self.args_bt,
                                      self.max_pages, ctypes.byref(self.hot.c), int(step), self.rows, self.stats,
                                      self.ws, self.ws_n, self.stream), "hs_resolve_plan")

    def gather_planned(self) -> None:
        nl, (_, R, P, K) = self.nl, self.shape
        _check(self.L.hs_gather_planned(self.pool.handle, self.lb, nl, R, P, K, ctypes.byref(self.hot.c), self.rows,
                                        self.ws, self.ws_n, self.gout, self.stream), "hs_gather_planned")

    def resolve_gather(self, topk: torch.Tensor, step: int) -> None:
        nl, (_, R, P, K) = self.nl, self.shape
        if tuple(topk.shape) != self.shape:
            raise ValueError("topk shape differs from the prepared shape")
        _check(self.L.hs_resolve_gather(self.pool.handle, self.lb, nl, R, P, K, _dev_i32(topk, "topk"), *self.args_bt,
                                        self.max_pages, ctypes.byref(self.hot.c), int(step), self.rows, self.stats,
                                        self.gout, self.ws, self.ws_n, self.stream), "hs_resolve_gather")

    def gather(self) -> None:
        if self.G == 1:
            _check(self.L.hs_gather_rows(self.pool.handle, self.lb, self.nl, self.rows, self.n_per_layer, self.gout,
                                         self.gstatus, self.stream), "hs_gather_rows")
            return
        # IndexShare: every layer of a group gathers the group's rows (one launch per layer)
        n, B = self.n_per_layer, self.pool.row_bytes
        for l in range(self.nl):
            _check(self.L.hs_gather_rows(self.pool.handle, self.lb + l, 1,
                                         ctypes.c_void_p(self.rows.value + 4 * n * (l // self.G)), n,
                                         ctypes.c_void_p(self.gout.value + n * B * l), self.gstatus, self.stream),
                   "hs_gather_rows")

    def offload(self, gpu_blocks: torch.Tensor, host_blocks: torch.Tensor, n: int) -> None:
        if n:
            _check(self.L.hs_offload_pages(self.pool.handle, _dev_i32(gpu_blocks, "gpu_blocks"),
                                           _dev_i32(host_blocks, "host_blocks"), int(n), None, self.stream),
                   "hs_offload_pages")
