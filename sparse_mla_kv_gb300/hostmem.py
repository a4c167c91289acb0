"""Pinned, device-mapped host memory for the host KV pool, backed by transparent huge pages.

The resolver's misses read single 656-byte rows from the pinned host pool with zero-copy loads,
scattered over the whole pool.  Each read needs an address translation for host memory, and with
small pages a pool of tens of GB has far more pages than the translation caches hold.  Measured on
a GB300 with 64 KB base pages (32K random misses per step): 117 GB/s from a 10 GB pool, 4 GB/s from
a 30 GB pool with base pages; with huge pages 122 GB/s at 10 GB, 96 GB/s at 20 GB, 33 GB/s at 40 GB,
24 GB/s at 80 GB.  Host pools are therefore allocated with mmap + madvise(MADV_HUGEPAGE) before the
pages are first touched (the system's transparent huge pages must allow madvise), then registered
with the CUDA runtime as portable and mapped.  Falls back to base pages where madvise is refused.

torch's own pinned allocator is not used: it rounds each allocation up to a power of two, which
doubles a pool of tens of GB.
"""
from __future__ import annotations

import ctypes
import mmap
import weakref

import numpy as np
import torch

_PROT_RW = mmap.PROT_READ | mmap.PROT_WRITE
_MAP_PRIVATE_ANON = mmap.MAP_PRIVATE | mmap.MAP_ANONYMOUS
_MADV_HUGEPAGE = 14
_CUDA_HOST_REGISTER_PORTABLE_MAPPED = 3

_libc = None


def _c():
    global _libc
    if _libc is None:
        L = ctypes.CDLL(None, use_errno=True)
        L.mmap.restype = ctypes.c_void_p
        L.mmap.argtypes = [ctypes.c_void_p, ctypes.c_size_t, ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_long]
        L.munmap.restype = ctypes.c_int
        L.munmap.argtypes = [ctypes.c_void_p, ctypes.c_size_t]
        L.madvise.restype = ctypes.c_int
        L.madvise.argtypes = [ctypes.c_void_p, ctypes.c_size_t, ctypes.c_int]
        _libc = L
    return _libc


def _release(ptr: int, base: int, span: int) -> None:
    try:
        torch.cuda.cudart().cudaHostUnregister(ptr)
    except Exception:
        pass
    _c().munmap(base, span)


def huge_page_bytes() -> int:
    """The transparent huge page size (2 MB with 4 KB base pages, 512 MB with 64 KB base pages)."""
    try:
        return int(open("/sys/kernel/mm/transparent_hugepage/hpage_pmd_size").read())
    except (OSError, ValueError):
        return 2 << 20


class _Mapping:
    """Owns one mapping, aligned to the huge page size; the tensor views keep it alive."""

    def __init__(self, nbytes: int, huge: bool = True):
        L = _c()
        hp = huge_page_bytes()
        span = nbytes + hp
        base = L.mmap(None, span, _PROT_RW, _MAP_PRIVATE_ANON, -1, 0)
        if base is None or base == ctypes.c_void_p(-1).value:
            raise MemoryError(f"mmap of {span} bytes failed")
        ptr = (base + hp - 1) // hp * hp
        self.huge = huge and L.madvise(ptr, nbytes, _MADV_HUGEPAGE) == 0
        rc = int(torch.cuda.cudart().cudaHostRegister(ptr, nbytes, _CUDA_HOST_REGISTER_PORTABLE_MAPPED))
        if rc != 0:
            L.munmap(base, span)
            raise RuntimeError(f"cudaHostRegister failed ({rc}) for {nbytes} bytes")
        self.ptr, self.nbytes = ptr, nbytes
        weakref.finalize(self, _release, ptr, base, span)


def _array(m: _Mapping, nbytes: int) -> np.ndarray:
    # the ctypes array holds the mapping; the numpy array holds the ctypes array; torch's storage holds
    # the numpy array: the mapping lives as long as any tensor view of it
    buf = (ctypes.c_uint8 * m.nbytes).from_address(m.ptr)
    buf._hs_mapping = m
    return np.ctypeslib.as_array(buf)[:nbytes]


def huge_page_fraction(t: torch.Tensor) -> float:
    """The share of a host tensor's resident bytes that the kernel backs with transparent huge pages
    (AnonHugePages / Rss of the mappings it spans, from /proc/self/smaps); -1.0 if it cannot be read."""
    lo = t.data_ptr()
    hi = lo + t.numel() * t.element_size()
    rss = huge = 0
    try:
        cur = None
        for line in open("/proc/self/smaps"):
            f = line.split()
            if "-" in f[0] and len(f) >= 5 and not f[0].endswith(":"):
                a, b = (int(x, 16) for x in f[0].split("-"))
                cur = a < hi and b > lo
            elif cur and f[0] == "Rss:":
                rss += int(f[1])
            elif cur and f[0] == "AnonHugePages:":
                huge += int(f[1])
    except (OSError, ValueError, IndexError):
        return -1.0
    return huge / rss if rss else -1.0


def pinned_host_pool(shape, dtype=torch.uint8, huge: bool = True) -> torch.Tensor:
    """A page-locked, device-mapped host tensor of exactly this size, backed by huge pages where the
    system allows (see the module docstring); huge=False keeps the base pages (for comparison).
    Contents are unspecified."""
    itemsize = torch.empty((), dtype=dtype).element_size()
    nbytes = max(int(np.prod(shape)) * itemsize, 1 << 16)
    m = _Mapping(nbytes, huge)
    return torch.from_numpy(_array(m, int(np.prod(shape)) * itemsize)).view(dtype).reshape(shape)
