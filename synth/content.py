"""Seeded row contents for the synthetic KV pools.

Every logical KV row has bytes fixed by a closed form, H(seed, layer, content_page, offset): the
row is row_bytes/4 little-endian 32-bit words, each a chain of MurmurHash3's public 32-bit
finaliser (fmix32) over the four coordinates and the word index.  Because the bytes of every
row are known without running any implementation, a test can check that each gathered or
offloaded row equals the source row of its logical token.

The rows stand in for the pages' FP8 sparse-MLA rows (512 B fp8 latent + 16 B fp32 scales +
128 B bf16 rope = 656 B); the resolver treats them as opaque bytes, so uniform random bytes are
as good as real ones.

This module holds no resolver arithmetic; it only makes inputs.  numpy and torch versions give
identical bytes (torch is used to fill large pools on the device).
"""
from __future__ import annotations

import numpy as np

MASK32 = 0xFFFFFFFF
_C1 = 0x85EBCA6B
_C2 = 0xC2B2AE35
_GOLD = 0x9E3779B9
_P2 = 0x27D4EB2F
_P3 = 0x165667B1


def fmix32_np(h: np.ndarray) -> np.ndarray:
    h = h.astype(np.uint64)  # products formed in 64 bits, then reduced mod 2^32
    m = np.uint64(MASK32)
    h ^= h >> np.uint64(16)
    h = (h * np.uint64(_C1)) & m
    h ^= h >> np.uint64(13)
    h = (h * np.uint64(_C2)) & m
    h ^= h >> np.uint64(16)
    return h.astype(np.uint32)


def _row_base_np(seed: int, layer, content_page, offset) -> np.ndarray:
    layer = np.asarray(layer, dtype=np.uint64)
    cp = np.asarray(content_page, dtype=np.uint64)
    off = np.asarray(offset, dtype=np.uint64)
    m = np.uint64(MASK32)
    b = fmix32_np(((np.uint64(seed) + np.uint64(_GOLD) * (layer + np.uint64(1))) & m).astype(np.uint32))
    b = fmix32_np(b ^ ((cp * np.uint64(_C1)) & m).astype(np.uint32))
    b = fmix32_np(b ^ ((off * np.uint64(_C2) + np.uint64(_P3)) & m).astype(np.uint32))
    return b


def rows_np(seed: int, layer, content_page, offset, row_bytes: int) -> np.ndarray:
    """Bytes of the rows (layer, content_page, offset) (broadcast together) -> uint8 [..., row_bytes]."""
    assert row_bytes % 4 == 0
    base = _row_base_np(seed, layer, content_page, offset)
    w = np.arange(row_bytes // 4, dtype=np.uint64)
    words = ((base[..., None].astype(np.uint64) + w * np.uint64(_P2)) & np.uint64(MASK32)).astype(np.uint32)
    words = fmix32_np(words)
    return words.astype("<u4").view(np.uint8).reshape(*base.shape, row_bytes)


def page_np(seed: int, layer: int, content_page: int, page_size: int, row_bytes: int) -> np.ndarray:
    """One page of rows -> uint8 [page_size, row_bytes]."""
    return rows_np(seed, layer, content_page, np.arange(page_size), row_bytes)


# ---------------------------------------------------------------- torch (device fill) version
def _mul32_t(x, c: int):
    """(x * c) mod 2^32 for int64 tensors holding values in [0, 2^32), without int64 overflow."""
    lo = c & 0xFFFF
    hi = c >> 16
    return (x * lo + (((x * hi) & 0xFFFF) << 16)) & MASK32


def fmix32_t(h):
    h = h ^ (h >> 16)
    h = _mul32_t(h, _C1)
    h = h ^ (h >> 13)
    h = _mul32_t(h, _C2)
    h = h ^ (h >> 16)
    return h


def rows_torch(seed: int, layer: int, content_page, offset, row_bytes: int):
    """torch twin of rows_np: content_page/offset int64 tensors (same device) -> uint8 [n, row_bytes]."""
    import torch

    cp = content_page.to(torch.int64)
    off = offset.to(torch.int64)
    b0 = (seed + _GOLD * (layer + 1)) & MASK32
    b = fmix32_t(torch.full_like(cp, b0))
    b = fmix32_t(b ^ _mul32_t(cp & MASK32, _C1))
    b = fmix32_t(b ^ ((_mul32_t(off & MASK32, _C2) + _P3) & MASK32))
    w = torch.arange(row_bytes // 4, dtype=torch.int64, device=cp.device)
    words = (b[:, None] + _mul32_t(w, _P2)[None, :]) & MASK32
    words = fmix32_t(words)
    # little-endian bytes of each 32-bit word
    shifts = torch.tensor([0, 8, 16, 24], dtype=torch.int64, device=cp.device)
    by = (words[..., None] >> shifts) & 0xFF
    return by.to(torch.uint8).reshape(cp.shape[0], row_bytes)
