"""Fill KV pools with the closed-form row contents (synth.content) using torch, on the device.

Input generation only: GPU pool blocks get the rows of the (request, page) they hold at the start;
pinned host pool blocks get the rows of their (request, page).  Large pools are filled in chunks on
the GPU (torch element-wise ops) and copied to pinned memory.  No resolver arithmetic here.
"""
from __future__ import annotations

import numpy as np
import torch

from . import content


def _rows_for_blocks(w, layer: int, owners: np.ndarray, device) -> torch.Tensor:
    """owners int64 [nb][2] (r, page) -> uint8 [nb, S, B] rows of those pages."""
    nb = owners.shape[0]
    cp = torch.from_numpy(w.content_page[owners[:, 0], owners[:, 1]].astype(np.int64)).to(device)
    cp = cp[:, None].expand(nb, w.S).reshape(-1)
    off = torch.arange(w.S, device=device, dtype=torch.int64)[None, :].expand(nb, w.S).reshape(-1)
    return content.rows_torch(w.content_seed, layer, cp, off, w.B).reshape(nb, w.S, w.B)


def fill_blocks(w, layer: int, dst: torch.Tensor, blocks: np.ndarray, owners: np.ndarray, device,
                chunk_blocks: int = 1024) -> None:
    """dst[blocks[i]] = rows of page owners[i] (dst: [num_blocks, S, B] uint8, GPU or pinned CPU)."""
    for i in range(0, len(blocks), chunk_blocks):
        b = blocks[i:i + chunk_blocks]
        rows = _rows_for_blocks(w, layer, owners[i:i + chunk_blocks], device)
        if dst.is_cuda:
            dst[torch.from_numpy(b.astype(np.int64)).to(dst.device)] = rows
        else:
            # pinned host pool: written by DMA straight from the device, one copy per run of
            # consecutive blocks (in a serving system the host pool is written by the GPU too --
            # offloads and prefill -- never by CPU stores)
            cuts = np.nonzero(np.diff(b) != 1)[0] + 1
            starts = np.concatenate([[0], cuts])
            ends = np.concatenate([cuts, [len(b)]])
            for a, e in zip(starts, ends):
                dst[int(b[a]):int(b[a]) + int(e - a)].copy_(rows[a:e])
            torch.cuda.synchronize(rows.device)


def fill_gpu_pool(w, layer: int, pool: torch.Tensor) -> None:
    own = w.gpu_block_owner()
    blocks = np.nonzero(own[:, 0] >= 0)[0]
    pool.zero_()
    fill_blocks(w, layer, pool, blocks, own[blocks], pool.device)


def fill_host_pool(w, layer: int, host: torch.Tensor, device) -> None:
    own = w.host_block_owner()
    blocks = np.nonzero(own[:, 0] >= 0)[0]
    order = np.argsort(blocks)
    fill_blocks(w, layer, host, blocks[order], own[blocks[order]], device, chunk_blocks=2048)


def expected_rows(w, layer: int, r_idx: torch.Tensor, ids: torch.Tensor) -> torch.Tensor:
    """Closed-form bytes of logical tokens ids (int64, device) of requests r_idx -> uint8 [n, B];
    ids == -1 gives zero rows."""
    dev = ids.device
    cached = getattr(w, "_content_page_dev", None)   # a device copy kept on the workload itself
    if cached is None or cached.device != dev:
        cached = torch.from_numpy(w.content_page.astype(np.int64)).to(dev)
        w._content_page_dev = cached
    cpt = cached
    valid = ids >= 0
    safe = torch.where(valid, ids, torch.zeros_like(ids))
    cp = cpt[r_idx, safe // w.S]
    rows = content.rows_torch(w.content_seed, layer, cp, safe % w.S, w.B)
    rows[~valid] = 0
    return rows


def pinned_empty(shape, dtype=torch.uint8) -> torch.Tensor:
    """A page-locked, device-mapped host tensor of exactly this size, huge-page backed (the library's
    host-pool allocator)."""
    from sparse_mla_kv_gb300.hostmem import pinned_host_pool
    return pinned_host_pool(shape, dtype)
