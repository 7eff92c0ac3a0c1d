"""Device-side helpers for paged KV caches: allocation and page tables (PyTorch memory).

No attention arithmetic lives here; these only size and place caller-owned buffers in the
layout the C ABI expects: cache [num_pages][n_kv_heads][16][head_dim] bf16, page table
int32 [B][max_pages].
"""
from __future__ import annotations

from typing import Optional

import torch

from . import PAGE_SIZE, g4attn_cache, make_cache


ROT_DIMS = 128            # rotated columns of a global head: dims 0-63 and 256-319


def untile(t: torch.Tensor) -> torch.Tensor:
    """A cache tensor in the tiled page layout as plain rows [pages][heads][16][D]
    (D = 256: [2][32][8][8] per page-head; D = 512: two such 256-dim halves)."""
    P, H = t.shape[0], t.shape[1]
    n = t[0, 0].numel()
    D = n // PAGE_SIZE
    if D == 256:
        return t.reshape(P, H, 2, 32, 8, 8).permute(0, 1, 2, 4, 3, 5).reshape(P, H, PAGE_SIZE, 256)
    halves = t.reshape(P, H, 2, 2, 32, 8, 8).permute(0, 1, 3, 5, 2, 4, 6)   # [P][H][kg][j8][half][dg][d8]
    return halves.reshape(P, H, PAGE_SIZE, 512)


def tile(rows: torch.Tensor) -> torch.Tensor:
    """Plain rows [pages][heads][16][D] in the tiled page layout (inverse of `untile`)."""
    P, H, D = rows.shape[0], rows.shape[1], rows.shape[3]
    if D == 256:
        return rows.reshape(P, H, 2, 8, 32, 8).permute(0, 1, 2, 4, 3, 5).contiguous().reshape(P, H, 2, 32, 8, 8)
    r = rows.reshape(P, H, 2, 8, 2, 32, 8)          # [P][H][kg][j8][half][dg][d8]
    return r.permute(0, 1, 4, 2, 5, 3, 6).contiguous().reshape(P, H, 2, 2, 32, 8, 8)


def untile_v256(t: torch.Tensor) -> torch.Tensor:
    """A sliding V tensor [pages][heads][2][2][16][8][8] (two 128-dim halves per page-head block)
    as plain rows [pages][heads][16][256]."""
    P, H = t.shape[0], t.shape[1]
    r = t.reshape(P, H, 2, 2, 16, 8, 8).permute(0, 1, 3, 5, 2, 4, 6)   # [P][H][kg][j8][half][dg][d8]
    return r.reshape(P, H, PAGE_SIZE, 256)


def tile_v256(rows: torch.Tensor) -> torch.Tensor:
    """Plain rows [pages][heads][16][256] in the sliding V layout (inverse of `untile_v256`)."""
    P, H = rows.shape[0], rows.shape[1]
    r = rows.reshape(P, H, 2, 8, 2, 16, 8)          # [P][H][kg][j8][half][dg][d8]
    return r.permute(0, 1, 4, 2, 5, 3, 6).contiguous().reshape(P, H, 2, 2, 16, 8, 8)


def untile_rot(t: torch.Tensor) -> torch.Tensor:
    """A global k_rot tensor [pages][4][2][2][8][8][8] as rows [pages][4][16][128] holding dims
    0-63 then 256-319."""
    P, H = t.shape[0], t.shape[1]
    r = t.reshape(P, H, 2, 2, 8, 8, 8).permute(0, 1, 3, 5, 2, 4, 6)    # [P][H][kg][j8][half][dg][d8]
    return r.reshape(P, H, PAGE_SIZE, ROT_DIMS)


class PagedKV:
    """One layer's paged cache, pages stored as 8x8 core-matrix tiles (see include/g4attn.h).
    `v` is None on K==V (global) layers, which carry `k_rot` (the roped rotated columns)."""

    def __init__(self, num_pages: int, n_kv_heads: int, head_dim: int, shared: bool, device="cuda",
                 fill: Optional[float] = float("nan")):
        if int(head_dim) == 256:
            shape = (int(num_pages), int(n_kv_heads), 2, 32, 8, 8)
        else:
            shape = (int(num_pages), int(n_kv_heads), 2, 2, 32, 8, 8)
        self.k = torch.empty(shape, dtype=torch.bfloat16, device=device)
        # sliding V: two contiguous 128-dim halves per page-head block (see untile_v256)
        self.v = None if shared else torch.empty((int(num_pages), int(n_kv_heads), 2, 2, 16, 8, 8),
                                                 dtype=torch.bfloat16, device=device)
        self.k_rot = (torch.empty((int(num_pages), int(n_kv_heads), 2, 2, 8, 8, 8), dtype=torch.bfloat16,
                                  device=device) if shared else None)
        if fill is not None:
            for t in (self.k, self.v, self.k_rot):
                if t is not None:
                    t.fill_(fill)
        self.num_pages = int(num_pages)

    @property
    def desc(self) -> g4attn_cache:
        return make_cache(self.k, self.v, self.num_pages, self.k_rot)

    def nbytes(self) -> int:
        return sum(t.numel() * 2 for t in (self.k, self.v, self.k_rot) if t is not None)


def device_int32(values, device="cuda") -> torch.Tensor:
    return torch.as_tensor(values, dtype=torch.int32).to(device)
