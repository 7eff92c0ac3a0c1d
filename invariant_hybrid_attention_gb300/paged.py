"""Device-side helpers for paged KV caches: allocation and page tables (PyTorch memory).

No attention arithmetic lives here; these only size and place caller-owned buffers in the
layout the C ABI expects: cache [num_pages][n_kv_heads][16][head_dim] bf16, page table
int32 [B][max_pages].
"""
from __future__ import annotations

from typing import Optional

import torch

from . import PAGE_SIZE, g4attn_cache, make_cache


def untile(t: torch.Tensor) -> torch.Tensor:
    """A cache tensor [pages][heads][2][D/8][8][8] as plain rows [pages][heads][16][D]."""
    P, H, D = t.shape[0], t.shape[1], t.shape[3] * 8
    return t.view(P, H, 2, D // 8, 8, 8).permute(0, 1, 2, 4, 3, 5).reshape(P, H, PAGE_SIZE, D)


def tile(rows: torch.Tensor) -> torch.Tensor:
    """Plain rows [pages][heads][16][D] in the cache's tiled layout [pages][heads][2][D/8][8][8]."""
    P, H, D = rows.shape[0], rows.shape[1], rows.shape[3]
    return rows.reshape(P, H, 2, 8, D // 8, 8).permute(0, 1, 2, 4, 3, 5).contiguous()


class PagedKV:
    """One layer's paged cache, pages stored as 8x8 core-matrix tiles (see include/g4attn.h).
    `v` is None on K==V (global) layers."""

    def __init__(self, num_pages: int, n_kv_heads: int, head_dim: int, shared: bool, device="cuda",
                 fill: Optional[float] = float("nan")):
        shape = (int(num_pages), int(n_kv_heads), 2, int(head_dim) // 8, 8, 8)
        self.k = torch.empty(shape, dtype=torch.bfloat16, device=device)
        self.v = None if shared else torch.empty(shape, dtype=torch.bfloat16, device=device)
        if fill is not None:
            self.k.fill_(fill)
            if self.v is not None:
                self.v.fill_(fill)
        self.num_pages = int(num_pages)

    @property
    def desc(self) -> g4attn_cache:
        return make_cache(self.k, self.v, self.num_pages)

    def nbytes(self) -> int:
        n = self.k.numel() * 2
        return n + (0 if self.v is None else self.v.numel() * 2)


def device_int32(values, device="cuda") -> torch.Tensor:
    return torch.as_tensor(values, dtype=torch.int32).to(device)
