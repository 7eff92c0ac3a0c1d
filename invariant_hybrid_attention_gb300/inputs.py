"""Seeded synthetic inputs, shared by the tests, the benchmark and the oracle checks.

This module draws numbers and lays them out; it holds none of the attention
arithmetic. Values come from a CPU ``torch.Generator`` seeded per call: fp32
standard-normal draws, multiplied by a scale, then cast to bf16 (round to
nearest even). Lengths and page permutations come from the same kind of
generator. Nothing here depends on a GPU.

The workload recipes (sizes, seeds, value scales) follow the five benchmark
configurations of the hybrid-attention build: a tiny two-sequence oracle case,
sliding-window prefill 4 x 4096, global K==V prefill 2 x 8192, a ragged 64-request
decode mix with 1k-32k contexts, and a batch-invariance stress.
"""
from __future__ import annotations

import dataclasses
from typing import List, Optional, Sequence

import torch

PAGE_SIZE = 16


def bf16_normal(shape: Sequence[int], seed: int, scale: float = 1.0) -> torch.Tensor:
    """N(0,1) fp32 draws from a CPU generator seeded with `seed`, times `scale`, cast to bf16."""
    g = torch.Generator(device="cpu")
    g.manual_seed(int(seed))
    x = torch.randn(*shape, generator=g, dtype=torch.float32)
    if scale != 1.0:
        x = x * scale
    return x.to(torch.bfloat16)


def bf16_normal_device(shape: Sequence[int], seed: int, scale: float = 1.0, device="cuda") -> torch.Tensor:
    """Same recipe as `bf16_normal`, drawn on the device from a seeded CUDA generator (used for
    the benchmark's multi-GB tensors; the values differ from the CPU generator's)."""
    g = torch.Generator(device=device)
    g.manual_seed(int(seed))
    x = torch.randn(*shape, generator=g, dtype=torch.float32, device=device)
    if scale != 1.0:
        x.mul_(scale)
    return x.to(torch.bfloat16)


def uniform_ints(n: int, lo: int, hi: int, seed: int) -> List[int]:
    """`n` integers uniform in [lo, hi] (both ends included)."""
    g = torch.Generator(device="cpu")
    g.manual_seed(int(seed))
    return [int(v) for v in torch.randint(lo, hi + 1, (n,), generator=g)]


def permutation(n: int, seed: int) -> torch.Tensor:
    g = torch.Generator(device="cpu")
    g.manual_seed(int(seed))
    return torch.randperm(n, generator=g)


@dataclasses.dataclass
class PagePlan:
    """Logical-to-physical page mapping for a batch of sequences.

    ``table[b][i]`` is the physical page holding keys ``16*i .. 16*i+15`` of
    sequence ``b``; unmapped entries are -1. ``num_pages`` is the number of
    physical pages the cache must hold.
    """

    table: torch.Tensor  # int32 [B][max_pages]
    num_pages: int

    @property
    def max_pages(self) -> int:
        return int(self.table.shape[1])


def make_page_plan(ctx_lens: Sequence[int], seed: int, max_pages: Optional[int] = None,
                   mapped_from: Optional[Sequence[int]] = None, spare_pages: int = 0) -> PagePlan:
    """Scatter every sequence's pages over a randomly permuted physical pool.

    ``mapped_from[b]`` (optional) is the first logical page that gets a physical
    page; earlier entries stay -1 (a sliding layer only needs its window).
    ``spare_pages`` extra physical pages are left unused in the pool.
    """
    B = len(ctx_lens)
    need = [(int(L) + PAGE_SIZE - 1) // PAGE_SIZE for L in ctx_lens]
    first = [0] * B if mapped_from is None else [int(m) for m in mapped_from]
    mp = max(need) if max_pages is None else int(max_pages)
    if mp < max(need):
        raise ValueError("max_pages smaller than the longest sequence")
    total = sum(n - f for n, f in zip(need, first)) + int(spare_pages)
    perm = permutation(max(total, 1), seed)
    table = torch.full((B, max(mp, 1)), -1, dtype=torch.int32)
    k = 0
    for b in range(B):
        for i in range(first[b], need[b]):
            table[b, i] = int(perm[k])
            k += 1
    return PagePlan(table=table, num_pages=max(total, 1))


@dataclasses.dataclass
class RowLayout:
    """Where each sequence's query rows sit in a packed or padded [T, H, D] tensor."""

    q_start: List[int]
    q_len: List[int]
    ctx_start: List[int]
    T: int


def packed_layout(q_lens: Sequence[int], ctx_starts: Optional[Sequence[int]] = None) -> RowLayout:
    starts, s = [], 0
    for L in q_lens:
        starts.append(s)
        s += int(L)
    cs = [0] * len(q_lens) if ctx_starts is None else [int(c) for c in ctx_starts]
    return RowLayout(q_start=starts, q_len=[int(L) for L in q_lens], ctx_start=cs, T=max(s, 1))


def padded_layout(q_lens: Sequence[int], ctx_starts: Optional[Sequence[int]] = None,
                  pad_to: Optional[int] = None) -> RowLayout:
    lmax = max(int(L) for L in q_lens) if pad_to is None else int(pad_to)
    starts = [b * lmax for b in range(len(q_lens))]
    cs = [0] * len(q_lens) if ctx_starts is None else [int(c) for c in ctx_starts]
    return RowLayout(q_start=starts, q_len=[int(L) for L in q_lens], ctx_start=cs,
                     T=max(lmax * len(q_lens), 1))


# ---- the benchmark workloads -------------------------------------------------------------

@dataclasses.dataclass(frozen=True)
class PrefillWorkload:
    name: str
    kind: str          # "sliding" | "global"
    n_seqs: int
    seq_len: int
    value_scale: float
    seed: int


SLIDING_PREFILL = PrefillWorkload("sliding-window prefill 4x4096 (Hq32/Hkv16/D256, W1024)",
                                  "sliding", 4, 4096, 0.5, 1)
GLOBAL_PREFILL = PrefillWorkload("global K==V prefill 2x8192 (Hq32/Hkv4/D512, p-RoPE 0.25)",
                                 "global", 2, 8192, 1.0, 2)


@dataclasses.dataclass(frozen=True)
class DecodeWorkload:
    name: str
    batch: int
    ctx_lo: int
    ctx_hi: int
    length_seed: int
    value_seed: int
    n_sliding: int
    n_global: int


DECODE_MIX = DecodeWorkload("ragged paged decode, B=64, ctx U[1024,32768], 5 sliding : 1 global",
                            64, 1024, 32768, 7, 8, 5, 1)


def prefill_tensors(kind: str, q_lens: Sequence[int], layout: RowLayout, n_q: int, n_kv: int, d: int,
                    seed: int, scale: float = 1.0, ctx_lens: Optional[Sequence[int]] = None):
    """Per-sequence raw projections for a prefill: q rows at the layout's places, plus every
    sequence's full key/value history (history rows first, then the new rows).

    Returns (q [T,n_q,d], hist_k list of [ctx,n_kv,d], hist_v list or None) as bf16 CPU tensors.
    Padding rows of q are filled with NaN so that any read of them shows up.
    """
    B = len(q_lens)
    ctx_lens = [layout.ctx_start[b] + int(q_lens[b]) for b in range(B)] if ctx_lens is None else ctx_lens
    q = torch.full((layout.T, n_q, d), float("nan"), dtype=torch.bfloat16)
    hist_k, hist_v = [], []
    for b in range(B):
        sb = seed * 1000003 + b * 7919
        qb = bf16_normal((int(q_lens[b]), n_q, d), sb + 1, scale)
        q[layout.q_start[b]:layout.q_start[b] + int(q_lens[b])] = qb
        hist_k.append(bf16_normal((int(ctx_lens[b]), n_kv, d), sb + 2, scale))
        if kind == "sliding":
            hist_v.append(bf16_normal((int(ctx_lens[b]), n_kv, d), sb + 3, scale))
    return q, hist_k, (hist_v if kind == "sliding" else None)


def rows_of(hist: List[torch.Tensor], layout: RowLayout, fill_nan: bool = True) -> torch.Tensor:
    """Gather each sequence's new rows (positions ctx_start .. ctx_start+q_len-1) of a per-sequence
    history into the layout's [T, H, D] tensor (padding rows NaN)."""
    n, d = hist[0].shape[1], hist[0].shape[2]
    out = torch.full((layout.T, n, d), float("nan") if fill_nan else 0.0, dtype=hist[0].dtype)
    for b, h in enumerate(hist):
        c0, L, s = layout.ctx_start[b], layout.q_len[b], layout.q_start[b]
        out[s:s + L] = h[c0:c0 + L]
    return out


# ---- the decode mix, one cache per layer ---------------------------------------------------

def decode_mix_lengths(wl: DecodeWorkload = DECODE_MIX) -> List[int]:
    """Context lengths of the decode mix (the new token included): `batch` integers uniform in
    [ctx_lo, ctx_hi], drawn with the workload's length seed."""
    return uniform_ints(wl.batch, wl.ctx_lo, wl.ctx_hi, wl.length_seed)


def decode_mix_first_keys(lens: Sequence[int], window: int) -> List[int]:
    """First key position each request's sliding cache holds: the page holding the window's first
    key (a sliding layer maps only the window's pages; earlier table entries stay -1)."""
    return [PAGE_SIZE * (max(0, int(L) - int(window)) // PAGE_SIZE) for L in lens]


def decode_mix_values(value_seed: int, layer: int, b: int, n_rows: int, n_kv: int, d: int, with_v: bool,
                      device="cuda"):
    """Key (and value) rows of request b of layer `layer` of the decode mix: the rows its cache holds,
    the new token's last. Seeded per (layer, request), so that any one request can be drawn again."""
    base = int(value_seed) * 1_000_000 + int(layer) * 10_000 + int(b) * 10
    k = bf16_normal_device((n_rows, n_kv, d), base + 1, device=device)
    v = bf16_normal_device((n_rows, n_kv, d), base + 2, device=device) if with_v else None
    return k, v


def decode_mix_queries(value_seed: int, layer: int, B: int, d: int, device="cuda") -> torch.Tensor:
    """The B decode queries [B, 32, d] of layer `layer` of the decode mix."""
    return bf16_normal_device((B, 32, d), int(value_seed) * 1_000_000 + int(layer) * 10_000 + 9999, device=device)
