"""Shared set-up for the GPU tests: seeded inputs, paged caches filled through the library,
and the oracle's answers on the same inputs. Nothing the oracle sees comes from the GPU."""
from __future__ import annotations

import numpy as np
import torch

import invariant_hybrid_attention_gb300 as g4
import oracle
from invariant_hybrid_attention_gb300 import inputs as gi
from invariant_hybrid_attention_gb300.paged import PagedKV, device_int32

# Tolerances of the build's numerical target: bf16 outputs with fp32 accumulation against
# the fp64 oracle.
TOL_MAX, TOL_MEAN = 2e-2, 2e-3

GEOM = {"sliding": dict(n_kv=16, d=256), "global": dict(n_kv=4, d=512)}


def layers(kind: str, window: int = 1024):
    if kind == "sliding":
        return g4.sliding_layer(window), oracle.with_window(oracle.SLIDING, window)
    return g4.global_layer(), oracle.GLOBAL


def f64(t: torch.Tensor) -> np.ndarray:
    return t.detach().float().cpu().double().numpy()


def errors(got: np.ndarray, want: np.ndarray):
    d = np.abs(got - want)
    return float(d.max()), float(d.mean())


def assert_close(got, want, what=""):
    mx, mean = errors(got, want)
    assert np.isfinite(got).all(), f"{what}: non-finite output"
    assert mx <= TOL_MAX and mean <= TOL_MEAN, f"{what}: max-abs {mx:.3e}, mean-abs {mean:.3e}"
    return mx, mean


class Norms:
    """Per-head norm weights drawn once (bf16, uniform in [0.5, 1.5]), as the library's argument
    struct (device tensors kept alive here) and as the oracle's Norms on the same bf16 values."""

    def __init__(self, kind, seed, q=True, k=True, v=True, eps=1e-6):
        d = GEOM[kind]["d"]
        g = torch.Generator().manual_seed(seed)
        draw = lambda: (torch.rand(d, generator=g, dtype=torch.float32) + 0.5).to(torch.bfloat16)
        self.wq = draw() if q else None
        self.wk = draw() if k else None
        self.dev = [None if w is None else w.cuda() for w in (self.wq, self.wk)]
        self.arg = g4.make_norms(self.dev[0], self.dev[1], v, eps)
        self.oracle = oracle.Norms(q_weight=None if self.wq is None else self.wq.double().numpy(),
                                   k_weight=None if self.wk is None else self.wk.double().numpy(), v_norm=v, eps=eps)


class Batch:
    """A prefill batch: per-sequence histories (positions 0 .. ctx_start+q_len-1) and the new rows."""

    def __init__(self, kind, q_lens, ctx_starts=None, padded=False, seed=0, scale=1.0, pad_to=None,
                 spare_pages=3, page_seed=None, spans=None):
        self.kind = kind
        self.spans = spans   # per sequence: its images as [s0, s1) position ranges, or None
        geo = GEOM[kind]
        self.n_kv, self.d = geo["n_kv"], geo["d"]
        self.q_lens = [int(x) for x in q_lens]
        self.ctx_starts = [0] * len(q_lens) if ctx_starts is None else [int(c) for c in ctx_starts]
        self.layout = (gi.padded_layout(self.q_lens, self.ctx_starts, pad_to) if padded
                       else gi.packed_layout(self.q_lens, self.ctx_starts))
        self.ctx_lens = [c + L for c, L in zip(self.ctx_starts, self.q_lens)]
        self.q, self.hist_k, self.hist_v = gi.prefill_tensors(kind, self.q_lens, self.layout, 32, self.n_kv,
                                                              self.d, seed, scale, self.ctx_lens)
        self.k_rows = gi.rows_of(self.hist_k, self.layout)
        self.v_rows = None if self.hist_v is None else gi.rows_of(self.hist_v, self.layout)
        self.plan = gi.make_page_plan(self.ctx_lens, seed=seed + 17 if page_seed is None else page_seed,
                                      spare_pages=spare_pages)

    def device_cache(self) -> PagedKV:
        return PagedKV(self.plan.num_pages, self.n_kv, self.d, shared=(self.kind == "global"))

    def append_history(self, layer, cache: PagedKV, table, norms=None):
        """Writes every sequence's rows before ctx_start into the cache with g4attn_kv_append."""
        if max(self.ctx_starts) == 0:
            return
        lens = list(self.ctx_starts)
        lay = gi.packed_layout([max(L, 0) for L in lens])
        k = gi.rows_of([h[:L] for h, L in zip(self.hist_k, lens)], lay, fill_nan=False).cuda()
        v = None if self.hist_v is None else gi.rows_of([h[:L] for h, L in zip(self.hist_v, lens)], lay,
                                                        fill_nan=False).cuda()
        rows = (device_int32(lay.q_start), device_int32(lay.q_len), device_int32([0] * len(lens)))
        if norms is None:
            g4.g4attn_kv_append(layer, k, v, *rows, cache.desc, table)
        else:
            g4.g4attn_kv_append_normed(layer, norms.arg, k, v, *rows, cache.desc, table)

    def span_rows(self) -> torch.Tensor:
        """int32 [T, 2]: each sequence row's image span, (0, 0) for text rows, and for gap rows
        values that would be refused if the kernels read them."""
        t = torch.tensor([[-7, 1 << 30]] * self.layout.T, dtype=torch.int32).reshape(-1, 2)
        for b, L in enumerate(self.q_lens):
            s, c = self.layout.q_start[b], self.ctx_starts[b]
            for r in range(L):
                t[s + r] = torch.tensor([0, 0])
                for s0, s1 in (self.spans[b] if self.spans else []):
                    if s0 <= c + r < s1:
                        t[s + r] = torch.tensor([s0, s1])
        return t

    def run(self, layer, out_fill=float("nan"), split=False, norms=None):
        """One prefill of the batch: g4attn_prefill; split="append": g4attn_kv_append then
        g4attn_prefill_attend on the raw queries (the launches of g4attn_prefill called apart);
        split=True: the staged form, g4attn_prefill_stage then g4attn_prefill_attend on the staged
        queries; with spans, g4attn_prefill_vision."""
        cache = self.device_cache()
        table = self.plan.table.cuda()
        self.append_history(layer, cache, table, norms)
        q = self.q.cuda()
        k = self.k_rows.cuda()
        v = None if self.v_rows is None else self.v_rows.cuda()
        out = torch.full_like(q, out_fill)
        rows = (device_int32(self.layout.q_start), device_int32(self.layout.q_len), device_int32(self.layout.ctx_start))
        if self.spans is not None:
            g4.g4attn_prefill_vision(layer, None if norms is None else norms.arg, q, k, v, *rows,
                                     self.span_rows().cuda(), cache.desc, table, out)
        elif norms is not None:
            g4.g4attn_prefill_normed(layer, norms.arg, q, k, v, *rows, cache.desc, table, out)
        elif split == "append":   # the two launches of g4attn_prefill called apart
            g4.g4attn_kv_append(layer, k, v, *rows, cache.desc, table)
            g4.g4attn_prefill_attend(layer, q, *rows, cache.desc, table, out)
        elif split:               # the staged form: roped queries staged in out, then attention
            g4.g4attn_prefill_stage(layer, q, k, v, *rows, cache.desc, table, out)
            g4.g4attn_prefill_attend(layer, None, *rows, cache.desc, table, out)
        else:
            g4.g4attn_prefill(layer, q, k, v, *rows, cache.desc, table, out)
        torch.cuda.synchronize()
        st = g4.g4attn_status_sync()
        assert st == g4.G4_OK, g4.status_string(st)
        return out, cache

    def oracle_rows(self, olayer, b, rows=None, norms=None):
        """fp64 answer for sequence b's new rows (all of them, or the given row indices)."""
        L, c, s = self.q_lens[b], self.ctx_starts[b], self.layout.q_start[b]
        idx = np.arange(L) if rows is None else np.asarray(rows)
        q = self.q[s + idx].double().numpy()
        v = None if self.hist_v is None else self.hist_v[b].double().numpy()
        return oracle.layer_rows(olayer, q, c + idx, self.hist_k[b].double().numpy(), v, 0,
                                 None if norms is None else norms.oracle,
                                 self.spans[b] if self.spans else None)


class DecodeBatch:
    """One decode step for B requests with contexts ctx_lens (the new token included)."""

    def __init__(self, kind, ctx_lens, seed=0, scale=1.0, window=1024, sliding_window_only=False,
                 page_seed=None):
        self.kind = kind
        geo = GEOM[kind]
        self.n_kv, self.d = geo["n_kv"], geo["d"]
        self.ctx_lens = [int(x) for x in ctx_lens]
        B = len(ctx_lens)
        self.hist_k, self.hist_v = [], []
        for b, L in enumerate(self.ctx_lens):
            sb = seed * 1000003 + b * 7919
            self.hist_k.append(gi.bf16_normal((L, self.n_kv, self.d), sb + 2, scale))
            if kind == "sliding":
                self.hist_v.append(gi.bf16_normal((L, self.n_kv, self.d), sb + 3, scale))
        self.q = torch.stack([gi.bf16_normal((32, self.d), seed * 1000003 + b * 7919 + 1, scale) for b in range(B)])
        first = None
        if sliding_window_only and kind == "sliding":
            first = [max(0, (L - window)) // 16 for L in self.ctx_lens]   # pages the window never reads stay -1
        self.plan = gi.make_page_plan(self.ctx_lens, seed=seed + 29 if page_seed is None else page_seed,
                                      mapped_from=first, spare_pages=5)
        self.first_page = first

    def run(self, layer, cache: PagedKV = None, norms=None, exact=False):
        """g4attn_decode (or g4attn_decode_normed); exact: g4attn_decode_exact on the smallest
        workspace it accepts."""
        B = len(self.ctx_lens)
        table = self.plan.table.cuda()
        if cache is None:
            cache = PagedKV(self.plan.num_pages, self.n_kv, self.d, shared=(self.kind == "global"))
            # history before the new token, written by the library itself
            lens = [L - 1 for L in self.ctx_lens]
            starts = [0] * B if self.first_page is None else [16 * f for f in self.first_page]
            lens = [L - s for L, s in zip(lens, starts)]
            lay = gi.packed_layout([max(L, 0) for L in lens], starts)
            if lay.T > 0 and sum(lens) > 0:
                k = gi.rows_of(self.hist_k, lay, fill_nan=False).cuda()
                v = None if self.kind == "global" else gi.rows_of(self.hist_v, lay, fill_nan=False).cuda()
                rows = (device_int32(lay.q_start), device_int32(lay.q_len), device_int32(lay.ctx_start))
                if norms is None:
                    g4.g4attn_kv_append(layer, k, v, *rows, cache.desc, table)
                else:
                    g4.g4attn_kv_append_normed(layer, norms.arg, k, v, *rows, cache.desc, table)
        k_new = torch.stack([h[L - 1] for h, L in zip(self.hist_k, self.ctx_lens)]).cuda()
        v_new = None if self.kind == "global" else torch.stack(
            [h[L - 1] for h, L in zip(self.hist_v, self.ctx_lens)]).cuda()
        q = self.q.cuda()
        out = torch.full_like(q, float("nan"))
        ws = torch.empty(g4.g4attn_decode_workspace_bytes(layer, B, self.plan.max_pages), dtype=torch.uint8,
                         device="cuda")
        if exact:
            ws = torch.empty(g4.g4attn_decode_exact_workspace_bytes(B), dtype=torch.uint8, device="cuda")
            g4.g4attn_decode_exact(layer, None if norms is None else norms.arg, q, k_new, v_new,
                                   device_int32(self.ctx_lens), cache.desc, table, out, ws)
        elif norms is None:
            g4.g4attn_decode(layer, q, k_new, v_new, device_int32(self.ctx_lens), cache.desc, table, out, ws)
        else:
            g4.g4attn_decode_normed(layer, norms.arg, q, k_new, v_new, device_int32(self.ctx_lens), cache.desc, table,
                                    out, ws)
        torch.cuda.synchronize()
        st = g4.g4attn_status_sync()
        assert st == g4.G4_OK, g4.status_string(st)
        return out, cache

    def oracle_row(self, olayer, b, norms=None):
        v = None if self.kind == "global" else self.hist_v[b].double().numpy()
        return oracle.decode_row(olayer, self.q[b].double().numpy(), self.hist_k[b].double().numpy(), v,
                                 None if norms is None else norms.oracle)
