#!/usr/bin/env python
"""Throughput of the hybrid batch-invariant attention hot path on GB300.

One step runs the whole path once over seeded synthetic inputs already resident in HBM:
  1. sliding-window prefill, 4 sequences x 4096 tokens (Q 32x256, KV 16x256, window 1024,
     RoPE theta 1e4, values N(0,1) x 0.5), paged cache with 16-token pages;
  2. global K==V prefill, 2 x 8192 (Q 32x512, 4 shared K=V heads x 512, p-RoPE 0.25, theta 1e6);
  3. one decode pass of the 5 sliding : 1 global mix: 64 requests, one query each, contexts
     uniform in [1024, 32768] (seed 7), one cache per layer filled through g4attn_kv_append, pages
     scattered by random permutations.
Each part is timed with CUDA events on the launching stream after an L2 flush (a 512 MB write); a
prefill part runs its two launches through g4attn_kv_append and g4attn_prefill_attend (exactly
g4attn_prefill) with an event between them, so the attention kernel is timed on its own. After the timed region, sampled outputs of the last step are checked against
the fp64 oracle; a miss ends the run without a result line. The end-to-end figures then time the
same parts through the public calls with host buffers (pinned host -> device inputs and device ->
host outputs inside the timed region).

Headline value: prefill TFLOP/s (credited FLOPs of parts 1+2 over their time); the decode part
reports KV GB/s. Both also as fractions of the measured GB300 peaks.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl g4attn|reference]

--impl reference times the fp64 CPU oracle (the method is published without installable code) on a bounded
sample of the same workload, on the host cores. With N > 1 (torchrun) every rank runs an
independent replica (the path has no exchange step); rank 0 prints one JSON line.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "prefill TFLOP/s & decode KV GB/s (% GB300 roofline), bitwise batch-invariant"
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0, "source": "fallback"}
WORKLOAD = ("hybrid attention step: sliding prefill 4x4096 (W1024) + global K==V prefill 2x8192 + "
            "decode mix B=64 ctx U[1024,32768] 5 sliding:1 global; Hq32, sliding Hkv16/D256, global Hkv4/D512")


def peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        d = json.load(open(p))
        return {"hbm_gbs": float(d["hbm_gbs"]), "bf16_tflops": float(d["bf16_tflops"]),
                "bf16_tflops_sustained": float(d.get("bf16_tflops_sustained", d["bf16_tflops"])),
                "source": "measured"}
    return dict(FALLBACK_PEAKS)


# ---------------------------------------------------------------- credited work (closed forms)

def sliding_pairs(L: int, W: int) -> int:
    """Visible (query, key) pairs of one causal sequence of length L with window W."""
    if W <= 0 or W >= L:
        return L * (L + 1) // 2
    return W * (W + 1) // 2 + (L - W) * W


def prefill_flops(D: int, Hq: int, lens, W: int) -> float:
    return 4.0 * D * Hq * sum(sliding_pairs(L, W) for L in lens)


# ---------------------------------------------------------------- clocks sampling

class Clocks:
    """nvidia-smi sampler (50 ms) started before the warm-up; summary() keeps the samples whose
    timestamps fall inside the timed region [t0, t1] (host wall clock)."""
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap,timestamp")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.path = None

    def __enter__(self):
        fd, self.path = tempfile.mkstemp(suffix=".csv")
        os.close(fd)
        try:
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}",
                                          "--format=csv,noheader,nounits", "-lms", "50"],
                                         stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
        except OSError:
            self.proc = None
        return self

    def __exit__(self, *exc):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    @staticmethod
    def _when(stamp: str):
        import datetime
        try:
            return datetime.datetime.strptime(stamp.strip(), "%Y/%m/%d %H:%M:%S.%f").timestamp()
        except ValueError:
            return None

    def summary(self, t0: float, t1: float):
        rows = []
        if self.path and os.path.exists(self.path):
            for line in open(self.path):
                f = [x.strip() for x in line.split(",")]
                if len(f) >= 10:
                    rows.append(f)
            os.unlink(self.path)
        inside = [r for r in rows if (self._when(r[9]) or 0.0) >= t0 and (self._when(r[9]) or 0.0) <= t1]
        rows = inside
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"], "samples": 0}

        def num(x):
            try:
                return float(x)
            except ValueError:
                return None
        sm = [num(r[1]) for r in rows if num(r[1]) is not None]
        mx = [num(r[2]) for r in rows if num(r[2]) is not None]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({n for r in rows for n, v in zip(names, r[5:9]) if v.strip().lower() == "active"})
        loaded = [s for s in sm if mx and s >= 0.5 * max(mx)] or sm
        return {"sm_mhz": statistics.median(loaded) if loaded else None, "sm_max_mhz": max(mx) if mx else None,
                "reasons": reasons, "samples": len(rows), "window_s": round(t1 - t0, 3),
                "power_w_max": max((num(r[3]) or 0.0) for r in rows)}


# ---------------------------------------------------------------- the GPU parts

def sample_rows(L: int, n: int, seed: int):
    """Sorted query rows of a length-L sequence to check: rows 0, 1023, 1024 and L-1, both rows at
    every 128-row tile edge, then seeded random rows up to n in all."""
    import numpy as np
    pick = {0, L - 1} | {r for r in (1023, 1024) if r < L}
    for t in range(128, L, 128):
        pick |= {t - 1, t}
    for r in np.random.default_rng(seed).permutation(L):
        if len(pick) >= n:
            break
        pick.add(int(r))
    return np.array(sorted(pick), dtype=np.int64)


class SlidingPrefill:
    """Sliding-window prefill, 4 causal sequences x 4096 (Q 32x256, KV 16x256, window 1024, RoPE
    theta 1e4), values N(0,1) x 0.5 drawn on the device (seed 1), pages scattered by a seeded
    permutation. The sequences are packed with ctx_start 0."""
    name = "sliding_prefill"
    kind = "sliding"

    def __init__(self, g4, gi, PagedKV, device_int32, n=4, L=4096, W=1024, seed=1, scale=0.5):
        import torch
        self.g4, self.layer, self.W = g4, g4.sliding_layer(W), W
        self.lens = [L] * n
        lay = gi.packed_layout(self.lens)
        self.T, self.q_start = lay.T, lay.q_start
        self.q = gi.bf16_normal_device((self.T, 32, 256), seed * 101 + 1, scale)
        self.k = gi.bf16_normal_device((self.T, 16, 256), seed * 101 + 2, scale)
        self.v = gi.bf16_normal_device((self.T, 16, 256), seed * 101 + 3, scale)
        self.plan = gi.make_page_plan(self.lens, seed=seed + 17)
        self.cache = PagedKV(self.plan.num_pages, 16, 256, shared=False, fill=None)
        self.table = self.plan.table.cuda()
        self.qs, self.ql, self.cs = (device_int32(x) for x in (lay.q_start, lay.q_len, lay.ctx_start))
        self.out = torch.empty_like(self.q)
        self.flops = prefill_flops(256, 32, self.lens, W)
        self.launches = 2   # the K'/V append by key groups, then attention

    def run(self):
        self.g4.g4attn_prefill(self.layer, self.q, self.k, self.v, self.qs, self.ql, self.cs, self.cache.desc,
                               self.table, self.out)

    def run_stage(self):   # launch 1 of g4attn_prefill: the cache append
        self.g4.g4attn_kv_append(self.layer, self.k, self.v, self.qs, self.ql, self.cs, self.cache.desc, self.table)

    def run_attend(self):  # launch 2: the attention kernel, rotating the raw queries itself
        self.g4.g4attn_prefill_attend(self.layer, self.q, self.qs, self.ql, self.cs, self.cache.desc, self.table,
                                      self.out)

    def host_io(self):
        return [self.q, self.k, self.v], [self.out]

    def oracle_layer(self):
        import oracle
        return oracle.with_window(oracle.SLIDING, self.W) if self.kind == "sliding" else oracle.GLOBAL

    def check(self, rows_per_seq: int, seed: int = 0):
        """(got, want) of sampled output rows of every sequence against the fp64 oracle, which sees
        the same input values (read back from the device) and nothing the library computed."""
        import oracle
        olayer = self.oracle_layer()
        res = []
        for b, L in enumerate(self.lens):
            s = self.q_start[b]
            rows = sample_rows(L, rows_per_seq, seed + b)
            k = self.k[s:s + L].float().cpu().double().numpy()
            v = None if self.v is None else self.v[s:s + L].float().cpu().double().numpy()
            q = self.q[s + rows].float().cpu().double().numpy()
            want = oracle.layer_rows(olayer, q, rows, k, v)
            got = self.out[s + rows].float().cpu().double().numpy()
            res.append((f"{self.name} seq {b}", rows, got, want))
        return res


class GlobalPrefill(SlidingPrefill):
    """Global K==V prefill, 2 causal sequences x 8192 (Q 32x512, 4 shared K=V heads x 512, p-RoPE
    partial 0.25, theta 1e6), N(0,1) values drawn on the device (seed 2)."""
    name = "global_prefill"
    kind = "global"

    def __init__(self, g4, gi, PagedKV, device_int32, n=2, L=8192, seed=2, scale=1.0):
        import torch
        self.g4, self.layer, self.W = g4, g4.global_layer(), 0
        self.lens = [L] * n
        lay = gi.packed_layout(self.lens)
        self.T, self.q_start = lay.T, lay.q_start
        self.q = gi.bf16_normal_device((self.T, 32, 512), seed * 101 + 1, scale)
        self.k = gi.bf16_normal_device((self.T, 4, 512), seed * 101 + 2, scale)
        self.v = None
        self.plan = gi.make_page_plan(self.lens, seed=seed + 17)
        self.cache = PagedKV(self.plan.num_pages, 4, 512, shared=True, fill=None)
        self.table = self.plan.table.cuda()
        self.qs, self.ql, self.cs = (device_int32(x) for x in (lay.q_start, lay.q_len, lay.ctx_start))
        self.out = torch.empty_like(self.q)
        self.flops = prefill_flops(512, 32, self.lens, 0)
        self.launches = 2

    def host_io(self):
        return [self.q, self.k], [self.out]


class DecodeMix:
    """One decode pass over the 5 sliding : 1 global mix: B = 64 requests, one query each, context
    lengths uniform in [1024, 32768] (seed 7), one cache per layer. Each cache is filled through
    g4attn_kv_append from seeded per-request key (and value) rows, so that it holds exactly what a
    prefill of those rows leaves (sliding K' = RoPE(k), V; global S and its roped columns). A sliding
    cache maps only the pages of each request's window, in a random permutation; the global cache
    maps every page. The timed decode call appends each request's last row (the new token) and
    attends."""
    name = "decode_mix"

    def __init__(self, g4, gi, PagedKV, device_int32, B=64, W=1024):
        import torch
        wl = gi.DECODE_MIX
        self.g4, self.gi, self.W, self.wl = g4, gi, W, wl
        self.lens = gi.decode_mix_lengths(wl)[:B]
        B = len(self.lens)
        self.B = B
        self.seq_len = device_int32(self.lens)
        self.sl, self.gl = g4.sliding_layer(W), g4.global_layer()
        self.n_sliding = wl.n_sliding
        self.layers = []
        for i in range(wl.n_sliding + wl.n_global):
            sliding = i < wl.n_sliding
            n_kv, d = (16, 256) if sliding else (4, 512)
            layer = self.sl if sliding else self.gl
            first = gi.decode_mix_first_keys(self.lens, W) if sliding else [0] * B
            plan = gi.make_page_plan(self.lens, seed=wl.length_seed * 31 + (i if sliding else 99),
                                     mapped_from=[f // 16 for f in first])
            cache = PagedKV(plan.num_pages, n_kv, d, shared=not sliding, fill=None)
            table = plan.table.cuda()
            ks, vs, k_new, v_new = [], [], [], []
            for b, L in enumerate(self.lens):
                k, v = gi.decode_mix_values(wl.value_seed, i, b, L - first[b], n_kv, d, sliding)
                ks.append(k[:-1])
                k_new.append(k[-1])
                if sliding:
                    vs.append(v[:-1])
                    v_new.append(v[-1])
            lay = gi.packed_layout([L - f - 1 for L, f in zip(self.lens, first)], first)
            rows = (device_int32(lay.q_start), device_int32(lay.q_len), device_int32(lay.ctx_start))
            g4.g4attn_kv_append(layer, torch.cat(ks), torch.cat(vs) if sliding else None, *rows, cache.desc, table)
            del ks, vs
            q = gi.decode_mix_queries(wl.value_seed, i, B, d)
            self.layers.append({"sliding": sliding, "layer": layer, "cache": cache, "table": table, "first": first,
                                "q": q, "k_new": torch.stack(k_new),
                                "v_new": torch.stack(v_new) if sliding else None, "out": torch.empty_like(q)})
        torch.cuda.synchronize()
        st = g4.g4attn_status_sync()
        if st != g4.G4_OK:
            raise SystemExit(f"device error while filling the decode caches: {g4.status_string(st)}")
        self.ws = {}
        for sliding, layer in ((True, self.sl), (False, self.gl)):
            mp = max(int(L["table"].shape[1]) for L in self.layers if L["sliding"] == sliding)
            self.ws[sliding] = torch.empty(g4.g4attn_decode_workspace_bytes(layer, B, mp), dtype=torch.uint8,
                                           device="cuda")
        qo_s = B * 32 * 256 * 2 * 2
        qo_g = B * 32 * 512 * 2 * 2
        self.bytes_sliding = sum(min(L, W) for L in self.lens) * 16 * 256 * 2 * 2 + qo_s
        self.bytes_global = sum(self.lens) * 4 * 512 * 2 + qo_g   # credited: S once (the k_rot reads are not)
        self.bytes = self.n_sliding * self.bytes_sliding + self.bytes_global
        self.launches = 3 * len(self.layers)

    def run_layer(self, i, exact=False):
        L = self.layers[i]
        if exact:
            self.g4.g4attn_decode_exact(L["layer"], None, L["q"], L["k_new"], L["v_new"], self.seq_len,
                                        L["cache"].desc, L["table"], L["out"], self.ws[L["sliding"]])
        else:
            self.g4.g4attn_decode(L["layer"], L["q"], L["k_new"], L["v_new"], self.seq_len, L["cache"].desc,
                                  L["table"], L["out"], self.ws[L["sliding"]])

    def run_sliding(self, i):
        self.run_layer(i)

    def run_global(self):
        self.run_layer(self.n_sliding)

    def run(self):
        for i in range(len(self.layers)):
            self.run_layer(i)

    # The same steps through g4attn_decode_exact (the prefill kernels on one-row chunks): rows with
    # a prefill's bits. Timed apart from the step, as the opt-in strict mode's cost.
    def run_sliding_exact(self, i):
        self.run_layer(i, exact=True)

    def run_global_exact(self):
        self.run_layer(self.n_sliding, exact=True)

    def host_io(self):
        ins = []
        for L in self.layers:
            ins += [L["q"], L["k_new"]] + ([L["v_new"]] if L["sliding"] else [])
        return ins, [L["out"] for L in self.layers]

    def check_request(self, i: int, b: int):
        """(got, want) of request b's output on layer i against the fp64 oracle, from the request's
        key (and value) rows drawn again with their seed."""
        import oracle
        L = self.layers[i]
        n_kv, d = (16, 256) if L["sliding"] else (4, 512)
        f, n = L["first"][b], self.lens[b]
        k, v = self.gi.decode_mix_values(self.wl.value_seed, i, b, n - f, n_kv, d, L["sliding"])
        olayer = oracle.with_window(oracle.SLIDING, self.W) if L["sliding"] else oracle.GLOBAL
        want = oracle.layer_rows(olayer, L["q"][b:b + 1].float().cpu().double().numpy(), [n - 1 - f],
                                 k.float().cpu().double().numpy(),
                                 None if v is None else v.float().cpu().double().numpy(), pos_offset=f)[0]
        return L["out"][b].float().cpu().double().numpy(), want


TOL_MAX, TOL_MEAN = 2e-2, 2e-3   # max-abs and mean-abs bars on bf16 outputs against the fp64 oracle


def verify_outputs(parts, dec, rows_per_seq: int = 8, requests: int = 4):
    """Checks sampled outputs of the step just timed against the fp64 oracle: rows_per_seq rows of
    every prefill sequence (its first and last among them) and `requests` requests of the first
    sliding layer and of the global layer of the decode mix (the longest among them). Returns a
    summary; raises SystemExit when any comparison misses the bars, so nothing is printed then."""
    import numpy as np
    cases = []
    for p in parts:
        cases += [(n, g, w) for n, _, g, w in p.check(rows_per_seq)]
    if dec is not None:
        longest = int(np.argmax(dec.lens))
        pick = sorted({longest} | set(range(min(requests - 1, dec.B))))
        for i in (0, dec.n_sliding):
            for b in pick:
                g, w = dec.check_request(i, b)
                cases.append((f"decode layer {i} request {b} (ctx {dec.lens[b]})", g, w))
    worst_max, worst_mean = 0.0, 0.0
    pick = pick if dec is not None else []
    for name, got, want in cases:
        d = np.abs(got - want)
        mx, mean = float(d.max()), float(d.mean())
        if not np.isfinite(got).all() or mx > TOL_MAX or mean > TOL_MEAN:
            raise SystemExit(f"output check failed: {name}: max-abs {mx:.3e}, mean-abs {mean:.3e}")
        worst_max, worst_mean = max(worst_max, mx), max(worst_mean, mean)
    return {"checked": len(cases), "max_abs": worst_max, "mean_abs_worst": worst_mean,
            "bars": {"max_abs": TOL_MAX, "mean_abs": TOL_MEAN}, "against": "fp64 oracle (oracle/core.py)",
            "what": f"{rows_per_seq} rows per prefill sequence; {len(pick)} requests "
                    f"of decode layers 0 (sliding) and {dec.n_sliding if dec is not None else '-'} (global)"}


# ---------------------------------------------------------------- timing helpers

def exact_decode_times(dec, flush, reps):
    """ms per layer of the decode mix through g4attn_decode_exact (after two warm-up calls each),
    CUDA events around each call, L2 flushed before each; outside the timed step."""
    import torch

    out = {}
    for name, fn in (("sliding_layer_ms", lambda: dec.run_sliding_exact(0)), ("global_layer_ms", dec.run_global_exact)):
        fn()
        fn()
        ts = []
        for _ in range(reps):
            flush()
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record()
            fn()
            b.record()
            torch.cuda.synchronize()
            ts.append(a.elapsed_time(b))
        out[name] = statistics.median(ts)
    st = dec.g4.g4attn_status_sync()
    if st != dec.g4.G4_OK:
        raise SystemExit(f"device error in the exact decode calls: {dec.g4.status_string(st)}")
    out["mix_ms"] = dec.n_sliding * out["sliding_layer_ms"] + out["global_layer_ms"]
    out["note"] = ("g4attn_decode_exact: rows bit-identical to a prefill's; 3 launches per call; "
                   "not part of the timed step")
    return out


def traffic_record(kernel: str):
    """DRAM bytes per launch from the committed ncu summary, if it was taken on the current sources
    (the hash covers every source file the kernel is built from); None otherwise."""
    p = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(p):
        return None
    rec = json.load(open(p)).get(kernel)
    if not rec:
        return None
    h = hashlib.sha256()
    for name in rec["sources"]:
        src = os.path.join(ROOT, "invariant_hybrid_attention_gb300", "csrc", name)
        if not os.path.exists(src):
            return None
        h.update(open(src, "rb").read())
    if h.hexdigest()[:16] != rec["sha256_16"]:
        return None
    return rec["dram_bytes_per_launch"]


# ---------------------------------------------------------------- the CPU oracle leg

def oracle_sample(budget_s: float, seed: int = 1):
    """The fp64 oracle, as it stands, on a bounded sample of the step's workload, about a third of
    `budget_s` on each part: sampled query rows of a sliding-prefill sequence (4096 keys, W 1024,
    values N(0,1) x 0.5), sampled rows of a global-prefill sequence (8192 keys), and whole decode
    requests of the decode mix (one sliding and one global layer, contexts of the mix). Inputs come
    from the CPU generator with the workloads' recipes. Returns a dict: prefill TFLOP/s (credited
    FLOPs of the rows done over their time), decode GB/s (credited bytes over time), and counts."""
    import numpy as np
    import oracle
    from invariant_hybrid_attention_gb300 import inputs as gi
    rng = np.random.default_rng(seed)
    part = budget_s / 3.0
    flops, pre_t, rows = 0.0, 0.0, {"sliding": 0, "global": 0}
    for kind, L, D, hkv, scale, W in (("sliding", 4096, 256, 16, 0.5, 1024), ("global", 8192, 512, 4, 1.0, 0)):
        lay = oracle.with_window(oracle.SLIDING, W) if kind == "sliding" else oracle.GLOBAL
        k = gi.bf16_normal((L, hkv, D), seed * 101 + 2, scale).double().numpy()
        v = gi.bf16_normal((L, hkv, D), seed * 101 + 3, scale).double().numpy() if kind == "sliding" else None
        spent = 0.0
        while spent < part:
            pos = np.sort(rng.choice(L, 16, replace=False))
            q = gi.bf16_normal((16, 32, D), int(rng.integers(1 << 30)), scale).double().numpy()
            hi = int(pos.max()) + 1
            t0 = time.perf_counter()
            oracle.layer_rows(lay, q, pos, k[:hi], None if v is None else v[:hi])
            spent += time.perf_counter() - t0
            flops += sum(4.0 * D * 32 * (min(int(p) + 1, W) if W else int(p) + 1) for p in pos)
            rows[kind] += 16
        pre_t += spent
    lens = gi.decode_mix_lengths()
    dec_bytes, dec_t, reqs = 0.0, 0.0, 0
    while dec_t < part:   # only the oracle calls are timed, not the drawing of their inputs
        b = int(rng.integers(len(lens)))
        n = lens[b]
        for kind in ("sliding", "global"):
            D, hkv = (256, 16) if kind == "sliding" else (512, 4)
            lay = oracle.with_window(oracle.SLIDING, 1024) if kind == "sliding" else oracle.GLOBAL
            f = gi.decode_mix_first_keys([n], 1024)[0] if kind == "sliding" else 0
            k = gi.bf16_normal((n - f, hkv, D), reqs * 2 + 1).double().numpy()
            v = gi.bf16_normal((n - f, hkv, D), reqs * 2 + 2).double().numpy() if kind == "sliding" else None
            q = gi.bf16_normal((1, 32, D), reqs * 2 + 3).double().numpy()
            t0 = time.perf_counter()
            oracle.layer_rows(lay, q, [n - 1 - f], k, v, pos_offset=f)
            dec_t += time.perf_counter() - t0
            dec_bytes += (min(n, 1024) * hkv * D * 2 * 2 if kind == "sliding" else n * hkv * D * 2) + 32 * D * 2 * 2
        reqs += 1
    return {"prefill_tflops": flops / pre_t / 1e12, "decode_gbs": dec_bytes / dec_t / 1e9,
            "rows": rows, "requests": reqs, "seconds": pre_t + dec_t}


def oracle_sample_text(r) -> str:
    return (f"fp64 oracle on {r['rows']['sliding']} query rows x 32 heads of the sliding prefill 4x4096 (W1024), "
            f"{r['rows']['global']} rows x 32 heads of the global prefill 2x8192, and {r['requests']} decode-mix "
            f"requests on one sliding and one global layer; {r['seconds']:.1f}s of CPU time")


def max_over_ranks(ms: dict, dist, device) -> dict:
    """Each named time (ms) as the maximum over all ranks: the job is as slow as its slowest rank."""
    import torch
    names = sorted(ms)
    t = torch.tensor([float(ms[n]) for n in names], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return dict(zip(names, (float(x) for x in t.tolist())))


def job_tflops(flops_per_step: float, steps: int, world: int, ms: float):
    """Whole-job throughput: the work of all ranks (replicas) over the max-over-ranks time."""
    return flops_per_step * steps * world / (ms * 1e-3) / 1e12 if ms > 0 else None


def cpu_cores():
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:
        return os.cpu_count() or 1


def run_reference(args, rank, world):
    if rank != 0:
        return 0
    per_step = max(3.0, min(20.0, 120.0 / max(1, args.steps + args.warmup)))
    for _ in range(args.warmup):
        oracle_sample(per_step / 4)
    res, ts = [], []
    for _ in range(args.steps):
        r = oracle_sample(per_step)
        res.append(r)
        ts.append(r["seconds"] * 1e3)
    val = statistics.median(r["prefill_tflops"] for r in res)
    tot = {"rows": {"sliding": sum(r["rows"]["sliding"] for r in res), "global": sum(r["rows"]["global"] for r in res)},
           "requests": sum(r["requests"] for r in res), "seconds": sum(r["seconds"] for r in res)}
    cores = cpu_cores()
    line = {"impl": "reference", "metric": METRIC, "value": val, "unit": "TFLOP/s", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": statistics.median(ts),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic (seeded N(0,1) bf16 values, CPU generator)",
            "config": {"workload": WORKLOAD, "reference": "fp64 numpy oracle (oracle/core.py), sampled rows"},
            "decode": {"value": statistics.median(r["decode_gbs"] for r in res), "unit": "GB/s"},
            "cpu_baseline": {"value": val, "unit": "TFLOP/s", "cores": cores, "kind": "oracle",
                             "sample": oracle_sample_text(tot)},
            "e2e": {"value": val, "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)
    return 0


# ---------------------------------------------------------------- main

def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=30)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", default="g4attn", choices=["g4attn", "reference"])
    ap.add_argument("--parts", default="sliding,global,decode")
    ap.add_argument("--cpu-budget", type=float, default=12.0, help="seconds of oracle time for cpu_baseline")
    ap.add_argument("--exact-decode-reps", type=int, default=5,
                    help="timed calls per layer kind of g4attn_decode_exact after the step (0: skip)")
    ap.add_argument("--decode-batch", type=int, default=64,
                    help="requests in the decode mix (64 is the measured workload; smaller only for profiling)")
    ap.add_argument("--check-rows", type=int, default=8,
                    help="output rows per prefill sequence checked against the fp64 oracle after the timed region")
    args = ap.parse_args()
    if args.warmup < 3:
        args.warmup = 3

    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if args.impl == "reference":
        return run_reference(args, rank, world)

    import torch
    torch.cuda.set_device(local)
    dist = None
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))

    # cpu_baseline first (rank 0, N = 1 only), before any large GPU work
    cpu = None
    if rank == 0 and world == 1 and args.cpu_budget > 0:
        r = oracle_sample(args.cpu_budget)
        cpu = {"value": r["prefill_tflops"], "unit": "TFLOP/s", "cores": cpu_cores(), "kind": "oracle",
               "decode": {"value": r["decode_gbs"], "unit": "GB/s"}, "sample": oracle_sample_text(r)}

    import invariant_hybrid_attention_gb300 as g4
    from invariant_hybrid_attention_gb300 import build as g4build
    from invariant_hybrid_attention_gb300 import inputs as gi
    from invariant_hybrid_attention_gb300.paged import PagedKV, device_int32
    g4build.build()
    g4.load()

    want = set(args.parts.split(","))
    parts = []
    if "sliding" in want:
        parts.append(SlidingPrefill(g4, gi, PagedKV, device_int32))
    if "global" in want:
        parts.append(GlobalPrefill(g4, gi, PagedKV, device_int32))
    dec = DecodeMix(g4, gi, PagedKV, device_int32, B=args.decode_batch) if "decode" in want else None
    flush_buf = torch.empty(512 * 1024 * 1024, dtype=torch.uint8, device="cuda")

    def flush():
        flush_buf.zero_()

    def step_parts():
        out = []
        for p in parts:
            out.append((p.name, (p.run_stage, p.run_attend)))
        if dec is not None:
            for i in range(dec.n_sliding):
                out.append((f"decode_sliding_{i}", lambda i=i: dec.run_layer(i)))
            out.append(("decode_global", lambda: dec.run_layer(dec.n_sliding)))
        return out

    sp = step_parts()
    clk = Clocks(local).__enter__()   # sampling from before the warm-up; summarised over the timed region
    def call(fn):
        if isinstance(fn, tuple):
            for f in fn:
                f()
        else:
            fn()

    for _ in range(args.warmup):
        for _, fn in sp:
            call(fn)
    torch.cuda.synchronize()
    st = g4.g4attn_status_sync()
    if st != g4.G4_OK:
        raise SystemExit(f"device error after warm-up: {g4.status_string(st)}")

    # ---- timed region: K steps, per-part CUDA events, L2 flushed before each part
    times = {n: [] for n, _ in sp}
    kern_times = {p.name: [] for p in parts}   # the attention launch of each prefill part
    if dist is not None:
        dist.barrier()
    torch.cuda.synchronize()
    t_start = time.time()
    for _ in range(args.steps):
        evs = []
        for n, fn in sp:
            flush()
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            m = None
            a.record()
            if isinstance(fn, tuple):   # prefill: stage, event, attend
                fn[0]()
                m = torch.cuda.Event(enable_timing=True)
                m.record()
                fn[1]()
            else:
                fn()
            b.record()
            evs.append((n, a, m, b))
        torch.cuda.synchronize()
        for n, a, m, b in evs:
            times[n].append(a.elapsed_time(b))
            if m is not None:
                kern_times[n].append(m.elapsed_time(b))
    torch.cuda.synchronize()
    t_end = time.time()
    clk.__exit__(None, None, None)
    if dist is not None:
        dist.barrier()
    clocks = clk.summary(t_start, t_end)
    st = g4.g4attn_status_sync()
    if st != g4.G4_OK:
        raise SystemExit(f"device error in the timed region: {g4.status_string(st)}")
    # the outputs of the last timed step, checked against the oracle before anything is reported
    check = verify_outputs(parts, dec, rows_per_seq=args.check_rows) if rank == 0 else None

    tot = {n: sum(v) for n, v in times.items()}          # ms over K steps
    ktot = {n: sum(v) for n, v in kern_times.items()}
    if dist is not None:
        tot = max_over_ranks(tot, dist, "cuda")
        ktot = max_over_ranks(ktot, dist, "cuda")
    K = args.steps
    pk = peaks()
    res = {}
    value = job_tflops(sum(p.flops for p in parts), K, world, sum(tot[p.name] for p in parts))

    # the attention kernel of each prefill part, timed on its own (event between the two launches)
    roofs = []
    for p in parts:
        call = tot[p.name] / K
        kern = ktot[p.name] / K
        ach = p.flops / (kern * 1e-3) / 1e12
        res[p.name] = {"ms": call, "stage_ms": call - kern, "attention_kernel_ms": kern,
                       "tflops_call": p.flops / (call * 1e-3) / 1e12, "tflops_kernel": ach,
                       "frac_of_measured_burst": ach / pk["bf16_tflops"],
                       "frac_of_measured_sustained": ach / pk["bf16_tflops_sustained"],
                       "credited_flops": p.flops}
        kname = "prefill_sliding_kernel" if p.name == "sliding_prefill" else "prefill_global_kernel"
        roofs.append((kern, {"kernel": kname, "bound": "tensor", "achieved": ach, "peak": pk["bf16_tflops"],
                             "unit": "TFLOP/s", "frac": ach / pk["bf16_tflops"],
                             "traffic": traffic_record(kname),
                             "peak_kind": f"bf16 dense burst, {pk['source']}"}))
    decode = None
    if dec is not None:
        s_ms = statistics.mean([tot[f"decode_sliding_{i}"] / K for i in range(dec.n_sliding)])
        g_ms = tot["decode_global"] / K
        d_ms = dec.n_sliding * s_ms + g_ms
        gbs = dec.bytes * world / (d_ms * 1e-3) / 1e9
        decode = {"value": gbs, "unit": "GB/s", "frac_of_measured_hbm": gbs / pk["hbm_gbs"],
                  "frac_of_8TBs_nominal": gbs / 8000.0, "ms": d_ms,
                  "sliding_layer": {"ms": s_ms, "gbs": dec.bytes_sliding / (s_ms * 1e-3) / 1e9,
                                    "credited_bytes": dec.bytes_sliding},
                  "global_layer": {"ms": g_ms, "gbs": dec.bytes_global / (g_ms * 1e-3) / 1e9,
                                   "credited_bytes": dec.bytes_global},
                  "note": "each decode call = append + chunk partials + ordered merge (3 launches)"}
        for nm, ms, by, kname in [("sliding", s_ms, dec.bytes_sliding, "decode_sliding_kernel"),
                                  ("global", g_ms, dec.bytes_global, "decode_global_kernel")]:
            ach = by / (ms * 1e-3) / 1e9
            roofs.append((ms, {"kernel": kname, "bound": "hbm", "achieved": ach, "peak": pk["hbm_gbs"],
                               "unit": "GB/s", "frac": ach / pk["hbm_gbs"], "traffic": traffic_record(kname),
                               "peak_kind": f"HBM copy, {pk['source']}",
                               "duration_from": "whole decode call (3 launches): a lower bound on the kernel"}))
        if args.exact_decode_reps > 0:
            decode["exact"] = exact_decode_times(dec, flush, args.exact_decode_reps)
            decode["exact"]["vs_fast_mix"] = decode["exact"]["mix_ms"] / d_ms
    # dominant kernel: the one the step spends the most time in (per step: decode sliding x5)
    weight = {"decode_sliding_kernel": dec.n_sliding if dec else 0}
    roofs.sort(key=lambda r: -r[0] * weight.get(r[1]["kernel"], 1))
    roofline = roofs[0][1] if roofs else None

    # ---- end to end through the public API with host buffers
    # A step of each group (the prefill parts; the decode mix) copies every part's inputs from pinned
    # host memory, runs the part through its public call (g4attn_prefill; g4attn_decode per layer)
    # and copies its outputs back. Copies run on a second stream, ordered by events: every input copy
    # is issued first, so that a part's inputs land while the parts before it compute, and a part's
    # outputs go back while the parts after it compute. Each group is timed on its own.
    def e2e_group(units):
        hosts = []
        for u in units:
            ins, outs = u.host_io()
            hosts.append((u, ins, outs, [t.cpu().pin_memory() for t in ins],
                          [torch.empty(o.shape, dtype=o.dtype, pin_memory=True) for o in outs]))
        main_s, copy_s = torch.cuda.current_stream(), torch.cuda.Stream()
        ms = []
        for it in range(args.steps + 1):
            flush()
            torch.cuda.synchronize()
            t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            t0.record(main_s)
            copy_s.wait_event(t0)
            landed = []
            with torch.cuda.stream(copy_s):
                for u, ins, outs, hin, hout in hosts:
                    for d, h in zip(ins, hin):
                        d.copy_(h, non_blocking=True)
                    e = torch.cuda.Event()
                    e.record(copy_s)
                    landed.append(e)
            for (u, ins, outs, hin, hout), e in zip(hosts, landed):
                main_s.wait_event(e)
                u.run()
                done = torch.cuda.Event()
                done.record(main_s)
                copy_s.wait_event(done)
                with torch.cuda.stream(copy_s):
                    for d, h in zip(outs, hout):
                        h.copy_(d, non_blocking=True)
            t1.record(copy_s)
            main_s.wait_stream(copy_s)
            torch.cuda.synchronize()
            if it > 0:
                ms.append(t0.elapsed_time(t1))
        st = g4.g4attn_status_sync()
        if st != g4.G4_OK:
            raise SystemExit(f"device error in the end-to-end steps: {g4.status_string(st)}")
        h2d = sum(t.numel() * t.element_size() for h in hosts for t in h[3])
        d2h = sum(t.numel() * t.element_size() for h in hosts for t in h[4])
        return statistics.median(ms), h2d, d2h

    e2e = None
    if parts or dec is not None:
        pm, ph2d, pd2h = e2e_group(parts) if parts else (0.0, 0, 0)
        dm, dh2d, dd2h = e2e_group([dec]) if dec is not None else (0.0, 0, 0)
        e2e = {"value": (sum(p.flops for p in parts) * world / (pm * 1e-3) / 1e12) if parts else None,
               "unit": "TFLOP/s", "h2d_bytes_per_step": ph2d + dh2d, "d2h_bytes_per_step": pd2h + dd2h,
               "ms_per_step": pm + dm, "prefill_ms": pm,
               "decode": ({"value": dec.bytes * world / (dm * 1e-3) / 1e9, "unit": "GB/s", "ms": dm,
                           "h2d_bytes": dh2d, "d2h_bytes": dd2h} if dec is not None else None),
               "covers": "every part: pinned host -> device inputs, the public call (g4attn_prefill; g4attn_decode "
                         "per layer), device -> host outputs; copies on a second stream overlap the other parts' "
                         "compute; the prefill parts and the decode mix timed as two groups"}

    launches = sum(p.launches for p in parts) + (dec.launches if dec else 0)
    ms_step = sum(tot.values()) / K
    line = {"metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": world, "steps": K,
            "warmup": args.warmup, "ms_per_step": ms_step, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "bf16",
            "data": "synthetic: seeded N(0,1) bf16 values (device generator), random page permutations",
            "config": {"workload": WORKLOAD, "parts": [n for n, _ in sp], "decode_batch": args.decode_batch,
                       "l2": "flushed before every part (512 MB write); inputs also exceed L2",
                       "parallelism": "replicas" if world > 1 else "single GPU"},
            "roofline": roofline, "prefill": res, "decode": decode, "cpu_baseline": cpu, "e2e": e2e,
            "verified": check,
            "gpu_launches": launches * K, "clocks": clocks, "peaks": pk}
    if rank == 0:
        print(json.dumps(line), flush=True)
    if dist is not None:
        dist.destroy_process_group()
    return 0


if __name__ == "__main__":
    sys.exit(main())
