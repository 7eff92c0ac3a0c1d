"""Batch-invariance stress on the GPU.

A fixed target request runs alone and inside 20 seeded mixed batches, and every output row it
gets must be bit-identical (torch.equal) across all of them. The target is a 3000-token
prefill followed by 64 decode steps, run for both layer kinds (RL-Kernel RFC "[RFC][Gemma-4-31B-it]
WS1/WS2 kernel roadmap", section 4 rule 6: a row is invariant to unrelated batch rows, padding,
packing and placement).

Each trial batch has B ~ U[1, 128] requests with prompt lengths U[1, 16384] and the target at a
random index. Pages are scattered by a fresh random permutation, and the cache starts as NaN.
Odd trials use a padded layout: each sequence's rows start at the next multiple of 256, and the
gap rows are NaN. The whole batch then decodes 64 steps together. The trials cycle through four
kinds of call: plain prefills; g4attn_prefill_vision, where the other requests carry images and
the target's rows are text; chunked prefills, where every other request continues a history
already in the cache (ctx_start > 0); and normed calls (per-head RMS norms on q, k and v, in the
prefill and in every decode step), whose target is compared with its own normed run alone. The
first three must give the target the plain run's bits.

A 131072-token global prefill must also give the same bits alone and inside batches; 64 of
its rows are checked against the fp64 oracle.
"""
import numpy as np
import pytest
import torch

import invariant_hybrid_attention_gb300 as g4
import oracle
from invariant_hybrid_attention_gb300 import inputs as gi
from invariant_hybrid_attention_gb300.paged import PagedKV, device_int32

from gpu_cases import GEOM, assert_close, f64, layers

pytestmark = pytest.mark.gpu

TARGET_LEN, DECODE_STEPS = 3000, 64
TRIAL_SEEDS = list(range(100, 120))


def device_normal(shape, seed, chunk_rows=65536):
    """Seeded N(0,1) bf16 on the device, drawn in chunks of rows (bounded fp32 scratch)."""
    t = torch.empty(shape, dtype=torch.bfloat16, device="cuda")
    g = torch.Generator(device="cuda")
    g.manual_seed(int(seed))
    flat = t.view(shape[0], -1)
    for r0 in range(0, shape[0], chunk_rows):
        r1 = min(shape[0], r0 + chunk_rows)
        flat[r0:r1] = torch.randn((r1 - r0, flat.shape[1]), generator=g, device="cuda").to(torch.bfloat16)
    return t


class Target:
    """The fixed request: prompt rows, decode queries, and its keys/values (device, bf16)."""

    def __init__(self, kind: str, seed: int = 77):
        n_kv, d = GEOM[kind]["n_kv"], GEOM[kind]["d"]
        L = TARGET_LEN + DECODE_STEPS
        self.q = gi.bf16_normal_device((TARGET_LEN, 32, d), seed)
        self.q_dec = gi.bf16_normal_device((DECODE_STEPS, 32, d), seed + 1)
        self.k = gi.bf16_normal_device((L, n_kv, d), seed + 2)
        self.v = None if kind == "global" else gi.bf16_normal_device((L, n_kv, d), seed + 3)


def layout_rows(lens, padded):
    starts, s = [], 0
    for b, L in enumerate(lens):
        if padded:
            s = (s + 255) // 256 * 256 + (128 if b % 2 else 0)
        starts.append(s)
        s += L
    return starts, max(s, 1)


MODES = ("plain", "vision", "chunked", "normed")


def stress_norms(kind):
    """Per-head norm weights (bf16, uniform in [0.5, 1.5]) on q and k, and the unit norm on v."""
    d = GEOM[kind]["d"]
    g = torch.Generator().manual_seed(4242)
    w = [(torch.rand(d, generator=g) + 0.5).to(torch.bfloat16).cuda() for _ in range(2)]
    return w, g4.make_norms(w[0], w[1], True, 1e-6)


def run_request_mix(kind, target, lens, at, padded, seed, mode="plain"):
    """Prefill the batch (target at index `at`) with a call of the given mode, then decode it
    DECODE_STEPS times. Returns the target's prefill output rows and its decode outputs."""
    layer, _ = layers(kind)
    n_kv, d = GEOM[kind]["n_kv"], GEOM[kind]["d"]
    B = len(lens)
    lens = [int(x) for x in lens]
    lens[at] = TARGET_LEN
    starts, T = layout_rows(lens, padded)
    st = starts[at]
    keep, norms = stress_norms(kind) if mode == "normed" else (None, None)
    # chunked: every other request continues a history of up to 2000 keys already in the cache
    hist = [0] * B
    if mode == "chunked":
        hist = [0 if b == at else h for b, h in enumerate(gi.uniform_ints(B, 1, 2000, seed + 3000))]

    q = device_normal((T, 32, d), seed * 7 + 1)
    k = device_normal((T, n_kv, d), seed * 7 + 2)
    v = None if kind == "global" else device_normal((T, n_kv, d), seed * 7 + 3)
    q[st:st + TARGET_LEN] = target.q
    k[st:st + TARGET_LEN] = target.k[:TARGET_LEN]
    if v is not None:
        v[st:st + TARGET_LEN] = target.v[:TARGET_LEN]
    if padded:   # gap rows: NaN
        covered = torch.zeros(T, dtype=torch.bool, device="cuda")
        for s0, L in zip(starts, lens):
            covered[s0:s0 + L] = True
        for t in (q, k, v):
            if t is not None:
                t[~covered] = float("nan")

    plan = gi.make_page_plan([h + L + DECODE_STEPS for h, L in zip(hist, lens)], seed=seed * 7 + 4, spare_pages=7)
    cache = PagedKV(plan.num_pages, n_kv, d, shared=(kind == "global"))   # NaN-filled
    table = plan.table.cuda()
    if mode == "chunked":   # the histories, appended first
        hl = gi.packed_layout(hist)
        hk = device_normal((hl.T, n_kv, d), seed * 7 + 5)
        hv = None if kind == "global" else device_normal((hl.T, n_kv, d), seed * 7 + 6)
        g4.g4attn_kv_append(layer, hk, hv, device_int32(hl.q_start), device_int32(hl.q_len),
                            device_int32([0] * B), cache.desc, table)
        del hk, hv
    out = torch.full_like(q, float("nan"))
    rows = (device_int32(starts), device_int32(lens), device_int32(hist))
    if mode == "vision":   # the other requests carry one image each; the target's rows are text
        span = torch.full((T, 2), 1 << 30, dtype=torch.int32)
        span[:, 0] = -7   # gap rows: spans that would be refused if read
        for b, (s0, L) in enumerate(zip(starts, lens)):
            span[s0:s0 + L] = 0
            if b != at and L >= 4:
                i0, i1 = L // 4, L // 4 + max(1, min(700, L // 2))
                span[s0 + i0:s0 + i1, 0] = i0
                span[s0 + i0:s0 + i1, 1] = i1
        g4.g4attn_prefill_vision(layer, None, q, k, v, *rows, span.cuda(), cache.desc, table, out)
    elif mode == "normed":
        g4.g4attn_prefill_normed(layer, norms, q, k, v, *rows, cache.desc, table, out)
    else:
        g4.g4attn_prefill(layer, q, k, v, *rows, cache.desc, table, out)
    pre = out[st:st + TARGET_LEN].clone()
    del q, k, v, out

    ws = torch.empty(g4.g4attn_decode_workspace_bytes(layer, B, int(table.shape[1])), dtype=torch.uint8,
                     device="cuda")
    dec = []
    for i in range(DECODE_STEPS):
        qd = gi.bf16_normal_device((B, 32, d), seed * 1000 + i)
        kn = gi.bf16_normal_device((B, n_kv, d), seed * 1000 + 500 + i)
        vn = None if kind == "global" else gi.bf16_normal_device((B, n_kv, d), seed * 1000 + 900 + i)
        qd[at] = target.q_dec[i]
        kn[at] = target.k[TARGET_LEN + i]
        if vn is not None:
            vn[at] = target.v[TARGET_LEN + i]
        o = torch.full_like(qd, float("nan"))
        sl = device_int32([h + L + i + 1 for h, L in zip(hist, lens)])
        if mode == "normed":
            g4.g4attn_decode_normed(layer, norms, qd, kn, vn, sl, cache.desc, table, o, ws)
        else:
            g4.g4attn_decode(layer, qd, kn, vn, sl, cache.desc, table, o, ws)
        dec.append(o[at].clone())
    torch.cuda.synchronize()
    st_ = g4.g4attn_status_sync()
    assert st_ == g4.G4_OK, g4.status_string(st_)
    return pre, torch.stack(dec)


def trial_shape(seed):
    B = gi.uniform_ints(1, 1, 128, seed)[0]
    lens = gi.uniform_ints(B, 1, 16384, seed + 1000)
    at = gi.uniform_ints(1, 0, B - 1, seed + 2000)[0]
    return lens, at, seed % 2 == 1


@pytest.mark.parametrize("kind", ["sliding", "global"])
def test_target_request_is_bit_identical_in_20_mixed_batches(kind):
    target = Target(kind)
    ref_pre, ref_dec = run_request_mix(kind, target, [TARGET_LEN], 0, False, seed=1)

    # the reference itself against the fp64 oracle (sampled prompt rows, first and last decode step)
    _, olayer = layers(kind)
    k_h = target.k.cpu().double().numpy()
    v_h = None if target.v is None else target.v.cpu().double().numpy()
    rows = np.array([0, 1, 127, 128, 1023, 1024, 2047, TARGET_LEN - 1])
    ri = torch.as_tensor(rows, device="cuda")
    want = oracle.layer_rows(olayer, target.q[ri].cpu().double().numpy(), rows, k_h[:TARGET_LEN],
                             None if v_h is None else v_h[:TARGET_LEN])
    assert_close(f64(ref_pre[ri]), want, f"{kind} target prompt rows")
    for i in (0, DECODE_STEPS - 1):
        L = TARGET_LEN + i + 1
        want = oracle.decode_row(olayer, target.q_dec[i].cpu().double().numpy(), k_h[:L],
                                 None if v_h is None else v_h[:L])
        assert_close(f64(ref_dec[i]), want, f"{kind} target decode step {i}")

    ref_n = run_request_mix(kind, target, [TARGET_LEN], 0, False, seed=2, mode="normed")   # the normed target alone
    for i, seed in enumerate(TRIAL_SEEDS):
        lens, at, padded = trial_shape(seed)
        mode = MODES[i % len(MODES)]
        pre, dec = run_request_mix(kind, target, lens, at, padded, seed, mode)
        want_pre, want_dec = ref_n if mode == "normed" else (ref_pre, ref_dec)
        assert torch.equal(pre, want_pre), (kind, seed, mode, len(lens), at, padded, "prefill")
        assert torch.equal(dec, want_dec), (kind, seed, mode, len(lens), at, padded, "decode")
        del pre, dec
        torch.cuda.empty_cache()


def test_global_prefill_131072_tokens_alone_and_in_batches():
    kind = "global"
    layer, olayer = layers(kind)
    L = 131072
    q_t = gi.bf16_normal_device((L, 32, 512), 501)
    k_t = gi.bf16_normal_device((L, 4, 512), 502)

    def run(lens, at, padded, seed):
        lens = list(lens)
        lens[at] = L
        starts, T = layout_rows(lens, padded)
        q = device_normal((T, 32, 512), seed)
        k = device_normal((T, 4, 512), seed + 1)
        q[starts[at]:starts[at] + L] = q_t
        k[starts[at]:starts[at] + L] = k_t
        plan = gi.make_page_plan(lens, seed=seed + 2, spare_pages=3)
        cache = PagedKV(plan.num_pages, 4, 512, shared=True)
        out = torch.full_like(q, float("nan"))
        g4.g4attn_prefill(layer, q, k, None, device_int32(starts), device_int32(lens), device_int32([0] * len(lens)),
                          cache.desc, plan.table.cuda(), out)
        torch.cuda.synchronize()
        st_ = g4.g4attn_status_sync()
        assert st_ == g4.G4_OK, g4.status_string(st_)
        return out[starts[at]:starts[at] + L].clone()

    alone = run([L], 0, False, 600)
    for lens, at, padded, seed in [([5000, L, 777], 1, False, 610), ([L, 3, 16384], 0, True, 620)]:
        other = run(lens, at, padded, seed)
        assert torch.equal(other, alone), (lens, at, padded)
        del other
    # 64 sampled rows (the first and last among them) against the oracle
    rng = np.random.default_rng(5)
    rows = np.unique(np.r_[0, L - 1, rng.choice(L, 62, replace=False)])
    ri = torch.as_tensor(rows, device="cuda")
    want = oracle.layer_rows(olayer, q_t[ri].cpu().double().numpy(), rows, k_t.cpu().double().numpy(), None)
    assert_close(f64(alone[ri]), want, "131072-token global prefill, sampled rows")
