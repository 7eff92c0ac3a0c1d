"""GPU parity: every CUDA entry point against the fp64 oracle on the same seeded inputs.

Bars: max-abs 2e-2 and mean-abs 2e-3 on bf16 outputs (fp32 accumulation); bit-exact where the
operation is a copy (p-RoPE's untouched pairs, V and S written into the cache).
"""
import numpy as np
import pytest
import torch

import invariant_hybrid_attention_gb300 as g4
import oracle
from invariant_hybrid_attention_gb300 import inputs as gi
from invariant_hybrid_attention_gb300.paged import PagedKV, device_int32, untile, untile_rot, untile_v256

from gpu_cases import GEOM, Batch, DecodeBatch, Norms, assert_close, f64, layers

pytestmark = pytest.mark.gpu


def bf16_round_bound(ref: np.ndarray) -> np.ndarray:
    """Half a bf16 ulp of |ref| plus a small fp32 slack: the bound on one RNE cast."""
    a = np.abs(ref)
    e = np.floor(np.log2(np.maximum(a, 1e-30)))
    return np.where(a > 0, 2.0 ** (e - 8), 0) + 1e-6 * (1 + a)


# ---------------------------------------------------------------- RoPE / p-RoPE

@pytest.mark.parametrize("kind", ["sliding", "global"])
def test_rope_apply_matches_oracle(kind):
    layer, olayer = layers(kind)
    D = GEOM[kind]["d"]
    T, H = 300, 7
    x = gi.bf16_normal((T, H, D), 3, 2.0)
    pos = torch.tensor(gi.uniform_ints(T, 0, oracle.MAX_POSITIONS - 1, 4), dtype=torch.int32)
    pos[:4] = torch.tensor([0, 1, 255, oracle.MAX_POSITIONS - 1], dtype=torch.int32)
    out = g4.g4attn_rope_apply(layer, x.cuda(), pos.cuda(), out=torch.empty((T, H, D), dtype=torch.bfloat16,
                                                                            device="cuda"))
    torch.cuda.synchronize()
    want = oracle.rope(x.double().numpy(), pos.numpy()[:, None], olayer.rope_theta, olayer.rope_partial)
    got = f64(out)
    assert (np.abs(got - want) <= bf16_round_bound(want) + 2e-6 * np.abs(want) + 1e-6).all()
    R = oracle.rope_rotated_pairs(D, olayer.rope_partial)
    keep = np.r_[R:D // 2, D // 2 + R:D]
    assert torch.equal(out.cpu()[:, :, keep], x[:, :, keep])          # untouched pairs: bit for bit
    # in place gives the same bits
    xi = x.cuda()
    g4.g4attn_rope_apply(layer, xi, pos.cuda())
    torch.cuda.synchronize()
    assert torch.equal(xi.cpu(), out.cpu())


# ---------------------------------------------------------------- cache append

@pytest.mark.parametrize("kind", ["sliding", "global"])
def test_kv_append_writes_the_contract_layout(kind):
    layer, olayer = layers(kind)
    bt = Batch(kind, [37, 5, 70], ctx_starts=[0, 20, 3], seed=5)
    cache = bt.device_cache()
    table = bt.plan.table.cuda()
    bt.append_history(layer, cache, table)
    g4.g4attn_kv_append(layer, bt.k_rows.cuda(), None if bt.v_rows is None else bt.v_rows.cuda(),
                        device_int32(bt.layout.q_start), device_int32(bt.layout.q_len),
                        device_int32(bt.layout.ctx_start), cache.desc, table)
    torch.cuda.synchronize()
    assert g4.g4attn_status_sync() == g4.G4_OK
    kc = untile(cache.k.cpu())
    vc = None if cache.v is None else untile_v256(cache.v.cpu())
    rc = None if cache.k_rot is None else untile_rot(cache.k_rot.cpu())
    R = oracle.rope_rotated_pairs(olayer.head_dim, olayer.rope_partial)
    rot_dims = np.r_[0:R, olayer.head_dim // 2:olayer.head_dim // 2 + R]
    for b, L in enumerate(bt.ctx_lens):
        for pos in range(L):
            page = int(bt.plan.table[b, pos // 16])
            stored = kc[page, :, pos % 16, :]
            raw = bt.hist_k[b][pos]
            if kind == "global":
                assert torch.equal(stored, raw)                          # S stored un-rotated
                # k_rot: p-RoPE(S) on the rotated dims, one bf16 rounding from the exact value
                want = oracle.rope(raw.double().numpy(), pos, olayer.rope_theta, olayer.rope_partial)[:, rot_dims]
                got = rc[page, :, pos % 16, :].double().numpy()
                assert (np.abs(got - want) <= bf16_round_bound(want) + 1e-6).all(), (b, pos)
            else:
                want = oracle.rope(raw.double().numpy(), pos, olayer.rope_theta, olayer.rope_partial)
                got = stored.double().numpy()
                assert (np.abs(got - want) <= bf16_round_bound(want) + 1e-6).all()
                assert torch.equal(vc[page, :, pos % 16, :], bt.hist_v[b][pos])


# ---------------------------------------------------------------- decode

DECODE_CASES = {
    "sliding-w1024": ("sliding", 1024, [1, 2, 17, 255, 256, 257, 1023, 1024, 1025, 3000, 4097]),
    "sliding-w64": ("sliding", 64, [1, 16, 63, 64, 65, 200, 513]),
    "global": ("global", 0, [1, 15, 16, 17, 1023, 1024, 1025, 2049, 5000]),
}


@pytest.mark.parametrize("case", list(DECODE_CASES))
def test_decode_matches_oracle(case):
    kind, window, lens = DECODE_CASES[case]
    layer, olayer = layers(kind, window if window else 1024)
    db = DecodeBatch(kind, lens, seed=11, window=window, sliding_window_only=(kind == "sliding"))
    out, _ = db.run(layer)
    got = f64(out)
    for b in range(len(lens)):
        assert_close(got[b], db.oracle_row(olayer, b), f"{case} request {b} (len {lens[b]})")


@pytest.mark.parametrize("kind", ["sliding", "global"])
def test_decode_is_batch_invariant(kind):
    """The same request (same data, same pages) alone and inside a larger ragged batch at a
    different index gives the same bits."""
    layer, _ = layers(kind)
    target_len = 2500
    alone = DecodeBatch(kind, [target_len], seed=21)
    out_a, _ = alone.run(layer)
    mixed_lens = [700, 3, target_len, 1500, 4000]
    mixed = DecodeBatch(kind, mixed_lens, seed=21)
    # give index 2 the target's data
    mixed.hist_k[2] = alone.hist_k[0]
    if kind == "sliding":
        mixed.hist_v[2] = alone.hist_v[0]
    mixed.q[2] = alone.q[0]
    out_m, _ = mixed.run(layer)
    assert torch.equal(out_a[0].cpu(), out_m[2].cpu())


# ---------------------------------------------------------------- sliding prefill

def check_prefill(bt: Batch, kind, window, sample=None):
    layer, olayer = layers(kind, window)
    out, _ = bt.run(layer)
    got = f64(out)
    covered = np.zeros(bt.layout.T, dtype=bool)
    for b, L in enumerate(bt.q_lens):
        s = bt.layout.q_start[b]
        covered[s:s + L] = True
        if L == 0:
            continue
        rows = None if sample is None or L <= sample else np.unique(
            np.r_[0, L - 1, np.random.default_rng(b).choice(L, sample, replace=False)])
        want = bt.oracle_rows(olayer, b, rows)
        idx = np.arange(L) if rows is None else rows
        assert_close(got[s + idx], want, f"sequence {b} (len {L}, ctx {bt.ctx_starts[b]})")
    # rows outside every sequence are never written
    assert np.isnan(got[~covered]).all()
    return out


def test_prefill_sliding_tiny_oracle_case():
    """Two causal sequences of 96 and 200 tokens, window shrunk to 64, N(0,1) inputs, seed 0."""
    check_prefill(Batch("sliding", [96, 200], seed=0), "sliding", 64)


@pytest.mark.parametrize("window", [1024, 64, 1])
@pytest.mark.parametrize("padded", [False, True], ids=["packed", "padded"])
def test_prefill_sliding_ragged(window, padded):
    bt = Batch("sliding", [1, 5, 127, 128, 129, 700, 1300], padded=padded, seed=3, scale=0.5)
    check_prefill(bt, "sliding", window, sample=96)


def test_prefill_sliding_chunked_with_history():
    """Chunks that start mid-sequence read earlier keys from the cache (written by kv_append)."""
    bt = Batch("sliding", [300, 64, 1, 200], ctx_starts=[1000, 77, 4000, 129], seed=4, scale=0.5)
    check_prefill(bt, "sliding", 1024, sample=96)


def test_prefill_sliding_batch_invariance():
    """A target sequence alone, packed among others and padded at another index: same bits."""
    layer, _ = layers("sliding", 1024)
    L = 1500
    alone = Batch("sliding", [L], seed=9, scale=0.5)
    out_a, _ = alone.run(layer)
    for lens, padded, at in [([200, L, 33], False, 1), ([L, 900], True, 0), ([5, 77, 1030, L], True, 3)]:
        bt = Batch("sliding", lens, padded=padded, seed=9 + len(lens), scale=0.5)
        bt.hist_k[at], bt.hist_v[at] = alone.hist_k[0], alone.hist_v[0]
        s = bt.layout.q_start[at]
        bt.q[s:s + L] = alone.q[:L]
        bt.k_rows = gi.rows_of(bt.hist_k, bt.layout)
        bt.v_rows = gi.rows_of(bt.hist_v, bt.layout)
        out_b, _ = bt.run(layer)
        assert torch.equal(out_a[:L].cpu(), out_b[s:s + L].cpu()), (lens, padded, at)


# ---------------------------------------------------------------- global (K==V) prefill

def test_prefill_global_tiny_oracle_case():
    """Two causal sequences of 96 and 200 tokens on the K==V layer, N(0,1) inputs, seed 0."""
    check_prefill(Batch("global", [96, 200], seed=0), "global", 0)


@pytest.mark.parametrize("padded", [False, True], ids=["packed", "padded"])
def test_prefill_global_ragged(padded):
    bt = Batch("global", [1, 5, 127, 128, 129, 700], padded=padded, seed=3, scale=0.5)
    check_prefill(bt, "global", 0, sample=64)


def test_prefill_global_chunked_with_history():
    """Chunks that start mid-sequence read earlier S and k_rot pages written by kv_append."""
    bt = Batch("global", [300, 64, 1, 200], ctx_starts=[1000, 77, 2500, 129], seed=4, scale=0.5)
    check_prefill(bt, "global", 0, sample=64)


def test_prefill_global_batch_invariance():
    """A target sequence alone, packed among others and padded at another index: same bits."""
    layer, _ = layers("global")
    L = 900
    alone = Batch("global", [L], seed=9, scale=0.5)
    out_a, _ = alone.run(layer)
    for lens, padded, at in [([200, L, 33], False, 1), ([L, 300], True, 0), ([5, 77, 530, L], True, 3)]:
        bt = Batch("global", lens, padded=padded, seed=9 + len(lens), scale=0.5)
        bt.hist_k[at] = alone.hist_k[0]
        s = bt.layout.q_start[at]
        bt.q[s:s + L] = alone.q[:L]
        bt.k_rows = gi.rows_of(bt.hist_k, bt.layout)
        out_b, _ = bt.run(layer)
        assert torch.equal(out_a[:L].cpu(), out_b[s:s + L].cpu()), (lens, padded, at)


@pytest.mark.parametrize("padded", [False, True], ids=["packed", "padded"])
@pytest.mark.parametrize("kind", ["sliding", "global"])
def test_prefill_split_steps_equal_prefill(kind, padded):
    """The queries rotated inside the attention kernel (g4attn_prefill, or g4attn_kv_append then
    g4attn_prefill_attend on the raw queries) and the staged form (g4attn_prefill_stage writes the
    roped queries into out, g4attn_prefill_attend reads them there) give the same bits: the same
    angles, rotation and bf16 cast at the declared roped-q cast point."""
    layer, _ = layers(kind, 1024)
    lens, starts = [300, 1, 129, 700], [0, 40, 256, 1000]
    mk = lambda: Batch(kind, lens, ctx_starts=starts, padded=padded, seed=21, scale=0.5)
    whole, cache_a = mk().run(layer)
    staged, cache_b = mk().run(layer, split=True)
    apart, cache_c = mk().run(layer, split="append")
    # bit patterns: rows outside every sequence and unwritten cache slots hold NaN in all three
    for other, cache in ((staged, cache_b), (apart, cache_c)):
        assert torch.equal(whole.cpu().view(torch.int16), other.cpu().view(torch.int16))
        assert torch.equal(cache_a.k.cpu().view(torch.int16), cache.k.cpu().view(torch.int16))


@pytest.mark.parametrize("kind", ["sliding", "global"])
def test_chunked_prefill_is_bit_identical_to_one_prefill(kind):
    """A sequence prefilled in chunks (each chunk reading the earlier keys from the cache) gives the
    same bits as one prefill of the whole sequence. Query tiles are aligned to absolute position
    and a key tile with no visible key adds exact zeros, so a row's arithmetic does not depend on
    where its chunk starts. Cuts fall mid-tile, on tile edges and one row from them; the last
    pattern ends in one-row chunks, i.e. decode steps run through g4attn_prefill."""
    layer, _ = layers(kind, 1024)
    L = 1500
    full = Batch(kind, [L], seed=31, scale=0.5)
    out_full, _ = full.run(layer)
    ref = out_full[:L].cpu().view(torch.int16)
    for cuts in ([700], [333, 1029], [1, 127, 128, 1281], [1497, 1498, 1499]):
        edges = [0] + cuts + [L]
        for a, b in zip(edges[:-1], edges[1:]):
            ch = Batch(kind, [b - a], ctx_starts=[a], seed=7 + a, scale=0.5)
            ch.hist_k = [full.hist_k[0][:b]]
            if full.hist_v is not None:
                ch.hist_v = [full.hist_v[0][:b]]
            ch.q[:b - a] = full.q[a:b]
            ch.k_rows = gi.rows_of(ch.hist_k, ch.layout)
            ch.v_rows = None if ch.hist_v is None else gi.rows_of(ch.hist_v, ch.layout)
            out_c, _ = ch.run(layer)
            got = out_c[:b - a].cpu().view(torch.int16)
            assert torch.equal(got, ref[a:b]), (kind, cuts, a, b)



def test_context_parallel_sliding_shards_with_window_halo_are_bit_identical():
    """Context parallelism of a sliding layer, simulated on one GPU: a 4096-token sequence split into
    four uneven shards (cuts mid-tile) as four ranks would hold it. Each shard's cache holds only
    its own keys and the pages of the W - 1 keys before them (the halo a rank would receive from the
    rank on its left); every other page-table entry is -1. Each shard is one prefill call at its
    absolute positions, and its rows are bit-identical to one prefill of the whole sequence."""
    layer, _ = layers("sliding", 1024)
    W, L = 1024, 4096
    full = Batch("sliding", [L], seed=81, scale=0.5)
    out_full, _ = full.run(layer)
    ref = out_full[:L].cpu().view(torch.int16)
    kh, vh = full.hist_k[0], full.hist_v[0]
    for a, b in [(0, 1000), (1000, 2100), (2100, 3333), (3333, 4096)]:
        p0 = max(0, a - (W - 1)) // 16                  # first page of the halo
        plan = gi.make_page_plan([b], seed=90 + a, mapped_from=[p0], spare_pages=1)
        table = plan.table.cuda()
        cache = PagedKV(plan.num_pages, 16, 256, shared=False)
        h = a - 16 * p0                                 # halo keys, from the page boundary
        if h > 0:
            g4.g4attn_kv_append(layer, kh[16 * p0:a].cuda(), vh[16 * p0:a].cuda(), device_int32([0]),
                                device_int32([h]), device_int32([16 * p0]), cache.desc, table)
        out = torch.full((b - a, 32, 256), float("nan"), dtype=torch.bfloat16, device="cuda")
        g4.g4attn_prefill(layer, full.q[a:b].cuda(), kh[a:b].cuda(), vh[a:b].cuda(), device_int32([0]),
                          device_int32([b - a]), device_int32([a]), cache.desc, table, out)
        torch.cuda.synchronize()
        assert g4.g4attn_status_sync() == g4.G4_OK
        assert torch.equal(out.cpu().view(torch.int16), ref[a:b]), (a, b)


# ---------------------------------------------------------------- per-head norms before RoPE

NORM_CASES = [("sliding", dict()), ("sliding", dict(k=False, v=False)), ("sliding", dict(q=False)),
              ("global", dict()), ("global", dict(k=False, v=False))]
NORM_IDS = ["sliding-all", "sliding-q", "sliding-kv", "global-all", "global-q"]


def scale_raw(bt, kind, norms, f=3.0):
    """Normed projections at f times unit scale, so that their norms have work to do. Un-normed
    ones stay at unit scale, as in the other parity tests: an un-normed q or k at scale 3 sharpens
    the logits until the declared bf16 casts alone reach the absolute tolerance, and an un-normed
    value sets the output's scale. On a K==V layer the keys are the values."""
    if norms.oracle.q_weight is not None:
        bt.q = bt.q * f
    if norms.oracle.k_weight is not None:
        bt.hist_k = [h * f for h in bt.hist_k]
        if hasattr(bt, "layout"):
            bt.k_rows = gi.rows_of(bt.hist_k, bt.layout)
    if norms.oracle.v_norm and kind == "sliding":
        bt.hist_v = [h * f for h in bt.hist_v]
        if hasattr(bt, "layout"):
            bt.v_rows = gi.rows_of(bt.hist_v, bt.layout)


@pytest.mark.parametrize("kind,which", NORM_CASES, ids=NORM_IDS)
def test_prefill_normed_matches_oracle(kind, which):
    """Raw projections normed in the stage; chunks whose history is appended with the same norms."""
    layer, olayer = layers(kind, 1024)
    norms = Norms(kind, seed=41, **which)
    bt = Batch(kind, [1, 5, 127, 129, 300], ctx_starts=[0, 40, 0, 1000, 129], seed=42)
    scale_raw(bt, kind, norms)
    out, _ = bt.run(layer, norms=norms)
    got = f64(out)
    for b, L in enumerate(bt.q_lens):
        s = bt.layout.q_start[b]
        rows = np.unique(np.r_[0, L - 1, np.random.default_rng(b).choice(L, min(L, 40), replace=False)])
        assert_close(got[s + rows], bt.oracle_rows(olayer, b, rows, norms), f"{kind} normed sequence {b}")


@pytest.mark.parametrize("kind,which", NORM_CASES, ids=NORM_IDS)
def test_decode_normed_matches_oracle(kind, which):
    layer, olayer = layers(kind, 1024)
    norms = Norms(kind, seed=43, **which)
    db = DecodeBatch(kind, [1, 17, 300, 1500], seed=44)
    scale_raw(db, kind, norms)
    out, _ = db.run(layer, norms=norms)
    got = f64(out)
    for b in range(len(db.ctx_lens)):
        assert_close(got[b], db.oracle_row(olayer, b, norms), f"{kind} normed decode request {b}")


@pytest.mark.parametrize("kind", ["sliding", "global"])
def test_prefill_normed_batch_invariance(kind):
    """With the norms on, a target sequence alone and inside batches gives the same bits."""
    layer, _ = layers(kind, 1024)
    norms = Norms(kind, seed=45)
    L = 700
    alone = Batch(kind, [L], seed=46, scale=2.0)
    out_a, _ = alone.run(layer, norms=norms)
    for lens, padded, at in [([200, L, 33], False, 1), ([5, 77, L], True, 2)]:
        bt = Batch(kind, lens, padded=padded, seed=47 + len(lens), scale=2.0)
        bt.hist_k[at] = alone.hist_k[0]
        if alone.hist_v is not None:
            bt.hist_v[at] = alone.hist_v[0]
        s = bt.layout.q_start[at]
        bt.q[s:s + L] = alone.q[:L]
        bt.k_rows = gi.rows_of(bt.hist_k, bt.layout)
        bt.v_rows = None if bt.hist_v is None else gi.rows_of(bt.hist_v, bt.layout)
        out_b, _ = bt.run(layer, norms=norms)
        assert torch.equal(out_a[:L].cpu(), out_b[s:s + L].cpu()), (kind, lens, padded, at)


# ---------------------------------------------------------------- decode with the prefill's bits

EXACT_LENS = {"sliding": [1, 17, 130, 700, 1500], "global": [1, 17, 130, 700, 2100]}


def full_prefill_last_rows(db: DecodeBatch, layer, norms=None, seed=0):
    """Each request's whole sequence prefilled in one batched call; returns the rows at each
    sequence's last position (the decode query there, random queries before it)."""
    lens = db.ctx_lens
    lay = gi.packed_layout(lens)
    qs = []
    for b, L in enumerate(lens):
        q = gi.bf16_normal((L, 32, db.d), seed * 7 + b, 0.5)
        q[L - 1] = db.q[b]
        qs.append(q)
    q = gi.rows_of(qs, lay, fill_nan=False).cuda()
    k = gi.rows_of(db.hist_k, lay, fill_nan=False).cuda()
    v = None if db.kind == "global" else gi.rows_of(db.hist_v, lay, fill_nan=False).cuda()
    cache = PagedKV(db.plan.num_pages, db.n_kv, db.d, shared=(db.kind == "global"))
    rows = (device_int32(lay.q_start), device_int32(lay.q_len), device_int32(lay.ctx_start))
    out = torch.full_like(q, float("nan"))
    if norms is None:
        g4.g4attn_prefill(layer, q, k, v, *rows, cache.desc, db.plan.table.cuda(), out)
    else:
        g4.g4attn_prefill_normed(layer, norms.arg, q, k, v, *rows, cache.desc, db.plan.table.cuda(), out)
    torch.cuda.synchronize()
    assert g4.g4attn_status_sync() == g4.G4_OK
    return torch.stack([out[s + L - 1] for s, L in zip(lay.q_start, lens)]).cpu()


@pytest.mark.parametrize("normed", [False, True], ids=["plain", "normed"])
@pytest.mark.parametrize("kind", ["sliding", "global"])
def test_decode_exact_has_the_prefill_bits(kind, normed):
    """g4attn_decode_exact gives, bit for bit, the row a prefill of the whole sequence computes at
    the decode position, and matches the oracle."""
    layer, olayer = layers(kind, 1024)
    norms = Norms(kind, 72) if normed else None
    db = DecodeBatch(kind, EXACT_LENS[kind], seed=71, scale=0.5)
    out, _ = db.run(layer, norms=norms, exact=True)
    want_bits = full_prefill_last_rows(db, layer, norms, seed=71)
    assert torch.equal(out.cpu(), want_bits)
    for b in range(len(db.ctx_lens)):
        assert_close(f64(out[b]), db.oracle_row(olayer, b, None if norms is None else norms), f"request {b}")


def test_decode_exact_bad_seq_len_is_reported():
    layer, _ = layers("sliding", 1024)
    db = DecodeBatch("sliding", [40, 64], seed=73)
    dcache = PagedKV(db.plan.num_pages, 16, 256, shared=False)
    q = db.q.cuda()
    kn = torch.stack([h[L - 1] for h, L in zip(db.hist_k, db.ctx_lens)]).cuda()
    vn = torch.stack([h[L - 1] for h, L in zip(db.hist_v, db.ctx_lens)]).cuda()
    ws = torch.empty(g4.g4attn_decode_exact_workspace_bytes(2), dtype=torch.uint8, device="cuda")
    out = torch.zeros_like(q)
    g4.g4attn_decode_exact(layer, None, q, kn, vn, device_int32([40, 0]), dcache.desc, db.plan.table.cuda(), out, ws)
    assert g4.g4attn_status_sync() == g4.G4_ERR_DEVICE
    assert g4.g4attn_status_sync() == g4.G4_OK
    assert (out[1] == 0).all()   # the request without a position is left untouched


# ---------------------------------------------------------------- vision-token mask

VISION_CASES = {
    # an image longer than the window and across query and key tiles, one touching the last row,
    # a one-token image, and (second sequence) an image that began in the cached history
    "sliding": dict(q_lens=[300, 517, 129], ctx=[0, 40, 0], window=96,
                    spans=[[(20, 150), (290, 300)], [(30, 90), (200, 201), (400, 557)], [(0, 129)]]),
    "global": dict(q_lens=[260, 130, 64], ctx=[0, 5, 0], window=0,
                   spans=[[(10, 200), (255, 260)], [(5, 6), (100, 135)], [(0, 64)]]),
}


@pytest.mark.parametrize("padded", [False, True], ids=["packed", "padded"])
@pytest.mark.parametrize("kind", ["sliding", "global"])
def test_prefill_vision_matches_oracle(kind, padded):
    c = VISION_CASES[kind]
    bt = Batch(kind, c["q_lens"], ctx_starts=c["ctx"], padded=padded, seed=61, scale=0.5, spans=c["spans"])
    check_prefill(bt, kind, c["window"])
    assert g4.g4attn_status_sync() == g4.G4_OK


@pytest.mark.parametrize("kind", ["sliding", "global"])
def test_prefill_vision_text_only_is_bit_identical_to_prefill(kind):
    """No image rows, or one-token images (which widen nothing), give the plain prefill's bits."""
    c = VISION_CASES[kind]
    layer, _ = layers(kind, c["window"] or 1024)
    plain = Batch(kind, c["q_lens"], ctx_starts=c["ctx"], seed=62, scale=0.5)
    out_p, _ = plain.run(layer)
    for spans in ([[] for _ in c["q_lens"]], [[(c0 + 3, c0 + 4)] for c0 in c["ctx"]]):
        vis = Batch(kind, c["q_lens"], ctx_starts=c["ctx"], seed=62, scale=0.5, spans=spans)
        out_v, _ = vis.run(layer)
        assert torch.equal(out_p.cpu(), out_v.cpu())


@pytest.mark.parametrize("kind", ["sliding", "global"])
def test_prefill_vision_batch_invariance(kind):
    """A sequence with images, alone and among other sequences with their own images: same bits."""
    window = 1024 if kind == "sliding" else 0
    layer, _ = layers(kind, window or 1024)
    L = 1400
    spans = [(100, 1300), (1350, 1360)]
    alone = Batch(kind, [L], seed=63, scale=0.5, spans=[spans])
    out_a, _ = alone.run(layer)
    for lens, padded, at, others in [([200, L, 33], False, 1, [[(0, 150)], None, [(5, 33)]]),
                                     ([L, 700], True, 0, [None, [(600, 700)]])]:
        bt = Batch(kind, lens, padded=padded, seed=64 + len(lens), scale=0.5,
                   spans=[spans if i == at else (o or []) for i, o in enumerate(others)])
        bt.hist_k[at] = alone.hist_k[0]
        if kind == "sliding":
            bt.hist_v[at] = alone.hist_v[0]
        s = bt.layout.q_start[at]
        bt.q[s:s + L] = alone.q[:L]
        bt.k_rows = gi.rows_of(bt.hist_k, bt.layout)
        if kind == "sliding":
            bt.v_rows = gi.rows_of(bt.hist_v, bt.layout)
        out_b, _ = bt.run(layer)
        assert torch.equal(out_a[:L].cpu(), out_b[s:s + L].cpu()), (lens, padded, at)


@pytest.mark.parametrize("kind", ["sliding", "global"])
def test_prefill_vision_bad_spans_are_reported(kind):
    """A span reaching past the call's rows, and rows of one image that disagree on its span, are
    seen on the device: the status says so, and the next call starts clean."""
    window = 1024 if kind == "sliding" else 0
    layer, _ = layers(kind, window or 1024)
    for spans in ([[(50, 400)]],                    # ends past the sequence's 300 keys
                  [[(10, 60)], ]):                  # consistent, as a control
        bt = Batch(kind, [300], seed=65, scale=0.5, spans=spans)
        cache = bt.device_cache()
        rows = (device_int32(bt.layout.q_start), device_int32(bt.layout.q_len), device_int32(bt.layout.ctx_start))
        out = torch.zeros_like(bt.q).cuda()
        sp = bt.span_rows()
        g4.g4attn_prefill_vision(layer, None, bt.q.cuda(), bt.k_rows.cuda(),
                                 None if bt.v_rows is None else bt.v_rows.cuda(), *rows, sp.cuda(), cache.desc,
                                 bt.plan.table.cuda(), out)
        want = g4.G4_ERR_DEVICE if spans[0][0][1] > 300 else g4.G4_OK
        assert g4.g4attn_status_sync() == want
    # rows 10..199 form one image, but row 127, the last of the first query tile, claims to be
    # text: that tile's key range then stops at key 127 while its rows 10..126 reach key 199
    bt = Batch(kind, [300], seed=65, scale=0.5, spans=[[(10, 200)]])
    sp = bt.span_rows()
    sp[127] = torch.tensor([0, 0])
    cache = bt.device_cache()
    rows = (device_int32(bt.layout.q_start), device_int32(bt.layout.q_len), device_int32(bt.layout.ctx_start))
    out = torch.zeros_like(bt.q).cuda()
    g4.g4attn_prefill_vision(layer, None, bt.q.cuda(), bt.k_rows.cuda(),
                             None if bt.v_rows is None else bt.v_rows.cuda(), *rows, sp.cuda(), cache.desc,
                             bt.plan.table.cuda(), out)
    assert g4.g4attn_status_sync() == g4.G4_ERR_DEVICE
    assert g4.g4attn_status_sync() == g4.G4_OK


# ---------------------------------------------------------------- the end of the position range

def test_sliding_prefill_and_decode_at_the_last_positions():
    """A 300-row chunk whose last row sits at position 262143, the last one a sequence may use, then a
    decode step that lands on it again from a one-row-shorter history: the RoPE angles are at their
    largest there. Only the window's pages are mapped (the rest of the 16384-entry table is -1),
    and the oracle is given just the window's keys, at their absolute positions."""
    layer, olayer = layers("sliding", 1024)
    n_max = oracle.MAX_POSITIONS
    L = 300
    c = n_max - L                                  # the chunk's first position
    p0 = ((c - 1024) // 16) * 16                   # first kept key: the window of the chunk's first row
    hist_len = n_max - p0
    k_hist = gi.bf16_normal((hist_len, 16, 256), 71, 0.5)
    v_hist = gi.bf16_normal((hist_len, 16, 256), 72, 0.5)
    q = gi.bf16_normal((L, 32, 256), 73, 0.5)
    plan = gi.make_page_plan([n_max], seed=74, mapped_from=[p0 // 16], spare_pages=2)
    table = plan.table.cuda()
    cache = PagedKV(plan.num_pages, 16, 256, shared=False)
    # history p0 .. c-1 through kv_append, then the chunk through prefill
    pre = c - p0
    g4.g4attn_kv_append(layer, k_hist[:pre].cuda(), v_hist[:pre].cuda(), device_int32([0]), device_int32([pre]),
                        device_int32([p0]), cache.desc, table)
    out = torch.full((L, 32, 256), float("nan"), dtype=torch.bfloat16, device="cuda")
    g4.g4attn_prefill(layer, q.cuda(), k_hist[pre:].cuda(), v_hist[pre:].cuda(), device_int32([0]),
                      device_int32([L]), device_int32([c]), cache.desc, table, out)
    torch.cuda.synchronize()
    assert g4.g4attn_status_sync() == g4.G4_OK
    rows = np.array([0, 1, 150, L - 2, L - 1])
    want = oracle.layer_rows(olayer, q[rows].double().numpy(), c - p0 + rows, k_hist.double().numpy(),
                             v_hist.double().numpy(), pos_offset=p0)
    assert_close(f64(out)[rows], want, "prefill rows at the end of the position range")
    # a decode step at position n_max - 1 over the same history (its own key rewritten identically)
    qd = gi.bf16_normal((1, 32, 256), 75, 0.5)
    ws = torch.empty(g4.g4attn_decode_workspace_bytes(layer, 1, plan.table.shape[1]), dtype=torch.uint8,
                     device="cuda")
    dout = torch.empty_like(qd).cuda()
    g4.g4attn_decode(layer, qd.cuda(), k_hist[-1:].cuda(), v_hist[-1:].cuda(), device_int32([n_max]), cache.desc,
                     table, dout, ws)
    torch.cuda.synchronize()
    assert g4.g4attn_status_sync() == g4.G4_OK
    want_d = oracle.layer_rows(olayer, qd.double().numpy(), [hist_len - 1], k_hist.double().numpy(),
                               v_hist.double().numpy(), pos_offset=p0)
    assert_close(f64(dout), want_d, "decode at the last position")
    # one position further is refused on the device (the status says so; the context stays usable)
    g4.g4attn_decode(layer, qd.cuda(), k_hist[-1:].cuda(), v_hist[-1:].cuda(), device_int32([n_max + 1]),
                     cache.desc, table, dout, ws)
    assert g4.g4attn_status_sync() == g4.G4_ERR_DEVICE
    assert g4.g4attn_status_sync() == g4.G4_OK


# ---------------------------------------------------------------- degenerate and faulty inputs

@pytest.mark.parametrize("kind", ["sliding", "global"])
def test_zero_length_sequences_in_a_batch(kind):
    """q_len 0 is allowed: such sequences produce and touch nothing, the others are exact."""
    bt = Batch(kind, [100, 0, 200, 0], ctx_starts=[0, 5, 0, 0], seed=51, scale=0.5)
    check_prefill(bt, kind, 0 if kind == "global" else 1024)


@pytest.mark.parametrize("kind", ["sliding", "global"])
def test_rows_past_the_end_of_q_are_refused(kind):
    """A sequence whose q_start + q_len reaches past the T rows of the call is refused on the
    device (the status word says so) and none of its rows is read or written: q, k, v and out carry
    40 guard rows past T here, and the guard rows of out stay NaN. The other sequence is exact."""
    layer, olayer = layers(kind, 1024)
    bt = Batch(kind, [100, 200], seed=91, scale=0.5)   # T = 300
    T, guard = 300, 40
    plan = gi.make_page_plan([100, 240], seed=92)
    cache = PagedKV(plan.num_pages, bt.n_kv, bt.d, shared=(kind == "global"))
    pad = lambda x: torch.cat([x, torch.zeros((guard,) + tuple(x.shape[1:]), dtype=x.dtype)]).cuda()
    q, k = pad(bt.q), pad(bt.k_rows)
    v = None if bt.v_rows is None else pad(bt.v_rows)
    out = torch.full((T + guard, 32, bt.d), float("nan"), dtype=torch.bfloat16, device="cuda")
    rows = (device_int32([0, 100]), device_int32([100, 230]), device_int32([0, 0]))   # 100 + 230 > T
    g4.g4attn_prefill(layer, q[:T], k[:T], None if v is None else v[:T], *rows, cache.desc, plan.table.cuda(),
                      out[:T])
    torch.cuda.synchronize()
    assert g4.g4attn_status_sync() == g4.G4_ERR_DEVICE
    assert g4.g4attn_status_sync() == g4.G4_OK
    assert torch.isnan(out[T:].float()).all()
    assert_close(f64(out[:100]), bt.oracle_rows(olayer, 0), "the valid sequence")


@pytest.mark.parametrize("kind", ["sliding", "global"])
def test_positions_past_the_limit_are_refused_without_overflow(kind):
    """A chunk whose ctx_start lies so close to 2^31 that ctx_start + q_len overflows int32 is
    refused on the device as a whole (none of its rows is read or written, the status says so),
    and the other sequence of the batch is exact."""
    layer, olayer = layers(kind, 1024)
    bt = Batch(kind, [100, 200], seed=93, scale=0.5)
    cache = bt.device_cache()
    out = torch.full_like(bt.q, float("nan")).cuda()
    rows = (device_int32(bt.layout.q_start), device_int32(bt.layout.q_len), device_int32([0, 2**31 - 150]))
    g4.g4attn_prefill(layer, bt.q.cuda(), bt.k_rows.cuda(), None if bt.v_rows is None else bt.v_rows.cuda(), *rows,
                      cache.desc, bt.plan.table.cuda(), out)
    torch.cuda.synchronize()
    assert g4.g4attn_status_sync() == g4.G4_ERR_DEVICE
    assert g4.g4attn_status_sync() == g4.G4_OK
    assert torch.isnan(out[100:].float()).all()
    assert_close(f64(out[:100]), bt.oracle_rows(olayer, 0), "the valid sequence")


def test_device_detected_errors_are_reported_and_cleared(lib):
    """A page-table entry outside the pool and a decode position beyond the page table are seen on
    the device: the work they touch is skipped, the status word says so, and the next call starts
    clean. Nothing traps; the context stays usable."""
    layer, _ = layers("sliding", 1024)
    bt = Batch("sliding", [300], seed=52, scale=0.5)
    cache = bt.device_cache()
    table = bt.plan.table.clone()
    table[0, 5] = bt.plan.num_pages + 7          # keys 80..95 point outside the pool
    rows = (device_int32(bt.layout.q_start), device_int32(bt.layout.q_len), device_int32(bt.layout.ctx_start))
    out = torch.zeros_like(bt.q).cuda()
    g4.g4attn_prefill(layer, bt.q.cuda(), bt.k_rows.cuda(), bt.v_rows.cuda(), *rows, cache.desc, table.cuda(), out)
    assert g4.g4attn_status_sync() == g4.G4_ERR_DEVICE
    assert g4.g4attn_status_sync() == g4.G4_OK   # read and cleared
    # the same prefill with a good table is clean and exact afterwards
    check_prefill(Batch("sliding", [300], seed=52, scale=0.5), "sliding", 1024)
    assert g4.g4attn_status_sync() == g4.G4_OK
    # decode: a request whose position lies beyond its page table
    db = DecodeBatch("sliding", [40, 64], seed=53)
    dcache = PagedKV(db.plan.num_pages, 16, 256, shared=False)
    dt = db.plan.table.cuda()
    q = db.q.cuda()
    kn = torch.stack([h[L - 1] for h, L in zip(db.hist_k, db.ctx_lens)]).cuda()
    vn = torch.stack([h[L - 1] for h, L in zip(db.hist_v, db.ctx_lens)]).cuda()
    ws = torch.empty(g4.g4attn_decode_workspace_bytes(layer, 2, db.plan.max_pages), dtype=torch.uint8, device="cuda")
    dout = torch.empty_like(q)
    too_far = [40, 16 * db.plan.max_pages + 1]
    g4.g4attn_decode(layer, q, kn, vn, device_int32(too_far), dcache.desc, dt, dout, ws)
    assert g4.g4attn_status_sync() == g4.G4_ERR_DEVICE
    assert g4.g4attn_status_sync() == g4.G4_OK
