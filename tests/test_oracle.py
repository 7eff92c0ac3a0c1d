"""Pins for the fp64 oracle: each check ties it to something other than itself.

* closed forms (q = 0 gives the mean of the visible values; frequency identities);
* library routines on special cases (torch scaled_dot_product_attention in fp64 for
  causal and banded masks, with and without GQA);
* textbook RoPE as complex multiplication;
* invariants (pair norms, relative position, perturbation outside the mask, K==V);
* the geometry table of the RFC's checkpoint fingerprint (tests/golden).

The last block plants mistakes in the oracle and checks that some pin catches each one.
"""
import math
import os

import numpy as np
import pytest
import torch
import torch.nn.functional as F

import oracle
from oracle import core as oa

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def rng(seed):
    return np.random.default_rng(seed)


def bf16ish(a):
    """Round fp64 values to bf16 so inputs look like the kernels' inputs."""
    return torch.from_numpy(np.asarray(a, np.float32)).to(torch.bfloat16).double().numpy()


# ---------------------------------------------------------------- checks (reused by controls)

def check_geometry(o):
    vals = {}
    with open(os.path.join(GOLDEN, "gemma4_31b_attention_geometry.txt")) as f:
        for line in f:
            line = line.strip()
            if line and not line.startswith("#"):
                k, v = line.split()
                vals[k] = float(v)
    S, G = o.SLIDING, o.GLOBAL
    assert S.n_q_heads == vals["q_heads"] and G.n_q_heads == vals["q_heads"]
    assert S.n_kv_heads == vals["sliding_kv_heads"] and S.head_dim == vals["sliding_head_dim"]
    assert S.window == vals["sliding_window"] and S.rope_theta == vals["sliding_rope_theta"]
    assert S.rope_partial == 1.0 and not S.kv_shared
    assert G.n_kv_heads == vals["global_kv_heads"] and G.head_dim == vals["global_head_dim"]
    assert G.kv_shared == bool(vals["global_k_eq_v"]) and G.window == 0
    assert G.rope_partial == vals["global_rope_partial"] and G.rope_theta == vals["global_rope_theta"]
    assert o.MAX_POSITIONS == vals["max_positions"]


def check_rope_complex(o, D, theta, partial, seed=0):
    """Textbook RoPE: z_t = x_t + i x_{t+D/2} is multiplied by exp(i pos f_t) for the first R
    pairs, f_t = theta^(-2t/D) evaluated with math.pow one pair at a time."""
    r = rng(seed)
    x = r.standard_normal((7, D))
    pos = np.array([0, 1, 2, 17, 1000, 65535, 262143])
    y = o.rope(x, pos, theta, partial)
    half = D // 2
    R = int(partial * D / 2)
    for n in range(x.shape[0]):
        for t in range(half):
            z = complex(x[n, t], x[n, t + half])
            if t < R:
                z *= complex(math.cos(pos[n] * math.pow(theta, -2.0 * t / D)),
                             math.sin(pos[n] * math.pow(theta, -2.0 * t / D)))
            assert abs(y[n, t] - z.real) < 1e-9 and abs(y[n, t + half] - z.imag) < 1e-9, (n, t)


def check_inv_freq_identities(o, D, theta):
    f = o.rope_inv_freq(D, theta)
    assert f.shape == (D // 2,)
    assert f[0] == 1.0
    assert abs(f[D // 4] - 1.0 / math.sqrt(theta)) < 1e-15 * 1e3
    # f_t * f_{D/2 - t} = 1/theta for every t in 1 .. D/2-1: the exponent's denominator is D
    prod = f[1:] * f[1:][::-1]
    assert np.allclose(prod, 1.0 / theta, rtol=1e-12, atol=0)


def check_sdpa_causal(o, seed=1):
    r = rng(seed)
    L, D = 37, 32
    q, k, v = (r.standard_normal((L, D)) for _ in range(3))
    scale = 0.17
    got = o.attention(q, k, v, np.arange(L), np.arange(L), 0, scale)
    t = lambda a: torch.from_numpy(a)[None, None]
    ref = F.scaled_dot_product_attention(t(q), t(k), t(v), is_causal=True, scale=scale)[0, 0].numpy()
    assert np.abs(got - ref).max() < 1e-12


def check_sdpa_band(o, W, seed=2):
    r = rng(seed)
    L, D = 50, 16
    q, k, v = (r.standard_normal((L, D)) for _ in range(3))
    scale = 0.25
    got = o.attention(q, k, v, np.arange(L), np.arange(L), W, scale)
    ones = torch.ones(L, L, dtype=torch.bool)
    band = torch.tril(ones) & torch.triu(ones, diagonal=-(W - 1))
    t = lambda a: torch.from_numpy(a)[None, None]
    ref = F.scaled_dot_product_attention(t(q), t(k), t(v), attn_mask=band, scale=scale)[0, 0].numpy()
    assert np.abs(got - ref).max() < 1e-12


def check_layer_vs_sdpa(o, layer, L=40, seed=3):
    """A whole layer (GQA, RoPE applied to q and k with the oracle's rope, pinned on its own)
    against SDPA on the rotated tensors with the GQA heads repeated by torch."""
    r = rng(seed)
    q = r.standard_normal((L, layer.n_q_heads, layer.head_dim))
    k = r.standard_normal((L, layer.n_kv_heads, layer.head_dim))
    v = None if layer.kv_shared else r.standard_normal((L, layer.n_kv_heads, layer.head_dim))
    got = o.layer_rows(layer, q, np.arange(L), k, v)
    pos = np.arange(L)[:, None]
    qr = o.rope(q, pos, layer.rope_theta, layer.rope_partial)
    kr = o.rope(k, pos, layer.rope_theta, layer.rope_partial)
    vv = k if layer.kv_shared else v
    tq = torch.from_numpy(qr).permute(1, 0, 2)[None]
    tk = torch.from_numpy(kr).permute(1, 0, 2).repeat_interleave(layer.group, dim=0)[None]
    tv = torch.from_numpy(vv).permute(1, 0, 2).repeat_interleave(layer.group, dim=0)[None]
    ones = torch.ones(L, L, dtype=torch.bool)
    mask = torch.tril(ones)
    if layer.window > 0:
        mask &= torch.triu(ones, diagonal=-(layer.window - 1))
    ref = F.scaled_dot_product_attention(tq, tk, tv, attn_mask=mask,
                                         scale=1.0 / math.sqrt(layer.head_dim))[0].permute(1, 0, 2).numpy()
    assert np.abs(got - ref).max() < 1e-11


def check_q_zero_mean(o, layer, L=150, seed=4):
    """With q = 0 every visible score is equal, so row i is the plain mean of the visible
    (un-rotated) values: the last min(i+1, W) of them."""
    r = rng(seed)
    q = np.zeros((L, layer.n_q_heads, layer.head_dim))
    k = r.standard_normal((L, layer.n_kv_heads, layer.head_dim))
    v = None if layer.kv_shared else r.standard_normal((L, layer.n_kv_heads, layer.head_dim))
    vals = k if layer.kv_shared else v
    got = o.layer_rows(layer, q, np.arange(L), k, v)
    for i in [0, 1, 2, layer.window - 2 if layer.window else 5, layer.window - 1 if layer.window else 60,
              layer.window if layer.window else 99, L - 1]:
        if i < 0 or i >= L:
            continue
        lo = 0 if layer.window <= 0 else max(0, i - layer.window + 1)
        for h in (0, layer.n_q_heads - 1):
            want = vals[lo:i + 1, h // layer.group].mean(axis=0)
            assert np.abs(got[i, h] - want).max() < 1e-12, (i, h)


def check_outside_perturbation(o, layer, L=90, seed=5):
    r = rng(seed)
    q = r.standard_normal((L, layer.n_q_heads, layer.head_dim))
    k = r.standard_normal((L, layer.n_kv_heads, layer.head_dim))
    v = None if layer.kv_shared else r.standard_normal((L, layer.n_kv_heads, layer.head_dim))
    i = L - 20
    base = o.layer_rows(layer, q[[i]], [i], k, v)
    outside = [j for j in range(L) if j > i or (layer.window > 0 and i - j > layer.window - 1)]
    inside = [j for j in range(L) if j not in outside]
    k2 = k.copy()
    k2[outside] += 3.0
    v2 = None if v is None else v.copy()
    if v2 is not None:
        v2[outside] -= 5.0
    assert np.array_equal(o.layer_rows(layer, q[[i]], [i], k2, v2), base)
    k3 = k.copy()
    k3[inside[0]] += 3.0
    assert np.abs(o.layer_rows(layer, q[[i]], [i], k3, v) - base).max() > 1e-6


def check_rms_norm_closed_form(o, seed=11):
    """The unit norm keeps each vector's direction and gives mean(y^2) = ms / (ms + eps), where
    ms is the input's mean square."""
    r = rng(seed)
    x = r.standard_normal((5, 3, 64)) * 3.0
    eps = 0.25
    y = o.rms_norm(x, None, eps)
    ms = (x * x).mean(axis=-1)
    assert np.allclose((y * y).mean(axis=-1), ms / (ms + eps), rtol=1e-12, atol=0)
    c = y / x
    assert (c > 0).all() and np.allclose(c, c[..., :1], rtol=1e-12, atol=0)


def check_rms_norm_vs_torch(o, seed=12):
    r = rng(seed)
    for D in (256, 512):
        x = r.standard_normal((4, 2, D)) * 2.0
        w = r.standard_normal(D)
        for weight in (w, None):
            ref = F.rms_norm(torch.from_numpy(x), (D,), weight=None if weight is None else torch.from_numpy(w),
                             eps=1e-6).numpy()
            assert np.abs(o.rms_norm(x, weight, 1e-6) - ref).max() < 1e-12


def normed_inputs(layer, L, seed, k_weight=True, q_weight=True, v_norm=True, eps=1e-6):
    r = rng(seed)
    D = layer.head_dim
    q = r.standard_normal((L, layer.n_q_heads, D)) * 1.7
    k = r.standard_normal((L, layer.n_kv_heads, D)) * 0.6
    v = None if layer.kv_shared else r.standard_normal((L, layer.n_kv_heads, D)) * 2.2
    norms = oracle.Norms(q_weight=r.uniform(0.5, 1.5, D) if q_weight else None,
                         k_weight=r.uniform(0.5, 1.5, D) if k_weight else None, v_norm=v_norm, eps=eps)
    return q, k, v, norms


def check_normed_layer_vs_torch(o, layer, L=24, seed=14, **kw):
    """A normed layer against torch: F.rms_norm on the raw projections (K==V: K = w_k n(S), V = n(S)),
    the oracle's own pinned rope, and SDPA with the GQA heads repeated by torch."""
    q, k, v, norms = normed_inputs(layer, L, seed, **kw)
    got = o.layer_rows(layer, q, np.arange(L), k, v, 0, norms)
    D = layer.head_dim

    def tn(x, w):
        return F.rms_norm(torch.from_numpy(x), (D,), weight=None if w is None else torch.from_numpy(w),
                          eps=norms.eps).numpy()
    qn = q if norms.q_weight is None else tn(q, norms.q_weight)
    kn = k if norms.k_weight is None else tn(k, norms.k_weight)
    vsrc = k if layer.kv_shared else v
    vn = tn(vsrc, None) if norms.v_norm else vsrc
    pos = np.arange(L)[:, None]
    qr = oracle.rope(qn, pos, layer.rope_theta, layer.rope_partial)
    kr = oracle.rope(kn, pos, layer.rope_theta, layer.rope_partial)
    tq = torch.from_numpy(qr).permute(1, 0, 2)[None]
    tk = torch.from_numpy(kr).permute(1, 0, 2).repeat_interleave(layer.group, dim=0)[None]
    tv = torch.from_numpy(vn).permute(1, 0, 2).repeat_interleave(layer.group, dim=0)[None]
    ones = torch.ones(L, L, dtype=torch.bool)
    mask = torch.tril(ones)
    if layer.window > 0:
        mask &= torch.triu(ones, diagonal=-(layer.window - 1))
    ref = F.scaled_dot_product_attention(tq, tk, tv, attn_mask=mask,
                                         scale=1.0 / math.sqrt(D))[0].permute(1, 0, 2).numpy()
    assert np.abs(got - ref).max() < 1e-11


def check_norm_scale_invariance(o, layer, L=30, seed=13):
    """With q, k and v normed (eps far below the inputs' mean square), scaling any raw q, k or v
    vector by a positive factor leaves every output unchanged; without the norms it does not."""
    q, k, v, norms = normed_inputs(layer, L, seed, eps=1e-14)
    r = rng(seed + 1)
    cq = r.uniform(0.1, 10.0, (L, layer.n_q_heads, 1))
    ck = r.uniform(0.1, 10.0, (L, layer.n_kv_heads, 1))
    v2 = None if v is None else v * r.uniform(0.1, 10.0, (L, layer.n_kv_heads, 1))
    base = o.layer_rows(layer, q, np.arange(L), k, v, 0, norms)
    got = o.layer_rows(layer, q * cq, np.arange(L), k * ck, v2, 0, norms)
    assert np.abs(got - base).max() < 1e-9
    raw = o.layer_rows(layer, q * cq, np.arange(L), k * ck, v2) - o.layer_rows(layer, q, np.arange(L), k, v)
    assert np.abs(raw).max() > 1e-3


# ---------------------------------------------------------------- the pins


def test_rms_norm_closed_form():
    check_rms_norm_closed_form(oracle)


def test_rms_norm_matches_torch():
    check_rms_norm_vs_torch(oracle)


@pytest.mark.parametrize("layer,kw", [
    (oracle.with_window(oracle.SLIDING, 8), {}),
    (oracle.with_window(oracle.SLIDING, 8), dict(k_weight=False, v_norm=False)),
    (oracle.with_window(oracle.SLIDING, 8), dict(q_weight=False)),
    (oracle.GLOBAL, {}),
    (oracle.GLOBAL, dict(k_weight=False, v_norm=False)),
], ids=["sliding-all", "sliding-q-only", "sliding-kv-only", "global-all", "global-q-only"])
def test_normed_layer_matches_torch(layer, kw):
    check_normed_layer_vs_torch(oracle, layer, **kw)


@pytest.mark.parametrize("layer", [oracle.with_window(oracle.SLIDING, 8), oracle.GLOBAL], ids=["sliding", "global"])
def test_normed_outputs_do_not_depend_on_input_scale(layer):
    check_norm_scale_invariance(oracle, layer)


def test_normed_decode_row_equals_prefill_row():
    for layer in (oracle.with_window(oracle.SLIDING, 16), oracle.GLOBAL):
        q, k, v, norms = normed_inputs(layer, 40, 15)
        rows = oracle.layer_rows(layer, q, np.arange(40), k, v, 0, norms)
        for p in (0, 17, 39):
            d = oracle.decode_row(layer, q[p], k[:p + 1], None if v is None else v[:p + 1], norms)
            assert np.abs(d - rows[p]).max() < 1e-12

def test_geometry_matches_checkpoint_fingerprint():
    check_geometry(oracle)


@pytest.mark.parametrize("D,theta,partial", [(256, 1e4, 1.0), (512, 1e6, 0.25), (64, 100.0, 0.5)])
def test_rope_is_complex_rotation(D, theta, partial):
    check_rope_complex(oracle, D, theta, partial)


@pytest.mark.parametrize("D,theta", [(256, 1e4), (512, 1e6)])
def test_inv_freq_identities(D, theta):
    check_inv_freq_identities(oracle, D, theta)


def test_rotated_pair_counts():
    assert oracle.rope_rotated_pairs(256, 1.0) == 128
    assert oracle.rope_rotated_pairs(512, 0.25) == 64


@pytest.mark.parametrize("layer", [oracle.SLIDING, oracle.GLOBAL], ids=["sliding", "global"])
def test_rope_norms_identity_and_untouched_dims(layer):
    r = rng(6)
    D = layer.head_dim
    x = bf16ish(r.standard_normal((64, D)))
    pos = r.integers(0, oracle.MAX_POSITIONS, size=64)
    pos[0] = 0
    y = oracle.rope(x, pos, layer.rope_theta, layer.rope_partial)
    half = D // 2
    assert np.allclose(x[:, :half] ** 2 + x[:, half:] ** 2, y[:, :half] ** 2 + y[:, half:] ** 2,
                       rtol=1e-12, atol=1e-12)
    assert np.array_equal(y[0], x[0])                       # position 0 is the identity
    R = oracle.rope_rotated_pairs(D, layer.rope_partial)
    untouched = np.r_[R:half, half + R:D]
    assert np.array_equal(y[:, untouched], x[:, untouched])  # bitwise, not just close
    moved = np.r_[0:R, half:half + R]
    assert (np.abs(y[1:, moved] - x[1:, moved]).max(axis=1) > 0).all()


@pytest.mark.parametrize("layer", [oracle.SLIDING, oracle.GLOBAL], ids=["sliding", "global"])
def test_rope_scores_depend_on_relative_position(layer):
    r = rng(7)
    D = layer.head_dim
    q, k = r.standard_normal(D), r.standard_normal(D)
    for i, j, delta in [(5, 3, 1000), (300, 0, 77777), (1023, 1000, 200000)]:
        a = oracle.rope(q, i, layer.rope_theta, layer.rope_partial) @ oracle.rope(k, j, layer.rope_theta, layer.rope_partial)
        b = oracle.rope(q, i + delta, layer.rope_theta, layer.rope_partial) @ \
            oracle.rope(k, j + delta, layer.rope_theta, layer.rope_partial)
        assert abs(a - b) < 1e-8 * (1 + abs(a))


def test_core_matches_sdpa_causal():
    check_sdpa_causal(oracle)


@pytest.mark.parametrize("W", [1, 2, 7, 49, 50, 64])
def test_core_matches_sdpa_band(W):
    check_sdpa_band(oracle, W)


@pytest.mark.parametrize("layer", [oracle.with_window(oracle.SLIDING, 16), oracle.GLOBAL], ids=["sliding", "global"])
def test_layer_matches_sdpa_gqa(layer):
    check_layer_vs_sdpa(oracle, layer)


@pytest.mark.parametrize("layer", [oracle.with_window(oracle.SLIDING, 64), oracle.GLOBAL], ids=["sliding", "global"])
def test_q_zero_gives_mean_of_visible_values(layer):
    check_q_zero_mean(oracle, layer)


@pytest.mark.parametrize("layer", [oracle.with_window(oracle.SLIDING, 32), oracle.GLOBAL], ids=["sliding", "global"])
def test_keys_outside_the_mask_do_not_matter(layer):
    check_outside_perturbation(oracle, layer)


def test_window_at_least_length_is_causal():
    r = rng(8)
    L = 60
    lay = oracle.with_window(oracle.SLIDING, 60)
    q = r.standard_normal((L, 32, 256))
    k = r.standard_normal((L, 16, 256))
    v = r.standard_normal((L, 16, 256))
    a = oracle.layer_rows(lay, q, np.arange(L), k, v)
    b = oracle.layer_rows(oracle.with_window(oracle.SLIDING, 0), q, np.arange(L), k, v)
    c = oracle.layer_rows(oracle.with_window(oracle.SLIDING, 10 ** 6), q, np.arange(L), k, v)
    assert np.array_equal(a, b) and np.array_equal(b, c)


@pytest.mark.parametrize("layer", [oracle.with_window(oracle.SLIDING, 24), oracle.GLOBAL], ids=["sliding", "global"])
def test_outputs_invariant_to_position_shift(layer):
    r = rng(9)
    L = 48
    q = r.standard_normal((L, 32, layer.head_dim))
    k = r.standard_normal((L, layer.n_kv_heads, layer.head_dim))
    v = None if layer.kv_shared else r.standard_normal((L, layer.n_kv_heads, layer.head_dim))
    a = oracle.layer_rows(layer, q, np.arange(L), k, v)
    b = oracle.layer_rows(layer, q, np.arange(L), k, v, pos_offset=123457)
    assert np.abs(a - b).max() < 1e-10


def test_k_eq_v_uses_unrotated_values():
    """The global layer fed S equals a two-tensor layer of the same geometry fed K := S, V := S
    (only K is rotated), and differs from one fed V := p-RoPE(S)."""
    r = rng(10)
    L = 70
    G = oracle.GLOBAL
    two = oracle.Layer("global", 32, 4, 512, 0, G.rope_theta, G.rope_partial, False)
    q = r.standard_normal((L, 32, 512))
    S = r.standard_normal((L, 4, 512))
    a = oracle.layer_rows(G, q, np.arange(L), S, None)
    b = oracle.layer_rows(two, q, np.arange(L), S, S)
    assert np.array_equal(a, b)
    S_rot = oracle.rope(S, np.arange(L)[:, None], G.rope_theta, G.rope_partial)
    c = oracle.layer_rows(two, q, np.arange(L), S, S_rot)
    assert np.abs(a - c).max() > 1e-3


@pytest.mark.parametrize("layer", [oracle.with_window(oracle.SLIDING, 64), oracle.GLOBAL], ids=["sliding", "global"])
def test_decode_row_equals_prefill_row(layer):
    r = rng(11)
    L = 130
    q = r.standard_normal((L, 32, layer.head_dim))
    k = r.standard_normal((L, layer.n_kv_heads, layer.head_dim))
    v = None if layer.kv_shared else r.standard_normal((L, layer.n_kv_heads, layer.head_dim))
    full = oracle.layer_rows(layer, q, np.arange(L), k, v)
    for p in (0, 1, 63, 64, L - 1):
        d = oracle.decode_row(layer, q[p], k[:p + 1], None if v is None else v[:p + 1])
        assert np.abs(d - full[p]).max() < 1e-12


def test_batched_prefill_matches_per_sequence_rows_and_chunks():
    """Packed rows, a chunk with history (ctx_start > 0) and a padding gap."""
    r = rng(12)
    lay = oracle.with_window(oracle.SLIDING, 20)
    lens, ctx = [30, 17], [0, 25]
    hist_k = [r.standard_normal((c + L, 16, 256)) for L, c in zip(lens, ctx)]
    hist_v = [r.standard_normal((c + L, 16, 256)) for L, c in zip(lens, ctx)]
    q = r.standard_normal((60, 32, 256))
    out = oracle.prefill(lay, q, hist_k, hist_v, [0, 40], lens, ctx)
    assert np.isnan(out[30:40]).all() and np.isnan(out[57:]).all()
    a = oracle.layer_rows(lay, q[40:57], np.arange(25, 42), hist_k[1], hist_v[1])
    assert np.array_equal(out[40:57], a)
    full = oracle.layer_rows(lay, np.concatenate([np.zeros((25, 32, 256)), q[40:57]]), np.arange(42),
                             hist_k[1], hist_v[1])
    assert np.abs(full[25:] - out[40:57]).max() < 1e-12


def test_credited_flops_closed_form():
    # Sliding 4 x 4096 with W = 1024: sum_i min(i+1, W) = W(W+1)/2 + (L-W) W per sequence.
    pairs = 1024 * 1025 // 2 + (4096 - 1024) * 1024
    assert pairs == 3670528
    got = oracle.credited_prefill_flops(oracle.SLIDING, [4096] * 4, [0] * 4)
    assert got == 4.0 * 256 * 32 * 4 * pairs
    got = oracle.credited_prefill_flops(oracle.GLOBAL, [8192] * 2, [0] * 2)
    assert got == 4.0 * 512 * 32 * 2 * (8192 * 8193 // 2)


# ---------------------------------------------------------------- vision-token mask

def token_type_mask(token_type: np.ndarray, base: torch.Tensor) -> torch.Tensor:
    """The usual construction of the vision mask from per-token types (1 = image token): each
    maximal run of image tokens is one image, numbered by a cumulative sum over run starts; a
    query and a key of the same image see each other; everything else keeps the base mask."""
    tt = torch.from_numpy(np.asarray(token_type, np.int64))
    starts = (tt == 1) & torch.cat([torch.ones(1, dtype=torch.bool), tt[:-1] == 0])
    group = torch.cumsum(starts.long(), 0)
    img = (tt[:, None] == 1) & (tt[None, :] == 1) & (group[:, None] == group[None, :])
    return base | img


def runs_of_ones(token_type):
    """[s0, s1) of each maximal run of 1s, by a plain scan."""
    spans, s0 = [], None
    for i, t in enumerate(list(token_type) + [0]):
        if t == 1 and s0 is None:
            s0 = i
        elif t != 1 and s0 is not None:
            spans.append((s0, i))
            s0 = None
    return spans


VISION_TYPES = {
    # two images, one longer than the test window, one touching the last row
    "mid": [0] * 5 + [1] * 13 + [0] * 6 + [1] * 4 + [0] * 9 + [1] * 3,
    # an image at the very start, and single-token images
    "edges": [1] * 7 + [0, 1, 0, 0, 1] + [0] * 10 + [1] * 9 + [0] * 12,
}


def check_vision_vs_sdpa(o, layer, types, seed=11):
    r = rng(seed)
    L = len(types)
    q = r.standard_normal((L, layer.n_q_heads, layer.head_dim))
    k = r.standard_normal((L, layer.n_kv_heads, layer.head_dim))
    v = None if layer.kv_shared else r.standard_normal((L, layer.n_kv_heads, layer.head_dim))
    got = o.layer_rows(layer, q, np.arange(L), k, v, spans=runs_of_ones(types))
    pos = np.arange(L)[:, None]
    qr = o.rope(q, pos, layer.rope_theta, layer.rope_partial)
    kr = o.rope(k, pos, layer.rope_theta, layer.rope_partial)
    vv = k if layer.kv_shared else v
    tq = torch.from_numpy(qr).permute(1, 0, 2)[None]
    tk = torch.from_numpy(kr).permute(1, 0, 2).repeat_interleave(layer.group, dim=0)[None]
    tv = torch.from_numpy(vv).permute(1, 0, 2).repeat_interleave(layer.group, dim=0)[None]
    ones = torch.ones(L, L, dtype=torch.bool)
    base = torch.tril(ones)
    if layer.window > 0:
        base &= torch.triu(ones, diagonal=-(layer.window - 1))
    mask = token_type_mask(np.asarray(types), base)
    ref = F.scaled_dot_product_attention(tq, tk, tv, attn_mask=mask,
                                         scale=1.0 / math.sqrt(layer.head_dim))[0].permute(1, 0, 2).numpy()
    assert np.abs(got - ref).max() < 1e-11


def check_whole_image_is_full_attention(o, L=24, seed=12):
    """A global layer whose every token belongs to one image attends without any mask."""
    layer = o.GLOBAL
    r = rng(seed)
    q = r.standard_normal((L, layer.n_q_heads, layer.head_dim))
    s = r.standard_normal((L, layer.n_kv_heads, layer.head_dim))
    got = o.layer_rows(layer, q, np.arange(L), s, None, spans=[(0, L)])
    pos = np.arange(L)[:, None]
    tq = torch.from_numpy(o.rope(q, pos, layer.rope_theta, layer.rope_partial)).permute(1, 0, 2)[None]
    tk = torch.from_numpy(o.rope(s, pos, layer.rope_theta, layer.rope_partial)).permute(1, 0, 2)
    tv = torch.from_numpy(s).permute(1, 0, 2)
    ref = F.scaled_dot_product_attention(tq, tk.repeat_interleave(layer.group, 0)[None],
                                         tv.repeat_interleave(layer.group, 0)[None], is_causal=False,
                                         scale=1.0 / math.sqrt(layer.head_dim))[0].permute(1, 0, 2).numpy()
    assert np.abs(got - ref).max() < 1e-11


@pytest.mark.parametrize("types", sorted(VISION_TYPES))
@pytest.mark.parametrize("layer", [oracle.with_window(oracle.SLIDING, 6), oracle.GLOBAL], ids=["sliding", "global"])
def test_vision_mask_matches_token_type_construction(layer, types):
    check_vision_vs_sdpa(oracle, layer, VISION_TYPES[types])


def test_whole_sequence_image_is_unmasked_attention():
    check_whole_image_is_full_attention(oracle)


def test_vision_spans_in_batched_prefill_match_per_sequence_rows():
    """prefill hands each sequence its own spans, also for a chunk that starts mid-context."""
    r = rng(13)
    layer = oracle.with_window(oracle.SLIDING, 8)
    lens, ctx = [30, 21], [0, 9]
    spans = [[(3, 14)], [(10, 25)]]
    hist = [r.standard_normal((c + n, layer.n_kv_heads, layer.head_dim)) for n, c in zip(lens, ctx)]
    vh = [r.standard_normal(h.shape) for h in hist]
    q = r.standard_normal((sum(lens), layer.n_q_heads, layer.head_dim))
    got = oracle.prefill(layer, q, hist, vh, [0, 30], lens, ctx, spans=spans)
    want1 = oracle.layer_rows(layer, q[30:], np.arange(9, 30), hist[1], vh[1], spans=spans[1])
    assert np.array_equal(got[30:], want1)
    plain = oracle.prefill(layer, q, hist, vh, [0, 30], lens, ctx)
    assert not np.allclose(got[:30], plain[:30])


# ---------------------------------------------------------------- planted mistakes

def _fails(fn, *a, **kw):
    try:
        fn(*a, **kw)
    except AssertionError:
        return True
    return False


def test_control_window_off_by_one(monkeypatch):
    good = oa.visible

    def wide(q_pos, k_pos, window):
        return good(q_pos, k_pos, window + 1 if window > 0 else 0)
    monkeypatch.setattr(oa, "visible", wide)
    assert _fails(check_q_zero_mean, oa, oracle.with_window(oracle.SLIDING, 64))
    assert _fails(check_sdpa_band, oa, 7)


def test_control_interleaved_pairs(monkeypatch):
    def interleaved(x, pos, theta, partial):
        x = np.asarray(x, np.float64)
        D = x.shape[-1]
        R = oa.rope_rotated_pairs(D, partial)
        ang = np.asarray(pos, np.float64)[..., None] * oa.rope_inv_freq(D, theta)[:R]
        y = x.copy()
        a, b = x[..., 0:2 * R:2], x[..., 1:2 * R:2]
        y[..., 0:2 * R:2] = a * np.cos(ang) - b * np.sin(ang)
        y[..., 1:2 * R:2] = b * np.cos(ang) + a * np.sin(ang)
        return y
    monkeypatch.setattr(oa, "rope", interleaved)
    assert _fails(check_rope_complex, oa, 512, 1e6, 0.25)


def test_control_rotation_direction(monkeypatch):
    good = oa.rope
    monkeypatch.setattr(oa, "rope", lambda x, pos, theta, partial: good(x, -np.asarray(pos), theta, partial))
    assert _fails(check_rope_complex, oa, 256, 1e4, 1.0)


def test_control_frequency_denominator(monkeypatch):
    # The other partial-RoPE reading: a spectrum over the rotated block only.
    monkeypatch.setattr(oa, "rope_inv_freq",
                        lambda D, theta: np.power(float(theta), -2.0 * np.arange(D // 2) / (D // 2)))
    assert _fails(check_inv_freq_identities, oa, 512, 1e6)
    assert _fails(check_rope_complex, oa, 512, 1e6, 0.25)


def test_control_values_rotated(monkeypatch):
    good = oa.keys_values

    def rotated_v(layer, k_hist, v_hist, pos_offset=0, norms=None):
        k_rot, v = good(layer, k_hist, v_hist, pos_offset, norms)
        return k_rot, (k_rot.copy() if layer.kv_shared else v)
    monkeypatch.setattr(oa, "keys_values", rotated_v)
    assert _fails(check_q_zero_mean, oa, oracle.GLOBAL)


def test_control_dropped_scale(monkeypatch):
    good = oa.attention
    monkeypatch.setattr(oa, "attention", lambda q, k, v, qp, kp, w, s: good(q, k, v, qp, kp, w, 1.0))
    assert _fails(check_sdpa_causal, oa)
    assert _fails(check_layer_vs_sdpa, oa, oracle.GLOBAL)


def test_control_gqa_mapping(monkeypatch):
    # Wrong head grouping: query head h reads KV head h % Hkv instead of h // G.
    def modulo_rows(layer, q_rows, q_pos, k_hist, v_hist, pos_offset=0):
        q_rows = np.asarray(q_rows, np.float64)
        k_rot, v = oa.keys_values(layer, k_hist, v_hist, pos_offset)
        qp = np.asarray(q_pos) + pos_offset
        q_rot = oa.rope(q_rows, qp[:, None], layer.rope_theta, layer.rope_partial)
        out = np.empty((q_rows.shape[0], layer.n_q_heads, v.shape[2]))
        kp = np.arange(k_rot.shape[0]) + pos_offset
        for h in range(layer.n_q_heads):
            g = h % layer.n_kv_heads
            out[:, h] = oa.attention(q_rot[:, h], k_rot[:, g], v[:, g], qp, kp, layer.window, layer.scale)
        return out
    monkeypatch.setattr(oa, "layer_rows", modulo_rows)
    assert _fails(check_layer_vs_sdpa, oa, oracle.GLOBAL)


def test_control_norm_weight_inside(monkeypatch):
    # The weight applied before the normalisation instead of after it.
    good = oa.rms_norm
    monkeypatch.setattr(oa, "rms_norm", lambda x, w, eps: good(np.asarray(x) * (1.0 if w is None else w), None, eps))
    assert _fails(check_normed_layer_vs_torch, oa, oracle.with_window(oracle.SLIDING, 8))
    assert _fails(check_normed_layer_vs_torch, oa, oracle.GLOBAL)


def test_control_k_eq_v_values_take_the_key_weight(monkeypatch):
    # K==V with V normed by the key's weighted norm instead of the unit norm.
    good = oa.normed_kv

    def wrong(layer, norms, k, v):
        kk, vv = good(layer, norms, k, v)
        return kk, (kk.copy() if layer.kv_shared and norms is not None and norms.k_weight is not None else vv)
    monkeypatch.setattr(oa, "normed_kv", wrong)
    assert _fails(check_normed_layer_vs_torch, oa, oracle.GLOBAL)


def test_control_norm_missing_on_queries(monkeypatch):
    monkeypatch.setattr(oa, "normed_q", lambda norms, q: np.asarray(q, np.float64))
    assert _fails(check_normed_layer_vs_torch, oa, oracle.GLOBAL)
    assert _fails(check_norm_scale_invariance, oa, oracle.with_window(oracle.SLIDING, 8))


def test_control_vision_forward_only(monkeypatch):
    good = oa.same_image
    monkeypatch.setattr(oa, "same_image", lambda qp, kp, sp: good(qp, kp, sp) &
                        (np.asarray(kp)[None, :] <= np.asarray(qp)[:, None]))
    assert _fails(check_vision_vs_sdpa, oa, oracle.GLOBAL, VISION_TYPES["mid"])
    assert _fails(check_whole_image_is_full_attention, oa)


def test_control_vision_leaks_to_text_rows(monkeypatch):
    def leaky(qp, kp, sp):
        kp = np.asarray(kp)[None, :]
        ok = np.zeros((len(qp), kp.shape[1]), dtype=bool)
        for s0, s1 in sp:
            ok |= (kp >= s0) & (kp < s1)
        return ok
    monkeypatch.setattr(oa, "same_image", leaky)
    assert _fails(check_vision_vs_sdpa, oa, oracle.GLOBAL, VISION_TYPES["mid"])


def test_control_vision_span_end_inclusive(monkeypatch):
    good = oa.same_image
    monkeypatch.setattr(oa, "same_image", lambda qp, kp, sp: good(qp, kp, [(a, b + 1) for a, b in sp]))
    assert _fails(check_vision_vs_sdpa, oa, oracle.with_window(oracle.SLIDING, 6), VISION_TYPES["edges"])
