"""Plain fp64 CPU oracle for the hybrid sliding/global decoder attention of Gemma-4-31B.

TEST INFRASTRUCTURE. Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU legs of
``bench.py`` (its ``cpu_baseline`` and ``--impl reference``) import this package. The
product path (the CUDA library and its binding) never does, and the two share no code.

Sources, cited by page title and section:

* RFC = "[RFC][Gemma-4-31B-it][CUDA/ROCm] WS1/WS2 kernel roadmap, ablation matrix and
  integration plan" (RL-Kernel issue 415).
  - §2 "Checkpoint fingerprint" table: 32 Q heads; sliding layers 16 KV heads of dim 256,
    window 1024, standard RoPE theta 1e4; global layers 4 KV heads of dim 512,
    ``attention_k_eq_v=true``, proportional p-RoPE with partial factor 0.25 and theta 1e6;
    5 sliding : 1 full schedule; 262144 max positions.
  - §5 work-item table rows ``sliding_rope_d256``, ``global_proportional_p_rope``,
    ``sliding_attention_core`` (causal local attention, window 1024),
    ``global_attention_core`` (full causal attention with K=V) and
    ``global_k_eq_v_projection`` (K=V is one projection).
* TF = TensorFold PR "cuda gemma4: images on the 31B, the image tower": its Gemma 4 engine
  commit keeps each sliding layer's last 1023 positions, so a query sees itself plus the
  1023 keys before it (window edge reading below).

Readings of points the pages leave open (each is listed in the design notes):

* RoPE pairs are half-split: element t pairs with t + D/2 for t < D/2. Pair t turns by
  ``pos * theta**(-2t/D)``; the exponent runs over the full head dim D, which is what makes
  the partial RoPE "proportional". Only the first ``R = floor(partial * D / 2)`` pairs turn
  (R = 128 of 128 on sliding layers, 64 of 256 on global layers); the rest pass unchanged.
* K==V: the cache holds one projection S per global layer. V is S as stored; K is
  p-RoPE(S). At position 0 the rotation is the identity, so K and V agree there.
* Window W: key j is visible to query i iff j <= i and i - j <= W - 1. Global layers: j <= i.
* Vision tokens (the model card's ``use_bidirectional_attention="vision"``; RFC §5 row
  ``multimodal_bidirectional_mask``): the tokens of one image see one another in both
  directions, on top of the layer's own mask. An image is a span [s0, s1) of positions. The RFC
  puts this mask in the global attention path; TensorFold's engine gives it to the sliding
  layers (an image row sees every row of its image past the window) and keeps global layers
  causal. Both readings are covered: the spans are an argument of either layer kind, and the
  caller passes them to the layers it wants. A decode query is a text token and takes none.
* Softmax scale defaults to 1/sqrt(D). No attention-logit soft cap (only the final logits
  are capped, RFC §2).
* Positions are the index within the sequence: 0 .. L-1; a decode query sits at L-1.
* GQA: KV head g serves query heads g*G .. g*G+G-1 with G = Hq / Hkv.
* Per-head norms (RFC §5 row ``qk_rmsnorm_d256_d512``; TensorFold's ``tf_qk_rows_once``, which
  "can norm v by a unit RMS norm"), optional and applied to the raw projections before RoPE:
  n(x) = x / sqrt(mean(x^2 over the head dim) + eps). q -> w_q * n(q) and k -> w_k * n(k) with
  per-dim weights; v -> n(v) (unit, no weight). On a K==V layer the one projection S gives
  K = w_k * n(S) and V = n(S). The pages do not give eps; it is a parameter (1e-6 by default).

Parity pins for every function here live in ``tests/test_oracle.py``.
"""
from __future__ import annotations

import math
from dataclasses import dataclass
from typing import Optional, Sequence

import numpy as np


@dataclass(frozen=True)
class Layer:
    kind: str            # "sliding" | "global"
    n_q_heads: int
    n_kv_heads: int
    head_dim: int
    window: int          # keys seen including self; 0 = unbounded (global)
    rope_theta: float
    rope_partial: float
    kv_shared: bool      # K==V (global layers)
    softmax_scale: Optional[float] = None

    @property
    def scale(self) -> float:
        return self.softmax_scale if self.softmax_scale is not None else 1.0 / math.sqrt(self.head_dim)

    @property
    def group(self) -> int:
        return self.n_q_heads // self.n_kv_heads


# RFC §2 checkpoint-fingerprint table.
SLIDING = Layer("sliding", 32, 16, 256, 1024, 1.0e4, 1.0, False)
GLOBAL = Layer("global", 32, 4, 512, 0, 1.0e6, 0.25, True)
MAX_POSITIONS = 262144


def with_window(layer: Layer, window: int) -> Layer:
    return Layer(layer.kind, layer.n_q_heads, layer.n_kv_heads, layer.head_dim, int(window),
                 layer.rope_theta, layer.rope_partial, layer.kv_shared, layer.softmax_scale)


# ---- per-head RMS norms (RFC §5 qk_rmsnorm_d256_d512) -------------------------------------

@dataclass(frozen=True)
class Norms:
    q_weight: Optional[np.ndarray] = None   # [D] multiplier of the query norm; None: q is not normed
    k_weight: Optional[np.ndarray] = None   # [D] multiplier of the key norm; None: k is not normed
    v_norm: bool = False                    # values (V, or S read as V) get a unit RMS norm
    eps: float = 1e-6


def rms_norm(x: np.ndarray, weight: Optional[np.ndarray], eps: float) -> np.ndarray:
    """x / sqrt(mean(x^2) + eps) over the last axis, times `weight` per element when given."""
    x = np.asarray(x, dtype=np.float64)
    y = x / np.sqrt(np.mean(x * x, axis=-1, keepdims=True) + float(eps))
    return y if weight is None else y * np.asarray(weight, dtype=np.float64)


def normed_q(norms: Optional[Norms], q: np.ndarray) -> np.ndarray:
    q = np.asarray(q, np.float64)
    if norms is None or norms.q_weight is None:
        return q
    return rms_norm(q, norms.q_weight, norms.eps)


def normed_kv(layer: "Layer", norms: Optional[Norms], k: np.ndarray, v: Optional[np.ndarray]):
    """The key source and the values after the norms, before RoPE. K==V: both come from S."""
    k = np.asarray(k, np.float64)
    if layer.kv_shared:
        kk = k if norms is None or norms.k_weight is None else rms_norm(k, norms.k_weight, norms.eps)
        vv = k if norms is None or not norms.v_norm else rms_norm(k, None, norms.eps)
        return kk, vv
    v = np.asarray(v, np.float64)
    kk = k if norms is None or norms.k_weight is None else rms_norm(k, norms.k_weight, norms.eps)
    vv = v if norms is None or not norms.v_norm else rms_norm(v, None, norms.eps)
    return kk, vv


# ---- RoPE / p-RoPE (RFC §5 rows sliding_rope_d256 and global_proportional_p_rope) ----------

def rope_inv_freq(head_dim: int, theta: float) -> np.ndarray:
    """theta ** (-2t/D) for t = 0 .. D/2-1; the denominator is the full head dim D."""
    t = np.arange(head_dim // 2, dtype=np.float64)
    return np.power(float(theta), -2.0 * t / float(head_dim))


def rope_rotated_pairs(head_dim: int, partial: float) -> int:
    """R = floor(partial * D / 2): the leading pairs that turn; 0.25 of 256 pairs -> 64."""
    return int(math.floor(partial * head_dim / 2 + 1e-9))


def rope(x: np.ndarray, pos, theta: float, partial: float) -> np.ndarray:
    """Rotate the leading R half-split pairs of the last axis of `x` by pos * inv_freq.

    x: [..., D] (any float dtype, computed in fp64); pos: integers broadcastable to x.shape[:-1].
    Pairs t >= R are copied unchanged.
    """
    x = np.asarray(x, dtype=np.float64)
    D = x.shape[-1]
    half = D // 2
    R = rope_rotated_pairs(D, partial)
    y = x.copy()
    if R == 0:
        return y
    ang = np.asarray(pos, dtype=np.float64)[..., None] * rope_inv_freq(D, theta)[:R]
    c, s = np.cos(ang), np.sin(ang)
    a = x[..., :R]
    b = x[..., half:half + R]
    y[..., :R] = a * c - b * s
    y[..., half:half + R] = b * c + a * s
    return y


# ---- masks and the attention core (RFC §5 sliding_attention_core / global_attention_core) --

def visible(q_pos: np.ndarray, k_pos: np.ndarray, window: int) -> np.ndarray:
    """Boolean [n_q, n_k]: causal, and with window W > 0 also i - j <= W - 1."""
    qp = np.asarray(q_pos, dtype=np.int64)[:, None]
    kp = np.asarray(k_pos, dtype=np.int64)[None, :]
    ok = kp <= qp
    if window > 0:
        ok &= (qp - kp) <= (window - 1)
    return ok


def same_image(q_pos: np.ndarray, k_pos: np.ndarray, spans) -> np.ndarray:
    """Boolean [n_q, n_k]: query and key are tokens of one image. spans lists the images as
    [s0, s1) position ranges; text tokens lie in none."""
    qp = np.asarray(q_pos, dtype=np.int64)[:, None]
    kp = np.asarray(k_pos, dtype=np.int64)[None, :]
    ok = np.zeros((qp.shape[0], kp.shape[1]), dtype=bool)
    for s0, s1 in spans:
        ok |= (qp >= s0) & (qp < s1) & (kp >= s0) & (kp < s1)
    return ok


def attention(q: np.ndarray, k: np.ndarray, v: np.ndarray, q_pos, k_pos, window: int,
              scale: float, spans=None) -> np.ndarray:
    """softmax_j(scale * q.k_j over visible j) . v_j for one head.

    q: [n, D] (already rotated); k: [m, D] (already rotated); v: [m, Dv]. Returns [n, Dv].
    Visible: the layer's mask (`visible`), or, with image spans, also a key of the query's own
    image. Every query must see at least one key.
    """
    s = (np.asarray(q, np.float64) @ np.asarray(k, np.float64).T) * scale
    vis = visible(q_pos, k_pos, window)
    if spans:
        vis = vis | same_image(q_pos, k_pos, spans)
    if not vis.any(axis=1).all():
        raise ValueError("a query row sees no key")
    s = np.where(vis, s, -np.inf)
    p = np.exp(s - s.max(axis=1, keepdims=True))
    p = np.where(vis, p, 0.0)
    return (p @ np.asarray(v, np.float64)) / p.sum(axis=1, keepdims=True)


def keys_values(layer: Layer, k_hist: np.ndarray, v_hist: Optional[np.ndarray], pos_offset: int = 0,
                norms: Optional[Norms] = None):
    """The rotated keys and the values of one sequence's history.

    k_hist: [L, Hkv, D] raw key projections (the shared S for a K==V layer);
    v_hist: [L, Hkv, D] or None for K==V. Keys sit at positions pos_offset + 0..L-1.
    Returns (k_rot [L, Hkv, D], v [L, Hkv, D]) in fp64.
    """
    k_hist = np.asarray(k_hist, np.float64)
    L = k_hist.shape[0]
    pos = np.arange(L, dtype=np.int64) + pos_offset
    if layer.kv_shared:
        if v_hist is not None:
            raise ValueError("a K==V layer takes no separate V")
    elif v_hist is None:
        raise ValueError("a sliding layer needs V")
    k_src, v = normed_kv(layer, norms, k_hist, v_hist)   # K==V without norms: V is S, un-rotated
    k_rot = rope(k_src, pos[:, None], layer.rope_theta, layer.rope_partial)
    return k_rot, v


def layer_rows(layer: Layer, q_rows: np.ndarray, q_pos: Sequence[int], k_hist: np.ndarray,
               v_hist: Optional[np.ndarray], pos_offset: int = 0, norms: Optional[Norms] = None,
               spans=None) -> np.ndarray:
    """Attention output of one sequence's query rows.

    q_rows: [n, Hq, D] raw query projections at positions q_pos (each < L, measured from the
    first key); k_hist / v_hist as in `keys_values`; spans: the sequence's images as [s0, s1)
    ranges of absolute positions (see `same_image`), or None. Returns [n, Hq, D] fp64.
    """
    q_rows = normed_q(norms, q_rows)
    q_pos = np.asarray(q_pos, dtype=np.int64)
    k_rot, v = keys_values(layer, k_hist, v_hist, pos_offset, norms)
    L = k_rot.shape[0]
    k_pos = np.arange(L, dtype=np.int64) + pos_offset
    qp = q_pos + pos_offset
    q_rot = rope(q_rows, qp[:, None], layer.rope_theta, layer.rope_partial)
    out = np.empty((q_rows.shape[0], layer.n_q_heads, v.shape[2]), dtype=np.float64)
    for h in range(layer.n_q_heads):
        g = h // layer.group
        if spans:
            out[:, h, :] = attention(q_rot[:, h, :], k_rot[:, g, :], v[:, g, :], qp, k_pos,
                                     layer.window, layer.scale, spans)
        else:
            out[:, h, :] = attention(q_rot[:, h, :], k_rot[:, g, :], v[:, g, :], qp, k_pos,
                                     layer.window, layer.scale)
    return out


def prefill(layer: Layer, q: np.ndarray, k_hist: Sequence[np.ndarray], v_hist, q_start: Sequence[int],
            q_len: Sequence[int], ctx_start: Sequence[int], norms: Optional[Norms] = None,
            spans=None) -> np.ndarray:
    """Batched prefill: rows q_start[b] .. +q_len[b] of q [T, Hq, D] are sequence b's positions
    ctx_start[b] .. ctx_start[b]+q_len[b]-1; k_hist[b] holds that sequence's keys at positions
    0 .. ctx_start[b]+q_len[b]-1. spans[b] (optional) lists sequence b's images as [s0, s1)
    position ranges. Rows of q outside every sequence come back as NaN."""
    q = np.asarray(q, np.float64)
    out = np.full((q.shape[0], layer.n_q_heads, layer.head_dim), np.nan)
    for b in range(len(q_len)):
        s, L, c = int(q_start[b]), int(q_len[b]), int(ctx_start[b])
        if L == 0:
            continue
        vb = None if v_hist is None else v_hist[b][:c + L]
        sp = None if spans is None else spans[b]
        out[s:s + L] = layer_rows(layer, q[s:s + L], np.arange(c, c + L), k_hist[b][:c + L], vb, 0, norms, sp)
    return out


def decode_row(layer: Layer, q_new: np.ndarray, k_hist: np.ndarray, v_hist: Optional[np.ndarray],
               norms: Optional[Norms] = None) -> np.ndarray:
    """One decode step: the query [Hq, D] sits at position L-1 where L = len(k_hist), and the
    history already holds the new token's key/value at L-1. Written head by head, key by key."""
    q_new = normed_q(norms, q_new)
    k_rot, v = keys_values(layer, k_hist, v_hist, 0, norms)
    L = k_rot.shape[0]
    p = L - 1
    qr = rope(q_new, np.full((layer.n_q_heads,), p), layer.rope_theta, layer.rope_partial)
    lo = 0 if layer.window <= 0 else max(0, p - layer.window + 1)
    out = np.empty((layer.n_q_heads, v.shape[2]), np.float64)
    for h in range(layer.n_q_heads):
        g = h // layer.group
        scores = np.array([qr[h] @ k_rot[j, g] * layer.scale for j in range(lo, p + 1)])
        w = np.exp(scores - scores.max())
        out[h] = (w[:, None] * v[lo:p + 1, g, :]).sum(axis=0) / w.sum()
    return out


def credited_prefill_flops(layer: Layer, q_len: Sequence[int], ctx_start: Sequence[int]) -> float:
    """4 * D * Hq * (number of visible (query, key) pairs): QK^T and PV, 2 flops per MAC."""
    pairs = 0
    for L, c in zip(q_len, ctx_start):
        for i in range(int(c), int(c) + int(L)):
            n = i + 1
            if layer.window > 0:
                n = min(n, layer.window)
            pairs += n
    return 4.0 * layer.head_dim * layer.n_q_heads * pairs
