"""Tensor parallelism over heads, simulated on one GPU (RL-Kernel RFC "[RFC][Gemma-4-31B-it] WS1/WS2
kernel roadmap", section 5 rows ws2_tp2, ws2_tp4 and ws2_tp8_kv_replication; section 4 rule 6: a
row is invariant to rank placement).

With tp ranks, rank r owns query heads 32 r / tp .. 32 (r + 1) / tp - 1 and the KV heads they read:
16 / tp sliding KV heads, and 4 / tp global ones, where at tp = 8 the 4 global KV heads are
replicated, ranks 2g and 2g + 1 both holding head g. Each rank's call runs on tensors and a paged
cache that hold only its heads, through a layer descriptor with the slice's head counts. Attention
has no exchange step between heads, so no collective is involved: the test runs the tp rank calls
one after another and checks that their outputs, side by side, are the full call's bits. The same
holds for a decode step over caches each rank filled itself. A rank slice also matches the fp64
oracle of its own geometry.
"""
import copy

import numpy as np
import pytest
import torch

import invariant_hybrid_attention_gb300 as g4
import oracle

from gpu_cases import Batch, DecodeBatch, assert_close, f64, layers

pytestmark = pytest.mark.gpu


def rank_heads(kind, tp, r):
    """(query head range, KV head range) of rank r of tp; query head h reads full KV head h // G."""
    G = 2 if kind == "sliding" else 8
    hq = 32 // tp
    q0, q1 = r * hq, (r + 1) * hq
    return (q0, q1), (q0 // G, (q1 - 1) // G + 1)


def rank_layer(kind, tp, window=1024):
    return g4.sliding_layer(window, tp=tp) if kind == "sliding" else g4.global_layer(tp=tp)


def slice_batch(bt, kind, tp, r):
    """A rank's copy of a prefill batch: its query heads and the KV heads they read."""
    (q0, q1), (k0, k1) = rank_heads(kind, tp, r)
    rb = copy.copy(bt)
    rb.q = bt.q[:, q0:q1].contiguous()
    rb.hist_k = [h[:, k0:k1].contiguous() for h in bt.hist_k]
    rb.k_rows = bt.k_rows[:, k0:k1].contiguous()
    if bt.hist_v is not None:
        rb.hist_v = [h[:, k0:k1].contiguous() for h in bt.hist_v]
        rb.v_rows = bt.v_rows[:, k0:k1].contiguous()
    rb.n_kv = k1 - k0
    return rb


@pytest.mark.parametrize("tp", [2, 4, 8])
@pytest.mark.parametrize("kind", ["sliding", "global"])
def test_rank_slices_of_a_prefill_are_the_full_call_bit_for_bit(kind, tp):
    layer, _ = layers(kind, 1024)
    bt = Batch(kind, [300, 130, 1], ctx_starts=[0, 200, 17], padded=True, seed=95, scale=0.5)
    full, _ = bt.run(layer)
    full = full.cpu().view(torch.int16)
    for r in range(tp):
        (q0, q1), _ = rank_heads(kind, tp, r)
        out, _ = slice_batch(bt, kind, tp, r).run(rank_layer(kind, tp))
        assert torch.equal(out.cpu().view(torch.int16), full[:, q0:q1]), (kind, tp, r)


@pytest.mark.parametrize("tp", [2, 8])
@pytest.mark.parametrize("kind", ["sliding", "global"])
def test_rank_slices_of_a_decode_step_are_the_full_call_bit_for_bit(kind, tp):
    layer, _ = layers(kind, 1024)
    db = DecodeBatch(kind, [5, 1500, 2049], seed=96)
    full, _ = db.run(layer)
    full = full.cpu().view(torch.int16)
    for r in range(tp):
        (q0, q1), (k0, k1) = rank_heads(kind, tp, r)
        rd = copy.copy(db)
        rd.q = db.q[:, q0:q1].contiguous()
        rd.hist_k = [h[:, k0:k1].contiguous() for h in db.hist_k]
        rd.hist_v = [h[:, k0:k1].contiguous() for h in db.hist_v]
        rd.n_kv = k1 - k0
        out, _ = rd.run(rank_layer(kind, tp))
        assert torch.equal(out.cpu().view(torch.int16), full[:, q0:q1]), (kind, tp, r)


@pytest.mark.parametrize("kind", ["sliding", "global"])
def test_a_tp8_rank_slice_matches_the_oracle_of_its_geometry(kind):
    """Rank 3 of 8 (query heads 12-15; sliding KV heads 6-7, global KV head 1, replicated) against the
    fp64 oracle of a layer with the slice's head counts."""
    tp, r = 8, 3
    window = 64 if kind == "sliding" else 0
    _, full_olayer = layers(kind, window or 1024)
    bt = Batch(kind, [200, 77], seed=97, scale=0.5)
    rb = slice_batch(bt, kind, tp, r)
    out, _ = rb.run(rank_layer(kind, tp, window or 1024))
    got = f64(out)
    (q0, q1), (k0, k1) = rank_heads(kind, tp, r)
    olayer = oracle.Layer(kind, q1 - q0, k1 - k0, full_olayer.head_dim, window, full_olayer.rope_theta,
                          full_olayer.rope_partial, full_olayer.kv_shared)
    for b, L in enumerate(rb.q_lens):
        s = rb.layout.q_start[b]
        assert_close(got[s:s + L], rb.oracle_rows(olayer, b), f"{kind} tp8 rank {r} sequence {b}")
