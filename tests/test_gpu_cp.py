"""Context parallelism of a global (K==V) layer over keys, simulated on one GPU (RL-Kernel RFC
"[RFC][Gemma-4-31B-it] WS1/WS2 kernel roadmap", section 5 rows ws2_tp4_cp2 and
cp_sliding_window_policy; section 4 rule 3: a split only with a fixed merge tree).

A sequence's keys are cut into contiguous ranges, one per "rank"; each rank's paged cache holds only
its own range (the cuts fall inside pages, so a page a rank shares with its neighbour holds NaN where
the neighbour's keys would be). Every rank computes g4attn_prefill_partial for all the query rows over
its own keys, and g4attn_merge_partials merges the partials in rank order. Checked: the merged rows
against the fp64 oracle of the whole layer; each rank's partial, divided by its sum, against the
oracle restricted to that rank's keys; a single range merged alone against g4attn_prefill, bit for
bit (the same arithmetic up to one multiplication by 2^0); and the sharded call's rows bit-identical
across batchings.
"""
import numpy as np
import pytest
import torch

import invariant_hybrid_attention_gb300 as g4
import oracle
from invariant_hybrid_attention_gb300 import inputs as gi
from invariant_hybrid_attention_gb300.paged import PagedKV, device_int32

from gpu_cases import Batch, assert_close, f64, layers

pytestmark = pytest.mark.gpu


def run_sharded(bt: Batch, cuts, layer, seed=0):
    """cuts[b]: the range edges of sequence b (0 = e_0 <= e_1 <= ... <= e_n = its context length), the
    same n for every sequence. Returns (merged output, list of (o_part, ml_part)) as device tensors."""
    n = len(cuts[0]) - 1
    assert all(len(c) == n + 1 for c in cuts)
    T = bt.layout.T
    rows = (device_int32(bt.layout.q_start), device_int32(bt.layout.q_len), device_int32(bt.layout.ctx_start))
    q = bt.q.cuda()
    parts = []
    for r in range(n):
        lo = [c[r] for c in cuts]
        hi = [c[r + 1] for c in cuts]
        plan = gi.make_page_plan(bt.ctx_lens, seed=seed + 31 * r + 5, mapped_from=[a // 16 for a in lo],
                                 spare_pages=2)
        cache = PagedKV(plan.num_pages, 4, 512, shared=True)   # NaN-filled: only this rank's keys are written
        table = plan.table.cuda()
        lay = gi.packed_layout([b - a for a, b in zip(lo, hi)], lo)
        k = gi.rows_of([h[:b] for h, b in zip(bt.hist_k, hi)], lay, fill_nan=False).cuda()
        g4.g4attn_kv_append(layer, k, None, device_int32(lay.q_start), device_int32(lay.q_len),
                            device_int32(lay.ctx_start), cache.desc, table)
        o = torch.full((T, 32, 512), float("nan"), dtype=torch.float32, device="cuda")
        ml = torch.full((T, 32, 2), float("nan"), dtype=torch.float32, device="cuda")
        g4.g4attn_prefill_partial(layer, q, *rows, device_int32(lo), device_int32(hi), cache.desc, table, o, ml)
        parts.append((o, ml))
    out = torch.full_like(q, float("nan"))
    g4.g4attn_merge_partials(layer, [o for o, _ in parts], [m for _, m in parts], rows[0], rows[1], out)
    torch.cuda.synchronize()
    st = g4.g4attn_status_sync()
    assert st == g4.G4_OK, g4.status_string(st)
    return out, parts


def restricted_oracle(olayer, bt, b, rows, k_lo, k_hi):
    """fp64 attention of sequence b's rows over its keys k_lo .. k_hi-1 only (causal): [n, 32, 512],
    NaN for rows that see none of them."""
    c = bt.ctx_starts[b]
    s = bt.layout.q_start[b]
    qpos = c + np.asarray(rows)
    k_rot, v = oracle.keys_values(olayer, bt.hist_k[b].double().numpy(), None)
    qr = oracle.rope(bt.q[s + np.asarray(rows)].double().numpy(), qpos[:, None], olayer.rope_theta, olayer.rope_partial)
    kp = np.arange(k_lo, k_hi)
    out = np.full((len(rows), 32, 512), np.nan)
    sees = qpos >= k_lo
    if not sees.any():
        return out
    for h in range(32):
        out[sees, h] = oracle.attention(qr[sees, h], k_rot[k_lo:k_hi, h // 8], v[k_lo:k_hi, h // 8], qpos[sees], kp, 0,
                                        olayer.scale)
    return out


def test_sharded_global_prefill_matches_the_oracle_and_each_part_its_range():
    layer, olayer = layers("global")
    bt = Batch("global", [700, 333], ctx_starts=[0, 100], seed=101, scale=0.5)
    cuts = [[0, 130, 383, 612, 700], [0, 1, 250, 299, 433]]   # inside pages; one range of a single key
    out, parts = run_sharded(bt, cuts, layer, seed=7)
    got = f64(out)
    for b, L in enumerate(bt.q_lens):
        s = bt.layout.q_start[b]
        assert_close(got[s:s + L], bt.oracle_rows(olayer, b), f"merged sequence {b}")
        rows = np.unique(np.r_[0, L - 1, np.random.default_rng(b).choice(L, 40, replace=False)])
        for r, (o, ml) in enumerate(parts):
            want = restricted_oracle(olayer, bt, b, rows, cuts[b][r], cuts[b][r + 1])
            mlr = ml[s + torch.as_tensor(rows)].cpu().double().numpy()
            orr = o[s + torch.as_tensor(rows)].cpu().double().numpy()
            empty = np.isnan(want[:, 0, 0])
            assert (mlr[empty, :, 0] == -np.inf).all() and (mlr[empty, :, 1] == 0).all() and (orr[empty] == 0).all()
            if (~empty).any():
                part = orr[~empty] / mlr[~empty, :, 1:2]
                assert_close(part, want[~empty], f"sequence {b} part {r}")
    assert np.isnan(got[bt.layout.T:]).all()


def test_a_single_range_merged_alone_is_the_prefill_bit_for_bit():
    layer, _ = layers("global")
    bt = Batch("global", [300, 5, 129], ctx_starts=[0, 40, 0], padded=True, seed=102, scale=0.5)
    whole, _ = bt.run(layer)
    one, _ = run_sharded(bt, [[0, c] for c in bt.ctx_lens], layer, seed=8)
    assert torch.equal(whole.cpu().view(torch.int16), one.cpu().view(torch.int16))


def test_sharded_rows_are_bit_identical_across_batchings():
    layer, _ = layers("global")
    L = 900
    cuts_t = [0, 200, 517, 900]
    alone = Batch("global", [L], seed=103, scale=0.5)
    out_a, _ = run_sharded(alone, [cuts_t], layer, seed=9)
    for lens, padded, at in [([60, L, 333], False, 1), ([L, 1000], True, 0)]:
        bt = Batch("global", lens, padded=padded, seed=104 + len(lens), scale=0.5)
        bt.hist_k[at] = alone.hist_k[0]
        s = bt.layout.q_start[at]
        bt.q[s:s + L] = alone.q[:L]
        bt.k_rows = gi.rows_of(bt.hist_k, bt.layout)
        cuts = [cuts_t if i == at else [0, Li // 3, 2 * Li // 3, Li] for i, Li in enumerate(bt.ctx_lens)]
        out_b, _ = run_sharded(bt, cuts, layer, seed=11 + len(lens))
        assert torch.equal(out_a[:L].cpu(), out_b[s:s + L].cpu()), (lens, padded, at)
