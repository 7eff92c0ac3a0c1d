"""The benchmark's three timed workloads, at their full shapes, against the fp64 oracle.

These run the very objects bench.py times (same shapes, seeds, value scales, page permutations and
calls), so the configurations it reports on are shown to compute the attention they claim:

  * sliding-window prefill: 4 causal sequences x 4096 tokens, Q 32x256, KV 16x256, window 1024,
    RoPE theta 1e4, N(0,1) x 0.5 values (seed 1), 16-token pages scattered by a random permutation;
  * global K==V prefill: 2 causal sequences x 8192 tokens, Q 32x512, 4 shared K=V heads x 512,
    p-RoPE partial 0.25 with theta 1e6, N(0,1) values (seed 2);
  * the decode mix: 64 requests, contexts uniform in [1024, 32768] (seed 7), values seed 8, one
    cache per layer of the 5 sliding : 1 global schedule, sliding caches mapping only the window's
    pages, every page scattered by a random permutation.

Each prefill sequence is checked on 256 sampled rows: rows 0, 1023, 1024 and the last, both rows at
every 128-row tile edge, and seeded random rows. Every request of every decode layer is checked.
The bars are max-abs 2e-2 and mean-abs 2e-3 on the bf16 outputs (fp32 accumulation inside).
"""
import numpy as np
import pytest
import torch

import bench
import invariant_hybrid_attention_gb300 as g4
from invariant_hybrid_attention_gb300 import inputs as gi
from invariant_hybrid_attention_gb300.paged import PagedKV, device_int32

from gpu_cases import assert_close

pytestmark = pytest.mark.gpu


@pytest.fixture(autouse=True)
def _loaded():
    g4.load()


def run_and_check_prefill(part):
    part.run()
    torch.cuda.synchronize()
    assert g4.g4attn_status_sync() == g4.G4_OK
    checked = part.check(256)
    assert len(checked) == len(part.lens)
    for name, rows, got, want in checked:
        L = part.lens[0]
        assert len(rows) >= 256 and rows[0] == 0 and rows[-1] == L - 1
        assert {1023, 1024} <= set(rows.tolist())
        assert set(range(127, L - 1, 128)) <= set(rows.tolist()) and set(range(128, L, 128)) <= set(rows.tolist())
        assert_close(got, want, name)


def test_sliding_prefill_4x4096_window_1024_matches_oracle():
    part = bench.SlidingPrefill(g4, gi, PagedKV, device_int32)
    assert part.lens == [4096] * 4 and part.W == 1024 and part.plan.num_pages == 4 * 256
    assert not torch.equal(part.plan.table.flatten().sort().values, part.plan.table.flatten())   # permuted
    run_and_check_prefill(part)


def test_global_prefill_2x8192_matches_oracle():
    part = bench.GlobalPrefill(g4, gi, PagedKV, device_int32)
    assert part.lens == [8192] * 2 and part.v is None
    run_and_check_prefill(part)


def test_decode_mix_b64_every_request_of_every_layer_matches_oracle():
    dec = bench.DecodeMix(g4, gi, PagedKV, device_int32)
    assert dec.B == 64 and len(dec.layers) == 6 and min(dec.lens) >= 1024 and max(dec.lens) <= 32768
    assert [L["sliding"] for L in dec.layers] == [True] * 5 + [False]
    for L in dec.layers[:5]:   # window-only maps: pages before the window are unmapped
        first = L["first"]
        t = L["table"].cpu()
        for b, f in enumerate(first):
            assert (t[b, :f // 16] == -1).all() and (t[b, f // 16:(dec.lens[b] + 15) // 16] >= 0).all()
    dec.run()
    torch.cuda.synchronize()
    assert g4.g4attn_status_sync() == g4.G4_OK
    for i in range(len(dec.layers)):
        for b in range(dec.B):
            got, want = dec.check_request(i, b)
            assert_close(got, want, f"decode layer {i} request {b} (ctx {dec.lens[b]})")
