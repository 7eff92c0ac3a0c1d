"""Fail closed when a kernel cannot make progress (RL-Kernel RFC "[RFC][Gemma-4-31B-it] WS1/WS2
kernel roadmap", section 4 rule 7).

Every spin-wait of the kernels' barrier protocols is bounded by a limit the host sets at launch
(g4attn_set_wait_limit_ns; 2 s by default). With the limit at 0, the first wait of each kernel whose
first poll fails gives up at once: the kernel sets the timeout bit of the device error word, lets the
copies and tensor-core operations it already issued finish, frees its tensor memory and returns.
Nothing here faults, traps or withholds an arrival: real waits simply run out.

Each case runs a small call with the default limit (the reference), then with the limit at 0, whose
status must be G4_ERR_TIMEOUT, then once more with the default limit: the status is clean again and
the output equals the reference bit for bit, so the context and the library's state survived.
"""
import pytest
import torch

import invariant_hybrid_attention_gb300 as g4
from invariant_hybrid_attention_gb300.paged import PagedKV, device_int32

from gpu_cases import Batch, DecodeBatch, layers

pytestmark = pytest.mark.gpu


def prefill_call(kind):
    layer, _ = layers(kind, 1024)
    bt = Batch(kind, [200, 77], seed=81, scale=0.5)

    def run():
        cache = bt.device_cache()
        out = torch.full_like(bt.q, float("nan")).cuda()
        rows = (device_int32(bt.layout.q_start), device_int32(bt.layout.q_len), device_int32(bt.layout.ctx_start))
        g4.g4attn_prefill(layer, bt.q.cuda(), bt.k_rows.cuda(), None if bt.v_rows is None else bt.v_rows.cuda(),
                          *rows, cache.desc, bt.plan.table.cuda(), out)
        torch.cuda.synchronize()
        return out, g4.g4attn_status_sync()
    return run


def decode_call(kind):
    layer, _ = layers(kind, 1024)
    db = DecodeBatch(kind, [900, 3000], seed=82)
    _, cache = db.run(layer)   # fills the cache (history and the new token) with the default limit
    q = db.q.cuda()
    k_new = torch.stack([h[L - 1] for h, L in zip(db.hist_k, db.ctx_lens)]).cuda()
    v_new = None if kind == "global" else torch.stack([h[L - 1] for h, L in zip(db.hist_v, db.ctx_lens)]).cuda()
    ws = torch.empty(g4.g4attn_decode_workspace_bytes(layer, 2, db.plan.max_pages), dtype=torch.uint8, device="cuda")

    def run():
        out = torch.full_like(q, float("nan"))
        g4.g4attn_decode(layer, q, k_new, v_new, device_int32(db.ctx_lens), cache.desc, db.plan.table.cuda(), out, ws)
        torch.cuda.synchronize()
        return out, g4.g4attn_status_sync()
    return run


CASES = {"decode-sliding": lambda: decode_call("sliding"), "decode-global": lambda: decode_call("global"),
         "prefill-sliding": lambda: prefill_call("sliding"), "prefill-global": lambda: prefill_call("global")}


@pytest.mark.parametrize("case", list(CASES))
def test_a_wait_that_runs_out_is_reported_and_the_next_call_is_exact(case):
    run = CASES[case]()
    assert g4.g4attn_wait_limit_ns() == g4.DEFAULT_WAIT_LIMIT_NS
    ref, st = run()
    assert st == g4.G4_OK
    g4.g4attn_set_wait_limit_ns(0)
    try:
        _, st = run()
    finally:
        g4.g4attn_set_wait_limit_ns(g4.DEFAULT_WAIT_LIMIT_NS)
    assert st == g4.G4_ERR_TIMEOUT, g4.status_string(st)
    assert g4.g4attn_status_sync() == g4.G4_OK   # read and cleared
    again, st = run()
    assert st == g4.G4_OK
    assert torch.equal(again.cpu().view(torch.int16), ref.cpu().view(torch.int16))
