"""g4attn_decode_static (the decode step on the library's static scratch, for callers that
cannot allocate device memory) against g4attn_decode with a caller workspace.

Two static calls in a row per layer kind, the first with the larger batch, so that whatever
the first call leaves in the shared scratch is still there when the second runs. Both entry
points run the same deterministic kernels on the same inputs, so each output must equal the
workspace entry point's bit for bit (a partly stale read of the shared scratch would show), and
it must also be finite. The file is named so that it is collected last; it passes alone in a
fresh process as well.
"""
import numpy as np
import pytest
import torch

import invariant_hybrid_attention_gb300 as g4
from invariant_hybrid_attention_gb300.paged import device_int32

from gpu_cases import DecodeBatch, f64, layers

pytestmark = pytest.mark.gpu

CALLS = {
    "sliding": [([3000, 1, 700, 1025, 4097, 256, 90], 31), ([5, 1500], 32)],
    "global": [([5000, 17, 1024, 2049, 300], 41), ([1, 1030], 42)],
}


def static_decode(db: DecodeBatch, layer, cache):
    B = len(db.ctx_lens)
    k_new = torch.stack([h[L - 1] for h, L in zip(db.hist_k, db.ctx_lens)]).cuda()
    v_new = None if db.kind == "global" else torch.stack(
        [h[L - 1] for h, L in zip(db.hist_v, db.ctx_lens)]).cuda()
    q = db.q.cuda()
    out = torch.full_like(q, float("nan"))
    assert out.shape[0] == B
    g4.g4attn_decode_static(layer, q, k_new, v_new, device_int32(db.ctx_lens), cache.desc, db.plan.table.cuda(), out)
    torch.cuda.synchronize()
    st = g4.g4attn_status_sync()
    assert st == g4.G4_OK, g4.status_string(st)
    return out


@pytest.mark.parametrize("kind", ["sliding", "global"])
def test_decode_static_matches_decode_on_two_calls_in_a_row(kind):
    layer, _ = layers(kind)
    for call, (lens, seed) in enumerate(CALLS[kind]):
        db = DecodeBatch(kind, lens, seed=seed)
        need = g4.g4attn_decode_workspace_bytes(layer, len(lens), db.plan.max_pages)
        assert 0 < need <= g4.DECODE_STATIC_SCRATCH_BYTES
        want, cache = db.run(layer)              # the workspace entry point (it also fills the cache)
        got = static_decode(db, layer, cache)    # re-appends the same token at the same slot
        assert np.isfinite(f64(got)).all(), f"call {call}: non-finite output"
        assert torch.equal(got, want), f"call {call}: the static-scratch decode differs from g4attn_decode"
