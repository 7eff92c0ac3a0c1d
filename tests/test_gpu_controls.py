"""Negative controls for the GPU parity check: the comparison the parity tests make (max-abs 2e-2,
mean-abs 2e-3 against the fp64 oracle) must tell the page's readings apart from plausible wrong ones.

The kernels are not touched. On the tiny oracle case (two causal sequences of 96 and 200 tokens,
N(0,1) inputs, seed 0; window 64 on the sliding layer) the library's output is compared once with the
oracle as written, which must pass, and then with the oracle carrying one planted mistake at a time,
each of which must fail the same bars. The mistakes are planted in the oracle, on the CPU:
  - the sliding layer's RoPE family (all pairs turn, theta 1e4) on the global layer;
  - V := p-RoPE(S) on the K==V layer, instead of the stored, un-rotated S;
  - the window one key wider or one key narrower;
  - interleaved pairs (2t, 2t+1) instead of half-split pairs (t, t + D/2).
"""
import dataclasses

import numpy as np
import pytest

import oracle
import oracle.core as oc

from gpu_cases import TOL_MAX, TOL_MEAN, Batch, errors, f64, layers

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def outputs():
    """The library's output of the tiny case, per layer kind: (batch, oracle layer, rows as fp64)."""
    res = {}
    for kind, window in (("sliding", 64), ("global", 0)):
        layer, olayer = layers(kind, window or 1024)
        bt = Batch(kind, [96, 200], seed=0)
        out, _ = bt.run(layer)
        res[kind] = (bt, olayer, f64(out))
    return res


def passes(bt, olayer, got) -> bool:
    """True when every sequence of the batch meets both bars against the (possibly planted) oracle."""
    for b, L in enumerate(bt.q_lens):
        s = bt.layout.q_start[b]
        mx, mean = errors(got[s:s + L], bt.oracle_rows(olayer, b))
        if not (mx <= TOL_MAX and mean <= TOL_MEAN):
            return False
    return True


def interleaved_rope(x, pos, theta, partial):
    x = np.asarray(x, np.float64)
    D = x.shape[-1]
    R = oc.rope_rotated_pairs(D, partial)
    ang = np.asarray(pos, np.float64)[..., None] * oc.rope_inv_freq(D, theta)[:R]
    y = x.copy()
    a, b = x[..., 0:2 * R:2], x[..., 1:2 * R:2]
    y[..., 0:2 * R:2] = a * np.cos(ang) - b * np.sin(ang)
    y[..., 1:2 * R:2] = b * np.cos(ang) + a * np.sin(ang)
    return y


@pytest.mark.parametrize("kind", ["sliding", "global"])
def test_the_oracle_as_written_passes(outputs, kind):
    bt, olayer, got = outputs[kind]
    assert passes(bt, olayer, got)


def test_sliding_rope_family_on_the_global_layer_fails(outputs):
    bt, olayer, got = outputs["global"]
    wrong = dataclasses.replace(olayer, rope_theta=oracle.SLIDING.rope_theta, rope_partial=1.0)
    assert not passes(bt, wrong, got)


def test_values_taken_as_the_rotated_keys_fail(outputs, monkeypatch):
    bt, olayer, got = outputs["global"]
    good = oc.keys_values

    def rotated_v(layer, k_hist, v_hist, pos_offset=0, norms=None):
        k_rot, v = good(layer, k_hist, v_hist, pos_offset, norms)
        return k_rot, (k_rot.copy() if layer.kv_shared else v)
    monkeypatch.setattr(oc, "keys_values", rotated_v)
    assert not passes(bt, olayer, got)


@pytest.mark.parametrize("delta", [-1, 1])
def test_window_off_by_one_fails(outputs, delta):
    bt, olayer, got = outputs["sliding"]
    assert not passes(bt, oracle.with_window(oracle.SLIDING, olayer.window + delta), got)


@pytest.mark.parametrize("kind", ["sliding", "global"])
def test_interleaved_pairs_fail(outputs, kind, monkeypatch):
    bt, olayer, got = outputs[kind]
    monkeypatch.setattr(oc, "rope", interleaved_rope)
    assert not passes(bt, olayer, got)
