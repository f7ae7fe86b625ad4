"""Pins of the oracle's rotary position embedding (CPU only).

The pages put no positional encoding inside the layer; rotary embedding is a
follow-on for real models (Qwen-family, rotate-half convention).  Pinned by a
hand-computed rotation, the identity at position 0, the relative-position
property, and layer-level cases where the rotation must not matter.
"""
import math

import numpy as np
import pytest

from diffusion_branch_speculative_gb300 import synth
from oracle import specfold_oracle as orc


def test_rope_hand_values():
    """hd = 4, theta = 100, position 1: frequencies 1 and 0.1; pairs (0, 2)
    and (1, 3) rotate by 1 and 0.1 radians."""
    x = np.array([1.0, 2.0, 3.0, 4.0])
    got = orc.rope(x, 1.0, 100.0)
    c1, s1, c2, s2 = math.cos(1.0), math.sin(1.0), math.cos(0.1), math.sin(0.1)
    want = [1 * c1 - 3 * s1, 2 * c2 - 4 * s2, 3 * c1 + 1 * s1, 4 * c2 + 2 * s2]
    np.testing.assert_allclose(got, want, rtol=1e-15, atol=1e-15)


def test_rope_position_zero_is_identity_and_norms_kept():
    rng = np.random.default_rng(0)
    x = rng.standard_normal((5, 3, 64))
    assert np.array_equal(orc.rope(x, 0.0, 10000.0), x)
    y = orc.rope(x, 123.0, 10000.0)
    np.testing.assert_allclose(np.linalg.norm(y, axis=-1), np.linalg.norm(x, axis=-1), rtol=1e-13)


def test_rope_scores_depend_on_relative_position_only():
    rng = np.random.default_rng(1)
    q, k = rng.standard_normal(128), rng.standard_normal(128)
    a = orc.rope(q, 40.0, 10000.0) @ orc.rope(k, 13.0, 10000.0)
    b = orc.rope(q, 40.0 + 977.0, 10000.0) @ orc.rope(k, 13.0 + 977.0, 10000.0)
    c = orc.rope(q, 27.0, 10000.0) @ orc.rope(k, 0.0, 10000.0)
    np.testing.assert_allclose([b, c], [a, a], rtol=1e-9)
    # and it does depend on the distance
    assert abs(orc.rope(q, 41.0, 10000.0) @ orc.rope(k, 13.0, 10000.0) - a) > 1e-6


def _small(P, L=6, levels=(1, 2, 1)):
    return synth.small_workload(d=64, n_q=4, n_kv=2, hd=16, F=96, P=P, L=L, levels=levels)


def test_rope_single_key_leaves_output_unchanged():
    """P = 0, L = 1: each row attends to its own key only, so the softmax
    weight is 1 and the output is v whatever the rotation: values are not
    rotated."""
    inp = synth.make_layer_inputs(_small(P=0, L=1, levels=(1, 1)), seed=3)
    d = inp.dims
    a = orc.layer_forward(inp.H, inp.parent, inp.weights, inp.prefix.K, inp.prefix.V, 0.05, d.eps, d.n_kv, d.hd)
    b = orc.layer_forward(inp.H, inp.parent, inp.weights, inp.prefix.K, inp.prefix.V, 0.05, d.eps, d.n_kv, d.hd,
                          rope_theta=10000.0)
    np.testing.assert_allclose(b["out"], a["out"], rtol=1e-12, atol=1e-12)


def test_rope_zero_queries_leave_output_unchanged():
    """W_q = 0 makes every score 0, so attention is a plain average whatever
    the rotation; rope touches only the scores."""
    inp = synth.make_layer_inputs(_small(P=8), seed=4)
    W = dict(inp.weights)
    W["w_q"] = np.zeros_like(W["w_q"])
    d = inp.dims
    a = orc.layer_forward(inp.H, inp.parent, W, inp.prefix.K, inp.prefix.V, 0.05, d.eps, d.n_kv, d.hd)
    b = orc.layer_forward(inp.H, inp.parent, W, inp.prefix.K, inp.prefix.V, 0.05, d.eps, d.n_kv, d.hd,
                          rope_theta=10000.0)
    np.testing.assert_allclose(b["out"], a["out"], rtol=1e-12, atol=1e-12)


def test_rope_changes_scores_when_it_should():
    inp = synth.make_layer_inputs(_small(P=8), seed=5)
    d = inp.dims
    a = orc.layer_forward(inp.H, inp.parent, inp.weights, inp.prefix.K, inp.prefix.V, 0.0, d.eps, d.n_kv, d.hd)
    b = orc.layer_forward(inp.H, inp.parent, inp.weights, inp.prefix.K, inp.prefix.V, 0.0, d.eps, d.n_kv, d.hd,
                          rope_theta=10000.0)
    assert np.max(np.abs(b["attnO"] - a["attnO"])) > 1e-6


@pytest.mark.parametrize("tau", [0.0, 0.05])
def test_rope_serialized_equals_packed(tau):
    inp = synth.make_layer_inputs(_small(P=8, L=8, levels=(1, 2, 2)), seed=6)
    d = inp.dims
    res = orc.layer_forward(inp.H, inp.parent, inp.weights, inp.prefix.K, inp.prefix.V, tau, d.eps, d.n_kv, d.hd,
                            rope_theta=500.0)
    ser = orc.layer_serialized(inp.H, inp.parent, inp.weights, inp.prefix.K, inp.prefix.V, tau, d.eps, d.n_kv,
                               d.hd, rope_theta=500.0)
    np.testing.assert_allclose(res["out"].reshape(ser.shape), ser, rtol=1e-11, atol=1e-11)
    if tau == 0.0:
        B = inp.H.shape[0]
        for b in range(B):
            dense = orc.dense_branch_forward(inp.H[b], inp.weights, inp.prefix.K, inp.prefix.V, d.eps, d.n_kv,
                                             d.hd, rope_theta=500.0)
            np.testing.assert_allclose(ser[b], dense, rtol=1e-11, atol=1e-11)


def test_rope_identical_children_equal_root():
    inp = synth.make_layer_inputs(_small(P=8, L=5, levels=(1, 2, 3)), seed=7, identical_children=True)
    d = inp.dims
    res = orc.layer_forward(inp.H, inp.parent, inp.weights, inp.prefix.K, inp.prefix.V, 0.05, d.eps, d.n_kv, d.hd,
                            rope_theta=10000.0)
    out = res["out"].reshape(inp.H.shape)
    assert np.array_equal(out[1:], np.broadcast_to(out[0], out[1:].shape))
