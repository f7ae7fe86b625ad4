"""Pins of the variant gate that compares a child with the row its parent's
output comes from (CPU only).

The explainer measures the child against its parent; a chain of folds can
then reuse an output whose input drifted further than tau.  The variant
compares with the computed source instead.  Pinned by a hand-built chain,
its equality with the parent gate where every parent is computed, and the
drift bound it guarantees.
"""
import math

import numpy as np
import pytest

from diffusion_branch_speculative_gb300 import synth
from oracle import specfold_oracle as orc


def test_gate_source_hand_chain():
    """root [1, 0] -> b1 [1, 0.08] -> b2 [1, 0.16], tau = 0.1: b1 folds onto
    the root (r = 0.08).  Against its parent b2 would fold too (r = 0.08 /
    |b1|), against the root it must not (r = 0.16)."""
    H = np.array([[[1.0, 0.0]], [[1.0, 0.08]], [[1.0, 0.16]]])
    parent = np.array([-1, 0, 1], np.int32)
    f_par, r_par = orc.gate(H, parent, 0.1)
    f_src, r_src = orc.gate_source(H, parent, 0.1)
    assert f_par[1:, 0].tolist() == [True, True]
    assert f_src[1:, 0].tolist() == [True, False]
    np.testing.assert_allclose(r_src[2, 0], 0.16, rtol=1e-15)
    np.testing.assert_allclose(r_par[2, 0], 0.08 / math.sqrt(1.0064), rtol=1e-15)
    # and the resolved sources: b2 is its own source under the variant
    assert orc.resolve(f_src, parent).tolist() == [0, 0, 2]


def test_gate_source_equals_parent_gate_on_a_star():
    """Every non-root node hangs off the root, which is always computed, so
    the computed source of each parent row is the parent itself."""
    w = synth.small_workload(d=32, n_q=2, n_kv=1, hd=16, F=64, P=0, L=12, levels=(1, 6))
    inp = synth.make_layer_inputs(w, seed=3)
    a = orc.gate(inp.H, inp.parent, 0.05)
    b = orc.gate_source(inp.H, inp.parent, 0.05)
    assert np.array_equal(a[0], b[0])
    np.testing.assert_array_equal(a[1], b[1])


@pytest.mark.parametrize("seed", [0, 1, 2])
def test_gate_source_bounds_the_drift(seed):
    """Every folded row's input is within tau of its resolved source's
    input (checked with numpy norms on the final src)."""
    w = synth.small_workload(d=48, n_q=2, n_kv=1, hd=16, F=64, P=0, L=16, levels=(1, 2, 3, 3, 2))
    inp = synth.make_layer_inputs(w, seed=seed)
    tau = 0.1
    fold, _ = orc.gate_source(inp.H, inp.parent, tau)
    src = orc.resolve(fold, inp.parent)
    B, L, d = inp.H.shape
    H2 = inp.H.reshape(B * L, d).astype(np.float64)
    for r in np.nonzero(fold.reshape(-1))[0]:
        s = src[r]
        assert np.linalg.norm(H2[r] - H2[s]) < tau * np.linalg.norm(H2[s])


def test_gate_source_force_feeds_later_sources():
    """Forcing b1 to recompute makes b2 compare against b1 itself."""
    H = np.array([[[1.0, 0.0]], [[1.0, 0.08]], [[1.0, 0.16]]])
    parent = np.array([-1, 0, 1], np.int32)
    force = np.array([[-1], [0], [-1]], np.int8)
    f, r = orc.gate_source(H, parent, 0.1, force)
    assert f[1:, 0].tolist() == [False, True]
    np.testing.assert_allclose(r[2, 0], 0.08 / math.sqrt(1.0064), rtol=1e-15)


@pytest.mark.parametrize("tau", [0.02, 0.1])
def test_gate_source_serialized_equals_packed(tau):
    w = synth.small_workload(d=64, n_q=4, n_kv=2, hd=16, F=96, P=8, L=8, levels=(1, 2, 2, 1))
    inp = synth.make_layer_inputs(w, seed=9)
    d = inp.dims
    res = orc.layer_forward(inp.H, inp.parent, inp.weights, inp.prefix.K, inp.prefix.V, tau, d.eps, d.n_kv, d.hd,
                            gate_ref="source")
    ser = orc.layer_serialized(inp.H, inp.parent, inp.weights, inp.prefix.K, inp.prefix.V, tau, d.eps, d.n_kv,
                               d.hd, gate_ref="source")
    np.testing.assert_allclose(res["out"].reshape(ser.shape), ser, rtol=1e-11, atol=1e-11)
