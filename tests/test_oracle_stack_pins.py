"""Pins of the oracle's stack of folded layers (CPU only).

The stack is a composition of the pinned single layer, so what needs pinning
is the composition itself: each layer reads the previous layer's output,
uses its own weights and prefix, and runs the gate again on its own input
(the "automatic release" of a fold, SpecFold explainer page, "mechanism"
paragraph).  The pins are a hand-built layer with a closed form, the dense
case against torch library routines, and exact invariants.
"""
import math

import numpy as np
import pytest
import torch
import torch.nn.functional as Fn

from diffusion_branch_speculative_gb300 import synth
from oracle import specfold_oracle as orc


def _scaling_layer(d: int, n_heads: int, c: float, F: int = 4) -> dict:
    """A layer whose output is h * (1 - c / rms(h)) for a one-token block
    with no prefix: with one key the softmax weight is 1, so attention returns
    v = rmsnorm(h) (W_v = I, MHA); W_o = -c I adds -c h / rms(h); W_down = 0
    turns the FFN off."""
    I = np.eye(d)
    return {
        "g1": np.ones(d), "w_q": np.zeros((d, d)), "w_k": np.zeros((d, d)), "w_v": I,
        "w_o": -c * I, "g2": np.ones(d),
        "w_gate": np.zeros((F, d)), "w_up": np.zeros((F, d)), "w_down": np.zeros((d, F)),
    }


def test_stack_release_closed_form():
    """A child row folds at layer 0 (r = 0.05 < tau = 0.1); layer 0 shrinks
    the parent row to a quarter, so at layer 1 the same difference is
    r = 0.2 > tau and the row is recomputed.  Every output is hand-computed."""
    d, nh = 8, 2
    hd = d // nh
    h = np.full(d, 2.0)                          # rms(h) = 2
    delta = 0.1 * np.array([1.0, -1.0] * (d // 2))  # orthogonal to h, |delta| / |h| = 0.05
    H = np.stack([h, h + delta])[:, None, :]     # B = 2, L = 1
    parent = np.array([-1, 0], np.int32)
    empty = np.zeros((0, nh, hd))
    c0, c1 = 1.5, 0.1
    layers = [(_scaling_layer(d, nh, c0), empty, empty), (_scaling_layer(d, nh, c1), empty, empty)]
    res = orc.stack_forward(H, parent, layers, 0.1, 0.0, nh, hd)
    assert res["fold"][0].tolist() == [[False], [True]]
    assert res["fold"][1].tolist() == [[False], [False]]
    assert res["n"] == [1, 2]
    np.testing.assert_allclose(res["rel"][0][1, 0], 0.05, rtol=1e-14)
    np.testing.assert_allclose(res["rel"][1][1, 0], 0.2, rtol=1e-14)
    # layer 0: root h -> h (1 - 1.5 / 2) = h / 4; the folded child keeps its delta
    np.testing.assert_allclose(res["inputs"][1][0, 0], h / 4, rtol=1e-15)
    np.testing.assert_allclose(res["inputs"][1][1, 0], h / 4 + delta, rtol=1e-15)
    # layer 1: both recomputed; rms(h/4) = 0.5, rms(h/4 + delta) = sqrt(0.26)
    x = h / 4 + delta
    np.testing.assert_allclose(res["out"][0, 0], (h / 4) * (1 - c1 / 0.5), rtol=1e-14)
    np.testing.assert_allclose(res["out"][1, 0], x * (1 - c1 / math.sqrt(0.26)), rtol=1e-14)


def test_stack_store_rounds_between_layers():
    """``store`` is applied to every layer's output before the next layer."""
    d, nh = 8, 2
    H = np.full((1, 1, d), 3.0)
    empty = np.zeros((0, nh, d // nh))
    layers = [(_scaling_layer(d, nh, 1.0), empty, empty)] * 2
    seen = []

    def store(x):
        seen.append(x.copy())
        return np.round(x, 1)

    res = orc.stack_forward(H, np.array([-1], np.int32), layers, 0.0, 0.0, nh, d // nh, store=store)
    # 3 -> 3 (1 - 1/3) = 2 -> stored 2.0 -> 2 (1 - 1/2) = 1
    np.testing.assert_allclose(seen[0], 2.0, rtol=1e-15)
    np.testing.assert_allclose(res["inputs"][1], 2.0, rtol=0)
    np.testing.assert_allclose(res["out"], 1.0, rtol=0)


def _torch_dense(Hb, W, eps, n_kv, hd):
    """Textbook pre-norm layer (no prefix) from torch library routines, fp64."""
    t = lambda a: torch.as_tensor(np.asarray(a, np.float64))
    h = t(Hb)
    L, d = h.shape
    x = Fn.rms_norm(h, (d,), weight=t(W["g1"]), eps=eps)
    q = Fn.linear(x, t(W["w_q"])).reshape(L, -1, hd).transpose(0, 1)
    k = Fn.linear(x, t(W["w_k"])).reshape(L, n_kv, hd).transpose(0, 1)
    v = Fn.linear(x, t(W["w_v"])).reshape(L, n_kv, hd).transpose(0, 1)
    o = Fn.scaled_dot_product_attention(q[None], k[None], v[None], enable_gqa=True)[0]
    a = h + Fn.linear(o.transpose(0, 1).reshape(L, -1), t(W["w_o"]))
    x2 = Fn.rms_norm(a, (d,), weight=t(W["g2"]), eps=eps)
    gg = Fn.silu(Fn.linear(x2, t(W["w_gate"]))) * Fn.linear(x2, t(W["w_up"]))
    return (a + Fn.linear(gg, t(W["w_down"]))).numpy()


def test_stack_tau_zero_is_dense_stack_torch():
    """tau = 0 folds nothing at any layer, so each branch runs the plain
    pre-norm stack; with no prefix that stack is torch's library layer
    applied once per layer, with that layer's weights."""
    w = synth.small_workload(d=64, n_q=4, n_kv=2, hd=16, F=96, P=0, L=6, levels=(1, 2, 1))
    st = synth.make_stack_inputs(w, seed=5, n_layers=3)
    d = st.dims
    layers = [(st.weights[l], st.prefixes[l].K, st.prefixes[l].V) for l in range(3)]
    res = orc.stack_forward(st.H, st.parent, layers, 0.0, d.eps, d.n_kv, d.hd)
    assert res["n"] == [st.H.shape[0] * st.H.shape[1]] * 3
    for b in range(st.H.shape[0]):
        x = st.H[b]
        for l in range(3):
            x = _torch_dense(x, st.weights[l], d.eps, d.n_kv, d.hd)
        np.testing.assert_allclose(res["out"][b], x, rtol=1e-10, atol=1e-10)


def test_stack_identical_children_equal_root_at_every_layer():
    """Children identical to their parents with tau > 0 fold at every layer
    (their difference stays exactly zero), so every child equals the root."""
    w = synth.small_workload(d=64, n_q=4, n_kv=2, hd=16, F=96, P=8, L=5, levels=(1, 2, 3))
    st = synth.make_stack_inputs(w, seed=2, n_layers=3, identical_children=True)
    d = st.dims
    layers = [(st.weights[l], st.prefixes[l].K, st.prefixes[l].V) for l in range(3)]
    res = orc.stack_forward(st.H, st.parent, layers, 0.05, d.eps, d.n_kv, d.hd)
    B, L, _ = st.H.shape
    for l in range(3):
        assert res["fold"][l][1:].all() and not res["fold"][l][0].any()
        assert res["n"][l] == L
        X = res["inputs"][l]
        assert np.array_equal(X[1:], np.broadcast_to(X[0], X[1:].shape))
    assert np.array_equal(res["out"][1:], np.broadcast_to(res["out"][0], res["out"][1:].shape))


def test_stack_gate_reads_each_layer_input():
    """Layer l's decisions are the closed-form gate (brute force, fsum) on
    layer l's own input, and that input is layer l-1's output."""
    w = synth.small_workload(d=64, n_q=4, n_kv=2, hd=16, F=96, P=8, L=8, levels=(1, 2, 2))
    st = synth.make_stack_inputs(w, seed=7, n_layers=3)
    d = st.dims
    tau = 0.05
    layers = [(st.weights[l], st.prefixes[l].K, st.prefixes[l].V) for l in range(3)]
    res = orc.stack_forward(st.H, st.parent, layers, tau, d.eps, d.n_kv, d.hd)
    B, L, _ = st.H.shape
    for l in range(3):
        X = res["inputs"][l]
        for b in range(1, B):
            p = int(st.parent[b])
            for i in range(L):
                num = math.fsum((X[b, i] - X[p, i]) ** 2)
                den = math.fsum(X[p, i] ** 2)
                assert res["fold"][l][b, i] == (num < tau * tau * den)
        assert res["n"][l] == int((~res["fold"][l]).sum())
        nxt = orc.layer_forward(X, st.parent, st.weights[l], st.prefixes[l].K, st.prefixes[l].V, tau,
                                d.eps, d.n_kv, d.hd)["out"].reshape(X.shape)
        ref = res["inputs"][l + 1] if l + 1 < 3 else res["out"]
        np.testing.assert_array_equal(nxt, ref)
