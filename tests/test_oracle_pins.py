"""Pins of the CPU oracle to things other than itself (CPU only).

Each test ties one part of the oracle to a closed form, a library routine, an
invariant the SpecFold pages fix, or brute force on tiny inputs, chosen so that
a dropped term, a wrong sign or index, or a transposed operand fails one of
them.
"""
import math

import numpy as np
import pytest
import torch
import torch.nn.functional as Fn

from oracle import specfold_oracle as orc
from diffusion_branch_speculative_gb300 import synth


def _tiny(seed=0, **kw):
    return synth.make_layer_inputs("tiny", seed=seed, **kw)


def _run(inp, tau, **kw):
    d = inp.dims
    return orc.layer_forward(inp.H, inp.parent, inp.weights, inp.prefix.K, inp.prefix.V,
                             tau, d.eps, d.n_kv, d.hd, **kw)


# ---------------------------------------------------------------- gate ------

def test_gate_hand_values():
    """Closed-form relative differences on 2-d rows (|p| = 5)."""
    p = [3.0, 4.0]
    rows = [
        ([3.0, 4.5], 0.1),            # |delta| = 0.5
        ([4.5, 6.0], 0.5),            # delta = 0.5 p exactly
        ([3.0, 4.0], 0.0),            # identical
        ([-3.0, -4.0], 2.0),          # sign flip: |delta| = 10
        ([3.0, 9.0], 1.0),            # |delta| = 5
    ]
    H = np.array([[p] * len(rows), [c for c, _ in rows]], dtype=np.float64)
    parent = np.array([-1, 0])
    for tau in (0.05, 0.2, 0.5, 1.5):
        fold, rel = orc.gate(H, parent, tau)
        assert not fold[0].any()
        assert np.all(rel[0] == -1.0)
        for i, (_, r) in enumerate(rows):
            assert rel[1, i] == pytest.approx(r, abs=1e-15)
            # delta = 0.5 p with tau = 0.5 is an exact tie: ties recompute
            expect = (r < tau) or (r == 0.0 and tau > 0)
            assert bool(fold[1, i]) == expect, (i, tau)


def test_gate_zero_parent_and_tau_zero():
    H = np.zeros((2, 3, 4))
    H[1, 1] = 1e-30           # parent row is zero, child not
    parent = np.array([-1, 0])
    fold, rel = orc.gate(H, parent, 0.1)
    assert fold[1, 0] and fold[1, 2] and not fold[1, 1]
    assert rel[1, 0] == 0.0 and rel[1, 1] == np.inf
    fold0, _ = orc.gate(H, parent, 0.0)
    assert not fold0.any()
    foldinf, _ = orc.gate(np.random.default_rng(1).standard_normal((3, 4, 8)), np.array([-1, 0, 1]), np.inf)
    assert foldinf[1:].all() and not foldinf[0].any()


def test_gate_brute_force_norm_ratio():
    """Decisions and r against numpy's 2-norm ratio, away from ties."""
    rng = np.random.default_rng(3)
    B, L, d = 6, 12, 40
    H = rng.standard_normal((B, L, d))
    parent = np.array([-1, 0, 0, 1, 2, 3])
    for b in range(1, B):
        H[b] = H[parent[b]] + rng.uniform(0, 0.3, (L, 1)) * rng.standard_normal((L, d)) / math.sqrt(d)
    tau = 0.1
    fold, rel = orc.gate(H, parent, tau)
    for b in range(1, B):
        for i in range(L):
            r = np.linalg.norm(H[b, i] - H[parent[b], i]) / np.linalg.norm(H[parent[b], i])
            assert rel[b, i] == pytest.approx(r, rel=1e-12)
            if abs(r - tau) > 1e-9:
                assert bool(fold[b, i]) == (r < tau)


def test_gate_force_override():
    inp = _tiny()
    fold, _ = orc.gate(inp.H, inp.parent, 0.05)
    force = np.full(fold.shape, -1, np.int8)
    force[2, 3] = 1 - int(fold[2, 3])
    f2, _ = orc.gate(inp.H, inp.parent, 0.05, force)
    assert f2[2, 3] != fold[2, 3]
    assert (f2 != fold).sum() == 1
    bad = np.full(fold.shape, -1, np.int8)
    bad[0, 0] = 1
    with pytest.raises(ValueError):
        orc.gate(inp.H, inp.parent, 0.05, bad)


# ------------------------------------------------------- resolve / pack ------

def _random_fold(rng, B, L, p_fold):
    fold = rng.random((B, L)) < p_fold
    fold[0] = False
    return fold


def test_resolve_matches_chain_walk_and_is_nearest_active_ancestor():
    rng = np.random.default_rng(5)
    for trial in range(20):
        levels = [1] + list(rng.integers(1, 4, size=rng.integers(1, 5)))
        g = synth.make_graph(levels, rng)
        B, L = len(g.parent), int(rng.integers(1, 9))
        fold = _random_fold(rng, B, L, 0.6)
        src = orc.resolve(fold, g.parent)
        for b in range(B):
            for i in range(L):
                r = b * L + i
                s = int(src[r])
                assert s == orc.walk_chain(fold, g.parent, b, i)
                sb, si = divmod(s, L)
                assert si == i and not fold[sb, si]
                # s is an ancestor-or-self, and every row strictly between is folded
                c = b
                while c != sb:
                    assert fold[c, i]
                    c = int(g.parent[c])
                    assert c >= 0


def test_pack_is_stream_compaction():
    rng = np.random.default_rng(7)
    for p in (0.0, 0.3, 0.9, 1.0):
        fold = _random_fold(rng, 9, 7, p)
        idx, slot, n = orc.pack(fold)
        flat = fold.reshape(-1)
        assert n == int((~flat).sum())
        assert np.all(np.diff(idx) > 0)
        assert np.all(~flat[idx])
        assert np.all(slot[idx] == np.arange(n))
        assert np.all(slot[flat] == -1)


# --------------------------------------------------- dense layer vs torch ----

def _torch_dense(Hb, W, pk, pv, eps, n_kv, hd):
    """Textbook pre-norm layer assembled from torch library routines (fp64)."""
    t = lambda a: torch.as_tensor(np.asarray(a, np.float64))
    h = t(Hb)
    L, d = h.shape
    x = Fn.rms_norm(h, (d,), weight=t(W["g1"]), eps=eps)
    q = Fn.linear(x, t(W["w_q"])).reshape(L, -1, hd).transpose(0, 1)
    k = Fn.linear(x, t(W["w_k"])).reshape(L, n_kv, hd)
    v = Fn.linear(x, t(W["w_v"])).reshape(L, n_kv, hd)
    K = torch.cat([t(pk), k], 0).transpose(0, 1)
    V = torch.cat([t(pv), v], 0).transpose(0, 1)
    o = Fn.scaled_dot_product_attention(q[None], K[None], V[None], enable_gqa=True)[0]
    a = h + Fn.linear(o.transpose(0, 1).reshape(L, -1), t(W["w_o"]))
    x2 = Fn.rms_norm(a, (d,), weight=t(W["g2"]), eps=eps)
    gg = Fn.silu(Fn.linear(x2, t(W["w_gate"]))) * Fn.linear(x2, t(W["w_up"]))
    return (a + Fn.linear(gg, t(W["w_down"]))).numpy()


@pytest.mark.parametrize("n_q,n_kv", [(4, 2), (4, 4), (6, 1)])
def test_dense_forward_matches_torch_library(n_q, n_kv):
    w = synth.small_workload(d=64, n_q=n_q, n_kv=n_kv, hd=16, F=96, P=24, L=8, levels=(1, 1))
    inp = synth.make_layer_inputs(w, seed=11)
    W = dict(inp.weights)
    rng = np.random.default_rng(2)
    W["g1"] = rng.uniform(0.5, 1.5, 64)     # non-unit gains so a dropped gain fails
    W["g2"] = rng.uniform(0.5, 1.5, 64)
    d = inp.dims
    ours = orc.dense_branch_forward(inp.H[0], W, inp.prefix.K, inp.prefix.V, d.eps, n_kv, d.hd)
    ref = _torch_dense(inp.H[0], W, inp.prefix.K, inp.prefix.V, d.eps, n_kv, d.hd)
    np.testing.assert_allclose(ours, ref, rtol=1e-10, atol=1e-10)


def test_attention_single_key_returns_value():
    """L = 1, P = 0: softmax over one key is 1, so the output is v."""
    rng = np.random.default_rng(4)
    q = rng.standard_normal((1, 4, 8))
    K = {0: rng.standard_normal((2, 8))}
    V = {0: rng.standard_normal((2, 8))}
    o = orc.attention_rows(q, np.array([0]), {0: [0]}, K, V, np.zeros((0, 2, 8)), np.zeros((0, 2, 8)), 2)
    np.testing.assert_allclose(o.reshape(4, 8), V[0][[0, 0, 1, 1]], rtol=0, atol=1e-15)


def test_silu_and_rmsnorm_closed_forms():
    assert orc.silu(np.array(0.0)) == 0.0
    assert orc.silu(np.array(1.0)) == pytest.approx(1.0 / (1.0 + math.exp(-1.0)))
    assert orc.silu(np.array(-1000.0)) == pytest.approx(0.0, abs=1e-300)
    x = np.array([3.0, 4.0])
    # mean(x^2) = 12.5
    np.testing.assert_allclose(orc.rmsnorm(x, np.ones(2), 0.0), x / math.sqrt(12.5), rtol=1e-15)
    np.testing.assert_allclose(orc.rmsnorm(x, np.array([2.0, 0.5]), 0.5), x * [2.0, 0.5] / math.sqrt(13.0),
                               rtol=1e-15)


# ------------------------------------------------------- layer invariants ----

@pytest.mark.parametrize("seed", [0, 1])
def test_I1_tau_zero_is_dense(seed):
    inp = _tiny(seed)
    d = inp.dims
    res = _run(inp, 0.0)
    assert res["n"] == inp.H.shape[0] * inp.H.shape[1]
    B, L, D = inp.H.shape
    out = res["out"].reshape(B, L, D)
    for b in range(B):
        dense = orc.dense_branch_forward(inp.H[b], inp.weights, inp.prefix.K, inp.prefix.V, d.eps, d.n_kv, d.hd)
        np.testing.assert_allclose(out[b], dense, rtol=1e-11, atol=1e-11)


def test_I2_identical_children_equal_root_exactly():
    inp = _tiny(2, identical_children=True)
    for tau in (np.inf, 1e6, 1e-3):
        res = _run(inp, tau)
        B, L, D = inp.H.shape
        out = res["out"].reshape(B, L, D)
        assert res["n"] == L
        for b in range(1, B):
            assert np.array_equal(out[b], out[0])


def test_I3_recomputed_rows_equal_dense_recompute():
    """Children differ from their parent only at revealed positions: each
    recomputed row equals a dense recompute of its own branch."""
    inp = _tiny(4, ripple=False, noise=False)
    d = inp.dims
    res = _run(inp, 0.05)
    B, L, D = inp.H.shape
    out = res["out"].reshape(B, L, D)
    fold = res["fold"]
    for b in range(1, B):
        rev = inp.branches.new_reveals[b]
        assert sorted(np.nonzero(~fold[b])[0].tolist()) == rev
        dense = orc.dense_branch_forward(inp.H[b], inp.weights, inp.prefix.K, inp.prefix.V, d.eps, d.n_kv, d.hd)
        for i in rev:
            np.testing.assert_allclose(out[b, i], dense[i], rtol=1e-11, atol=1e-11)


@pytest.mark.parametrize("seed,tau", [(0, 0.05), (1, 0.02), (5, 0.1), (6, 0.3)])
def test_I4_serialized_equals_packed(seed, tau):
    inp = _tiny(seed)
    d = inp.dims
    res = _run(inp, tau)
    ser = orc.layer_serialized(inp.H, inp.parent, inp.weights, inp.prefix.K, inp.prefix.V, tau, d.eps,
                               d.n_kv, d.hd)
    np.testing.assert_allclose(res["out"], ser.reshape(res["out"].shape), rtol=1e-11, atol=1e-11)


def test_I4_serialized_equals_packed_branchy_graph():
    w = synth.small_workload(d=64, n_q=4, n_kv=2, hd=16, F=96, P=16, L=8, levels=(1, 3, 4),
                             reveals=(1, 2), second_parent=True)
    inp = synth.make_layer_inputs(w, seed=9)
    d = inp.dims
    res = _run(inp, 0.05)
    assert 0 < res["n"] < inp.H.shape[0] * inp.H.shape[1]
    ser = orc.layer_serialized(inp.H, inp.parent, inp.weights, inp.prefix.K, inp.prefix.V, 0.05, d.eps,
                               d.n_kv, d.hd)
    np.testing.assert_allclose(res["out"], ser.reshape(res["out"].shape), rtol=1e-11, atol=1e-11)


def test_I6_folded_rows_keep_their_residual():
    inp = _tiny(0)
    res = _run(inp, 0.05)
    B, L, D = inp.H.shape
    H = inp.H.reshape(B * L, D).astype(np.float64)
    out = res["out"]
    src = res["src"]
    folded = np.nonzero(src != np.arange(B * L))[0]
    assert len(folded) > 0
    for r in folded:
        s = src[r]
        np.testing.assert_allclose(out[r] - H[r], out[s] - H[s], rtol=0, atol=1e-12)


def test_row_subset_matches_full():
    inp = _tiny(1)
    d = inp.dims
    full = _run(inp, 0.05)
    rows = [0, 17, 20, 33, 63]
    sub = _run(inp, 0.05, rows=rows)
    # BLAS blocks differently for a different row count: equal to round-off
    np.testing.assert_allclose(sub["out"], full["out"][rows], rtol=1e-12, atol=1e-12)


def test_tiny_expected_fold_structure():
    """tau = 0.05 with ripple 0.3 exp(-d/2): a child recomputes exactly the
    positions within distance 3 of its new reveal (0.3 e^{-3/2} = 0.067 >
    0.05 > 0.3 e^{-2} = 0.041), clipped to the block."""
    inp = _tiny(0)
    res = _run(inp, 0.05)
    fold = res["fold"]
    L = inp.H.shape[1]
    for b in range(1, inp.H.shape[0]):
        (rv,) = inp.branches.new_reveals[b]
        expect = [i for i in range(L) if abs(i - rv) <= 3]
        assert sorted(np.nonzero(~fold[b])[0].tolist()) == expect


def test_near_tau_rows():
    rel = np.array([[-1.0, -1.0], [0.05, 0.0500049]])
    m = orc.near_tau_rows(rel, 0.05)
    assert m.tolist() == [[False, False], [True, True]]
    m2 = orc.near_tau_rows(np.array([[-1.0], [0.0500051]]), 0.05)
    assert not m2.any()


def test_golden_regression_fixture():
    import json, os
    from tests.golden.make_golden import summary
    path = os.path.join(os.path.dirname(__file__), "golden", "tiny_oracle_seed0.json")
    with open(path) as f:
        want = json.load(f)
    got = summary(want["seed"], want["tau"])
    for k in ("parent", "fold", "src", "packed_idx", "n"):
        assert got[k] == want[k], k
    np.testing.assert_allclose(got["out_row_sums"], want["out_row_sums"], rtol=1e-9, atol=1e-9)
    np.testing.assert_allclose(got["out_first8_row0"], want["out_first8_row0"], rtol=1e-9, atol=1e-12)
