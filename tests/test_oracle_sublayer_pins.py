"""Pins of the oracle's two variant readings (CPU only): the literal
attention correction for folded rows ("attn_rematch": a folded position's
attention output is matched again against its branch's own keys and values,
SpecFold explainer page, implementation note) and one gate per sublayer
("ffn_gate").  Pinned by hand-built layers with closed forms, by torch
library routines row by row, and by the invariants that define the folded
rows.
"""
import math

import numpy as np
import pytest
import torch
import torch.nn.functional as Fn

from diffusion_branch_speculative_gb300 import synth
from oracle import specfold_oracle as orc


def _t(a):
    return torch.as_tensor(np.asarray(a, np.float64))


def _run(inp, tau, **kw):
    d = inp.dims
    return orc.layer_forward_sublayers(inp.H, inp.parent, inp.weights, inp.prefix.K, inp.prefix.V, tau,
                                       d.eps, d.n_kv, d.hd, **kw)


def _chain_src(fold, parent, b, i):
    """Walk the fold chain of (b, i) up through first parents (test's own)."""
    while fold[b, i]:
        b = int(parent[b])
    return b


def _ffn_torch(A, W, eps):
    """out = A + down(silu(gate(x2)) * up(x2)), x2 = rmsnorm(A): torch routines."""
    a = _t(A)
    x2 = Fn.rms_norm(a, (a.shape[-1],), weight=_t(W["g2"]), eps=eps)
    gg = Fn.silu(Fn.linear(x2, _t(W["w_gate"]))) * Fn.linear(x2, _t(W["w_up"]))
    return (a + Fn.linear(gg, _t(W["w_down"]))).numpy()


def _layer(d, w_o, F=4, w_gate=None, w_up=None, w_down=None):
    """Hand-built layer: zero queries and keys (uniform attention), W_v = I
    (MHA, so the attention output is the mean of the keys' normalised rows),
    unit gains, the given W_o and FFN (off by default)."""
    I = np.eye(d)
    return {
        "g1": np.ones(d), "w_q": np.zeros((d, d)), "w_k": np.zeros((d, d)), "w_v": I, "w_o": w_o,
        "g2": np.ones(d),
        "w_gate": np.zeros((F, d)) if w_gate is None else w_gate,
        "w_up": np.zeros((F, d)) if w_up is None else w_up,
        "w_down": np.zeros((d, F)) if w_down is None else w_down,
    }


def _unit(h):
    return h / math.sqrt(float(np.mean(h * h)))


# ------------------------------------------------------------ closed forms --

def test_rematch_closed_form_ripple():
    """B = 2, L = 2, no prefix.  Row (1, 0) equals its parent row and folds;
    row (1, 1) is far from (0, 1) and is recomputed.  With uniform attention
    and W_v = I the attention output of a row of branch b is the mean of its
    block's normalised source rows.  The base reading copies the root's output
    to (1, 0); the literal correction lets (1, 0) see branch 1's own block,
    so the recomputed (1, 1) reaches it."""
    d, nh, c = 8, 2, 0.75
    h00 = np.full(d, 2.0)
    h01 = 3.0 * np.array([1.0, -1.0] * 4)
    h11 = np.array([0.0, 4.0] * 4)
    H = np.stack([[h00, h01], [h00, h11]])
    parent = np.array([-1, 0], np.int32)
    W = _layer(d, c * np.eye(d))
    empty = np.zeros((0, nh, d // nh))
    base = orc.layer_forward_sublayers(H, parent, W, empty, empty, 0.1, 0.0, nh, d // nh)
    fix = orc.layer_forward_sublayers(H, parent, W, empty, empty, 0.1, 0.0, nh, d // nh, attn_rematch=True)
    for res in (base, fix):
        assert res["fold"].tolist() == [[False, False], [True, False]]
        assert res["n"] == 3
    x00, x01, x11 = _unit(h00), _unit(h01), _unit(h11)
    root0 = h00 + c * (x00 + x01) / 2
    np.testing.assert_allclose(base["out"][0], root0, rtol=1e-14)
    np.testing.assert_allclose(base["out"][2], root0, rtol=1e-14)           # copied
    np.testing.assert_allclose(fix["out"][2], h00 + c * (x00 + x11) / 2, rtol=1e-14)
    np.testing.assert_allclose(fix["out"][3], h11 + c * (x00 + x11) / 2, rtol=1e-14)
    np.testing.assert_allclose(base["out"][3], fix["out"][3], rtol=1e-15)
    assert fix["attn_rows"].tolist() == [0, 1, 2, 3]


def test_ffn_gate_recomputes_what_attention_folded():
    """L = 1, no prefix.  The attention sublayer maps h to h (1 - 1.5 / rms(h)),
    shrinking the root row to a quarter, so a child folded by the first gate
    (r = 0.05 < tau = 0.1) is 0.2 away from the root after it: the FFN gate
    recomputes its FFN on its own A.  Hand-computed with a one-unit FFN
    silu(x2[0]) * x2[1] * e."""
    d, nh = 8, 2
    e = np.arange(1.0, d + 1) / d
    wg = np.zeros((1, d)); wg[0, 0] = 1.0
    wu = np.zeros((1, d)); wu[0, 1] = 1.0
    W = _layer(d, -1.5 * np.eye(d), F=1, w_gate=wg, w_up=wu, w_down=e[:, None])
    h = np.full(d, 2.0)
    delta = 0.1 * np.array([1.0, -1.0] * 4)
    H = np.stack([h, h + delta])[:, None, :]
    parent = np.array([-1, 0], np.int32)
    empty = np.zeros((0, nh, d // nh))
    silu = lambda z: float(Fn.silu(torch.tensor(z, dtype=torch.float64)))
    A_root = h / 4
    A_child = h / 4 + delta                     # attention folded: keeps its difference
    x2r, x2c = _unit(A_root), _unit(A_child)
    out_root = A_root + silu(x2r[0]) * x2r[1] * e
    gated = orc.layer_forward_sublayers(H, parent, W, empty, empty, 0.1, 0.0, nh, d // nh, ffn_gate=True)
    plain = orc.layer_forward_sublayers(H, parent, W, empty, empty, 0.1, 0.0, nh, d // nh)
    for res in (gated, plain):
        assert res["fold"].tolist() == [[False], [True]]
        np.testing.assert_allclose(res["A"], np.stack([A_root, A_child]), rtol=1e-14)
        np.testing.assert_allclose(res["out"][0], out_root, rtol=1e-14)
    assert gated["fold_ffn"].tolist() == [[False], [False]] and gated["n_ffn"] == 2
    np.testing.assert_allclose(gated["rel_ffn"][1, 0], 0.2, rtol=1e-14)
    np.testing.assert_allclose(gated["out"][1], A_child + silu(x2c[0]) * x2c[1] * e, rtol=1e-14)
    np.testing.assert_allclose(plain["out"][1], out_root + delta, rtol=1e-14)


def test_ffn_gate_folds_what_attention_recomputed():
    """L = 1.  W_o = -u u^T removes about half of a child's difference along
    u (the alternating direction): the child (r = 0.15 > tau) is recomputed
    through attention, but its A is within tau of the root's, so the FFN
    gate folds it: out = out_root + (A_child - A_root)."""
    d, nh = 8, 2
    u = np.array([1.0, -1.0] * 4) / math.sqrt(d)
    e = np.arange(1.0, d + 1) / d
    wg = np.zeros((1, d)); wg[0, 0] = 1.0
    wu = np.zeros((1, d)); wu[0, 1] = 1.0
    W = _layer(d, -np.outer(u, u), F=1, w_gate=wg, w_up=wu, w_down=e[:, None])
    h = np.full(d, 2.0)
    hc = h + 0.3 * math.sqrt(d) * u
    H = np.stack([h, hc])[:, None, :]
    parent = np.array([-1, 0], np.int32)
    empty = np.zeros((0, nh, d // nh))
    silu = lambda z: float(Fn.silu(torch.tensor(z, dtype=torch.float64)))
    A_root = h                                   # u^T ones = 0
    k = 1.0 / math.sqrt(float(np.mean(hc * hc)))
    A_child = hc - (0.3 * math.sqrt(d) * k) * u
    gated = orc.layer_forward_sublayers(H, parent, W, empty, empty, 0.1, 0.0, nh, d // nh, ffn_gate=True)
    plain = orc.layer_forward_sublayers(H, parent, W, empty, empty, 0.1, 0.0, nh, d // nh)
    for res in (gated, plain):
        assert res["fold"].tolist() == [[False], [False]]
        np.testing.assert_allclose(res["A"], np.stack([A_root, A_child]), rtol=1e-14)
    np.testing.assert_allclose(gated["rel"][1, 0], 0.15, rtol=1e-14)
    np.testing.assert_allclose(gated["rel_ffn"][1, 0], 0.15 * (1 - k), rtol=1e-13)
    assert gated["fold_ffn"].tolist() == [[False], [True]] and gated["n_ffn"] == 1
    x2r, x2c = _unit(A_root), _unit(A_child)
    out_root = A_root + silu(x2r[0]) * x2r[1] * e
    np.testing.assert_allclose(gated["out"][1], out_root + (A_child - A_root), rtol=1e-14)
    np.testing.assert_allclose(plain["out"][1], A_child + silu(x2c[0]) * x2c[1] * e, rtol=1e-14)


# ------------------------------------------------- seeded, against torch --

def _inputs(seed, P=12, wo_scale=1.0):
    """Seeded small layer.  ``wo_scale`` (a power of two) strengthens the
    attention sublayer: with the default weights (std 0.02) it moves the
    state so little that both gates take the same decisions everywhere."""
    w = synth.small_workload(d=64, n_q=4, n_kv=2, hd=16, F=96, P=P, L=6, levels=(1, 2, 3))
    inp = synth.make_layer_inputs(w, seed=seed)
    inp.weights["w_o"] = inp.weights["w_o"] * wo_scale
    return inp


def test_both_off_is_the_base_layer():
    inp = _inputs(1)
    d = inp.dims
    ref = orc.layer_forward(inp.H, inp.parent, inp.weights, inp.prefix.K, inp.prefix.V, 0.05, d.eps, d.n_kv, d.hd)
    res = _run(inp, 0.05)
    assert np.array_equal(res["fold"], ref["fold"]) and np.array_equal(res["src"], ref["src"])
    assert np.array_equal(res["fold_ffn"], ref["fold"]) and res["n_ffn"] == ref["n"]
    np.testing.assert_allclose(res["out"], ref["out"], rtol=1e-12, atol=1e-12)


@pytest.mark.parametrize("flags", [(True, False), (False, True), (True, True)])
def test_tau_zero_is_dense_torch(flags):
    """tau = 0 folds nothing at either gate: every branch runs the plain
    pre-norm layer, here assembled from torch routines."""
    inp = _inputs(2)
    d = inp.dims
    res = _run(inp, 0.0, attn_rematch=flags[0], ffn_gate=flags[1])
    B, L, D = inp.H.shape
    assert res["n"] == B * L and res["n_ffn"] == B * L
    W = inp.weights
    for b in range(B):
        h = _t(inp.H[b])
        x = Fn.rms_norm(h, (D,), weight=_t(W["g1"]), eps=d.eps)
        q = Fn.linear(x, _t(W["w_q"])).reshape(L, -1, d.hd).transpose(0, 1)
        k = Fn.linear(x, _t(W["w_k"])).reshape(L, d.n_kv, d.hd)
        v = Fn.linear(x, _t(W["w_v"])).reshape(L, d.n_kv, d.hd)
        K = torch.cat([_t(inp.prefix.K), k], 0).transpose(0, 1)
        V = torch.cat([_t(inp.prefix.V), v], 0).transpose(0, 1)
        o = Fn.scaled_dot_product_attention(q[None], K[None], V[None], enable_gqa=True)[0]
        a = h + Fn.linear(o.transpose(0, 1).reshape(L, -1), _t(W["w_o"]))
        np.testing.assert_allclose(res["out"][b * L:(b + 1) * L], _ffn_torch(a.numpy(), W, d.eps),
                                   rtol=1e-10, atol=1e-10)


def test_rematch_rows_against_torch_sdpa():
    """Every row's A under the literal correction, rebuilt in the test: the
    query of the row's chain end, keys and values of its own branch's block
    (each block position's chain end), torch SDPA, then W_o and the residual.
    The FFN rows follow torch's FFN; every other row keeps the FFN delta of
    its source exactly."""
    inp = _inputs(3)
    d = inp.dims
    W = inp.weights
    tau = 0.05
    res = _run(inp, tau, attn_rematch=True)
    base = _run(inp, tau)
    B, L, D = inp.H.shape
    fold, parent = res["fold"], inp.parent
    assert 0 < res["n"] < B * L
    H2 = inp.H.reshape(B * L, D)

    def qkv(r):
        x = Fn.rms_norm(_t(H2[r]), (D,), weight=_t(W["g1"]), eps=d.eps)
        return (Fn.linear(x, _t(W["w_q"])).reshape(-1, d.hd), Fn.linear(x, _t(W["w_k"])).reshape(d.n_kv, d.hd),
                Fn.linear(x, _t(W["w_v"])).reshape(d.n_kv, d.hd))

    rippled = 0
    for b in range(B):
        ks = torch.stack([qkv(_chain_src(fold, parent, b, j) * L + j)[1] for j in range(L)])
        vs = torch.stack([qkv(_chain_src(fold, parent, b, j) * L + j)[2] for j in range(L)])
        K = torch.cat([_t(inp.prefix.K), ks], 0).transpose(0, 1)
        V = torch.cat([_t(inp.prefix.V), vs], 0).transpose(0, 1)
        for i in range(L):
            s = _chain_src(fold, parent, b, i) * L + i
            q = qkv(s)[0][:, None, :]
            o = Fn.scaled_dot_product_attention(q[None], K[None], V[None], enable_gqa=True)[0]
            a = _t(H2[b * L + i]) + Fn.linear(o.reshape(-1), _t(W["w_o"]))
            np.testing.assert_allclose(res["A"][b * L + i], a.numpy(), rtol=1e-10, atol=1e-10)
            if s != b * L + i and not np.allclose(res["out"][b * L + i], base["out"][b * L + i], rtol=1e-9):
                rippled += 1
    assert rippled > 0, "no folded row saw a different block: the case does not exercise the correction"
    act = res["ffn_rows"]
    np.testing.assert_allclose(res["out"][act], _ffn_torch(res["A"][act], W, d.eps), rtol=1e-10, atol=1e-10)
    for r in range(B * L):
        s = int(res["src_ffn"][r])
        if s != r:
            np.testing.assert_allclose(res["out"][r] - res["A"][r], res["out"][s] - res["A"][s],
                                       rtol=1e-12, atol=1e-12)


@pytest.mark.parametrize("rematch,tau", [(False, 0.17), (True, 0.07)])
def test_ffn_gate_invariants(rematch, tau):
    """The FFN gate's decisions are the closed-form rule (brute force, fsum)
    on the A rows against the parent's A; without the correction an
    attention-folded row's A is its source's plus its own input difference;
    FFN rows follow torch; FFN-folded rows keep the FFN delta of their FFN
    source."""
    inp = _inputs(4, wo_scale=128.0)
    d = inp.dims
    W = inp.weights
    res = _run(inp, tau, attn_rematch=rematch, ffn_gate=True)
    B, L, D = inp.H.shape
    A = res["A"].reshape(B, L, D)
    for b in range(1, B):
        p = int(inp.parent[b])
        for i in range(L):
            num = math.fsum((A[b, i] - A[p, i]) ** 2)
            den = math.fsum(A[p, i] ** 2)
            assert res["fold_ffn"][b, i] == (num < tau * tau * den)
    assert not res["fold_ffn"][0].any()
    assert res["n_ffn"] == int((~res["fold_ffn"]).sum())
    assert not np.array_equal(res["fold_ffn"], res["fold"]), "the two gates agree everywhere: weak case"
    H2 = inp.H.reshape(B * L, D)
    if not rematch:
        for r in range(B * L):
            s = int(res["src"][r])
            if s != r:
                np.testing.assert_allclose(res["A"][r], res["A"][s] + (H2[r] - H2[s]), rtol=1e-13, atol=1e-13)
    act = res["ffn_rows"]
    np.testing.assert_allclose(res["out"][act], _ffn_torch(res["A"][act], W, d.eps), rtol=1e-10, atol=1e-10)
    for r in range(B * L):
        s = int(res["src_ffn"][r])
        assert s == _chain_src(res["fold_ffn"], inp.parent, r // L, r % L) * L + r % L
        if s != r:
            np.testing.assert_allclose(res["out"][r] - res["A"][r], res["out"][s] - res["A"][s],
                                       rtol=1e-12, atol=1e-12)
