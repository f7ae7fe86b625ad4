"""The seeded input generator: determinism, dtype exactness, graph shape."""
import numpy as np
import pytest

from diffusion_branch_speculative_gb300 import synth


def test_round_bf16_known_values():
    x = np.array([1.0, 1.0 + 2 ** -8, 1.0 + 3 * 2 ** -9, -2.5, 0.0, 3.140625], np.float32)
    y = synth.round_bf16(x)
    # 1 + 2^-8 is a tie between 1 and 1 + 2^-7: ties go to the even mantissa (1.0)
    assert y.tolist() == [1.0, 1.0, 1.0 + 2 ** -7, -2.5, 0.0, 3.140625]
    assert np.array_equal(synth.round_bf16(y), y)


def test_deterministic_and_bf16_exact():
    a = synth.make_layer_inputs("tiny", seed=3, dtype="bf16")
    b = synth.make_layer_inputs("tiny", seed=3, dtype="bf16")
    assert np.array_equal(a.H, b.H)
    for k in a.weights:
        assert np.array_equal(a.weights[k], b.weights[k])
        assert np.array_equal(synth.round_bf16(a.weights[k]), a.weights[k])
    assert np.array_equal(synth.round_bf16(a.H), a.H)
    c = synth.make_layer_inputs("tiny", seed=4, dtype="bf16")
    assert not np.array_equal(a.H, c.H)


@pytest.mark.parametrize("name", list(synth.WORKLOADS))
def test_graph_shapes(name):
    w = synth.WORKLOADS[name]
    g = synth.make_graph(w.levels, np.random.default_rng(0), w.max_fanout, w.second_parent)
    assert len(g.parent) == w.B
    assert g.parent[0] == -1
    assert all(0 <= g.parent[b] < b for b in range(1, w.B))
    for b in range(1, w.B):
        assert g.level[g.parent[b]] == g.level[b] - 1
        if g.second[b] >= 0:
            assert g.second[b] != g.parent[b] and g.level[g.second[b]] == g.level[b] - 1
    if w.max_fanout:
        assert np.bincount(g.parent[1:], minlength=w.B).max() <= w.max_fanout
    assert [int((g.level == lv).sum()) for lv in range(len(w.levels))] == list(w.levels)


def test_forced_fraction_counts():
    w = synth.small_workload(d=64, L=8, levels=(1, 3, 4))
    for f in (0.0, 0.25, 1.0):
        inp = synth.make_layer_inputs(w, seed=1, forced_frac=f)
        H = inp.H.astype(np.float64)
        big = 0
        for b in range(1, w.B):
            p = inp.parent[b]
            r = np.linalg.norm(H[b] - H[p], axis=1) / np.linalg.norm(H[p], axis=1)
            assert np.all((np.abs(r - 0.5) < 0.01) | (r < 0.01))
            big += int((r > 0.1).sum())
        assert big == round(f * (w.B - 1) * w.L)


def test_ripple_profile():
    inp = synth.make_layer_inputs("tiny", seed=0, dtype="f32")
    H = inp.H.astype(np.float64)
    for b in range(1, 4):
        p = inp.parent[b]
        (rv,) = inp.branches.new_reveals[b]
        r = np.linalg.norm(H[b] - H[p], axis=1) / np.linalg.norm(H[p], axis=1)
        for i in range(16):
            dist = abs(i - rv)
            s = 1.0 if dist == 0 else 0.3 * np.exp(-dist / 2.0)
            # u and w are independent random unit vectors (nearly orthogonal in 256-d)
            assert r[i] == pytest.approx(np.hypot(s, 1e-3), rel=2e-2, abs=3e-4)


def test_prefix_view_is_strided_slice():
    inp = synth.make_layer_inputs("tiny", seed=0)
    pk, pv = inp.prefix.K, inp.prefix.V
    assert pk.shape == (64, 2, 64) and pv.shape == (64, 2, 64)
    assert np.shares_memory(pk, inp.prefix.cache)
    assert pk.strides[0] == 2 * 2 * 64 * 4
