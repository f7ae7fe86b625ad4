"""CUDA path vs the CPU oracle, through the C-ABI (GPU only).

Bars: gate decisions, provenance and packed index lists are
bit-exact (rows within 1e-4 relative of tau are reported and take the GPU's
decision on both sides); bf16 outputs are within 2e-2 relative L2.
"""
import numpy as np
import pytest
import torch

from diffusion_branch_speculative_gb300 import binding, synth
from oracle import specfold_oracle as orc
from tests.gpu_cases import (TOL, DeviceInputs, bf16, check_layer, f32, oracle_with_gpu_decisions,
                             read_intermediates, rel_l2, run_layer, to_np)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    binding.lib()


# ------------------------------------------------------------ GEMM engine --

@pytest.mark.parametrize("M,N,K", [(1, 128, 64), (100, 256, 512), (300, 384, 1024), (129, 3584, 3584),
                                   (64, 3584, 18944), (2048, 1024, 4096),
                                   (2560, 2048, 1024)])   # 160 tiles: the last 8 split along K
def test_linear_matches_fp64(M, N, K):
    rng = np.random.default_rng(M + N + K)
    X = synth.round_bf16(rng.standard_normal((M, K)).astype(np.float32))
    W = synth.round_bf16((rng.standard_normal((N, K)) * 0.02).astype(np.float32))
    Xd, Wd = bf16(X), bf16(W)
    Y = torch.empty(M, N, dtype=torch.bfloat16, device="cuda")
    ws = binding.alloc_workspace(binding.linear_workspace_size(M, N))
    binding.specfold_linear(Xd, Wd, Y, ws)
    ref = X.astype(np.float64) @ W.astype(np.float64).T
    assert rel_l2(to_np(Y), ref) < 5e-3
    # a second call reuses the self-resetting split-K counters
    Y2 = torch.empty_like(Y)
    binding.specfold_linear(Xd, Wd, Y2, ws)
    assert torch.equal(Y, Y2)
    assert binding.specfold_get_status(ws) == 0


# ------------------------------------------------ standalone S1/S2/S3 calls --

@pytest.mark.parametrize("name,tau", [("tiny", 0.05), ("7b_layer", 0.05), ("3b_layer", 0.05)])
def test_gate_resolve_pack_standalone(name, tau):
    inp = synth.make_layer_inputs(name, seed=1, dtype="bf16")
    dev = DeviceInputs(inp)
    B, L, D = inp.H.shape
    R = B * L
    fold = torch.empty(R, dtype=torch.uint8, device="cuda")
    rel = torch.empty(R, dtype=torch.float32, device="cuda")
    binding.specfold_gate(dev.H, dev.parent, tau, fold, rel)
    f0, r0 = orc.gate(inp.H, inp.parent, np.float32(tau))
    near = orc.near_tau_rows(r0, float(np.float32(tau)))
    fg = fold.cpu().numpy().astype(bool).reshape(B, L)
    assert np.array_equal(fg[~near], f0[~near])
    # resolve/pack on the oracle's decisions (GPU's at near-tau rows)
    f_use = np.where(near, fg, f0)
    fold_d = torch.from_numpy(f_use.reshape(-1).astype(np.uint8)).cuda()
    src = torch.empty(R, dtype=torch.int32, device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    binding.specfold_resolve(fold_d, dev.parent, B, L, src, status)
    assert np.array_equal(src.cpu().numpy(), orc.resolve(f_use, inp.parent))
    pidx = torch.empty(R, dtype=torch.int32, device="cuda")
    slot = torch.empty(R, dtype=torch.int32, device="cuda")
    n_dev = torch.empty(1, dtype=torch.int32, device="cuda")
    X1 = torch.empty(R, D, dtype=torch.bfloat16, device="cuda")
    binding.specfold_pack(fold_d, dev.H, dev.W["g1"], inp.dims.eps, pidx, slot, n_dev, X1)
    idx, sl, n = orc.pack(f_use)
    assert int(n_dev.item()) == n
    assert np.array_equal(pidx.cpu().numpy()[:n], idx)
    assert np.array_equal(slot.cpu().numpy(), sl)
    x1 = orc.rmsnorm(inp.H.reshape(R, D)[idx], inp.weights["g1"], inp.dims.eps)
    assert rel_l2(to_np(X1[:n]), x1) < 5e-3
    assert int(status.item()) == 0


def test_bad_parent_sets_status():
    inp = synth.make_layer_inputs("tiny", seed=0, dtype="bf16")
    B, L = 4, 16
    fold = torch.ones(B * L, dtype=torch.uint8, device="cuda")
    parent = torch.tensor([-1, 0, 2, 1], dtype=torch.int32, device="cuda")   # parent[2] = 2 is invalid
    src = torch.empty(B * L, dtype=torch.int32, device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    binding.specfold_resolve(fold, parent, B, L, src, status)
    s = src.cpu().numpy().reshape(B, L)
    assert int(status.item()) & binding.DEV_BAD_PARENT
    assert np.all(s[0] == np.arange(L)) and np.all(s[1] == np.arange(L))
    assert np.all(s[2] == 2 * L + np.arange(L))          # chain stops at the bad link
    assert np.all(s[3] == np.arange(L))                  # 3 -> 1 -> 0


# --------------------------------------------------------- whole layer ----

@pytest.mark.parametrize("tau", [0.0, 0.05, 0.2])
def test_layer_small(tau):
    w = synth.small_workload(d=256, n_q=4, n_kv=2, hd=64, F=512, P=64, L=16, levels=(1, 2, 2))
    m, _, _ = check_layer(synth.make_layer_inputs(w, seed=3), tau)
    if tau == 0.0:
        assert m["n"] == 5 * 16


def test_layer_ragged_hd128():
    """P and L not multiples of the tiles, several branches per query tile."""
    w = synth.small_workload(d=512, n_q=8, n_kv=2, hd=128, F=384, P=100, L=12, levels=(1, 3, 4, 3),
                             reveals=(1, 2), second_parent=True)
    check_layer(synth.make_layer_inputs(w, seed=5), 0.05)


def test_layer_no_prefix():
    w = synth.small_workload(d=256, n_q=4, n_kv=2, hd=64, F=256, P=0, L=8, levels=(1, 2))
    check_layer(synth.make_layer_inputs(w, seed=2), 0.05)


@pytest.mark.parametrize("levels,L,tau", [
    ((1, 8, 55, 64), 32, 0.05),   # 4096 rows: several rows per warp (rows re-read for RMSNorm1)
    ((1, 1), 320, 0.05),          # more block positions than CTAs: positions grouped in turn
    ((1,), 16, 0.05),             # the main branch alone: every row recomputed
    ((1, 3, 9), 32, 0.0),         # tau = 0: nothing folds
])
def test_layer_gate_pack_shapes(levels, L, tau):
    """The fused gate / resolve / pack launch on shapes that take its other
    code paths, against the oracle (decisions, sources, packed list exact;
    outputs within tolerance)."""
    w = synth.small_workload(d=256, n_q=4, n_kv=2, hd=64, F=256, P=64, L=L, levels=levels)
    m, _, _ = check_layer(synth.make_layer_inputs(w, seed=11), tau)
    if tau == 0.0 or len(levels) == 1:
        assert m["n"] == sum(levels) * L


TOL_F32 = 1e-4   # relative L2 for the fp32 path (fp32 storage and accumulation)


def check_layer_f32(inp, tau, rope_theta=0.0, gate_ref=0, prefix=None):
    """The fp32 path against the oracle: decisions, provenance and packed
    lists bit-exact; every fp32 intermediate and the output within 1e-4."""
    dev = DeviceInputs(inp, rope_theta=rope_theta, gate_ref=gate_ref)
    pk, pv = (dev.pk, dev.pv) if prefix is None else prefix
    lay = binding.FoldedLayer(dev.dims, dev.W, dev.B, dev.L, pk, pv)
    out = lay.forward(dev.H, dev.parent, tau)
    torch.cuda.synchronize()
    assert lay.status() == 0
    gi = read_intermediates(lay, dev)
    res, _, bad = oracle_with_gpu_decisions(inp, tau, gi["fold"], rope_theta=rope_theta, gate_ref=gate_ref)
    assert bad == 0
    assert np.array_equal(gi["src"], res["src"]) and gi["n"] == res["n"]
    assert np.array_equal(gi["packed_idx"], res["packed_idx"])
    act = res["act_rows"]
    k = gi["slot"][act]
    m = {"X1": rel_l2(gi["X1"][k], res["X1"]), "Q": rel_l2(gi["Q"][k], res["Q"]),
         "K": rel_l2(gi["bK"][act], np.stack([res["K_rows"][r] for r in act])),
         "attnO": rel_l2(gi["attnO"][k], res["attnO"]), "A": rel_l2(gi["A"][k], res["A"]),
         "X2": rel_l2(gi["X2"][k], res["X2"]), "G": rel_l2(gi["G"][k], res["G"])}
    B, L, D = inp.H.shape
    Hg = to_np(out).reshape(B * L, D)
    Hin = inp.H.reshape(B * L, D).astype(np.float64)
    m["H_out"] = rel_l2(Hg, res["out"])
    m["delta"] = rel_l2(Hg - Hin, res["out"] - Hin)
    for key, val in m.items():
        assert val < TOL_F32, (key, val, m)
    return m


@pytest.mark.parametrize("tau", [0.05, 0.0, 0.2])
def test_layer_tiny_fp32(tau):
    """The tiny fp32 configuration (d 256, 4/2 x 64, F 1024, P 64, L 16, a
    4-branch chain) through the fp32 path."""
    m = check_layer_f32(synth.make_layer_inputs("tiny", seed=0), tau)
    print(m)


def test_layer_tiny_fp32_rope_paged_variant():
    inp = synth.make_layer_inputs("tiny", seed=1)
    pk, pv, _pool, _table = _paged(inp, 16, poison=True, as_f32=True)
    check_layer_f32(inp, 0.05, rope_theta=10000.0, gate_ref=1, prefix=(pk, pv))


def test_linear_fp32_matches_fp64():
    rng = np.random.default_rng(8)
    M, N, K = 70, 96, 256
    X = rng.standard_normal((M, K)).astype(np.float32)
    W = (rng.standard_normal((N, K)) * 0.02).astype(np.float32)
    Y = torch.empty(M, N, dtype=torch.float32, device="cuda")
    ws = binding.alloc_workspace(binding.linear_workspace_size(M, N))
    binding.specfold_linear(f32(X), f32(W), Y, ws)
    assert rel_l2(to_np(Y), X.astype(np.float64) @ W.astype(np.float64).T) < 1e-5


def test_layer_tiny_workload_bf16():
    check_layer(synth.make_layer_inputs("tiny", seed=0, dtype="bf16"), 0.05)


@pytest.mark.parametrize("tau", [0.0, 0.02, 0.05, 0.1])
def test_layer_7b(tau):
    m, _, _ = check_layer(synth.make_layer_inputs("7b_layer", seed=0), tau)
    print("7b", tau, m)


def test_layer_3b():
    m, _, _ = check_layer(synth.make_layer_inputs("3b_layer", seed=0), 0.05)
    print("3b", m)


@pytest.mark.parametrize("frac,n_expect", [(0.0, 32), (0.1, 234), (0.25, 536), (0.5, 1040), (1.0, 2048)])
def test_layer_stress_all_rows(frac, n_expect):
    """The stress workload (prefix 8192, 64 branches) at five recompute
    fractions: every output row, and every packed row's intermediates (so
    every m-tile of each GEMM and every query tile of the attention), row by
    row against the oracle.  n = 234 splits every attention tile's key
    range in two (104 units); n = 1040 runs 228 whole tiles, two waves."""
    inp = synth.make_layer_inputs("stress", seed=0, forced_frac=frac)
    m, _, _ = check_layer(inp, 0.05)
    assert m["n"] == n_expect
    print("stress", frac, m)


# the draft-budget points of the 7B-like layer (level sizes; node 0 is the main branch)
BUDGET_7B = {4: (1, 1, 2), 16: (1, 4, 11), 32: (1, 4, 6, 6, 6, 5, 4)}


@pytest.mark.parametrize("B", [4, 16, 32])
def test_layer_7b_budget(B):
    """The 7B-like layer (prefix 512, L 32) over 4, 16 and 32 branches: all
    rows against the oracle."""
    base = synth.WORKLOADS["7b_layer"]
    w = synth.Workload(f"7b_budget{B}", base.dims, P=base.P, L=base.L, levels=BUDGET_7B[B],
                       max_fanout=4 if B == 16 else None, second_parent=True, reveals=base.reveals,
                       ripple_len=base.ripple_len, taus=(0.05,), dtype="bf16")
    m, _, _ = check_layer(synth.make_layer_inputs(w, seed=B), 0.05)
    print("7b budget", B, m)


def test_deterministic_bitwise():
    inp = synth.make_layer_inputs("7b_layer", seed=4)
    dev = DeviceInputs(inp)
    lay = binding.FoldedLayer(dev.dims, dev.W, dev.B, dev.L, dev.pk, dev.pv)
    a = lay.forward(dev.H, dev.parent, 0.05).clone()
    b = lay.forward(dev.H, dev.parent, 0.05).clone()
    torch.cuda.synchronize()
    assert torch.equal(a, b)


def test_timeout_selftest_reports_and_context_survives():
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    binding.specfold_selftest_timeout(status, 20_000_000)
    torch.cuda.synchronize()
    assert int(status.item()) & binding.DEV_TIMEOUT
    assert binding.timeout_sites(int(status.item())) == ["timeout probe"]
    x = torch.ones(4, device="cuda")
    assert float((x * 2).sum().item()) == 8.0


@pytest.mark.parametrize("name", ["7b_layer", "small"])
def test_standalone_stage_calls_chain(name):
    """S1..S10 through the per-stage entry points (gate, resolve, pack, qkv,
    attention, out_proj, ffn) match the oracle and the fused layer call."""
    if name == "small":
        w = synth.small_workload(d=512, n_q=8, n_kv=2, hd=128, F=384, P=100, L=12, levels=(1, 3, 4))
        inp = synth.make_layer_inputs(w, seed=8)
    else:
        inp = synth.make_layer_inputs(name, seed=2)
    tau = 0.05
    dev = DeviceInputs(inp)
    d = inp.dims
    B, L, D = inp.H.shape
    R = B * L
    g = d.n_q // d.n_kv
    ws = binding.alloc_workspace(binding.workspace_size(dev.dims, B, L))
    cw = binding.make_weights(dev.W)
    i32 = dict(dtype=torch.int32, device="cuda")
    bf = dict(dtype=torch.bfloat16, device="cuda")
    fold = torch.empty(R, dtype=torch.uint8, device="cuda")
    src, pidx, slot = torch.empty(R, **i32), torch.empty(R, **i32), torch.empty(R, **i32)
    n_dev = torch.empty(1, **i32)
    X1 = torch.empty(R, D, **bf)
    Q = torch.empty(d.n_kv, R * g, d.hd, **bf)
    bK, bV = torch.zeros(R, d.n_kv, d.hd, **bf), torch.zeros(R, d.n_kv, d.hd, **bf)
    O = torch.empty(R, d.n_q * d.hd, **bf)
    A = torch.empty(R, D, **bf)
    Hout = torch.empty_like(dev.H)
    binding.specfold_gate(dev.H, dev.parent, tau, fold)
    binding.specfold_resolve(fold, dev.parent, B, L, src)
    binding.specfold_pack(fold, dev.H, dev.W["g1"], d.eps, pidx, slot, n_dev, X1)
    binding.specfold_qkv(dev.dims, cw, X1, pidx, n_dev, B, L, Q, bK, bV, ws)
    binding.specfold_attention(dev.dims, Q, dev.pk, dev.pv, dev.P, bK, bV, src, pidx, n_dev, B, L, O, ws)
    binding.specfold_out_proj(dev.dims, cw, O, pidx, n_dev, dev.H, B, L, A, ws)
    binding.specfold_ffn(dev.dims, cw, A, pidx, n_dev, dev.H, src, fold, B, L, Hout, ws)
    torch.cuda.synchronize()
    assert binding.specfold_get_status(ws) == 0
    gf = fold.cpu().numpy().astype(bool)
    res, _, n_bad = oracle_with_gpu_decisions(inp, tau, gf)
    assert n_bad == 0
    assert np.array_equal(src.cpu().numpy(), res["src"])
    n = int(n_dev.item())
    assert n == res["n"]
    assert rel_l2(to_np(A[:n]), res["A"]) < TOL
    assert rel_l2(to_np(Hout).reshape(R, D), res["out"]) < TOL
    # same result as the fused layer call
    lay, out = run_layer(dev, tau)
    assert rel_l2(to_np(Hout), to_np(out)) < 2e-3


def test_graph_replay_matches_eager_and_tracks_inputs():
    inp = synth.make_layer_inputs("7b_layer", seed=6)
    dev = DeviceInputs(inp)
    lay = binding.FoldedLayer(dev.dims, dev.W, dev.B, dev.L, dev.pk, dev.pv)
    eager = lay.forward(dev.H, dev.parent, 0.05).clone()
    H = dev.H.clone()
    out = torch.empty_like(H)
    g = lay.graph(H, dev.parent, 0.05, out)
    n0 = binding.specfold_launch_count()
    g.launch()
    torch.cuda.synchronize()
    assert binding.specfold_launch_count() - n0 >= 6   # at least one launch per stage kernel
    assert torch.equal(out, eager)
    # new inputs written into the captured buffer are picked up by the replay
    inp2 = synth.make_layer_inputs("7b_layer", seed=7)
    H.copy_(bf16(inp2.H))
    g.launch()
    torch.cuda.synchronize()
    eager2 = lay.forward(H, dev.parent, 0.05)
    torch.cuda.synchronize()
    assert torch.equal(out, eager2)
    g.close()


def test_graph_with_stage_events():
    inp = synth.make_layer_inputs("small" if False else "tiny", seed=1, dtype="bf16")
    dev = DeviceInputs(inp)
    lay = binding.FoldedLayer(dev.dims, dev.W, dev.B, dev.L, dev.pk, dev.pv)
    out = torch.empty_like(dev.H)
    ev = [torch.cuda.Event(enable_timing=True) for _ in range(binding.STAGE_EVENTS)]
    for e in ev:
        e.record()
    g = lay.graph(dev.H, dev.parent, 0.05, out, events=ev)
    for _ in range(3):
        g.launch()
        ev[-1].synchronize()
        times = [ev[i].elapsed_time(ev[i + 1]) for i in range(binding.STAGE_EVENTS - 1)]
        assert all(t >= 0 for t in times) and sum(times) > 0
    g.close()
    assert torch.equal(out, lay.forward(dev.H, dev.parent, 0.05))


# ------------------------------------------------------------ rotary embedding --

@pytest.mark.parametrize("tau,theta", [(0.05, 10000.0), (0.0, 500.0)])
def test_layer_rope_small(tau, theta):
    w = synth.small_workload(d=256, n_q=4, n_kv=2, hd=64, F=512, P=72, L=24, levels=(1, 2, 3))
    m, _, _ = check_layer(synth.make_layer_inputs(w, seed=21), tau, rope_theta=theta)
    print(m)


def test_layer_rope_7b_sampled():
    """7B layer with the Qwen2.5 rope base (1e6), sampled rows."""
    inp = synth.make_layer_inputs("7b_layer", seed=2)
    B, L, _ = inp.H.shape
    rng = np.random.default_rng(3)
    rows = np.unique(np.concatenate([np.arange(L), rng.choice(np.arange(L, B * L), 24, replace=False)]))
    check_layer(inp, 0.05, rows=rows, inter=False, rope_theta=1.0e6)


def test_rope_standalone_matches_oracle():
    """specfold_rope on given Q / block-K layouts against the oracle's rope,
    at positions up to the stress prefix (P 8192)."""
    R, L, P, n_q, n_kv, hd = 96, 32, 8192, 8, 2, 128
    g = n_q // n_kv
    rng = np.random.default_rng(5)
    Q = synth.round_bf16(rng.standard_normal((n_kv, R * g, hd)).astype(np.float32))
    K = synth.round_bf16(rng.standard_normal((R, n_kv, hd)).astype(np.float32))
    n = 70
    pidx = np.sort(rng.choice(R, size=n, replace=False)).astype(np.int32)
    dims = binding.make_dims(256, n_q, n_kv, hd, 512, 1e-6, binding.BF16, 1.0e6)
    Qd, Kd = bf16(Q), bf16(K)
    pid = torch.from_numpy(np.concatenate([pidx, np.full(R - n, -1, np.int32)])).cuda()
    n_dev = torch.tensor([n], dtype=torch.int32, device="cuda")
    binding.specfold_rope(dims, Qd, Kd, pid, n_dev, R // L, L, P)
    torch.cuda.synchronize()
    Qg, Kg = to_np(Qd), to_np(Kd)
    for k in range(n):
        r = int(pidx[k])
        pos = P + r % L
        q_ref = orc.rope(Q[:, k * g:(k + 1) * g, :], pos, 1.0e6)
        assert rel_l2(Qg[:, k * g:(k + 1) * g, :], q_ref) < 1e-2
        assert rel_l2(Kg[r], orc.rope(K[r], pos, 1.0e6)) < 1e-2
    # rows beyond n and keys of unpacked rows are untouched
    assert np.array_equal(Qg[:, n * g:, :], Q[:, n * g:, :])
    untouched = np.setdiff1d(np.arange(R), pidx)
    assert np.array_equal(Kg[untouched], K[untouched])


# ------------------------------------------------------------ paged prefix --

def _paged(inp, page_size, spare_pages=3, seed=0, poison=True, as_f32=False):
    """Scatter the seeded prefix K/V into a fused page pool
    [pages * page_size, 2, n_kv, hd] in shuffled page order; unused pool
    tokens hold NaN (they must never be read)."""
    P = inp.prefix.P
    d = inp.dims
    need = (P + page_size - 1) // page_size
    pages = need + spare_pages
    rng = np.random.default_rng(seed)
    table = rng.permutation(pages)[:need].astype(np.int32)
    pool = np.full((pages * page_size, 2, d.n_kv, d.hd), np.nan if poison else 0.0, np.float32)
    for t in range(P):
        tok = table[t // page_size] * page_size + t % page_size
        pool[tok, 0] = inp.prefix.K[t]
        pool[tok, 1] = inp.prefix.V[t]
    pool_d = f32(pool) if as_f32 else bf16(pool)
    table_d = torch.from_numpy(table).cuda()
    return (binding.PagedPrefix(pool_d[:, 0], table_d, page_size, P),
            binding.PagedPrefix(pool_d[:, 1], table_d, page_size, P), pool_d, table_d)


@pytest.mark.parametrize("P,page_size", [(200, 16), (512, 128), (300, 256), (72, 8)])
def test_layer_paged_prefix(P, page_size):
    """The layer on a paged prefix (shuffled pages, NaN in every unused pool
    token) against the oracle on the logical prefix."""
    w = synth.small_workload(d=256, n_q=4, n_kv=2, hd=128, F=512, P=P, L=16, levels=(1, 2, 2))
    inp = synth.make_layer_inputs(w, seed=31)
    pk, pv, _pool, _table = _paged(inp, page_size)
    dev = DeviceInputs(inp)
    lay = binding.FoldedLayer(dev.dims, dev.W, dev.B, dev.L, pk, pv)
    out = lay.forward(dev.H, dev.parent, 0.05)
    torch.cuda.synchronize()
    assert lay.status() == 0
    gi = read_intermediates(lay, dev)
    res, _, bad = oracle_with_gpu_decisions(inp, 0.05, gi["fold"])
    assert bad == 0
    k = gi["slot"][res["act_rows"]]
    assert rel_l2(gi["attnO"][k], res["attnO"]) < TOL
    # the same layer on the contiguous view gives the same bits
    lay2 = binding.FoldedLayer(dev.dims, dev.W, dev.B, dev.L, dev.pk, dev.pv)
    out2 = lay2.forward(dev.H, dev.parent, 0.05)
    torch.cuda.synchronize()
    assert torch.equal(out, out2)


def test_paged_prefix_bad_page_sets_status():
    """A block-table entry outside the pool reads as zeros and sets
    SPECFOLD_DEV_BAD_PAGE; the context stays usable."""
    w = synth.small_workload(d=256, n_q=4, n_kv=2, hd=64, F=512, P=96, L=16, levels=(1, 2))
    inp = synth.make_layer_inputs(w, seed=32)
    pk, pv, pool, table = _paged(inp, 16, poison=False)
    table[2] = 10_000
    dev = DeviceInputs(inp)
    lay = binding.FoldedLayer(dev.dims, dev.W, dev.B, dev.L, pk, pv)
    out = lay.forward(dev.H, dev.parent, 0.05)
    torch.cuda.synchronize()
    assert lay.status() & binding.DEV_BAD_PAGE
    assert torch.isfinite(out.float()).all()
    assert lay.status() == 0   # cleared by the read


# ------------------------------------------------- variant: gate vs source --

@pytest.mark.parametrize("name,tau", [("7b_layer", 0.05), ("3b_layer", 0.05), ("tiny", 0.1), ("stress", 0.05)])
def test_gate_source_standalone(name, tau):
    """Decisions of the variant gate bit-exact against the oracle (rows
    within 1e-4 of tau take the GPU's decision), r within fp32 rounding."""
    inp = synth.make_layer_inputs(name, seed=4, dtype="bf16")
    dev = DeviceInputs(inp)
    B, L, _ = inp.H.shape
    R = B * L
    fold = torch.empty(R, dtype=torch.uint8, device="cuda")
    rel = torch.empty(R, dtype=torch.float32, device="cuda")
    binding.specfold_gate_source(dev.H, dev.parent, tau, fold, rel)
    torch.cuda.synchronize()
    fg = fold.cpu().numpy().astype(bool)
    t32 = np.float32(tau)
    f0, r0 = orc.gate_source(inp.H, inp.parent, t32)
    for _ in range(2):
        near = orc.near_tau_rows(r0, float(t32))
        force = np.where(near, fg.reshape(B, L).astype(np.int8), np.int8(-1)).astype(np.int8)
        f0, r0 = orc.gate_source(inp.H, inp.parent, t32, force)
    near = orc.near_tau_rows(r0, float(t32))
    assert np.array_equal(fg.reshape(B, L)[~near], f0[~near])
    rg = rel.cpu().numpy().reshape(B, L)
    fin = np.isfinite(r0) & (r0 >= 0)
    np.testing.assert_allclose(rg[fin], r0[fin], rtol=1e-4, atol=1e-6)
    # it differs from the parent gate somewhere on deep graphs (or equals it)
    fp = np.zeros(R, np.uint8)
    fpd = torch.empty(R, dtype=torch.uint8, device="cuda")
    binding.specfold_gate(dev.H, dev.parent, tau, fpd)
    print(name, "rows folded: source", int(fg.sum()), "parent", int(fpd.sum().item()))


@pytest.mark.parametrize("tau", [0.05, 0.1])
def test_layer_gate_source_small(tau):
    w = synth.small_workload(d=256, n_q=4, n_kv=2, hd=64, F=512, P=64, L=16, levels=(1, 2, 3, 2, 1))
    m, _, _ = check_layer(synth.make_layer_inputs(w, seed=41), tau, gate_ref=1)
    print(m)


def test_layer_gate_source_3b_sampled():
    inp = synth.make_layer_inputs("3b_layer", seed=1)
    B, L, _ = inp.H.shape
    rng = np.random.default_rng(2)
    rows = np.unique(np.concatenate([np.arange(L), rng.choice(np.arange(L, B * L), 24, replace=False)]))
    check_layer(inp, 0.05, rows=rows, inter=False, gate_ref=1)


# ------------------------------------------ S1-S3 in one launch (entry point) --

def _gate_pack_case(levels, L, d, frac, tau=0.05, fanout=None):
    base = synth.small_workload(d=d, n_q=4, n_kv=2, hd=64, F=256, P=0, L=L, levels=levels, max_fanout=fanout)
    return synth.make_layer_inputs(base, seed=9, forced_frac=frac)


@pytest.mark.parametrize("levels,L,d,frac", [
    ((1, 8, 55), 32, 3584, 1.0),        # the stress size, every row recomputed
    ((1, 8, 55), 32, 3584, 0.25),
    ((1, 8, 64, 439), 32, 256, 0.25),   # 16384 rows (the row limit): many rows per CTA
    ((1, 2, 3, 2), 32, 3584, 0.25),     # 8 branches, depth 3: the dependents lists built by one warp
    ((1, 4, 11, 16), 32, 3584, 0.5),    # 32 branches: the largest graph the one-warp lists take
])
def test_gate_pack_entry_point(levels, L, d, frac):
    """specfold_gate_pack against the oracle: decisions, sources, packed list
    and n exactly, RMSNorm1 row by row; the dependents lists are a partition
    of the folded rows by source."""
    inp = _gate_pack_case(levels, L, d, frac, fanout=8)
    dev = DeviceInputs(inp)
    B, L, D = inp.H.shape
    R = B * L
    ws = binding.alloc_workspace(binding.workspace_size(dev.dims, B, L))
    binding.specfold_gate_pack(dev.dims, dev.W["g1"], dev.H, dev.parent, 0.05, ws)
    torch.cuda.synchronize()
    assert binding.specfold_get_status(ws) == 0
    lo = binding.workspace_layout(dev.dims, B, L)

    def view(name, dtype, n):
        off = getattr(lo, name)
        es = torch.empty((), dtype=dtype).element_size()
        return ws[off:off + n * es].view(dtype)
    fold = view("fold", torch.uint8, R).cpu().numpy().astype(bool)
    f0, r0 = orc.gate(inp.H, inp.parent, np.float32(0.05))
    near = orc.near_tau_rows(r0, float(np.float32(0.05)))
    assert np.array_equal(fold.reshape(B, L)[~near], f0[~near])
    f_use = fold.reshape(B, L)
    src = view("src", torch.int32, R).cpu().numpy()
    assert np.array_equal(src, orc.resolve(f_use, inp.parent))
    idx, sl, n = orc.pack(f_use)
    assert int(view("n_packed", torch.int32, 1).item()) == n
    assert np.array_equal(view("packed_idx", torch.int32, R).cpu().numpy()[:n], idx)
    assert np.array_equal(view("slot_of_row", torch.int32, R).cpu().numpy(), sl)
    x1 = view("x1", torch.bfloat16, R * D).view(R, D)[:n].float().cpu().numpy()
    ref = orc.rmsnorm(inp.H.reshape(R, D)[idx], inp.weights["g1"], inp.dims.eps)
    from tests.gpu_cases import rel_rows
    assert float(rel_rows(x1, ref).max()) < 5e-3
    # dependents: every folded row exactly once, in the range of its source
    rng = view("dep_rng", torch.int32, 2 * R).view(R, 2).cpu().numpy()
    deps = view("dep_rows", torch.int32, R).cpu().numpy()
    seen = np.zeros(R, int)
    for s in idx:
        b_, e_ = rng[s]
        for r in deps[b_:e_]:
            assert src[r] == s and r != s
            seen[r] += 1
    folded = np.nonzero(src != np.arange(R))[0]
    assert np.all(seen[folded] == 1) and seen.sum() == len(folded)
