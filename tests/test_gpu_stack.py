"""Stack of folded layers on the GPU (specfold_stack_forward), through the C-ABI.

What is checked:
  * composition: the stack equals the same layers called one by one with
    specfold_layer_forward, bit for bit (states between layers, per-layer
    decisions and packed counts), eagerly and as a replayed graph;
  * per-layer parity against the oracle: the oracle runs the stack itself
    from the seeded inputs, storing each layer's output in bf16 (the stack's
    storage precision), and every layer of the CUDA path is checked on the
    oracle's own input to that layer, with the single-layer bars (decisions,
    provenance and packed lists bit-exact; bf16 outputs within 2e-2 relative
    L2);
  * end-to-end drift of the CUDA stack against the float64 oracle stack;
  * at the full 28-layer 7B-class size: composition, and the exact identical-
    children invariant at every layer.
"""
import numpy as np
import pytest
import torch

from diffusion_branch_speculative_gb300 import binding, synth
from oracle import specfold_oracle as orc
from tests.gpu_cases import TOL, DeviceInputs, bf16, check_layer, rel_l2, to_np

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    binding.lib()


class DeviceStack:
    """Seeded stack inputs on the device, and a FoldedStack over them."""

    def __init__(self, st: synth.StackInputs):
        self.st = st
        d = st.dims
        self.dims = binding.make_dims(d.d, d.n_q, d.n_kv, d.hd, d.F, d.eps, binding.BF16)
        self.H = bf16(st.H)
        self.parent = torch.from_numpy(st.parent.astype(np.int32)).cuda()
        self.W = [{k: bf16(v) for k, v in w.items()} for w in st.weights]
        self.caches = [bf16(p.cache) for p in st.prefixes]
        P, off = st.prefixes[0].P, st.prefixes[0].offset
        self.pk = [c[off:off + P, 0] if P else None for c in self.caches]
        self.pv = [c[off:off + P, 1] if P else None for c in self.caches]
        self.B, self.L, _ = st.H.shape
        self.stack = binding.FoldedStack(self.dims, self.W, self.B, self.L, self.pk, self.pv)


def chained_layers(dims, weights, H, parent, pk, pv, tau, ws):
    """The same layers called one at a time; returns (inputs of layers 1..n,
    final output, per-layer fold, per-layer n)."""
    cw = [binding.make_weights(w) for w in weights]
    P = 0 if pk[0] is None else pk[0].shape[0]
    B, L, _ = H.shape
    lo = binding.workspace_layout(dims, B, L)
    states, folds, ns = [], [], []
    x = H
    for l in range(len(weights)):
        y = torch.empty_like(H)
        binding.specfold_layer_forward(dims, cw[l], x, parent, pk[l], pv[l], P, tau, y, ws)
        folds.append(ws[lo.fold:lo.fold + B * L].clone())
        ns.append(int(ws[lo.n_packed:lo.n_packed + 4].view(torch.int32).item()))
        states.append(y)
        x = y
    torch.cuda.synchronize()
    return states[:-1], states[-1], folds, ns


def assert_stack_equals_chain(ds, tau, graph=False):
    s = ds.stack
    out = torch.empty_like(ds.H)
    if graph:
        g = s.graph(ds.H, ds.parent, tau, out, record=True)
        g.launch()
        g.launch()   # a replay is repeatable
    else:
        s.forward(ds.H, ds.parent, tau, out, record=True)
    torch.cuda.synchronize()
    assert s.status() == 0
    states, final, folds, ns = chained_layers(ds.dims, ds.W, ds.H, ds.parent, ds.pk, ds.pv, tau, s.ws)
    assert torch.equal(out, final)
    for l, x in enumerate(states):
        assert torch.equal(s.hidden[l], x), l
    for l in range(s.n_layers):
        assert torch.equal(s.fold[l].reshape(-1), folds[l]), l
    assert s.n_packed.cpu().tolist() == ns
    # without records the states ping-pong through the workspace: same output
    out2 = torch.empty_like(ds.H)
    s.forward(ds.H, ds.parent, tau, out2, record=False)
    torch.cuda.synchronize()
    assert torch.equal(out2, out)
    return ns


def _small(levels=(1, 2, 2), P=64, L=16, d=256, n_q=4, n_kv=2, hd=64, F=512):
    return synth.small_workload(d=d, n_q=n_q, n_kv=n_kv, hd=hd, F=F, P=P, L=L, levels=levels)


def test_stack_one_layer_equals_layer_forward():
    st = synth.make_stack_inputs(_small(), seed=4, n_layers=1)
    ds = DeviceStack(st)
    ns = assert_stack_equals_chain(ds, 0.05)
    assert ns[0] == int((ds.stack.fold[0] == 0).sum().item())


@pytest.mark.parametrize("tau", [0.0, 0.05, 0.2])
def test_stack_equals_chained_layers(tau):
    st = synth.make_stack_inputs(_small(levels=(1, 3, 2, 2), L=24), seed=6, n_layers=4)
    ds = DeviceStack(st)
    ns = assert_stack_equals_chain(ds, tau)
    if tau == 0.0:
        assert ns == [ds.B * ds.L] * 4


def test_stack_graph_equals_chained_layers():
    st = synth.make_stack_inputs(_small(levels=(1, 2, 3)), seed=8, n_layers=3)
    assert_stack_equals_chain(DeviceStack(st), 0.05, graph=True)


def oracle_chain(st: synth.StackInputs, tau: float, upto: int):
    """The oracle's own stack over layers [0, upto), each output stored in
    bf16: returns the inputs of layers 0..upto (float32, bf16-exact)."""
    d = st.dims
    layers = [(st.weights[l], st.prefixes[l].K, st.prefixes[l].V) for l in range(upto)]
    res = orc.stack_forward(st.H, st.parent, layers, tau, d.eps, d.n_kv, d.hd, store=synth.round_bf16)
    return [x.astype(np.float32) for x in res["inputs"]] + [res["out"].astype(np.float32)]


def layer_case(st: synth.StackInputs, l: int, H: np.ndarray) -> synth.LayerInputs:
    br = synth.BranchInputs(H=H, graph=st.branches.graph, revealed=st.branches.revealed,
                            new_reveals=st.branches.new_reveals)
    return synth.LayerInputs(workload=st.workload, dims=st.dims, branches=br, weights=st.weights[l],
                             prefix=st.prefixes[l], dtype=st.dtype)


@pytest.mark.parametrize("tau,levels,L,hd", [(0.05, (1, 2, 2), 16, 64), (0.1, (1, 3, 4), 24, 128),
                                            (0.02, (1, 1, 1, 1, 1), 32, 64)])
def test_stack_per_layer_parity(tau, levels, L, hd):
    n_layers = 3
    w = _small(levels=levels, L=L, hd=hd, n_q=4, n_kv=2, d=256 if hd == 64 else 512)
    st = synth.make_stack_inputs(w, seed=12, n_layers=n_layers)
    inputs = oracle_chain(st, tau, n_layers - 1)
    ns = []
    for l in range(n_layers):
        m, _, _ = check_layer(layer_case(st, l, inputs[l]), tau)
        ns.append(m["n"])
    print("n per layer", ns)


def test_stack_end_to_end_drift_dense():
    """tau = 0: no decisions, so the CUDA stack and the float64 oracle stack
    differ by rounding only; every layer's state stays within 2e-2."""
    n_layers = 4
    st = synth.make_stack_inputs(_small(levels=(1, 2, 1)), seed=3, n_layers=n_layers)
    ds = DeviceStack(st)
    out = ds.stack.forward(ds.H, ds.parent, 0.0, record=True)
    torch.cuda.synchronize()
    d = st.dims
    layers = [(st.weights[l], st.prefixes[l].K, st.prefixes[l].V) for l in range(n_layers)]
    ref = orc.stack_forward(st.H, st.parent, layers, 0.0, d.eps, d.n_kv, d.hd)
    errs = [rel_l2(to_np(ds.stack.hidden[l - 1]), ref["inputs"][l]) for l in range(1, n_layers)]
    errs.append(rel_l2(to_np(out), ref["out"]))
    print("end-to-end rel-L2 per layer", errs)
    assert max(errs) < TOL


def test_stack_end_to_end_decisions_folded():
    """tau > 0: decisions of the CUDA stack (on its own bf16 states) agree
    with the float64 oracle stack's except for rows whose oracle r lies
    within 25 % of tau (the bf16 drift of earlier layers moves r by a few
    per cent near tau, where child and parent states nearly cancel)."""
    n_layers = 3
    tau = 0.05
    st = synth.make_stack_inputs(_small(levels=(1, 2, 2)), seed=9, n_layers=n_layers)
    ds = DeviceStack(st)
    ds.stack.forward(ds.H, ds.parent, tau, record=True)
    torch.cuda.synchronize()
    d = st.dims
    layers = [(st.weights[l], st.prefixes[l].K, st.prefixes[l].V) for l in range(n_layers)]
    ref = orc.stack_forward(st.H, st.parent, layers, tau, d.eps, d.n_kv, d.hd)
    for l in range(n_layers):
        fg = ds.stack.fold[l].cpu().numpy().astype(bool)
        band = np.abs(ref["rel"][l] - tau) <= 0.25 * tau
        band[0] = False
        assert np.array_equal(fg[~band], ref["fold"][l][~band]), l


# ---------------------------------------------------- 7B-class stack sizes --

def test_stack_7b_two_layers_parity_sampled():
    """The 28-layer stack's shapes (7B dims, prefix 2048, 16 branches in a
    fanout-4 tree): layers 0 and 1 against the oracle on sampled rows, and
    the two-layer stack against the chained layer calls."""
    tau = 0.05
    st = synth.make_stack_inputs("7b_stack", seed=0, n_layers=2)
    inputs = oracle_chain(st, tau, 1)
    B, L, _ = st.H.shape
    rng = np.random.default_rng(1)
    rows = np.unique(np.concatenate([np.arange(L), rng.choice(np.arange(L, B * L), 24, replace=False)]))
    for l in range(2):
        check_layer(layer_case(st, l, inputs[l]), tau, rows=rows, inter=False)
    assert_stack_equals_chain(DeviceStack(st), tau)


@pytest.fixture(scope="module")
def stack28():
    """28 layers of 7B-class weights drawn on the device by torch's seeded
    generator (these are only compared with the library itself)."""
    w = synth.WORKLOADS["7b_stack"]
    d = w.dims
    weights, caches = synth.torch_stack_params(d, w.n_layers, w.P, seed=0)
    off = synth.PREFIX_OFFSET
    pk = [c[off:off + w.P, 0] for c in caches]
    pv = [c[off:off + w.P, 1] for c in caches]
    dims = binding.make_dims(d.d, d.n_q, d.n_kv, d.hd, d.F, d.eps, binding.BF16)
    yield w, dims, weights, pk, pv
    del weights, caches
    torch.cuda.empty_cache()


def test_stack_7b_28_layers_equals_chained_layers(stack28):
    w, dims, weights, pk, pv = stack28
    br = synth.make_branches(w, np.random.default_rng(0))
    ds = type("DS", (), {})()
    ds.dims, ds.W, ds.pk, ds.pv = dims, weights, pk, pv
    ds.H = bf16(br.H)
    ds.parent = torch.from_numpy(br.graph.parent.astype(np.int32)).cuda()
    ds.B, ds.L = w.B, w.L
    ds.stack = binding.FoldedStack(dims, weights, w.B, w.L, pk, pv)
    ns = assert_stack_equals_chain(ds, 0.05, graph=True)
    print("n per layer", ns)
    assert all(w.L <= n <= w.B * w.L for n in ns)


def test_stack_7b_28_layers_identical_children(stack28):
    """Children identical to their parents fold at every layer and stay equal
    to the root exactly, through all 28 layers."""
    w, dims, weights, pk, pv = stack28
    br = synth.make_branches(w, np.random.default_rng(1), identical_children=True)
    H = bf16(br.H)
    parent = torch.from_numpy(br.graph.parent.astype(np.int32)).cuda()
    s = binding.FoldedStack(dims, weights, w.B, w.L, pk, pv)
    out = s.forward(H, parent, 0.05, record=True)
    torch.cuda.synchronize()
    assert s.status() == 0
    assert s.n_packed.cpu().tolist() == [w.L] * w.n_layers
    assert bool((s.fold[:, 1:] == 1).all()) and bool((s.fold[:, 0] == 0).all())
    for x in list(s.hidden) + [out]:
        assert torch.equal(x[1:], x[:1].expand_as(x[1:]))
