"""GPU parity of the variant sublayer path: the literal attention correction
for folded rows (attn_rematch) and a gate of its own for the FFN sublayer
(ffn_gate), against the oracle's ``layer_forward_sublayers``."""
import numpy as np
import pytest
import torch

from diffusion_branch_speculative_gb300 import binding, synth
from oracle import specfold_oracle as orc
from tests.gpu_cases import check_layer, check_layer_sublayers, rel_l2, to_np
from tests.test_gpu_stack import DeviceStack, assert_stack_equals_chain

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    binding.lib()


FLAGS = [(1, 0), (0, 1), (1, 1)]


def _small(seed, L=32, levels=(1, 2, 3, 2), wo_scale=1.0, **kw):
    """R = 256 rows (two GEMM row tiles), P 64.  wo_scale (a power of two)
    strengthens the attention sublayer so the two gates disagree on rows."""
    w = synth.small_workload(d=256, n_q=4, n_kv=2, hd=64, F=512, P=64, L=L, levels=levels, **kw)
    inp = synth.make_layer_inputs(w, seed=seed)
    inp.weights["w_o"] = synth.round_bf16((inp.weights["w_o"] * wo_scale).astype(np.float32))
    return inp


def _base_out(inp, tau):
    d = inp.dims
    return orc.layer_forward(inp.H, inp.parent, inp.weights, inp.prefix.K, inp.prefix.V, tau, d.eps, d.n_kv,
                             d.hd)["out"]


@pytest.mark.parametrize("flags", FLAGS)
@pytest.mark.parametrize("tau", [0.05, 0.0])
def test_sublayers_small(flags, tau):
    m, res, _, _ = check_layer_sublayers(_small(3), tau, *flags)
    print(flags, tau, m)
    if tau == 0.0:
        assert m["n"] == m["n_ffn"] == 256


def test_rematch_changes_folded_rows():
    """The correction is live: a folded row's attention output on the GPU is
    its own (its source's query over its own branch's block), not its
    source's.  Checked on the attention output, where the difference is not
    hidden under the residual state."""
    inp = _small(5)
    m, res, lay, _ = check_layer_sublayers(inp, 0.05, 1, 0)
    d = inp.dims
    R = res["A"].shape[0]
    F = np.nonzero(res["src"] != np.arange(R))[0]
    assert F.size > 0
    ao = to_np(lay.view("attn_o", torch.bfloat16, (R, d.n_q * d.hd)))
    own = res["attnO"][F]                 # attn_rows are all rows, in row order
    of_src = res["attnO"][res["src"][F]]  # what the base layer would reuse
    err = rel_l2(ao[F], own)
    assert err < 1e-2
    assert rel_l2(own, of_src) > 5 * err, (rel_l2(own, of_src), err)


@pytest.mark.parametrize("rematch,tau", [(0, 0.14), (1, 0.08), (1, 0.03)])
def test_ffn_gate_strong_attention(rematch, tau):
    """W_o x 128: the attention sublayer moves the state enough that the FFN
    gate folds rows the first gate recomputed and recomputes rows it
    folded."""
    m, res, _, _ = check_layer_sublayers(_small(3, wo_scale=128.0), tau, rematch, 1)
    print(rematch, tau, m)
    assert (res["fold_ffn"] != res["fold"]).sum() > 0


def test_sublayers_gate_source_rope():
    inp = _small(41, L=16, levels=(1, 2, 3, 2, 1))
    m, _, _, _ = check_layer_sublayers(inp, 0.05, 1, 1, rope_theta=10000.0, gate_ref=1)
    print(m)


def test_sublayers_flags_off_is_base_layer():
    """attn_rematch = ffn_gate = 0 takes the fused path; the same flags
    through the sublayer path's oracle agree with the base layer."""
    inp = _small(7)
    m, lay, out = check_layer(inp, 0.05)
    d = inp.dims
    res = orc.layer_forward_sublayers(inp.H, inp.parent, inp.weights, inp.prefix.K, inp.prefix.V, 0.05, d.eps,
                                      d.n_kv, d.hd)
    np.testing.assert_allclose(res["out"], _base_out(inp, 0.05), rtol=1e-10, atol=1e-10)


def test_sublayers_tiny_fp32():
    inp = synth.make_layer_inputs("tiny", seed=2)
    for flags in FLAGS:
        m, _, _, _ = check_layer_sublayers(inp, 0.05, *flags)
        print(flags, m)


@pytest.mark.parametrize("rematch,fgate,tau", [(0, 1, 0.05), (1, 0, 0.1), (1, 1, 0.05)])
def test_sublayers_7b(rematch, fgate, tau):
    """The 7B layer (d 3584, 28/4 x 128, F 18944, P 512, B 8, L 32) under each
    variant on its own and both together: the FFN gate's unpack-and-fill path
    without the correction, the correction without the FFN gate, and both."""
    inp = synth.make_layer_inputs("7b_layer", seed=0)
    m, _, _, _ = check_layer_sublayers(inp, tau, rematch, fgate)
    print(m)


@pytest.mark.parametrize("graph", [False, True])
def test_sublayers_stack_composition(graph):
    """A stack with both variant flags equals the chained single-layer calls
    bit for bit (states, decisions, packed counts), eagerly and as a graph."""
    st = synth.make_stack_inputs(synth.small_workload(d=256, n_q=4, n_kv=2, hd=64, F=512, P=32, L=16,
                                                      levels=(1, 2, 2)), seed=3, n_layers=3)
    ds = DeviceStack(st)
    d = st.dims
    ds.dims = binding.make_dims(d.d, d.n_q, d.n_kv, d.hd, d.F, d.eps, binding.BF16, 0.0, 0, 1, 1)
    ds.stack = binding.FoldedStack(ds.dims, ds.W, ds.B, ds.L, ds.pk, ds.pv)
    assert_stack_equals_chain(ds, 0.05, graph=graph)
