"""The C-ABI library: builds, loads, exports every declared symbol, and
rejects bad arguments on the host before touching a GPU (CPU only)."""
import ctypes
import os
import re
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def L():
    from diffusion_branch_speculative_gb300 import build, binding
    build.build()
    return binding.lib()


def test_exports_every_declared_symbol(L):
    from diffusion_branch_speculative_gb300 import binding
    names = binding.header_functions()
    assert len(names) == len(binding._SIG)
    out = subprocess.run(["nm", "-D", "--defined-only", binding.LIB_PATH], capture_output=True, text=True).stdout
    exported = {line.split()[-1] for line in out.splitlines() if line.strip()}
    missing = [n for n in names if n not in exported]
    assert not missing, missing
    for n in names:
        assert hasattr(L, n)
    # every declared function has a binding signature
    assert set(names) == set(binding._SIG)


def test_status_strings(L):
    from diffusion_branch_speculative_gb300 import binding
    assert binding.status_string(0) == "ok"
    assert "align" in binding.status_string(binding.EALIGN)
    assert binding.status_string(12345) == "unknown status"


def _dims(**kw):
    from diffusion_branch_speculative_gb300 import binding
    base = dict(d=3584, n_q=28, n_kv=4, hd=128, F=18944)
    base.update(kw)
    return binding.make_dims(base["d"], base["n_q"], base["n_kv"], base["hd"], base["F"])


def test_workspace_layout_host_only(L):
    from diffusion_branch_speculative_gb300 import binding
    d = _dims()
    lo = binding.workspace_layout(d, 8, 32)
    R = 256
    assert lo.total == binding.workspace_size(d, 8, 32)
    variant = ("q_all", "all_idx", "n_all", "a_all", "fold_ffn", "rel_ffn", "src_ffn", "packed_ffn", "slot_ffn",
               "n_ffn", "dep_rng_ffn", "dep_rows_ffn")
    names = [f for f, _ in binding.specfold_ws_layout._fields_]
    # the base path reserves no variant-path regions
    assert all(getattr(lo, f) == 0 for f in variant)
    offs = [getattr(lo, f) for f in names if f not in variant]
    assert all(o % 256 == 0 for o in offs)
    assert offs == sorted(offs)
    assert lo.dep_rows - lo.dep_rng >= R * 8
    assert lo.x1 - lo.sync >= 4 + 4 * 160
    assert lo.q - lo.x1 >= R * 3584 * 2
    assert lo.gemm_scratch - lo.x2 >= R * 3584 * 2 + R * 18944 * 2
    # with a variant flag every region is reserved, in order
    dv = binding.make_dims(3584, 28, 4, 128, 18944, 1e-6, binding.BF16, 0.0, 0, 1, 1)
    lv = binding.workspace_layout(dv, 8, 32)
    offs_v = [getattr(lv, f) for f in names]
    assert all(o % 256 == 0 for o in offs_v) and offs_v == sorted(offs_v)
    assert lv.q_all - lv.g >= R * 18944 * 2
    assert lv.a_all - lv.n_all >= 256 and lv.fold_ffn - lv.a_all >= R * 3584 * 2
    assert lv.dep_rows_ffn - lv.dep_rng_ffn >= R * 8
    assert lv.total > lo.total
    # invalid shapes give 0 / an error code
    assert binding.workspace_size(_dims(hd=96), 8, 32) == 0
    assert binding.workspace_size(_dims(n_q=27), 8, 32) == 0
    assert binding.workspace_size(d, 0, 32) == 0
    assert binding.workspace_size(d, 1024, 32) == 0     # beyond SPECFOLD_MAX_ROWS
    lo2 = binding.specfold_ws_layout()
    assert L.specfold_workspace_layout(ctypes.byref(_dims(d=300)), 8, 32, ctypes.byref(lo2)) == binding.EUNSUPPORTED


def test_host_argument_errors_launch_nothing(L):
    from diffusion_branch_speculative_gb300 import binding
    before = L.specfold_launch_count()
    P = ctypes.c_void_p
    good = P(0x10000)
    odd = P(0x10001)
    f32 = ctypes.c_float
    # gate: null pointers, NaN/negative tau, misaligned H, unsupported d
    assert L.specfold_gate(0, None, good, 8, 32, 3584, f32(0.05), good, None, None) == binding.EINVAL
    assert L.specfold_gate(0, good, good, 8, 32, 3584, f32(-0.1), good, None, None) == binding.EINVAL
    assert L.specfold_gate(0, good, good, 8, 32, 3584, f32(float("nan")), good, None, None) == binding.EINVAL
    assert L.specfold_gate(0, odd, good, 8, 32, 3584, f32(0.05), good, None, None) == binding.EALIGN
    assert L.specfold_gate(0, good, good, 8, 32, 3000, f32(0.05), good, None, None) == binding.EUNSUPPORTED
    assert L.specfold_gate(7, good, good, 8, 32, 3584, f32(0.05), good, None, None) == binding.EINVAL
    assert L.specfold_gate(0, good, good, 0, 32, 3584, f32(0.05), good, None, None) == binding.EINVAL
    assert L.specfold_gate(0, good, good, 1024, 32, 3584, f32(0.05), good, None, None) == binding.ECAPACITY
    assert L.specfold_resolve(None, good, 8, 32, good, None, None) == binding.EINVAL
    # layer forward: workspace too small, misaligned weights, bad view strides
    d = _dims()
    w = binding.specfold_weights(*([0x20000] * 9))
    view = binding.specfold_kv_view(0x30000, 2 * 4 * 128, 128)
    size = binding.workspace_size(d, 8, 32)
    args = lambda **kw: dict(dict(H=good, parent=good, view=view, P=512, tau=0.05, out=good, ws=good, wsb=size), **kw)

    def call(**kw):
        a = args(**kw)
        return L.specfold_layer_forward(ctypes.byref(d), ctypes.byref(w), a["H"], a["parent"], 8, 32, a["view"],
                                        a["view"], a["P"], f32(a["tau"]), a["out"], a["ws"], a["wsb"], None, None)
    assert call(wsb=size - 1) == binding.ECAPACITY
    assert call(tau=-1.0) == binding.EINVAL
    assert call(H=odd) == binding.EALIGN
    assert call(P=-1) == binding.EINVAL
    for bad in ({"attn_rematch": 2}, {"ffn_gate": -1}, {"gate_ref": 3}):
        db = binding.make_dims(3584, 28, 4, 128, 18944, **bad)
        assert L.specfold_layer_forward(ctypes.byref(db), ctypes.byref(w), good, good, 8, 32, view, view, 512,
                                        f32(0.05), good, good, size, None, None) == binding.EINVAL
    assert call(view=binding.specfold_kv_view(0x30000, 1028, 128)) == binding.EALIGN
    assert call(view=binding.specfold_kv_view(0x30008, 1024, 128)) == binding.EALIGN
    w_bad = binding.specfold_weights(*([0x20000] * 8 + [0x20004]))
    assert L.specfold_layer_forward(ctypes.byref(d), ctypes.byref(w_bad), good, good, 8, 32, view, view, 512,
                                    f32(0.05), good, good, size, None, None) == binding.EALIGN
    w_null = binding.specfold_weights(*([0x20000] * 8 + [None]))
    assert L.specfold_layer_forward(ctypes.byref(d), ctypes.byref(w_null), good, good, 8, 32, view, view, 512,
                                    f32(0.05), good, good, size, None, None) == binding.EINVAL
    # linear: unsupported shapes
    assert L.specfold_linear(0, good, good, 128, 100, 64, good, good, 1 << 30, None) == binding.EUNSUPPORTED
    assert L.specfold_linear(0, good, good, 128, 128, 60, good, good, 1 << 30, None) == binding.EUNSUPPORTED
    assert L.specfold_linear(1, good, good, 128, 100, 64, good, good, 1 << 30, None) == binding.EUNSUPPORTED
    assert L.specfold_linear(7, good, good, 128, 128, 64, good, good, 1 << 30, None) == binding.EINVAL
    assert L.specfold_selftest_timeout(None, 1000, None) == binding.EINVAL
    assert L.specfold_launch_count() == before


def test_stack_host_checks_launch_nothing(L):
    """Stack entry point: sizes and every host-side rejection, with no GPU."""
    from diffusion_branch_speculative_gb300 import binding
    before = L.specfold_launch_count()
    P = ctypes.c_void_p
    f32 = ctypes.c_float
    d = _dims()
    layer = binding.workspace_size(d, 16, 32)
    stack = binding.stack_workspace_size(d, 16, 32)
    assert stack == layer + 16 * 32 * 3584 * 2          # one bf16 state buffer, already 256-byte multiple
    assert binding.stack_workspace_size(_dims(hd=96), 16, 32) == 0
    good_w = binding.specfold_weights(*([0x20000] * 9))
    bad_w = binding.specfold_weights(*([0x20000] * 8 + [0x20004]))
    view = binding.specfold_kv_view(0x30000, 2 * 4 * 128, 128)
    W = (binding.specfold_weights * 3)(good_w, good_w, bad_w)
    V = (binding.specfold_kv_view * 3)(view, view, view)
    H, par, out, ws = P(0x100000), P(0x10000), P(0x200000), P(0x400000)

    def call(n=3, w=W, h=H, o=out, wsb=stack, tau=0.05, trace=None):
        return L.specfold_stack_forward(ctypes.byref(d), n, w, h, par, 16, 32, V, V, 2048, f32(tau), o, trace, ws,
                                        wsb, None)
    assert call(n=0) == binding.EINVAL
    assert call(w=None) == binding.EINVAL
    assert call() == binding.EALIGN                     # layer 2's w_down is misaligned
    assert call(n=2, wsb=stack - 1) == binding.ECAPACITY
    assert call(n=2, wsb=layer) == binding.ECAPACITY    # no room for the state buffer
    assert call(n=2, o=H) == binding.EINVAL             # H_out aliasing H_in
    assert call(n=2, tau=float("nan")) == binding.EINVAL
    overlap = binding.specfold_stack_trace(0x100000 - 64, None, None)
    assert call(n=2, trace=ctypes.byref(overlap)) == binding.EINVAL
    odd = binding.specfold_stack_trace(0x800008, None, None)
    assert call(n=2, trace=ctypes.byref(odd)) == binding.EALIGN
    assert L.specfold_launch_count() == before


def test_product_path_has_no_oracle_import():
    """The package never imports the oracle (it is test infrastructure)."""
    pkg = os.path.join(ROOT, "diffusion_branch_speculative_gb300")
    for f in os.listdir(pkg):
        if f.endswith(".py"):
            txt = open(os.path.join(pkg, f)).read()
            assert not re.search(r"^\s*(from|import)\s+oracle", txt, re.M), f
            assert "specfold_oracle" not in txt, f


def test_binding_fails_loudly_without_library(tmp_path):
    code = ("import sys; sys.path.insert(0, %r)\n"
            "from diffusion_branch_speculative_gb300 import binding\n"
            "binding._lib = None\n"
            "try:\n    binding.lib(%r)\nexcept RuntimeError as e:\n    print('RAISED', e)\n") % (
        ROOT, str(tmp_path / "nope.so"))
    out = subprocess.run([sys.executable, "-c", code], capture_output=True, text=True)
    assert "RAISED" in out.stdout
