"""Helpers shared by the GPU parity tests: move seeded inputs to the device,
run the CUDA path through the C-ABI binding, read its intermediates back, and
compare them with the CPU oracle."""
from __future__ import annotations

import numpy as np
import torch

from diffusion_branch_speculative_gb300 import binding, synth
from oracle import specfold_oracle as orc

TOL = 2e-2          # relative L2 bound for bf16 outputs
NEAR_TAU = 1e-4     # rows within this relative distance of tau are excluded from decision parity


def rel_l2(a, b) -> float:
    a = np.asarray(a, np.float64)
    b = np.asarray(b, np.float64)
    den = np.linalg.norm(b)
    return float(np.linalg.norm(a - b) / (den if den > 0 else 1.0))


def rel_rows(a, b) -> np.ndarray:
    """Relative L2 error of every row (axis 0), so that one wrong row (a bad
    tile, split slot or gathered key) cannot hide in a whole-tensor norm."""
    a = np.asarray(a, np.float64).reshape(len(a), -1)
    b = np.asarray(b, np.float64).reshape(len(b), -1)
    den = np.linalg.norm(b, axis=1)
    return np.linalg.norm(a - b, axis=1) / np.where(den > 0, den, 1.0)


def check_rows_out(Hg, ref, Hin, tol=TOL, floors=3.0):
    """Per-row bound on a bf16 layer output: the error of row r is at most tol
    of the layer's own contribution |ref_r - Hin_r| plus `floors` times the
    bf16 rounding floor of the row (a folded row passes three roundings: its
    source's A and output, and its own output).  Returns the worst ratio of
    error to bound."""
    Hg = np.asarray(Hg, np.float64)
    ref = np.asarray(ref, np.float64)
    err = np.linalg.norm(Hg - ref, axis=1)
    contrib = np.linalg.norm(ref - Hin, axis=1)
    floor = np.linalg.norm(synth.round_bf16(ref.astype(np.float32)).astype(np.float64) - ref, axis=1)
    bound = tol * contrib + floors * floor
    worst = int(np.argmax(err / np.maximum(bound, 1e-30)))
    assert np.all(err <= bound), (worst, float(err[worst]), float(bound[worst]), float(contrib[worst]),
                                  float(floor[worst]))
    return float(np.max(err / np.maximum(bound, 1e-30)))


def bf16(x: np.ndarray, device="cuda") -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(x, np.float32)).to(device).to(torch.bfloat16)


def to_np(t: torch.Tensor) -> np.ndarray:
    return t.detach().float().cpu().numpy()


def f32(x: np.ndarray, device="cuda") -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(x, np.float32)).to(device)


class DeviceInputs:
    """Seeded inputs on the device, in the workload's dtype (bf16, or fp32
    for the tiny fp32 configuration)."""

    def __init__(self, inp: synth.LayerInputs, device="cuda", rope_theta: float = 0.0, gate_ref: int = 0,
                 attn_rematch: int = 0, ffn_gate: int = 0):
        self.inp = inp
        d = inp.dims
        self.fp32 = inp.dtype == "f32"
        conv = f32 if self.fp32 else bf16
        self.tdtype = torch.float32 if self.fp32 else torch.bfloat16
        self.dims = binding.make_dims(d.d, d.n_q, d.n_kv, d.hd, d.F, d.eps, binding.F32 if self.fp32 else binding.BF16,
                                      rope_theta, gate_ref, attn_rematch, ffn_gate)
        self.H = conv(inp.H, device)
        self.parent = torch.from_numpy(inp.parent.astype(np.int32)).to(device)
        self.W = {k: conv(v, device) for k, v in inp.weights.items()}
        self.cache = conv(inp.prefix.cache, device)
        pre = inp.prefix
        self.P = pre.P
        self.pk = self.cache[pre.offset:pre.offset + pre.P, 0] if pre.P > 0 else None
        self.pv = self.cache[pre.offset:pre.offset + pre.P, 1] if pre.P > 0 else None
        self.B, self.L, _ = inp.H.shape


def run_layer(dev: DeviceInputs, tau: float):
    lay = binding.FoldedLayer(dev.dims, dev.W, dev.B, dev.L, dev.pk, dev.pv)
    out = lay.forward(dev.H, dev.parent, tau)
    torch.cuda.synchronize()
    return lay, out


def read_intermediates(lay: binding.FoldedLayer, dev: DeviceInputs) -> dict:
    d = dev.inp.dims
    R = dev.B * dev.L
    n = lay.n_packed()
    g = d.n_q // d.n_kv
    v = lay.view
    et = dev.tdtype
    res = {
        "n": n,
        "fold": v("fold", torch.uint8, (R,)).cpu().numpy().astype(bool),
        "rel": v("rel", torch.float32, (R,)).cpu().numpy(),
        "src": v("src", torch.int32, (R,)).cpu().numpy(),
        "packed_idx": v("packed_idx", torch.int32, (R,)).cpu().numpy()[:n],
        "slot": v("slot_of_row", torch.int32, (R,)).cpu().numpy(),
        "X1": to_np(v("x1", et, (R, d.d))[:n]),
        "Q": to_np(v("q", et, (d.n_kv, R, g, d.hd))[:, :n].permute(1, 0, 2, 3).reshape(n, -1)),
        "bK": to_np(v("block_k", et, (R, d.n_kv, d.hd))),
        "bV": to_np(v("block_v", et, (R, d.n_kv, d.hd))),
        "attnO": to_np(v("attn_o", et, (R, d.n_q * d.hd))[:n]),
        "A": to_np(v("a", et, (R, d.d))[:n]),
        "X2": to_np(v("x2", et, (R, d.d))[:n]),
        "G": to_np(v("g", et, (R, d.F))[:n]),
    }
    return res


def oracle_with_gpu_decisions(inp: synth.LayerInputs, tau: float, gpu_fold: np.ndarray, rows=None,
                              rope_theta: float = 0.0, gate_ref: int = 0):
    """Run the oracle; rows within NEAR_TAU of tau take the GPU's decision
    (spec rule: such rows are reported and excluded from decision
    parity).  Returns (oracle result, number of near-tau rows, mismatches
    outside the near-tau band).  With the variant gate (gate_ref 1) a forced
    decision changes the sources later rows compare with, so the near-tau
    set is found again after forcing (twice)."""
    d = inp.dims
    B, L, _ = inp.H.shape
    t32 = np.float32(tau)
    gf = gpu_fold.reshape(B, L)
    if gate_ref == 1:
        f0, rel = orc.gate_source(inp.H, inp.parent, t32)
        for _ in range(2):
            near = orc.near_tau_rows(rel, float(t32), NEAR_TAU)
            force = np.where(near, gf.astype(np.int8), np.int8(-1)).astype(np.int8)
            f0, rel = orc.gate_source(inp.H, inp.parent, t32, force)
        near = orc.near_tau_rows(rel, float(t32), NEAR_TAU)
    else:
        f0, rel = orc.gate(inp.H, inp.parent, t32)
        near = orc.near_tau_rows(rel, float(t32), NEAR_TAU)
    bad = (gf != f0) & ~near
    force = np.where(near, gf.astype(np.int8), np.int8(-1)).astype(np.int8)
    res = orc.layer_forward(inp.H, inp.parent, inp.weights, inp.prefix.K, inp.prefix.V, float(t32),
                            d.eps, d.n_kv, d.hd, force=force, rows=rows, rope_theta=rope_theta,
                            gate_ref="source" if gate_ref == 1 else "parent")
    return res, int(near.sum()), int(bad.sum())


def check_layer(inp, tau, rows=None, inter=True, rope_theta: float = 0.0, gate_ref: int = 0):
    dev = DeviceInputs(inp, rope_theta=rope_theta, gate_ref=gate_ref)
    lay, out = run_layer(dev, tau)
    assert lay.status() == 0
    gi = read_intermediates(lay, dev)
    res, n_near, n_bad = oracle_with_gpu_decisions(inp, tau, gi["fold"], rows, rope_theta=rope_theta,
                                                   gate_ref=gate_ref)
    assert n_bad == 0, f"{n_bad} gate decisions differ away from tau"
    B, L, D = inp.H.shape
    R = B * L
    # S1: relative differences (fp32 on the GPU) and decisions
    nonroot = np.arange(R) >= L
    rg, ro = gi["rel"][nonroot], res["rel"].reshape(-1)[nonroot]
    fin = np.isfinite(ro)
    np.testing.assert_allclose(rg[fin], ro[fin], rtol=1e-4, atol=1e-6)
    assert np.array_equal(gi["fold"], res["fold"].reshape(-1))
    # S2/S3: provenance and packed list, bit-exact
    assert np.array_equal(gi["src"], res["src"])
    assert gi["n"] == res["n"]
    assert np.array_equal(gi["packed_idx"], res["packed_idx"])
    assert np.array_equal(gi["slot"], res["slot"])
    m = {"n": gi["n"], "near_tau": n_near}
    rows_max = {}
    if inter:
        act = res["act_rows"]
        k = gi["slot"][act]
        pairs = {"X1": (gi["X1"][k], res["X1"]), "Q": (gi["Q"][k], res["Q"]),
                 "K": (gi["bK"][act], np.stack([res["K_rows"][r] for r in act])),
                 "V": (gi["bV"][act], np.stack([res["V_rows"][r] for r in act])),
                 "attnO": (gi["attnO"][k], res["attnO"]), "A": (gi["A"][k], res["A"]),
                 "X2": (gi["X2"][k], res["X2"]), "G": (gi["G"][k], res["G"])}
        for key, (g_, o_) in pairs.items():
            m[key] = rel_l2(g_, o_)
            rows_max[key] = float(rel_rows(g_, o_).max())
    Hg = to_np(out).reshape(R, D)
    Hin = inp.H.reshape(R, D).astype(np.float64)
    rr = res["out_rows"]
    m["H_out"] = rel_l2(Hg[rr], res["out"])
    m["delta"] = rel_l2(Hg[rr] - Hin[rr], res["out"] - Hin[rr])
    # The layer's own contribution (H_out - H_in) can be small next to H, so
    # the bf16 rounding of H_out alone may exceed 2e-2 of it: bound the error
    # by 2e-2 of the contribution plus twice that rounding floor.
    err = np.linalg.norm(Hg[rr] - res["out"])
    floor = np.linalg.norm(synth.round_bf16(res["out"].astype(np.float32)) - res["out"])
    assert err <= TOL * np.linalg.norm(res["out"] - Hin[rr]) + 2.0 * floor, m
    # and row by row (every output row the oracle computed)
    m["H_out_row_worst"] = check_rows_out(Hg[rr], res["out"], Hin[rr])
    for key, val in m.items():
        if key not in ("n", "near_tau", "delta", "H_out_row_worst"):
            assert val < TOL, (key, val, m)
    for key, val in rows_max.items():
        assert val < TOL, ("per-row", key, val, rows_max)
    m["rows_max"] = rows_max
    return m, lay, out


# ---------------------------------------------------------------------------
# the variant sublayer path (attn_rematch / ffn_gate)
# ---------------------------------------------------------------------------

# The FFN-sublayer gate decides on A, which the GPU stores in bf16 and the
# oracle keeps in float64, so the two compare slightly different rows.  The
# error of r = |A_b - A_p| / |A_p| is the part of A's error along the
# direction of A_b - A_p, over |A_p|.  Independent per-element errors give
# about sqrt(2) u / sqrt(d) (u = 2^-9 / sqrt(3) for bf16 storage), 1e-4 at
# d = 256; an error shared by a whole row (a scale error of the attention
# output, which the strong-attention cases below amplify into most of A - H)
# does not average out and gives about u itself.  Measured on GB300: up to
# 1.6e-3.  Rows with |r - tau| below 2e-3 in bf16 (1e-5 in fp32) take the
# GPU's decision (reported, excluded from decision parity), and the measured
# error must stay inside that band.
def ffn_near_abs(dtype: str, d: int) -> float:
    return 2e-3 if dtype == "bf16" else 1e-5


def read_sublayers(lay: binding.FoldedLayer, dev: DeviceInputs) -> dict:
    d = dev.inp.dims
    R = dev.B * dev.L
    v = lay.view
    n_f = int(v("n_ffn", torch.int32)[0].item())
    et = dev.tdtype
    return {
        "fold_ffn": v("fold_ffn", torch.uint8, (R,)).cpu().numpy().astype(bool),
        "rel_ffn": v("rel_ffn", torch.float32, (R,)).cpu().numpy(),
        "src_ffn": v("src_ffn", torch.int32, (R,)).cpu().numpy(),
        "packed_ffn": v("packed_ffn", torch.int32, (R,)).cpu().numpy()[:n_f],
        "n_ffn": n_f,
        "A_all": to_np(v("a_all", et, (R, d.d))),
        "X2": to_np(v("x2", et, (R, d.d))[:n_f]),
        "G": to_np(v("g", et, (R, d.F))[:n_f]),
    }


def oracle_sublayers_with_gpu_decisions(inp, tau, gpu_fold, gpu_fold_ffn, attn_rematch, ffn_gate,
                                        rope_theta=0.0, gate_ref=0, ffn_band=None):
    """The variant oracle with the GPU's decisions on near-tau rows of both
    gates.  Returns (result, near-tau rows of the first gate, mismatches
    outside its band, near-tau rows of the FFN gate, mismatches outside
    that band)."""
    d = inp.dims
    B, L, _ = inp.H.shape
    t32 = float(np.float32(tau))
    gf = gpu_fold.reshape(B, L)
    gff = gpu_fold_ffn.reshape(B, L)
    ref = "source" if gate_ref == 1 else "parent"
    gate_fn = orc.gate_source if gate_ref == 1 else orc.gate
    f0, rel = gate_fn(inp.H, inp.parent, t32)
    for _ in range(2 if gate_ref == 1 else 0):
        near = orc.near_tau_rows(rel, t32, NEAR_TAU)
        f0, rel = gate_fn(inp.H, inp.parent, t32, np.where(near, gf.astype(np.int8), np.int8(-1)).astype(np.int8))
    near = orc.near_tau_rows(rel, t32, NEAR_TAU)
    bad = int(((gf != f0) & ~near).sum())
    force = np.where(near, gf.astype(np.int8), np.int8(-1)).astype(np.int8)

    def run(force_ffn):
        return orc.layer_forward_sublayers(inp.H, inp.parent, inp.weights, inp.prefix.K, inp.prefix.V, t32, d.eps,
                                           d.n_kv, d.hd, attn_rematch=bool(attn_rematch), ffn_gate=bool(ffn_gate),
                                           force=force, force_ffn=force_ffn, rope_theta=rope_theta, gate_ref=ref)

    res = run(None)
    n_near_f, bad_f = 0, 0
    if ffn_gate:
        band = ffn_near_abs(inp.dtype, d.d) if ffn_band is None else ffn_band
        band = band if t32 > 0 else 0.0   # tau = 0 folds nothing: no band
        t_div = t32 if t32 > 0 else 1.0
        for _ in range(2 if gate_ref == 1 else 1):
            near_f = orc.near_tau_rows(res["rel_ffn"], t32, band / t_div)
            res = run(np.where(near_f, gff.astype(np.int8), np.int8(-1)).astype(np.int8))
        near_f = orc.near_tau_rows(res["rel_ffn"], t32, band / t_div)
        n_near_f = int(near_f.sum())
        bad_f = int(((gff != res["fold_ffn"]) & ~near_f).sum())
    return res, int(near.sum()), bad, n_near_f, bad_f


def check_layer_sublayers(inp, tau, attn_rematch, ffn_gate, rope_theta=0.0, gate_ref=0, prefix=None,
                          ffn_band=None):
    """The variant sublayer path against ``layer_forward_sublayers``: both
    gates' decisions, sources and packed lists exact (near-tau rows aside);
    A of every row, X2 and G of the FFN rows and H_out within tolerance."""
    dev = DeviceInputs(inp, rope_theta=rope_theta, gate_ref=gate_ref, attn_rematch=attn_rematch,
                       ffn_gate=ffn_gate)
    pk, pv = (dev.pk, dev.pv) if prefix is None else prefix
    lay = binding.FoldedLayer(dev.dims, dev.W, dev.B, dev.L, pk, pv)
    out = lay.forward(dev.H, dev.parent, tau)
    torch.cuda.synchronize()
    assert lay.status() == 0
    gi = read_intermediates(lay, dev)
    gs = read_sublayers(lay, dev)
    res, n_near, bad, n_near_f, bad_f = oracle_sublayers_with_gpu_decisions(
        inp, tau, gi["fold"], gs["fold_ffn"] if ffn_gate else gi["fold"], attn_rematch, ffn_gate, rope_theta,
        gate_ref, ffn_band)
    assert bad == 0, f"{bad} first-gate decisions differ away from tau"
    assert bad_f == 0, f"{bad_f} FFN-gate decisions differ away from tau"
    d = inp.dims
    B, L, D = inp.H.shape
    R = B * L
    assert np.array_equal(gi["fold"], res["fold"].reshape(-1))
    assert np.array_equal(gi["src"], res["src"])
    assert gi["n"] == res["n"] and np.array_equal(gi["packed_idx"], res["packed_idx"])
    m0 = {}
    if ffn_gate:
        assert np.array_equal(gs["fold_ffn"], res["fold_ffn"].reshape(-1))
        nonroot = np.arange(R) >= L
        ro = res["rel_ffn"].reshape(-1)[nonroot]
        fin = np.isfinite(ro)
        m0["rel_ffn_err"] = float(np.max(np.abs(gs["rel_ffn"][nonroot][fin] - ro[fin])))
        band = ffn_near_abs(inp.dtype, d.d) if ffn_band is None else ffn_band
        print("FFN gate: max |r_gpu - r_oracle|", m0["rel_ffn_err"], "band", band, "near-tau rows", n_near_f, "of", R)
        assert m0["rel_ffn_err"] < band, (m0["rel_ffn_err"], band)
        # the band excuses few rows: at most 5 % of the rows (and 2 rows on tiny layers)
        assert n_near_f <= max(2, R // 20), (n_near_f, R, m0["rel_ffn_err"], band)
    assert np.array_equal(gs["src_ffn"], res["src_ffn"])
    assert gs["n_ffn"] == res["n_ffn"] and np.array_equal(gs["packed_ffn"], res["packed_ffn"])
    tol = 1e-4 if dev.fp32 else TOL
    Hin = inp.H.reshape(R, D).astype(np.float64)
    m = {"n": gi["n"], "n_ffn": gs["n_ffn"], "near_tau": n_near, "near_tau_ffn": n_near_f, **m0}
    # attention output: every row with the correction, else the packed rows
    if attn_rematch:
        ao = to_np(lay.view("attn_o", dev.tdtype, (R, d.n_q * d.hd)))
    else:
        ao = gi["attnO"][gi["slot"][res["attn_rows"]]]
    m["attnO"] = rel_l2(ao, res["attnO"])
    m["X2"] = rel_l2(gs["X2"], res["X2"])
    m["G"] = rel_l2(gs["G"], res["G"])
    for key in ("attnO", "X2", "G"):
        assert m[key] < tol, (key, m)
    # row by row as well
    for key, (g_, o_) in (("attnO", (ao, res["attnO"])), ("X2", (gs["X2"], res["X2"])), ("G", (gs["G"], res["G"]))):
        worst = float(rel_rows(g_, o_).max()) if len(o_) else 0.0
        m[key + "_row_max"] = worst
        assert worst < tol, ("per-row", key, worst)
    Hg = to_np(out).reshape(R, D)
    m["A_delta"] = rel_l2(gs["A_all"] - Hin, res["A"] - Hin)
    m["delta"] = rel_l2(Hg - Hin, res["out"] - Hin)
    # A and H_out: the sublayers' own contributions (A - H_in, H_out - H_in)
    # can be small next to the state, so the bf16 rounding of the stored rows
    # alone may exceed 2e-2 of them: the bound is 2e-2 of the contribution plus
    # twice that rounding floor
    for got, ref, key in ((gs["A_all"], res["A"], "A_delta"), (Hg, res["out"], "delta")):
        if dev.fp32:
            assert m[key] < tol, (key, m)
            assert float(rel_rows(got - Hin, ref - Hin).max()) < 10 * tol, key
        else:
            floor = np.linalg.norm(synth.round_bf16(ref.astype(np.float32)) - ref)
            assert np.linalg.norm(got - ref) <= TOL * np.linalg.norm(ref - Hin) + 2.0 * floor, (key, m)
            m[key + "_row_worst"] = check_rows_out(got, ref, Hin)
    return m, res, lay, out
