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


def bf16(x: np.ndarray, device="cuda") -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(x, np.float32)).to(device).to(torch.bfloat16)


def to_np(t: torch.Tensor) -> np.ndarray:
    return t.detach().float().cpu().numpy()


class DeviceInputs:
    def __init__(self, inp: synth.LayerInputs, device="cuda"):
        self.inp = inp
        d = inp.dims
        self.dims = binding.make_dims(d.d, d.n_q, d.n_kv, d.hd, d.F, d.eps, binding.BF16)
        self.H = bf16(inp.H, device)
        self.parent = torch.from_numpy(inp.parent.astype(np.int32)).to(device)
        self.W = {k: bf16(v, device) for k, v in inp.weights.items()}
        self.cache = bf16(inp.prefix.cache, device)
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
    res = {
        "n": n,
        "fold": v("fold", torch.uint8, (R,)).cpu().numpy().astype(bool),
        "rel": v("rel", torch.float32, (R,)).cpu().numpy(),
        "src": v("src", torch.int32, (R,)).cpu().numpy(),
        "packed_idx": v("packed_idx", torch.int32, (R,)).cpu().numpy()[:n],
        "slot": v("slot_of_row", torch.int32, (R,)).cpu().numpy(),
        "X1": to_np(v("x1", torch.bfloat16, (R, d.d))[:n]),
        "Q": to_np(v("q", torch.bfloat16, (d.n_kv, R, g, d.hd))[:, :n].permute(1, 0, 2, 3).reshape(n, -1)),
        "bK": to_np(v("block_k", torch.bfloat16, (R, d.n_kv, d.hd))),
        "bV": to_np(v("block_v", torch.bfloat16, (R, d.n_kv, d.hd))),
        "attnO": to_np(v("attn_o", torch.bfloat16, (R, d.n_q * d.hd))[:n]),
        "A": to_np(v("a", torch.bfloat16, (R, d.d))[:n]),
        "X2": to_np(v("x2", torch.bfloat16, (R, d.d))[:n]),
        "G": to_np(v("g", torch.bfloat16, (R, d.F))[:n]),
    }
    return res


def oracle_with_gpu_decisions(inp: synth.LayerInputs, tau: float, gpu_fold: np.ndarray, rows=None):
    """Run the oracle; rows within NEAR_TAU of tau take the GPU's decision
    (spec rule: such rows are reported and excluded from decision
    parity).  Returns (oracle result, number of near-tau rows, mismatches
    outside the near-tau band)."""
    d = inp.dims
    B, L, _ = inp.H.shape
    f0, rel = orc.gate(inp.H, inp.parent, np.float32(tau))
    near = orc.near_tau_rows(rel, float(np.float32(tau)), NEAR_TAU)
    gf = gpu_fold.reshape(B, L)
    bad = (gf != f0) & ~near
    force = np.where(near, gf.astype(np.int8), np.int8(-1)).astype(np.int8)
    res = orc.layer_forward(inp.H, inp.parent, inp.weights, inp.prefix.K, inp.prefix.V, float(np.float32(tau)),
                            d.eps, d.n_kv, d.hd, force=force, rows=rows)
    return res, int(near.sum()), int(bad.sum())
