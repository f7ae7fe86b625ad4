"""Write the oracle regression fixture for the tiny fp32 workload.

Calls only the oracle (and the seeded input generator).  The fixture guards
the oracle against unintended changes; it is not an independent pin (those
are in test_oracle_pins.py).  Run from the repository root:

    python tests/golden/make_golden.py
"""
import json
import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
sys.path.insert(0, ROOT)

from oracle import specfold_oracle as orc  # noqa: E402
from diffusion_branch_speculative_gb300 import synth  # noqa: E402


def summary(seed=0, tau=0.05):
    inp = synth.make_layer_inputs("tiny", seed=seed)
    d = inp.dims
    res = orc.layer_forward(inp.H, inp.parent, inp.weights, inp.prefix.K, inp.prefix.V,
                            tau, d.eps, d.n_kv, d.hd)
    out = res["out"]
    return {
        "workload": "tiny", "seed": seed, "tau": tau,
        "parent": [int(x) for x in inp.parent],
        "fold": res["fold"].astype(int).tolist(),
        "src": [int(x) for x in res["src"]],
        "packed_idx": [int(x) for x in res["packed_idx"]],
        "n": int(res["n"]),
        "out_row_sums": [float(x) for x in out.sum(axis=1)],
        "out_first8_row0": [float(x) for x in out[0, :8]],
    }


if __name__ == "__main__":
    path = os.path.join(os.path.dirname(os.path.abspath(__file__)), "tiny_oracle_seed0.json")
    with open(path, "w") as f:
        json.dump(summary(), f, indent=1)
    print("wrote", path)
