"""Benchmark: verified branch-tokens/s of the folded verification layer.

One step = one folded-layer call (gate, resolve, pack + RMSNorm1, QKV, folded
attention, output projection + RMSNorm2, SwiGLU, down projection, fold-fill),
replayed as the library's CUDA graph of specfold_layer_forward
over one batch of B branches x L block tokens, on the 7B-like single-layer
workload: d 3584, 28/4 heads x 128, SwiGLU 18944, prefix 512, L 32, 8
branches on a depth-3 directed draft graph, seeded synthetic inputs.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--tau T] [--impl ours|reference]

Prints one JSON line (rank 0).  value = B*L*steps*N / (max over ranks of the
summed device time of the K steps), inputs resident in HBM; L2 is flushed
between steps (a 256 MiB write, then a 256 MiB read so the written lines are
evicted too), outside the timed events.  e2e = the same
metric through the public API with pinned host buffers, including the
host->device copy of H_in/parent and the device->host copy of H_out.
--impl reference times the CPU oracle on this host's cores instead.
Multi-GPU: independent replicas, one per rank (no data-path collective).
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402

METRIC = "verified branch-tokens/s per layer"
UNIT = "branch-tokens/s"
FLUSH_BYTES = 256 << 20
PEAKS_FALLBACK = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0}


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default="7b_layer")
    ap.add_argument("--tau", type=float, default=0.05)
    ap.add_argument("--frac", type=float, default=None, help="forced recompute fraction (stress workload)")
    ap.add_argument("--seed", type=int, default=0)
    ap.add_argument("--no-sweep", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-stress", action="store_true", help="skip the stress-workload recompute-fraction sweep")
    ap.add_argument("--no-budget", action="store_true", help="skip the draft-budget sweep")
    ap.add_argument("--no-stack", action="store_true", help="skip the 28-layer stack tau sweep")
    ap.add_argument("--no-3b", action="store_true", help="skip the 3B-class layer leg")
    ap.add_argument("--no-gate-pack", action="store_true", help="skip the fused gate/pack size sweep")
    return ap.parse_args()


def workload_desc(w, tau, frac=None):
    d = w.dims
    s = (f"{w.name}: d={d.d} heads={d.n_q}/{d.n_kv}x{d.hd} ffn={d.F} P={w.P} L={w.L} B={w.B} "
         f"levels={'/'.join(map(str, w.levels))} tau={tau}")
    if frac is not None:
        s += f" forced_frac={frac}"
    return s


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            p = json.load(f)
        return {"hbm_gbs": float(p["hbm_gbs"]), "bf16_tflops": float(p["bf16_tflops"]), "src": "measured"}
    except Exception:
        return dict(PEAKS_FALLBACK, src="fallback")


# ------------------------------------------------------------------ clocks --
class ClockSampler:
    """nvidia-smi clock/throttle samples while the timed region runs."""
    Q = ("timestamp,index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None
        self.lines = []

    def start(self):
        try:
            self.proc = subprocess.Popen(["nvidia-smi", f"--id={self.index}", f"--query-gpu={self.Q}",
                                          "--format=csv,noheader,nounits", "-lms", "100"],
                                         stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.t = threading.Thread(target=self._read, daemon=True)
            self.t.start()
        except Exception:
            self.proc = None

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append((time.time(), line.strip()))

    def stop(self, t0, t1):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        rows = [l for (t, l) in self.lines if t0 - 0.15 <= t <= t1 + 0.15] or [l for _, l in self.lines[-5:]]
        sm, mx, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for l in rows:
            f = [x.strip() for x in l.split(",")]
            try:
                sm.append(float(f[2]))
                mx = float(f[3])
                for nm, v in zip(names, f[6:10]):
                    if v.lower().startswith("active"):
                        reasons.add(nm)
            except (ValueError, IndexError):
                continue
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": mx, "reasons": sorted(reasons), "samples": len(sm)}


# ---------------------------------------------------------- roofline data --
def kernel_source_hash():
    h = hashlib.sha256()
    for f in ("gemm_tc.cu", "sf_device.cuh"):
        with open(os.path.join(ROOT, "diffusion_branch_speculative_gb300", "csrc", f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


def committed_traffic(kernel: str, workload: str):
    """dram bytes per launch from a committed ncu summary, if it was taken on
    the current kernel source (profiles/<kernel>__<workload>.md)."""
    path = os.path.join(ROOT, "profiles", f"{kernel}__{workload}.md")
    try:
        txt = open(path).read()
    except OSError:
        return None
    vals = {}
    for line in txt.splitlines():
        if ":" in line and line.strip().startswith("- "):
            k, v = line.strip()[2:].split(":", 1)
            vals[k.strip()] = v.strip().strip("`")
    if vals.get("kernel_source_sha") != kernel_source_hash():
        return None
    try:
        return float(vals["dram_bytes_per_launch"])
    except (KeyError, ValueError):
        return None


def stage_roofline(name, dims, n, R, us, peaks):
    """Algorithmic work of one launch of a stage and its bound."""
    d, F, e = dims.d, dims.F, 2
    nq, nkv = dims.n_q * dims.hd, dims.n_kv * dims.hd
    if name == "gate_up":
        flops = 2.0 * n * d * 2 * F
        byts = 2 * F * d * e + n * d * e + n * F * e
    elif name == "down":
        flops = 2.0 * n * F * d
        byts = d * F * e + n * F * e + 2 * n * d * e + n * 4
    elif name == "qkv":
        flops = 2.0 * n * d * (nq + 2 * nkv)
        byts = (nq + 2 * nkv) * d * e + n * d * e + n * (nq + 2 * nkv) * e
    elif name == "out_proj_norm":
        flops = 2.0 * n * nq * d
        byts = d * nq * e + n * nq * e + 2 * n * d * e
    else:
        return None
    t = us * 1e-6
    t_mem = byts / (peaks["hbm_gbs"] * 1e9)
    t_tc = flops / (peaks["bf16_tflops"] * 1e12)
    if t_mem >= t_tc:
        a = byts / t / 1e9
        return {"bound": "hbm", "achieved": round(a, 1), "peak": peaks["hbm_gbs"], "unit": "GB/s",
                "frac": round(a / peaks["hbm_gbs"], 4), "algorithmic_bytes": int(byts)}
    a = flops / t / 1e12
    return {"bound": "tensor", "achieved": round(a, 1), "peak": peaks["bf16_tflops"], "unit": "TFLOP/s",
            "frac": round(a / peaks["bf16_tflops"], 4), "algorithmic_flops": flops}


# ------------------------------------------------------ replica plumbing ----
def reduce_max(value: float, world: int, device: str = "cuda") -> float:
    """Max of one float over the ranks (one all-reduce); the value itself on
    one rank.  device "cuda" for NCCL, "cpu" for gloo."""
    if world <= 1:
        return value
    import torch
    import torch.distributed as dist
    t = torch.tensor([value], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def aggregate_rate(units_per_step: int, steps: int, world: int, total_ms_max: float) -> float:
    """Whole-job throughput of N replicas: every rank processed units_per_step
    per step; the job took the slowest rank's time."""
    return units_per_step * steps * world / (total_ms_max * 1e-3)


# ------------------------------------------------------------- our arm ----
def run_ours(args, rank, world):
    import torch

    from diffusion_branch_speculative_gb300 import binding, synth

    dev_index = int(os.environ.get("LOCAL_RANK", "0"))
    torch.cuda.set_device(dev_index)
    w = synth.WORKLOADS[args.workload]
    inp = synth.make_layer_inputs(w, seed=args.seed + rank, forced_frac=args.frac)
    d = inp.dims
    B, L, D = inp.H.shape
    R = B * L
    dims = binding.make_dims(d.d, d.n_q, d.n_kv, d.hd, d.F, d.eps, binding.BF16)
    to = lambda a: torch.from_numpy(np.ascontiguousarray(a, np.float32)).cuda().to(torch.bfloat16)
    H = to(inp.H)
    parent = torch.from_numpy(inp.parent.astype(np.int32)).cuda()
    W = {k: to(v) for k, v in inp.weights.items()}
    cache = to(inp.prefix.cache)
    o, P = inp.prefix.offset, inp.prefix.P
    pk, pv = (cache[o:o + P, 0], cache[o:o + P, 1]) if P else (None, None)
    lay = binding.FoldedLayer(dims, W, B, L, pk, pv)
    Hout = torch.empty_like(H)
    flush_w = torch.empty(FLUSH_BYTES, dtype=torch.uint8, device="cuda")
    flush_r = torch.ones(FLUSH_BYTES // 4, dtype=torch.float32, device="cuda")

    def flush():
        # write a buffer larger than L2, then read another one so the dirty
        # lines of the first are written back before the timed region starts
        flush_w.zero_()
        flush_r.sum()
    stream = torch.cuda.current_stream()
    peaks = load_peaks()

    def barrier():
        if world > 1:
            import torch.distributed as dist
            dist.barrier()

    def timed_steps(tau, steps, warmup, stage_events=False, only=None):
        """K replays of the layer's CUDA graph, L2 flushed before each.

        Without stage events the step is bracketed by events recorded on the
        stream around the graph launch (the flush ahead of it keeps the GPU
        busy while the host submits).  With stage events the graph itself
        carries event-record nodes at every stage boundary, for the per-stage
        breakdown."""
        ev = None
        if stage_events:
            ev = [torch.cuda.Event(enable_timing=True) for _ in range(binding.STAGE_EVENTS)]
            for e in ev:  # torch creates the CUDA event at its first record
                e.record(stream)
        if only is not None:  # just the boundaries around one stage
            ev = [e if i in (only, only + 1) else None for i, e in enumerate(ev)]
        graph = lay.graph(H, parent, tau, Hout, events=ev)
        for _ in range(warmup):
            flush()
            graph.launch()
        torch.cuda.synchronize()
        barrier()
        torch.cuda.synchronize()
        l0 = binding.specfold_launch_count()
        t0 = time.time()
        ms = []
        st_sum = [0.0] * (binding.STAGE_EVENTS - 1)
        a = torch.cuda.Event(enable_timing=True)
        b = torch.cuda.Event(enable_timing=True)
        for i in range(steps):
            flush()
            if stage_events and only is not None:
                graph.launch()
                ev[only + 1].synchronize()
                st_sum[only] += ev[only].elapsed_time(ev[only + 1])
            elif stage_events:
                graph.launch()
                ev[-1].synchronize()
                ms.append(ev[0].elapsed_time(ev[-1]))
                for si in range(binding.STAGE_EVENTS - 1):
                    st_sum[si] += ev[si].elapsed_time(ev[si + 1])
            else:
                a.record(stream)
                graph.launch()
                b.record(stream)
                b.synchronize()
                ms.append(a.elapsed_time(b))
        torch.cuda.synchronize()
        barrier()
        t1 = time.time()
        launches = binding.specfold_launch_count() - l0
        graph.close()
        stages = {nm: st_sum[si] / steps * 1e3 for si, nm in enumerate(binding.STAGE_NAMES)} if stage_events else None
        if only is not None:
            stages = {binding.STAGE_NAMES[only]: st_sum[only] / steps * 1e3}
        return sum(ms), ms, launches, stages, (t0, t1)

    # headline: tau from the command line, stage events on
    sampler = ClockSampler(dev_index)
    sampler.start()
    time.sleep(0.3)
    total_ms, ms, launches, _, (t0, t1) = timed_steps(args.tau, args.steps, args.warmup)
    clocks = sampler.stop(t0, t1)
    # per-stage breakdown (graph with event-record nodes at stage boundaries)
    _, _, _, stages, _ = timed_steps(args.tau, max(50, min(args.steps, 500)), 5, stage_events=True)
    st = lay.status()
    assert st == 0, f"device status {st:#x}: {binding.timeout_sites(st)}"
    n = lay.n_packed()
    total_ms_max = reduce_max(total_ms, world)
    value = aggregate_rate(B * L, args.steps, world, total_ms_max)

    # dominant kernel of the step
    gemm_stages = ("qkv", "out_proj_norm", "gate_up", "down")
    top = max(stages, key=stages.get)
    rf = stage_roofline(top, d, n, R, stages[top], peaks) if top in gemm_stages else None
    if rf is None:
        top = max(gemm_stages, key=lambda s: stages[s])
        rf = stage_roofline(top, d, n, R, stages[top], peaks)
    # re-time that stage with event nodes only at its two boundaries (each
    # event node in a graph costs microseconds of its own)
    only = binding.STAGE_NAMES.index(top)
    _, _, _, st_top, _ = timed_steps(args.tau, max(50, min(args.steps, 500)), 5, stage_events=True, only=only)
    rf = stage_roofline(top, d, n, R, st_top[top], peaks)
    rf["kernel"] = f"gemm_kernel ({top})"
    rf["us_per_launch"] = round(st_top[top], 2)
    rf["peak_src"] = f"{peaks['src']} ({'MEASURED_PEAKS.json burst' if peaks['src'] == 'measured' else 'recipe fallback'})"
    rf["traffic"] = committed_traffic(f"gemm_{top}", args.workload)
    rf["stage_share"] = round(stages[top] / sum(stages.values()), 3)

    # e2e through the public API with pinned host buffers.  A serving loop:
    # every step copies its inputs in from pinned host memory, runs the
    # layer and copies the output back; two buffer sets and three streams
    # let step i+1's input copy and step i-1's output copy overlap step i's
    # layer.  No L2 flush here: the layer's weights (466 MB for the 7B
    # layer) are larger than L2, so every step streams them from HBM.
    NBUF = 2
    H_host = torch.empty(H.shape, dtype=torch.bfloat16, pin_memory=True)
    H_host.copy_(H.cpu())
    par_host = parent.cpu().pin_memory()
    out_host = [torch.empty(H.shape, dtype=torch.bfloat16, pin_memory=True) for _ in range(NBUF)]
    H_e = [torch.empty_like(H) for _ in range(NBUF)]
    par_e = [torch.empty_like(parent) for _ in range(NBUF)]
    out_e = [torch.empty_like(H) for _ in range(NBUF)]
    for j in range(NBUF):
        H_e[j].copy_(H)
        par_e[j].copy_(parent)
    graphs = [lay.graph(H_e[j], par_e[j], args.tau, out_e[j]) for j in range(NBUF)]
    s_in, s_out = torch.cuda.Stream(), torch.cuda.Stream()
    ev_in = [torch.cuda.Event() for _ in range(NBUF)]
    ev_comp = [torch.cuda.Event() for _ in range(NBUF)]
    ev_out = [torch.cuda.Event() for _ in range(NBUF)]
    for e in ev_in + ev_comp + ev_out:
        e.record(stream)
    torch.cuda.synchronize()

    def e2e_run(steps):
        t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        t0.record(s_in)
        for i in range(steps):
            j = i % NBUF
            with torch.cuda.stream(s_in):
                s_in.wait_event(ev_comp[j])           # buffer j's last layer has read its input
                H_e[j].copy_(H_host, non_blocking=True)
                par_e[j].copy_(par_host, non_blocking=True)
                ev_in[j].record(s_in)
            stream.wait_event(ev_in[j])
            stream.wait_event(ev_out[j])               # buffer j's last output has been read out
            graphs[j].launch(stream)
            ev_comp[j].record(stream)
            with torch.cuda.stream(s_out):
                s_out.wait_event(ev_comp[j])
                out_host[j].copy_(out_e[j], non_blocking=True)
                ev_out[j].record(s_out)
        s_out.wait_event(ev_out[(steps - 1) % NBUF])
        t1.record(s_out)
        torch.cuda.synchronize()
        return t0.elapsed_time(t1)

    e2e_steps = max(NBUF, min(args.steps, 500))
    e2e_run(3 * NBUF)
    barrier()
    e_total = e2e_run(e2e_steps)
    for g in graphs:
        g.close()
    e_total = reduce_max(e_total, world)
    for j in range(NBUF):
        assert torch.equal(out_host[j].cuda(), Hout), "e2e output differs from the resident run"
    e2e = {"value": round(aggregate_rate(B * L, e2e_steps, world, e_total), 1), "unit": UNIT,
           "h2d_bytes_per_step": int(H.numel() * 2 + parent.numel() * 4),
           "d2h_bytes_per_step": int(Hout.numel() * 2), "steps": e2e_steps,
           "loop": f"{NBUF} buffer sets, input copy / layer / output copy on three streams, no L2 flush "
                   f"(weights > L2)"}
    # the device-only rate under the e2e loop's L2 policy (back-to-back
    # replays, no flush), so e2e is compared like with like
    g_nf = lay.graph(H, parent, args.tau, Hout)
    for _ in range(3):
        g_nf.launch()
    torch.cuda.synchronize()
    barrier()
    ea, eb = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    ea.record(stream)
    for _ in range(e2e_steps):
        g_nf.launch()
    eb.record(stream)
    eb.synchronize()
    nf_ms = reduce_max(ea.elapsed_time(eb), world)
    g_nf.close()
    e2e["device_no_flush"] = {"value": round(aggregate_rate(B * L, e2e_steps, world, nf_ms), 1),
                              "us_per_step": round(nf_ms / e2e_steps * 1e3, 2),
                              "note": "the same replays with inputs resident and no copies, back to back (no L2 "
                                      "flush), the e2e loop's L2 policy"}

    # recompute-fraction sweep (tau = 0 is the dense multi-branch verify)
    sweep = []
    if not args.no_sweep:
        for tau in ([0.0] + list(w.taus)):
            steps_s = max(50, min(args.steps, 300))
            tot, _, _, _, _ = timed_steps(tau, steps_s, 5)
            _, _, _, st, _ = timed_steps(tau, steps_s, 5, stage_events=True)
            nn = lay.n_packed()
            sweep.append({"tau": tau, "gate_ref": "parent", "n_packed": nn, "rho": round(nn / R, 4),
                          "us_per_step": round(tot / steps_s * 1e3, 2),
                          "tokens_per_s": round(R * steps_s / (tot * 1e-3), 1),
                          "stages_us": {k: round(v, 2) for k, v in st.items()}})
        dense = next(s for s in sweep if s["tau"] == 0.0)["us_per_step"]
        for s in sweep:
            s["time_vs_dense"] = round(s["us_per_step"] / dense, 4)
        # variant readings on the same layer: the gate against the parent's
        # computed source; folded rows' attention matched again against their
        # own branch; a gate of its own for the FFN sublayer
        variants = [("source", 1, 0, 0), ("parent", 0, 1, 0), ("parent", 0, 0, 1), ("parent", 0, 1, 1)]
        for ref, gref, rematch, fgate in variants:
            vdims = binding.make_dims(d.d, d.n_q, d.n_kv, d.hd, d.F, d.eps, binding.BF16, 0.0, gref, rematch, fgate)
            vlay = binding.FoldedLayer(vdims, W, B, L, pk, pv)
            vout = torch.empty_like(H)
            for tau in w.taus:
                g = vlay.graph(H, parent, tau, vout)
                for _ in range(3):
                    flush()
                    g.launch()
                torch.cuda.synchronize()
                ea, eb = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                steps_s = max(50, min(args.steps, 300))
                tot = 0.0
                for _ in range(steps_s):
                    flush()
                    ea.record(stream)
                    g.launch()
                    eb.record(stream)
                    eb.synchronize()
                    tot += ea.elapsed_time(eb)
                g.close()
                nn = vlay.n_packed()
                row = {"tau": tau, "gate_ref": ref, "n_packed": nn, "rho": round(nn / R, 4),
                       "us_per_step": round(tot / steps_s * 1e3, 2),
                       "tokens_per_s": round(R * steps_s / (tot * 1e-3), 1),
                       "time_vs_dense": round(tot / steps_s * 1e3 / dense, 4)}
                if rematch or fgate:
                    row["attn_rematch"] = rematch
                    row["ffn_gate"] = fgate
                    row["n_ffn"] = int(vlay.view("n_ffn", torch.int32)[0].item())
                sweep.append(row)
            assert vlay.status() == 0, "device status set"
            del vlay
    budget = [] if (args.no_budget or args.workload != "7b_layer") else budget_sweep(args, lay.dims, W, pk, pv, flush,
                                                                                       barrier)
    leg3b = None if (args.no_3b or args.workload != "7b_layer") else layer_leg(args, "3b_layer", flush, barrier)
    gp = None if (args.no_gate_pack or args.workload != "7b_layer") else gate_pack_sweep(args, flush, barrier)
    stress = [] if args.no_stress else stress_sweep(args, flush, barrier)
    del lay
    torch.cuda.empty_cache()
    stack = None if args.no_stack else stack_sweep(args, flush, barrier)
    return {
        "gate_pack_sweep": gp,
        "layer_3b": leg3b,
        "stack_sweep": stack,
        "budget_sweep": budget,
        "stress_sweep": stress,
        "value": value, "ms_per_step": total_ms_max / args.steps, "n_packed": n, "R": R, "w": w,
        "stages": stages, "roofline": rf, "e2e": e2e, "gpu_launches": launches, "clocks": clocks,
        "sweep": sweep, "inp": inp,
    }


# Draft graphs of growing budget for the 7B-like layer (level sizes; node 0 is
# the main branch).
BUDGET_LEVELS = {4: ((1, 1, 2), None), 8: ((1, 2, 3, 2), None), 16: ((1, 4, 11), 4),
                 32: ((1, 4, 6, 6, 6, 5, 4), None), 64: ((1, 8, 55), 8)}


def budget_sweep(args, dims, W, pk, pv, flush, barrier):
    """µs per verify step against the draft budget B (the explainer's Fig. 3
    question): the same 7B-like layer (prefix 512, L 32) over B branches,
    dense (tau = 0, every branch fully recomputed) and folded (tau = 0.05)."""
    import torch

    from diffusion_branch_speculative_gb300 import binding, synth
    base = synth.WORKLOADS["7b_layer"]
    to = lambda a: torch.from_numpy(np.ascontiguousarray(a, np.float32)).cuda().to(torch.bfloat16)
    stream = torch.cuda.current_stream()
    steps = max(20, min(args.steps, 200))
    rows = []
    for B, (levels, fanout) in BUDGET_LEVELS.items():
        w = synth.Workload(f"7b_budget{B}", base.dims, P=base.P, L=base.L, levels=levels, max_fanout=fanout,
                           second_parent=True, reveals=base.reveals, ripple_len=base.ripple_len, taus=(0.05,),
                           dtype="bf16")
        br = synth.make_branches(w, np.random.default_rng(args.seed + B))
        H = to(br.H)
        parent = torch.from_numpy(br.graph.parent.astype(np.int32)).cuda()
        out = torch.empty_like(H)
        lay = binding.FoldedLayer(dims, W, B, base.L, pk, pv)
        row = {"B": B}
        for tau, key in ((0.0, "dense"), (0.05, "folded")):
            g = lay.graph(H, parent, tau, out)
            for _ in range(3):
                flush()
                g.launch()
            torch.cuda.synchronize()
            barrier()
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            tot = 0.0
            for _ in range(steps):
                flush()
                a.record(stream)
                g.launch()
                b.record(stream)
                b.synchronize()
                tot += a.elapsed_time(b)
            g.close()
            row[f"{key}_us"] = round(tot / steps * 1e3, 2)
            if key == "folded":
                row["n_packed"] = lay.n_packed()
                row["rho"] = round(row["n_packed"] / (B * base.L), 4)
        row["folded_vs_dense"] = round(row["folded_us"] / row["dense_us"], 4)
        rows.append(row)
        del lay
    return rows


def stage_times(lay, H, parent, tau, out, flush, steps):
    """Mean µs of every stage of one layer call: a graph of the call with an
    event-record node at each stage boundary, replayed `steps` times after
    an L2 flush each."""
    import torch

    from diffusion_branch_speculative_gb300 import binding
    stream = torch.cuda.current_stream()
    ev = [torch.cuda.Event(enable_timing=True) for _ in range(binding.STAGE_EVENTS)]
    for e in ev:  # torch creates the CUDA event at its first record
        e.record(stream)
    g = lay.graph(H, parent, tau, out, events=ev)
    for _ in range(3):
        flush()
        g.launch()
    torch.cuda.synchronize()
    acc = [0.0] * (binding.STAGE_EVENTS - 1)
    for _ in range(steps):
        flush()
        g.launch()
        ev[-1].synchronize()
        for si in range(binding.STAGE_EVENTS - 1):
            acc[si] += ev[si].elapsed_time(ev[si + 1])
    g.close()
    return {nm: acc[si] / steps * 1e3 for si, nm in enumerate(binding.STAGE_NAMES)}


def layer_leg(args, name, flush, barrier):
    """One more single-layer workload (the 3B-class layer: d 3072, 24/8 heads,
    F 8192, prefix 4096, 32 branches): µs per step folded and dense, the
    stage breakdown and each stage against its bound."""
    import torch

    from diffusion_branch_speculative_gb300 import binding, synth
    w = synth.WORKLOADS[name]
    inp = synth.make_layer_inputs(w, seed=args.seed)
    d = inp.dims
    B, L, D = inp.H.shape
    dims = binding.make_dims(d.d, d.n_q, d.n_kv, d.hd, d.F, d.eps, binding.BF16)
    to = lambda a: torch.from_numpy(np.ascontiguousarray(a, np.float32)).cuda().to(torch.bfloat16)
    H = to(inp.H)
    parent = torch.from_numpy(inp.parent.astype(np.int32)).cuda()
    W = {k: to(v) for k, v in inp.weights.items()}
    cache = to(inp.prefix.cache)
    o, P = inp.prefix.offset, inp.prefix.P
    lay = binding.FoldedLayer(dims, W, B, L, cache[o:o + P, 0], cache[o:o + P, 1])
    out = torch.empty_like(H)
    stream = torch.cuda.current_stream()
    peaks = load_peaks()
    steps = max(20, min(args.steps, 200))
    res = {"workload": workload_desc(w, w.taus[0])}
    for tau, key in ((0.0, "dense"), (w.taus[0], "folded")):
        g = lay.graph(H, parent, tau, out)
        for _ in range(5):
            flush()
            g.launch()
        torch.cuda.synchronize()
        barrier()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        tot = 0.0
        for _ in range(steps):
            flush()
            a.record(stream)
            g.launch()
            b.record(stream)
            b.synchronize()
            tot += a.elapsed_time(b)
        g.close()
        res[f"{key}_us"] = round(tot / steps * 1e3, 2)
        if key == "folded":
            nn = lay.n_packed()
            st = stage_times(lay, H, parent, tau, out, flush, max(10, steps // 2))
            res.update({"n_packed": nn, "rho": round(nn / (B * L), 4),
                        "tokens_per_s": round(B * L * steps / (tot * 1e-3), 1),
                        "stages_us": {k: round(v, 2) for k, v in st.items()}})
            res["stage_roofline"] = {nm: stage_roofline(nm, d, nn, B * L, st[nm], peaks)
                                     for nm in ("qkv", "out_proj_norm", "gate_up", "down")}
            att_flops = 4.0 * nn * d.n_q * d.hd * (P + L)
            tf = att_flops / (st["attention"] * 1e-6) / 1e12
            res["stage_roofline"]["attention"] = {"bound": "tensor", "achieved": round(tf, 1),
                                                  "peak": peaks["bf16_tflops"], "unit": "TFLOP/s",
                                                  "frac": round(tf / peaks["bf16_tflops"], 4)}
    res["time_vs_dense"] = round(res["folded_us"] / res["dense_us"], 4)
    st = lay.status()
    assert st == 0, f"device status {st:#x}: {binding.timeout_sites(st)}"
    del lay, W, cache
    torch.cuda.empty_cache()
    return res


# draft graphs for the gate/pack sweep: fanout 8, level sizes summing to B
GATE_PACK_LEVELS = {64: (1, 8, 55), 128: (1, 8, 64, 55), 256: (1, 8, 64, 183), 512: (1, 8, 64, 439)}


def gate_pack_sweep(args, flush, barrier):
    """The fused gate / resolve / pack launch alone (specfold_gate_pack), 7B
    rows (d 3584, bf16), L 32, from the stress size (64 branches, 2048 rows) to
    the row limit (512 branches, 16384 rows): µs per launch from CUDA events
    around single launches after an L2 flush, and the achieved rate of its
    algorithmic bytes (H read once, X1 written for the packed rows, the
    row lists) against the measured copy peak."""
    import torch

    from diffusion_branch_speculative_gb300 import binding, synth
    peaks = load_peaks()
    d = synth.DIMS_7B
    dims = binding.make_dims(d.d, d.n_q, d.n_kv, d.hd, d.F, d.eps, binding.BF16)
    g1 = torch.ones(d.d, dtype=torch.bfloat16, device="cuda")
    stream = torch.cuda.current_stream()
    reps = 30
    rows = []
    for B in (64, 128, 256, 512):
        for frac in ((1.0, 0.25) if B in (64, 512) else (1.0,)):
            w = synth.Workload("gate_pack", d, P=0, L=32, levels=GATE_PACK_LEVELS[B], max_fanout=8,
                               second_parent=False, reveals=(1,), ripple_len=2.0, taus=(0.05,), dtype="bf16")
            br = synth.make_branches(w, np.random.default_rng(args.seed + B), forced_frac=frac)
            H = torch.from_numpy(np.ascontiguousarray(br.H, np.float32)).cuda().to(torch.bfloat16)
            parent = torch.from_numpy(br.graph.parent.astype(np.int32)).cuda()
            R = B * 32
            ws = binding.alloc_workspace(binding.workspace_size(dims, B, 32))
            for _ in range(3):
                binding.specfold_gate_pack(dims, g1, H, parent, 0.05, ws)
            torch.cuda.synchronize()
            barrier()
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            tot = 0.0
            for _ in range(reps):
                flush()
                a.record(stream)
                binding.specfold_gate_pack(dims, g1, H, parent, 0.05, ws)
                b.record(stream)
                b.synchronize()
                tot += a.elapsed_time(b)
            assert binding.specfold_get_status(ws) == 0, "device status set"
            lo = binding.workspace_layout(dims, B, 32)
            n = int(ws[lo.n_packed:lo.n_packed + 4].view(torch.int32).item())
            us = tot / reps * 1e3
            byts = R * d.d * 2 + n * d.d * 2 + 13 * R
            gbs = byts / (us * 1e-6) / 1e9
            rows.append({"B": B, "rows": R, "forced_frac": frac, "n_packed": n, "us": round(us, 2),
                         "algorithmic_bytes": int(byts), "achieved_gbs": round(gbs, 1),
                         "frac_of_hbm_peak": round(gbs / peaks["hbm_gbs"], 4)})
            del H, ws
    torch.cuda.empty_cache()
    return rows


def stress_sweep(args, flush, barrier):
    """µs per verify step against the recompute fraction on the stress
    workload (prefix 8192, 64 branches): forced fractions of non-root rows
    above tau = 0.05, and tau = 0 (dense multi-branch verify) for reference."""
    import torch

    from diffusion_branch_speculative_gb300 import binding, synth
    w = synth.WORKLOADS["stress"]
    base = synth.make_layer_inputs(w, seed=args.seed, forced_frac=0.0)
    d = base.dims
    B, L, D = base.H.shape
    dims = binding.make_dims(d.d, d.n_q, d.n_kv, d.hd, d.F, d.eps, binding.BF16)
    to = lambda a: torch.from_numpy(np.ascontiguousarray(a, np.float32)).cuda().to(torch.bfloat16)
    W = {k: to(v) for k, v in base.weights.items()}
    cache = to(base.prefix.cache)
    o, P = base.prefix.offset, base.prefix.P
    lay = binding.FoldedLayer(dims, W, B, L, cache[o:o + P, 0], cache[o:o + P, 1])
    H = torch.empty(B, L, D, dtype=torch.bfloat16, device="cuda")
    parent = torch.empty(B, dtype=torch.int32, device="cuda")
    out = torch.empty_like(H)
    stream = torch.cuda.current_stream()
    steps = max(20, min(args.steps, 100))
    peaks = load_peaks()
    rows = []
    for frac, tau in [(0.0, 0.0)] + [(f, 0.05) for f in w.forced_fracs]:
        br = synth.make_branches(w, np.random.default_rng(args.seed + 17), forced_frac=frac)
        H.copy_(to(br.H))
        parent.copy_(torch.from_numpy(br.graph.parent.astype(np.int32)))
        g = lay.graph(H, parent, tau, out)
        for _ in range(10):
            flush()
            g.launch()
        torch.cuda.synchronize()
        barrier()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        tot = 0.0
        for _ in range(steps):
            flush()
            a.record(stream)
            g.launch()
            b.record(stream)
            b.synchronize()
            tot += a.elapsed_time(b)
        g.close()
        nn = lay.n_packed()
        stages = stage_times(lay, H, parent, tau, out, flush, max(10, steps // 2))
        row = {"forced_frac": frac if tau > 0 else None, "tau": tau, "n_packed": nn,
               "rho": round(nn / (B * L), 4), "us_per_step": round(tot / steps * 1e3, 2),
               "tokens_per_s": round(B * L * steps / (tot * 1e-3), 1),
               "stages_us": {k: round(v, 2) for k, v in stages.items()}}
        # each GEMM stage and the attention against its bound (stage times come
        # from event nodes in the graph, which add a few microseconds each)
        row["stage_roofline"] = {nm: stage_roofline(nm, d, nn, B * L, stages[nm], peaks)
                                 for nm in ("qkv", "out_proj_norm", "gate_up", "down")}
        att_flops = 4.0 * nn * d.n_q * d.hd * (P + L)
        row["stage_roofline"]["attention"] = {
            "bound": "tensor", "achieved": round(att_flops / (stages["attention"] * 1e-6) / 1e12, 1),
            "peak": peaks["bf16_tflops"], "unit": "TFLOP/s",
            "frac": round(att_flops / (stages["attention"] * 1e-6) / 1e12 / peaks["bf16_tflops"], 4)}
        rows.append(row)
    dense = rows[0]["us_per_step"]
    for r in rows:
        r["time_vs_dense"] = round(r["us_per_step"] / dense, 4)
    del lay, W, cache
    torch.cuda.empty_cache()
    return rows


def stack_sweep(args, flush, barrier):
    """The 28-layer 7B-like stack (prefix 2048, 16 branches in a fanout-4
    tree): one verify step runs every layer, each re-gating on its own input.
    Per tau: µs per step, branch-tokens/s per layer and the recompute fraction
    of every layer (the explainer's appendix D question).  Weights are drawn
    on the device by torch's seeded generator (28 x 466 MB)."""
    import torch

    from diffusion_branch_speculative_gb300 import binding, synth
    w = synth.WORKLOADS["7b_stack"]
    d = w.dims
    dims = binding.make_dims(d.d, d.n_q, d.n_kv, d.hd, d.F, d.eps, binding.BF16)
    weights, caches = synth.torch_stack_params(d, w.n_layers, w.P, seed=args.seed + 101)
    o = synth.PREFIX_OFFSET
    pk = [c[o:o + w.P, 0] for c in caches]
    pv = [c[o:o + w.P, 1] for c in caches]
    br = synth.make_branches(w, np.random.default_rng(args.seed + 29))
    H = torch.from_numpy(np.ascontiguousarray(br.H, np.float32)).cuda().to(torch.bfloat16)
    parent = torch.from_numpy(br.graph.parent.astype(np.int32)).cuda()
    out = torch.empty_like(H)
    stack = binding.FoldedStack(dims, weights, w.B, w.L, pk, pv)
    stream = torch.cuda.current_stream()
    steps = max(10, min(args.steps, 30))
    R = w.B * w.L
    rows = []
    for tau in w.taus:
        g = stack.graph(H, parent, tau, out)
        for _ in range(3):
            flush()
            g.launch()
        torch.cuda.synchronize()
        barrier()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        tot = 0.0
        for _ in range(steps):
            flush()
            a.record(stream)
            g.launch()
            b.record(stream)
            b.synchronize()
            tot += a.elapsed_time(b)
        g.close()
        ns = stack.n_packed.cpu().tolist()
        us = tot / steps * 1e3
        rows.append({"tau": tau, "us_per_step": round(us, 1), "us_per_layer": round(us / w.n_layers, 2),
                     "tokens_per_s_per_layer": round(R * w.n_layers / (us * 1e-6), 1),
                     "rho_mean": round(sum(ns) / (R * w.n_layers), 4),
                     "rho_per_layer": [round(n / R, 4) for n in ns]})
    assert stack.status() == 0, "device status set"
    # depth profile at the command-line tau (one recorded, untimed step): how
    # far the state and the child/parent differences move with depth, and how
    # many rows change decision against layer 0 (released or newly folded)
    stack.forward(H, parent, args.tau, out, record=True)
    torch.cuda.synchronize()
    states = [H] + [stack.hidden[l] for l in range(w.n_layers - 1)]
    par = br.graph.parent
    root_rms, r_med, r_p10, r_p90 = [], [], [], []
    for x in states:
        xf = x.float()
        root_rms.append(round(float(xf[0].pow(2).mean().sqrt()), 3))
        diff = (xf[1:] - xf[torch.from_numpy(par[1:].astype(np.int64)).cuda()]).norm(dim=-1)
        base = xf[torch.from_numpy(par[1:].astype(np.int64)).cuda()].norm(dim=-1)
        r = (diff / base).flatten()
        q = torch.quantile(r, torch.tensor([0.1, 0.5, 0.9], device=r.device))
        r_p10.append(round(float(q[0]), 4))
        r_med.append(round(float(q[1]), 4))
        r_p90.append(round(float(q[2]), 4))
    f0 = stack.fold[0]
    changed = [int((stack.fold[l] != f0).sum()) for l in range(w.n_layers)]
    profile = {"tau": args.tau, "root_rms": root_rms, "r_p10": r_p10, "r_median": r_med, "r_p90": r_p90,
               "rows_changed_vs_layer0": changed}
    dense = rows[0]["us_per_step"] if rows and rows[0]["tau"] == 0.0 else None
    for r in rows:
        r["time_vs_dense"] = round(r["us_per_step"] / dense, 4) if dense else None
    del stack, weights, caches
    torch.cuda.empty_cache()
    return {"taus": rows, "depth_profile": profile}


# -------------------------------------------------------- oracle on CPU ----
def oracle_sample(inp, tau, rows_per_step, steps, budget_s=None):
    """Time the CPU oracle producing `rows_per_step` output rows per step."""
    from oracle import specfold_oracle as orc
    d = inp.dims
    W64 = {k: np.asarray(v, np.float64) for k, v in inp.weights.items()}
    pk = np.asarray(inp.prefix.K, np.float64)
    pv = np.asarray(inp.prefix.V, np.float64)
    H = inp.H.astype(np.float64)
    R = H.shape[0] * H.shape[1]
    rng = np.random.default_rng(7)
    done, t_total = 0, 0.0
    for i in range(steps):
        rows = rng.choice(R, size=rows_per_step, replace=False)
        t0 = time.perf_counter()
        orc.layer_forward(H, inp.parent, W64, pk, pv, float(np.float32(tau)), d.eps, d.n_kv, d.hd, rows=rows)
        t_total += time.perf_counter() - t0
        done += rows_per_step
        if budget_s is not None and t_total > budget_s:
            break
    return done, t_total


def oracle_one_core(workload, tau, seed, frac, budget_s):
    """The oracle timed with every BLAS and OpenMP pool held to one thread,
    in a child process (the pools size themselves when numpy loads)."""
    env = dict(os.environ, OPENBLAS_NUM_THREADS="1", OMP_NUM_THREADS="1", MKL_NUM_THREADS="1",
               BLIS_NUM_THREADS="1", VECLIB_MAXIMUM_THREADS="1")
    code = ("import json, sys; sys.path.insert(0, %r); import bench; "
            "from diffusion_branch_speculative_gb300 import synth; "
            "inp = synth.make_layer_inputs(%r, seed=%d, forced_frac=%r); "
            "done, secs = bench.oracle_sample(inp, %r, 8, 1000, budget_s=%r); "
            "print(json.dumps([done, secs]))") % (ROOT, workload, seed, frac, tau, budget_s)
    try:
        r = subprocess.run([sys.executable, "-c", code], env=env, capture_output=True, text=True, timeout=300)
        done, secs = json.loads(r.stdout.strip().splitlines()[-1])
        return {"value": round(done / secs, 3), "unit": UNIT, "cores": 1, "kind": "oracle",
                "sample": f"{done} seeded output rows (8 per oracle call), numpy float64, one BLAS thread, "
                          f"~{budget_s:.0f} s"}
    except Exception as e:  # reported, not fatal
        return {"unavailable": f"single-core oracle run failed: {type(e).__name__}"}


def main():
    args = parse()
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    if args.impl == "reference":
        if rank != 0:
            return 0
        from diffusion_branch_speculative_gb300 import synth
        w = synth.WORKLOADS[args.workload]
        inp = synth.make_layer_inputs(w, seed=args.seed, forced_frac=args.frac)
        R = w.B * w.L
        from oracle import specfold_oracle as orc
        fold0, _ = orc.gate(inp.H, inp.parent, float(np.float32(args.tau)))
        n_ref = int(orc.pack(fold0)[2])
        rows_per_step = 1
        oracle_sample(inp, args.tau, rows_per_step, max(1, min(args.warmup, 2)))
        done, secs = oracle_sample(inp, args.tau, rows_per_step, args.steps)
        val = done / secs
        print(json.dumps({
            "impl": "reference", "metric": METRIC, "value": round(val, 3), "unit": UNIT, "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(secs / args.steps * 1e3, 3),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": workload_desc(w, args.tau, args.frac), "B": w.B, "L": w.L, "P": w.P,
                       "tau": args.tau, "n_packed": n_ref, "recompute_fraction": round(n_ref / R, 4),
                       "l2": "n/a (CPU)", "parallelism": f"replicas x{args.gpus}"},
            "cpu_baseline": {"value": round(val, 3), "unit": UNIT, "cores": os.cpu_count(), "kind": "oracle",
                             "sample": f"{rows_per_step} seeded output row(s) of the {R}-row step per timed step "
                                       f"(numpy float64, all BLAS threads)"},
            "e2e": {"value": round(val, 3), "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
        }))
        return 0

    if world > 1:
        import torch
        import torch.distributed as dist
        torch.cuda.set_device(int(os.environ.get("LOCAL_RANK", "0")))
        dist.init_process_group("nccl")
    r = run_ours(args, rank, world)
    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        rows_per_step = 8
        done, secs = oracle_sample(r["inp"], args.tau, rows_per_step, 1000, budget_s=15.0)
        cpu = {"value": round(done / secs, 3), "unit": UNIT, "cores": os.cpu_count(), "kind": "oracle",
               "sample": f"{done} seeded output rows ({rows_per_step} per oracle call) of the "
                         f"{r['R']}-row step, numpy float64, all BLAS threads, ~15 s",
               "one_core": oracle_one_core(args.workload, args.tau, args.seed, args.frac, 10.0)}
    if rank == 0:
        w = r["w"]
        line = {
            "metric": METRIC, "value": round(r["value"], 1), "unit": UNIT, "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": round(r["ms_per_step"], 5), "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
            "config": {"workload": workload_desc(w, args.tau, args.frac), "B": w.B, "L": w.L, "P": w.P,
                       "tau": args.tau, "n_packed": r["n_packed"], "recompute_fraction": round(r["n_packed"] / r["R"], 4),
                       "l2": "flushed between steps (256 MiB write + 256 MiB read, outside the timed events)",
                       "parallelism": f"replicas x{world}"},
            "us_per_step": round(r["ms_per_step"] * 1e3, 2),
            "roofline": r["roofline"],
            "cpu_baseline": cpu,
            "e2e": r["e2e"],
            "gpu_launches": r["gpu_launches"],
            "clocks": r["clocks"],
            "stages_us": {k: round(v, 2) for k, v in r["stages"].items()},
            "sweep": r["sweep"],
            "stress_sweep": r["stress_sweep"],
            "budget_sweep": r["budget_sweep"],
            "stack_sweep": r["stack_sweep"],
            "layer_3b": r["layer_3b"],
            "gate_pack_sweep": r["gate_pack_sweep"],
        }
        print(json.dumps(line))
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()
    return 0


if __name__ == "__main__":
    sys.exit(main())
