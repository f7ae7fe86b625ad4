"""Seeded synthetic inputs for the folded multi-branch verification layer.

This module only draws inputs: draft graphs, branch hidden states, weights and a
shared prefix KV cache.  It holds none of the layer's arithmetic (no norm, no
projection, no attention), so the CPU oracle and the CUDA path can both take
their inputs from it without sharing any of the method.

What the inputs stand in for (SpecFold blog post, "observation" and "residual
ripple" paragraphs, Fig. 2): a child branch's layer input is close to its
parent's everywhere except near the positions the child newly revealed; the
difference is large at a revealed position and spreads to its neighbours with
a decay.  The pages measure on trained diffusion LMs over public benchmarks;
none of those are available, so these seeded branches replace them.

All floating-point arrays are returned as float32 holding values that are
exactly representable in the workload's dtype (bf16 values are rounded to
nearest-even once, here), so both sides see bit-identical inputs.
"""
from __future__ import annotations

import dataclasses
import math
from typing import List, Optional, Sequence

import numpy as np


# --------------------------------------------------------------------------
# bf16 rounding (input preparation only)
# --------------------------------------------------------------------------

def round_bf16(x: np.ndarray) -> np.ndarray:
    """Round float values to the nearest bf16 (ties to even); return float32."""
    a = np.ascontiguousarray(x, dtype=np.float32)
    u = a.view(np.uint32).astype(np.uint64)
    lsb = (u >> np.uint64(16)) & np.uint64(1)
    u = (u + np.uint64(0x7FFF) + lsb) >> np.uint64(16)
    out = (u << np.uint64(16)).astype(np.uint32).view(np.float32)
    return out.reshape(a.shape)


def bf16_bits(x: np.ndarray) -> np.ndarray:
    """Upper 16 bits of float32 values that are already bf16-exact."""
    a = np.ascontiguousarray(x, dtype=np.float32)
    return (a.view(np.uint32) >> np.uint32(16)).astype(np.uint16)


# --------------------------------------------------------------------------
# workload descriptions
# --------------------------------------------------------------------------

@dataclasses.dataclass(frozen=True)
class LayerDims:
    d: int            # hidden size
    n_q: int          # query heads
    n_kv: int         # key/value heads
    hd: int           # head dimension
    F: int            # SwiGLU inner width
    eps: float = 1e-6

    @property
    def group(self) -> int:
        return self.n_q // self.n_kv


@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    dims: LayerDims
    P: int                      # shared prefix length
    L: int                      # block length
    levels: Sequence[int]       # draft-graph level sizes (level 0 = root)
    max_fanout: Optional[int]   # cap on children per node (None = no cap)
    second_parent: bool         # record a second parent (ignored by resolve)
    reveals: Sequence[int]      # choices for new reveals per child
    ripple_len: float           # ripple decay length lambda
    taus: Sequence[float]
    dtype: str                  # "bf16" or "f32"
    n_layers: int = 1
    forced_fracs: Sequence[float] = ()

    @property
    def B(self) -> int:
        return int(sum(self.levels))

    @property
    def rows(self) -> int:
        return self.B * self.L


DIMS_TINY = LayerDims(d=256, n_q=4, n_kv=2, hd=64, F=1024)
DIMS_7B = LayerDims(d=3584, n_q=28, n_kv=4, hd=128, F=18944)
DIMS_3B = LayerDims(d=3072, n_q=24, n_kv=8, hd=128, F=8192)

WORKLOADS = {
    # tiny fp32 chain root -> b1 -> b2 -> b3, one reveal per child
    "tiny": Workload("tiny", DIMS_TINY, P=64, L=16, levels=(1, 1, 1, 1), max_fanout=None,
                     second_parent=False, reveals=(1,), ripple_len=2.0, taus=(0.05,), dtype="f32"),
    # 7B-like single layer, 8 branches, depth-3 directed draft graph
    "7b_layer": Workload("7b_layer", DIMS_7B, P=512, L=32, levels=(1, 2, 3, 2), max_fanout=None,
                         second_parent=True, reveals=(1, 2), ripple_len=2.0,
                         taus=(0.02, 0.05, 0.1), dtype="bf16"),
    # 7B-like 28-layer stack, 16 branches, fanout-4 tree
    "7b_stack": Workload("7b_stack", DIMS_7B, P=2048, L=32, levels=(1, 4, 11), max_fanout=4,
                         second_parent=False, reveals=(1,), ripple_len=2.0,
                         taus=(0.0, 0.025, 0.05, 0.075, 0.1, 0.125, 0.15, 0.175, 0.2),
                         dtype="bf16", n_layers=28),
    # 3B-class layer, 32 branches, depth-6 directed draft graph
    "3b_layer": Workload("3b_layer", DIMS_3B, P=4096, L=32, levels=(1, 4, 6, 6, 6, 5, 4),
                         max_fanout=None, second_parent=True, reveals=(1,), ripple_len=3.0,
                         taus=(0.05,), dtype="bf16"),
    # stress: 7B-like layer, prefix 8192, 64 branches (fanout 8, depth 2), forced fractions
    "stress": Workload("stress", DIMS_7B, P=8192, L=32, levels=(1, 8, 55), max_fanout=8,
                       second_parent=False, reveals=(1,), ripple_len=2.0, taus=(0.05,),
                       dtype="bf16", forced_fracs=(0.0, 0.10, 0.25, 0.50, 1.0)),
}

# Relative size of the forced deltas in the stress workload: well away from
# tau = 0.05 on both sides so no row sits near the threshold.
FORCED_ACTIVE_REL = 0.5
FORCED_QUIET_REL = 1e-3
NOISE_REL = 1e-3
RIPPLE_AMP = 0.3
WEIGHT_STD = 0.02
PREFIX_OFFSET = 8      # the prefix view starts this many tokens into the cache
PREFIX_SLACK = 8       # extra cache tokens after the view


# --------------------------------------------------------------------------
# draft graph
# --------------------------------------------------------------------------

@dataclasses.dataclass
class DraftGraph:
    parent: np.ndarray          # int32 [B], first parent, -1 for the root
    second: np.ndarray          # int32 [B], second parent or -1 (recorded, unused)
    level: np.ndarray           # int32 [B]


def make_graph(levels: Sequence[int], rng: np.random.Generator,
               max_fanout: Optional[int] = None, second_parent: bool = False) -> DraftGraph:
    """Nodes numbered level by level (so parent[b] < b); root is node 0."""
    if levels[0] != 1:
        raise ValueError("level 0 must hold exactly the root")
    B = int(sum(levels))
    parent = np.full(B, -1, np.int32)
    second = np.full(B, -1, np.int32)
    level = np.zeros(B, np.int32)
    prev = [0]
    nxt = 1
    for lv, count in enumerate(levels[1:], start=1):
        cur = []
        kids = {p: 0 for p in prev}
        for _ in range(count):
            cands = [p for p in prev if max_fanout is None or kids[p] < max_fanout]
            if not cands:
                raise ValueError("fanout cap too small for the level sizes")
            p = int(cands[rng.integers(len(cands))])
            kids[p] += 1
            parent[nxt] = p
            level[nxt] = lv
            if second_parent and len(prev) > 1 and rng.random() < 0.5:
                others = [q for q in prev if q != p]
                second[nxt] = int(others[rng.integers(len(others))])
            cur.append(nxt)
            nxt += 1
        prev = cur
    return DraftGraph(parent=parent, second=second, level=level)


# --------------------------------------------------------------------------
# inputs
# --------------------------------------------------------------------------

def _unit_rows(rng: np.random.Generator, n: int, d: int) -> np.ndarray:
    v = rng.standard_normal((n, d))
    return v / np.linalg.norm(v, axis=1, keepdims=True)


def _finish(x: np.ndarray, dtype: str) -> np.ndarray:
    return round_bf16(x) if dtype == "bf16" else np.ascontiguousarray(x, dtype=np.float32)


@dataclasses.dataclass
class BranchInputs:
    H: np.ndarray               # float32 [B, L, d]
    graph: DraftGraph
    revealed: List[set]         # per node: positions revealed so far
    new_reveals: List[List[int]]


def make_branches(w: Workload, rng: np.random.Generator, dtype: Optional[str] = None,
                  forced_frac: Optional[float] = None,
                  identical_children: bool = False,
                  ripple: bool = True, noise: bool = True) -> BranchInputs:
    """Branch hidden states H[B, L, d] on a seeded draft graph.

    Root H ~ N(0, 1).  Child = parent + delta, per position i:
      delta_i = s_i * |H_p[i]| * u_i + 1e-3 * |H_p[i]| * w_i
    with s = 1 at the child's new reveals and 0.3 exp(-dist/lambda) elsewhere
    (dist = distance to the nearest new reveal).  With ``forced_frac`` set,
    exactly round(f * (B-1) * L) seeded non-root rows get |delta| = 0.5 |H_p|
    and the rest 1e-3 |H_p|.  ``identical_children`` makes every child equal
    to its parent; ``ripple=False`` / ``noise=False`` drop those terms.
    """
    dtype = dtype or w.dtype
    d, L = w.dims.d, w.L
    g = make_graph(w.levels, rng, w.max_fanout, w.second_parent)
    B = len(g.parent)
    H = np.zeros((B, L, d), np.float64)
    H[0] = _finish(rng.standard_normal((L, d)), dtype)
    revealed: List[set] = [set()]
    new_rev: List[List[int]] = [[]]
    forced_rows = None
    if forced_frac is not None:
        k = int(round(forced_frac * (B - 1) * L))
        forced_rows = set(int(r) for r in rng.choice((B - 1) * L, size=k, replace=False))
    for b in range(1, B):
        p = int(g.parent[b])
        hp = H[p]
        pn = np.linalg.norm(hp, axis=1)
        free = [i for i in range(L) if i not in revealed[p]]
        R = int(w.reveals[rng.integers(len(w.reveals))])
        R = min(R, len(free))
        new = sorted(int(x) for x in rng.choice(free, size=R, replace=False)) if R else []
        revealed.append(revealed[p] | set(new))
        new_rev.append(new)
        u = _unit_rows(rng, L, d)
        wv = _unit_rows(rng, L, d)
        if identical_children:
            H[b] = hp
            continue
        if forced_rows is not None:
            s = np.array([FORCED_ACTIVE_REL if ((b - 1) * L + i) in forced_rows else FORCED_QUIET_REL
                          for i in range(L)])
            delta = (s * pn)[:, None] * u
        else:
            pos = np.arange(L)
            if new:
                dist = np.min(np.abs(pos[:, None] - np.array(new)[None, :]), axis=1)
            else:
                dist = np.full(L, 10 ** 6)
            s = np.where(dist == 0, 1.0, RIPPLE_AMP * np.exp(-dist / w.ripple_len))
            if not ripple:
                s = np.where(dist == 0, 1.0, 0.0)
            delta = (s * pn)[:, None] * u
            if noise:
                delta = delta + (NOISE_REL * pn)[:, None] * wv
        H[b] = _finish(hp + delta, dtype)
    return BranchInputs(H=H.astype(np.float32), graph=g, revealed=revealed, new_reveals=new_rev)


def make_weights(dims: LayerDims, rng: np.random.Generator, dtype: str = "bf16") -> dict:
    """Layer weights, nn.Linear layout [out, in]; RMSNorm gains are 1.

    Projections are N(0, 0.02) (rounded to the workload dtype).
    """
    d, hq, hkv, F = dims.d, dims.n_q * dims.hd, dims.n_kv * dims.hd, dims.F

    def lin(o, i):
        return _finish(rng.standard_normal((o, i), dtype=np.float32) * np.float32(WEIGHT_STD), dtype)

    return {
        "g1": np.ones(d, np.float32),
        "w_q": lin(hq, d), "w_k": lin(hkv, d), "w_v": lin(hkv, d),
        "w_o": lin(d, hq),
        "g2": np.ones(d, np.float32),
        "w_gate": lin(F, d), "w_up": lin(F, d), "w_down": lin(d, F),
    }


@dataclasses.dataclass
class PrefixCache:
    """A fused KV cache [T, 2, n_kv, hd]; the prefix view is tokens [off, off+P)."""
    cache: np.ndarray
    offset: int
    P: int

    @property
    def K(self) -> np.ndarray:      # [P, n_kv, hd] strided view, no copy
        return self.cache[self.offset:self.offset + self.P, 0]

    @property
    def V(self) -> np.ndarray:
        return self.cache[self.offset:self.offset + self.P, 1]


def make_prefix(dims: LayerDims, P: int, rng: np.random.Generator, dtype: str = "bf16") -> PrefixCache:
    """Shared prefix K/V ~ N(0, s^2), s = 0.02 sqrt(d) (the spread of a
    projected unit-RMS row under N(0, 0.02) weights).  Stored inside a larger
    fused cache so the kernels read it through a strided view."""
    T = P + PREFIX_OFFSET + PREFIX_SLACK
    s = WEIGHT_STD * math.sqrt(dims.d)
    cache = _finish(rng.standard_normal((T, 2, dims.n_kv, dims.hd), dtype=np.float32) * np.float32(s), dtype)
    return PrefixCache(cache=cache, offset=PREFIX_OFFSET, P=P)


@dataclasses.dataclass
class LayerInputs:
    workload: Workload
    dims: LayerDims
    branches: BranchInputs
    weights: dict
    prefix: PrefixCache
    dtype: str

    @property
    def H(self) -> np.ndarray:
        return self.branches.H

    @property
    def parent(self) -> np.ndarray:
        return self.branches.graph.parent


def make_layer_inputs(name_or_workload, seed: int = 0, dtype: Optional[str] = None,
                      forced_frac: Optional[float] = None, P: Optional[int] = None,
                      **branch_kw) -> LayerInputs:
    """Everything one layer call needs, from one seed (numpy default_rng)."""
    w = WORKLOADS[name_or_workload] if isinstance(name_or_workload, str) else name_or_workload
    dtype = dtype or w.dtype
    rng = np.random.default_rng(seed)
    br = make_branches(w, rng, dtype=dtype, forced_frac=forced_frac, **branch_kw)
    wts = make_weights(w.dims, rng, dtype=dtype)
    pre = make_prefix(w.dims, w.P if P is None else P, rng, dtype=dtype)
    return LayerInputs(workload=w, dims=w.dims, branches=br, weights=wts, prefix=pre, dtype=dtype)


def small_workload(d=256, n_q=4, n_kv=2, hd=64, F=512, P=64, L=16, levels=(1, 2, 2),
                   reveals=(1,), ripple_len=2.0, dtype="bf16", second_parent=False,
                   max_fanout=None, name="small") -> Workload:
    """A reduced workload for fast parity cases (several tiles plus ragged tails)."""
    return Workload(name, LayerDims(d=d, n_q=n_q, n_kv=n_kv, hd=hd, F=F), P=P, L=L,
                    levels=tuple(levels), max_fanout=max_fanout, second_parent=second_parent,
                    reveals=tuple(reveals), ripple_len=ripple_len, taus=(0.05,), dtype=dtype)


# --------------------------------------------------------------------------
# stacks of layers
# --------------------------------------------------------------------------

@dataclasses.dataclass
class StackInputs:
    """Inputs of an n-layer stack: the branch states entering layer 0 and,
    per layer, its own weights and prefix cache.  The draft deltas are drawn
    at layer 0 only; deeper layers see whatever the stack propagates."""
    workload: Workload
    dims: LayerDims
    branches: BranchInputs
    weights: List[dict]
    prefixes: List[PrefixCache]
    dtype: str

    @property
    def H(self) -> np.ndarray:
        return self.branches.H

    @property
    def parent(self) -> np.ndarray:
        return self.branches.graph.parent

    @property
    def n_layers(self) -> int:
        return len(self.weights)

    def layer(self, l: int) -> LayerInputs:
        """Layer l's weights and prefix with the layer-0 branch states."""
        return LayerInputs(workload=self.workload, dims=self.dims, branches=self.branches,
                           weights=self.weights[l], prefix=self.prefixes[l], dtype=self.dtype)


def make_stack_inputs(name_or_workload, seed: int = 0, n_layers: Optional[int] = None,
                      dtype: Optional[str] = None, P: Optional[int] = None, **branch_kw) -> StackInputs:
    """A seeded stack: branches, then (weights, prefix) of layer 0, 1, ... from
    one numpy generator, so a one-layer stack draws exactly the inputs of
    make_layer_inputs with the same seed."""
    w = WORKLOADS[name_or_workload] if isinstance(name_or_workload, str) else name_or_workload
    dtype = dtype or w.dtype
    n_layers = w.n_layers if n_layers is None else int(n_layers)
    if n_layers < 1:
        raise ValueError("a stack needs at least one layer")
    rng = np.random.default_rng(seed)
    br = make_branches(w, rng, dtype=dtype, **branch_kw)
    weights, prefixes = [], []
    for _ in range(n_layers):
        weights.append(make_weights(w.dims, rng, dtype=dtype))
        prefixes.append(make_prefix(w.dims, w.P if P is None else P, rng, dtype=dtype))
    return StackInputs(workload=w, dims=w.dims, branches=br, weights=weights, prefixes=prefixes, dtype=dtype)


def torch_stack_params(dims: LayerDims, n_layers: int, P: int, seed: int, device="cuda"):
    """Per-layer bf16 weights and fused prefix caches drawn with torch's own
    seeded generator on ``device`` (same distributions as make_weights /
    make_prefix, nn.Linear layout).  Used where a full-size stack is only timed
    or compared with itself: drawing 28 layers of 7B-class weights with numpy
    takes minutes.  Returns (list of weight dicts, list of caches
    [P + offset + slack, 2, n_kv, hd])."""
    import torch  # local: the numpy generators above do not need torch

    gen = torch.Generator(device=device)
    gen.manual_seed(int(seed))
    d, hq, hkv, F = dims.d, dims.n_q * dims.hd, dims.n_kv * dims.hd, dims.F

    def lin(o, i):
        t = torch.randn((o, i), generator=gen, device=device, dtype=torch.float32)
        return t.mul_(WEIGHT_STD).to(torch.bfloat16)

    ws, caches = [], []
    T = P + PREFIX_OFFSET + PREFIX_SLACK
    s = WEIGHT_STD * math.sqrt(d)
    for _ in range(n_layers):
        ws.append({
            "g1": torch.ones(d, device=device, dtype=torch.bfloat16),
            "w_q": lin(hq, d), "w_k": lin(hkv, d), "w_v": lin(hkv, d), "w_o": lin(d, hq),
            "g2": torch.ones(d, device=device, dtype=torch.bfloat16),
            "w_gate": lin(F, d), "w_up": lin(F, d), "w_down": lin(d, F),
        })
        c = torch.randn((T, 2, dims.n_kv, dims.hd), generator=gen, device=device, dtype=torch.float32)
        caches.append(c.mul_(s).to(torch.bfloat16))
    return ws, caches
