"""CPU oracle for SpecFold's folded multi-branch verification layer.

TEST INFRASTRUCTURE.  Only the test suite, the package smoke check and the
benchmark's CPU-baseline leg may import or run this module; the product path
never does.  It shares no code with the CUDA path: it takes plain numpy arrays
(float32 values, usually bf16-exact) and computes everything in float64 with
numpy, in the order the method is described, with no blocking or fusion.

Sources (all on the SpecFold explainer page, blog.ontle.kr/blog/358, unless
noted):
  * gate      -- "observation" paragraph (Fig. 2): the relative difference
                 |H_child - H_parent| / |H_parent| measured on the layer input;
                 the "mechanism" paragraph: tokens above tau are recomputed.
  * resolve   -- implementation note: the provenance kernel follows fold chains
                 to the parent state that was actually computed.
  * pack      -- "mechanism" paragraph and implementation note: every
                 recomputed (branch, position) of every branch goes into one
                 packed batch that the heavy layer runs on once.
  * attention -- implementation note: FlashAttention-style streaming over the
                 shared prefix cache (zero-copy strided view) plus the branch's
                 own block keys/values; GQA.
  * FFN/fold  -- implementation note and "measure diff -> reuse parent -> keep
                 own diff" sentence; page 4 (iitog.ru, "SpecFold ...до 1,99x",
                 key facts): folded attention and FFN keep the residual hidden
                 states.  Folded rows take out = out_src + (H_in - H_in,src).
  * variants  -- ``layer_forward_sublayers``: the implementation note's
                 correction read literally (folded positions' attention
                 matched again against their own branch's keys and values)
                 and one gate per sublayer.

Readings where the pages are silent or garbled:
  fold iff r < tau (so tau = 0 folds nothing); the comparison is done squared
  (|d|^2 < tau^2 |p|^2) and an all-zero parent row folds only an identical
  child; the gate compares against the first parent of a multi-parent node;
  no positional rotation inside the layer; attention is bidirectional over the
  whole prefix and the branch's own block, never across branches; block keys
  and values of a folded position are those of its resolved source row.

Parity pins: see tests/test_oracle_pins.py (and the *_pins.py files beside it).  The outputs of folded rows are
pinned only by the invariants that define them (I2, I6); their quality against
an unfolded model is an accuracy question the pages leave to task benchmarks,
so that comparison is "parity unpinned" by design.
"""
from __future__ import annotations

import math
from typing import Dict, Iterable, List, Optional

import numpy as np

F64 = np.float64


# ---------------------------------------------------------------------------
# elementwise pieces (textbook definitions)
# ---------------------------------------------------------------------------

def rmsnorm(x: np.ndarray, g: np.ndarray, eps: float) -> np.ndarray:
    """RMSNorm over the last axis: x * g / sqrt(mean(x^2) + eps)."""
    x = np.asarray(x, F64)
    ms = np.mean(x * x, axis=-1, keepdims=True)
    return x * np.asarray(g, F64) / np.sqrt(ms + eps)


def silu(z: np.ndarray) -> np.ndarray:
    """silu(z) = z / (1 + e^-z)."""
    with np.errstate(over="ignore"):
        return z / (1.0 + np.exp(-z))


def softmax_rows(s: np.ndarray) -> np.ndarray:
    m = np.max(s, axis=-1, keepdims=True)
    e = np.exp(s - m)
    return e / np.sum(e, axis=-1, keepdims=True)


# ---------------------------------------------------------------------------
# S1 gate
# ---------------------------------------------------------------------------

def rope(x: np.ndarray, pos, theta: float) -> np.ndarray:
    """Rotary position embedding in the rotate-half convention (the one of the
    Qwen/Llama model families): for j < hd/2 the pair (x[j], x[j + hd/2]) is
    rotated by the angle pos * theta^(-2j/hd).  x [..., hd] (last axis one
    head); pos broadcasts against x[..., 0]."""
    x = np.asarray(x, F64)
    hd = x.shape[-1]
    half = hd // 2
    freq = float(theta) ** (-2.0 * np.arange(half) / hd)
    ang = np.asarray(pos, F64)[..., None] * freq
    c, s = np.cos(ang), np.sin(ang)
    x1, x2 = x[..., :half], x[..., half:]
    return np.concatenate([x1 * c - x2 * s, x2 * c + x1 * s], axis=-1)


def gate(H: np.ndarray, parent: np.ndarray, tau: float,
         force: Optional[np.ndarray] = None):
    """Per (branch b, position i): fold flag and relative difference.

    r(b, i) = |H_b[i] - H_p[i]| / |H_p[i]| with p = parent[b] (first parent).
    Fold iff sum(delta^2) < tau^2 * sum(H_p^2), or the child row is identical
    to its parent row and tau > 0.  Root rows (b = 0) are never folded and get
    r = -1.  ``force`` (int8 [B, L], -1 = no override, 0 = recompute,
    1 = fold) overrides individual non-root decisions.
    Returns (fold bool [B, L], rel float64 [B, L]).
    """
    H = np.asarray(H, F64)
    B, L, _ = H.shape
    tau = float(tau)
    fold = np.zeros((B, L), dtype=bool)
    rel = np.full((B, L), -1.0)
    for b in range(1, B):
        p = int(parent[b])
        delta = H[b] - H[p]
        num = np.sum(delta * delta, axis=1)
        den = np.sum(H[p] * H[p], axis=1)
        with np.errstate(invalid="ignore"):
            below = num < (tau * tau) * den
        below = np.where(np.isnan(below), False, below)
        fold[b] = below | ((num == 0.0) & (tau > 0.0))
        with np.errstate(divide="ignore", invalid="ignore"):
            rel[b] = np.where(den > 0, np.sqrt(num / np.where(den > 0, den, 1.0)),
                              np.where(num == 0, 0.0, np.inf))
    if force is not None:
        force = np.asarray(force)
        if np.any(force[0] >= 0):
            raise ValueError("root rows cannot be forced")
        fold = np.where(force >= 0, force == 1, fold)
    return fold, rel


def gate_source(H: np.ndarray, parent: np.ndarray, tau: float,
                force: Optional[np.ndarray] = None):
    """Variant gate: compare child row (b, i) with the row its parent's
    output at position i actually comes from, s = src(parent[b], i), instead
    of the parent's own input: r = |H_b[i] - H_s[i]| / |H_s[i]|, same fold
    rule as ``gate``.  A fold then never reuses an output whose input is more
    than tau away, however long the chain.  Branches are visited in
    topological order, so src of every parent is known; a forced decision
    (``force``) feeds the later sources too.  Returns (fold, rel) like
    ``gate``."""
    H = np.asarray(H, F64)
    B, L, _ = H.shape
    tau = float(tau)
    fold = np.zeros((B, L), dtype=bool)
    rel = np.full((B, L), -1.0)
    srcb = np.zeros((B, L), dtype=np.int64)   # branch whose row is reused
    frc = None if force is None else np.asarray(force)
    if frc is not None and np.any(frc[0] >= 0):
        raise ValueError("root rows cannot be forced")
    for b in range(1, B):
        p = int(parent[b])
        for i in range(L):
            s = int(srcb[p, i])
            delta = H[b, i] - H[s, i]
            num = float(np.sum(delta * delta))
            den = float(np.sum(H[s, i] * H[s, i]))
            f = (num < (tau * tau) * den) or (num == 0.0 and tau > 0.0)
            if frc is not None and frc[b, i] >= 0:
                f = bool(frc[b, i] == 1)
            fold[b, i] = f
            rel[b, i] = math.sqrt(num / den) if den > 0 else (0.0 if num == 0 else math.inf)
            srcb[b, i] = s if f else b
    return fold, rel


# ---------------------------------------------------------------------------
# S2 resolve
# ---------------------------------------------------------------------------

def resolve(fold: np.ndarray, parent: np.ndarray) -> np.ndarray:
    """src(b, i) = b*L + i if (b, i) is recomputed, else src(parent[b], i).

    Branches come in topological order (parent[b] < b), so every parent's
    sources are known when its children are visited.  Returns int64 [B*L].
    """
    B, L = fold.shape
    src = np.empty(B * L, dtype=np.int64)
    for b in range(B):
        for i in range(L):
            r = b * L + i
            if not fold[b, i]:
                src[r] = r
            else:
                p = int(parent[b])
                src[r] = src[p * L + i]
    return src


def walk_chain(fold: np.ndarray, parent: np.ndarray, b: int, i: int) -> int:
    """The same source, found by walking up one row's own chain."""
    while fold[b, i]:
        b = int(parent[b])
    return b * fold.shape[1] + i


# ---------------------------------------------------------------------------
# S3 pack
# ---------------------------------------------------------------------------

def pack(fold: np.ndarray):
    """Packed batch: recomputed rows r = b*L + i in increasing r (branch-major,
    position-ascending).  Returns (packed_idx int64 [n], slot_of_row int64
    [B*L] with -1 for folded rows, n)."""
    flat = np.asarray(fold).reshape(-1)
    packed = [r for r in range(flat.size) if not flat[r]]
    slot = np.full(flat.size, -1, dtype=np.int64)
    for k, r in enumerate(packed):
        slot[r] = k
    return np.array(packed, dtype=np.int64), slot, len(packed)


# ---------------------------------------------------------------------------
# S4..S10 on the packed rows
# ---------------------------------------------------------------------------

def _w(W: dict, k: str) -> np.ndarray:
    return np.asarray(W[k], F64)


def attention_rows(q_rows: np.ndarray, branch_of_row: np.ndarray, kv_src: np.ndarray,
                   K_rows: Dict[int, np.ndarray], V_rows: Dict[int, np.ndarray],
                   prefK: np.ndarray, prefV: np.ndarray, n_kv: int) -> np.ndarray:
    """Attention for query rows q_rows [m, n_q, hd].

    Row k of branch b attends to every prefix key (shared, one copy) and to the
    L block keys of its own branch, block key j being the K/V of source row
    kv_src[b][j].  No mask inside the block (bidirectional), scale 1/sqrt(hd).
    Returns [m, n_q * hd].
    """
    m, n_q, hd = q_rows.shape
    g = n_q // n_kv
    pk = np.asarray(prefK, F64)
    pv = np.asarray(prefV, F64)
    out = np.zeros((m, n_q, hd))
    for b in np.unique(branch_of_row):
        sel = np.nonzero(branch_of_row == b)[0]
        bk = np.stack([K_rows[int(s)] for s in kv_src[int(b)]])      # [L, n_kv, hd]
        bv = np.stack([V_rows[int(s)] for s in kv_src[int(b)]])
        keys = np.concatenate([pk, bk], axis=0)                      # [P+L, n_kv, hd]
        vals = np.concatenate([pv, bv], axis=0)
        for h in range(n_q):
            hk = h // g
            s = q_rows[sel, h, :] @ keys[:, hk, :].T / math.sqrt(hd)  # [ms, P+L]
            out[sel, h, :] = softmax_rows(s) @ vals[:, hk, :]
    return out.reshape(m, n_q * hd)


def layer_forward(H, parent, W, prefK, prefV, tau, eps, n_kv, hd,
                  force=None, rows: Optional[Iterable[int]] = None, rope_theta: float = 0.0,
                  gate_ref: str = "parent") -> dict:
    """Folded layer over all branches, in the packed order.

    With ``rows`` given, only those output rows are produced (plus what they
    need: their sources, and the block K/V of the sources' branches), so a
    sample of a full-size workload can be checked row by row.

    Returns a dict with gate/resolve/pack results over all rows, and for the
    computed rows (increasing row id, listed in "act_rows"): X1, Q, attnO, A,
    X2, G, out_act; K/V per source row; and "out" for the requested rows
    (in "out_rows" order).

    rope_theta > 0 rotates the queries and the block keys (``rope``, position
    P + i for block position i); the prefix keys are taken as already
    rotated, as a KV cache stores them.  Values are never rotated.

    gate_ref "source" runs the variant gate (``gate_source``) instead.
    """
    H = np.asarray(H, F64)
    B, L, d = H.shape
    fold, rel = (gate_source if gate_ref == "source" else gate)(H, parent, tau, force)
    src = resolve(fold, parent)
    packed_idx, slot, n = pack(fold)
    H2 = H.reshape(B * L, d)
    want = list(range(B * L)) if rows is None else sorted(set(int(r) for r in rows))
    act = sorted({int(src[r]) for r in want})
    kv_src = {b: [int(src[b * L + j]) for j in range(L)] for b in {r // L for r in act}}
    kv_need = sorted({s for b in kv_src for s in kv_src[b]} | set(act))
    g1, g2 = W["g1"], W["g2"]
    wq, wk, wv, wo = _w(W, "w_q"), _w(W, "w_k"), _w(W, "w_v"), _w(W, "w_o")
    wg, wu, wd = _w(W, "w_gate"), _w(W, "w_up"), _w(W, "w_down")
    # S3: RMSNorm1 of recomputed rows
    X1 = {r: rmsnorm(H2[r], g1, eps) for r in kv_need}
    # S4: projections
    Xk = np.stack([X1[r] for r in kv_need])
    Kp = Xk @ wk.T
    Vp = Xk @ wv.T
    P = np.asarray(prefK).shape[0]
    K_rows = {r: Kp[t].reshape(n_kv, hd) for t, r in enumerate(kv_need)}
    if rope_theta > 0:
        K_rows = {r: rope(k, P + r % L, rope_theta) for r, k in K_rows.items()}
    V_rows = {r: Vp[t].reshape(n_kv, hd) for t, r in enumerate(kv_need)}
    Xa = np.stack([X1[r] for r in act])
    Q = Xa @ wq.T
    n_q = Q.shape[1] // hd
    if rope_theta > 0:
        pos = np.array([P + r % L for r in act], F64)[:, None]
        Q = rope(Q.reshape(len(act), n_q, hd), pos, rope_theta).reshape(len(act), n_q * hd)
    # S5: attention over prefix + own branch block
    attnO = attention_rows(Q.reshape(len(act), n_q, hd), np.array([r // L for r in act]),
                           kv_src, K_rows, V_rows, prefK, prefV, n_kv)
    # S6: output projection + residual
    A = H2[act] + attnO @ wo.T
    # S7: RMSNorm2
    X2 = rmsnorm(A, g2, eps)
    # S8: SwiGLU
    G = silu(X2 @ wg.T) * (X2 @ wu.T)
    # S9: down projection + residual
    out_act = A + G @ wd.T
    out_of = {r: out_act[t] for t, r in enumerate(act)}
    # S10: folded rows keep their own residual difference
    out = np.stack([out_of[r] if int(src[r]) == r else
                    out_of[int(src[r])] + (H2[r] - H2[int(src[r])]) for r in want])
    return {
        "fold": fold, "rel": rel, "src": src, "packed_idx": packed_idx, "slot": slot, "n": n,
        "act_rows": np.array(act, dtype=np.int64),
        "X1": np.stack([X1[r] for r in act]), "Q": Q, "K_rows": K_rows, "V_rows": V_rows,
        "attnO": attnO, "A": A, "X2": X2, "G": G, "out_act": out_act,
        "out_rows": np.array(want, dtype=np.int64), "out": out,
    }


# ---------------------------------------------------------------------------
# variant readings of the attention correction and of the gate's scope
# ---------------------------------------------------------------------------

def layer_forward_sublayers(H, parent, W, prefK, prefV, tau, eps, n_kv, hd,
                            attn_rematch: bool = False, ffn_gate: bool = False,
                            force=None, force_ffn=None, rope_theta: float = 0.0,
                            gate_ref: str = "parent") -> dict:
    """The folded layer under two variant readings, over all B*L rows.

    attn_rematch -- the implementation note's correction taken literally:
      "the attention output of a folded position is matched again against
      its branch's own keys and values".  Every folded row (b, i) runs
      attention: its query is its source's query (the row whose state it
      reuses), its keys and values are the prefix plus branch b's own block
      (block key j being the K/V of row src(b, j), as for every row).  Its
      attention sublayer output A = H + attnO W_o^T is therefore its own, and a
      change elsewhere in the branch reaches it (the "ripple" of the paper's
      section 4.4).  Its FFN sublayer stays folded: out = A + (out_s - A_s).
    ffn_gate -- one gate per sublayer: the FFN sublayer has a gate of its own
      on the attention sublayer's output A (same rule, same tau, same
      reference row: the parent, or the source with gate_ref "source"), with
      its own sources and packed list.  Rows it folds take
      out = out_s + (A - A_s), s their FFN source; the others run the FFN on
      their own A.  Without attn_rematch an attention-folded row keeps its
      residual difference through the attention sublayer:
      A = A_s + (H - H_s), s its attention source.

    With both flags off this is the layer of ``layer_forward``:
    out = out_s + (A - A_s) = out_s + (H - H_s) there.  ``force_ffn`` overrides
    FFN-gate decisions like ``force`` does the first gate's.

    Returns the first gate's fold / rel / src / packed_idx / slot / n, its
    computed rows "act_rows" with X1 and Q, K_rows / V_rows, attnO for the
    rows in "attn_rows", A [B*L, d], the FFN gate's fold_ffn / rel_ffn /
    src_ffn / packed_ffn / slot_ffn / n_ffn, X2 and G of the FFN's computed
    rows ("ffn_rows"), and out [B*L, d].
    """
    H = np.asarray(H, F64)
    B, L, d = H.shape
    R = B * L
    gate_fn = gate_source if gate_ref == "source" else gate
    fold, rel = gate_fn(H, parent, tau, force)
    src = resolve(fold, parent)
    packed_idx, slot, n = pack(fold)
    H2 = H.reshape(R, d)
    act = [int(r) for r in packed_idx]
    wq, wk, wv, wo = _w(W, "w_q"), _w(W, "w_k"), _w(W, "w_v"), _w(W, "w_o")
    wg, wu, wd = _w(W, "w_gate"), _w(W, "w_up"), _w(W, "w_down")
    P = np.asarray(prefK).shape[0]
    # attention sublayer inputs of the computed rows
    X1 = rmsnorm(H2[act], W["g1"], eps)
    Q = X1 @ wq.T
    n_q = Q.shape[1] // hd
    Kp = (X1 @ wk.T).reshape(n, n_kv, hd)
    Vp = (X1 @ wv.T).reshape(n, n_kv, hd)
    if rope_theta > 0:
        pos = np.array([P + r % L for r in act], F64)[:, None]
        Q = rope(Q.reshape(n, n_q, hd), pos, rope_theta).reshape(n, n_q * hd)
        Kp = rope(Kp, pos, rope_theta)
    K_rows = {r: Kp[t] for t, r in enumerate(act)}
    V_rows = {r: Vp[t] for t, r in enumerate(act)}
    q_of = {r: Q[t] for t, r in enumerate(act)}
    kv_src = {b: [int(src[b * L + j]) for j in range(L)] for b in range(B)}
    if attn_rematch:
        attn_rows = list(range(R))
        q_rows = np.stack([q_of[int(src[r])] for r in attn_rows]).reshape(R, n_q, hd)
        attnO = attention_rows(q_rows, np.arange(R) // L, kv_src, K_rows, V_rows, prefK, prefV, n_kv)
        A = H2 + attnO @ wo.T
    else:
        attn_rows = act
        attnO = attention_rows(Q.reshape(n, n_q, hd), np.array(act) // L, kv_src, K_rows, V_rows,
                               prefK, prefV, n_kv)
        A = np.zeros((R, d))
        A[act] = H2[act] + attnO @ wo.T
        for r in range(R):
            s = int(src[r])
            if s != r:
                A[r] = A[s] + (H2[r] - H2[s])
    # FFN sublayer
    if ffn_gate:
        fold_f, rel_f = gate_fn(A.reshape(B, L, d), parent, tau, force_ffn)
        src_f = resolve(fold_f, parent)
        packed_f, slot_f, n_f = pack(fold_f)
    else:
        fold_f, rel_f, src_f, packed_f, slot_f, n_f = fold, rel, src, packed_idx, slot, n
    ffn_rows = [int(r) for r in packed_f]
    X2 = rmsnorm(A[ffn_rows], W["g2"], eps)
    G = silu(X2 @ wg.T) * (X2 @ wu.T)
    out = np.zeros((R, d))
    out[ffn_rows] = A[ffn_rows] + G @ wd.T
    for r in range(R):
        s = int(src_f[r])
        if s != r:
            out[r] = out[s] + (A[r] - A[s])
    return {
        "fold": fold, "rel": rel, "src": src, "packed_idx": packed_idx, "slot": slot, "n": n,
        "act_rows": np.array(act, dtype=np.int64), "X1": X1, "Q": Q, "K_rows": K_rows, "V_rows": V_rows,
        "attn_rows": np.array(attn_rows, dtype=np.int64), "attnO": attnO, "A": A,
        "fold_ffn": fold_f, "rel_ffn": rel_f, "src_ffn": src_f, "packed_ffn": packed_f, "slot_ffn": slot_f,
        "n_ffn": n_f, "ffn_rows": np.array(ffn_rows, dtype=np.int64), "X2": X2, "G": G, "out": out,
    }


# ---------------------------------------------------------------------------
# modes used as cross-checks
# ---------------------------------------------------------------------------

def dense_branch_forward(Hb, W, prefK, prefV, eps, n_kv, hd, rope_theta: float = 0.0) -> np.ndarray:
    """Plain pre-norm layer over one branch's L rows with no folding."""
    Hb = np.asarray(Hb, F64)
    L, d = Hb.shape
    x = rmsnorm(Hb, W["g1"], eps)
    q = (x @ _w(W, "w_q").T).reshape(L, -1, hd)
    k = (x @ _w(W, "w_k").T).reshape(L, n_kv, hd)
    if rope_theta > 0:
        pos = np.asarray(prefK).shape[0] + np.arange(L, dtype=F64)[:, None]
        q = rope(q, pos, rope_theta)
        k = rope(k, pos, rope_theta)
    v = (x @ _w(W, "w_v").T).reshape(L, n_kv, hd)
    keys = np.concatenate([np.asarray(prefK, F64), k], axis=0)
    vals = np.concatenate([np.asarray(prefV, F64), v], axis=0)
    n_q = q.shape[1]
    g = n_q // n_kv
    o = np.zeros_like(q)
    for h in range(n_q):
        s = q[:, h, :] @ keys[:, h // g, :].T / math.sqrt(hd)
        o[:, h, :] = softmax_rows(s) @ vals[:, h // g, :]
    A = Hb + o.reshape(L, -1) @ _w(W, "w_o").T
    x2 = rmsnorm(A, W["g2"], eps)
    G = silu(x2 @ _w(W, "w_gate").T) * (x2 @ _w(W, "w_up").T)
    return A + G @ _w(W, "w_down").T


def layer_serialized(H, parent, W, prefK, prefV, tau, eps, n_kv, hd, force=None,
                     rope_theta: float = 0.0, gate_ref: str = "parent") -> np.ndarray:
    """Serialized evaluation: one row at a time, straight from the definition,
    with no packed batch and no scan (the check the SpecFold authors describe
    in their appendix C).  Small inputs only.  Returns out [B, L, d]."""
    H = np.asarray(H, F64)
    B, L, d = H.shape
    fold, _ = (gate_source if gate_ref == "source" else gate)(H, parent, tau, force)
    g1 = W["g1"]
    cache: Dict[int, np.ndarray] = {}

    P = np.asarray(prefK).shape[0]

    def kv_of(r):
        x = rmsnorm(H.reshape(B * L, d)[r], g1, eps)
        k = (x @ _w(W, "w_k").T).reshape(n_kv, hd)
        if rope_theta > 0:
            k = rope(k, P + r % L, rope_theta)
        return (k, (x @ _w(W, "w_v").T).reshape(n_kv, hd))

    def computed_out(b, i):
        r = b * L + i
        if r in cache:
            return cache[r]
        h = H[b, i]
        x = rmsnorm(h, g1, eps)
        q = (x @ _w(W, "w_q").T).reshape(-1, hd)
        if rope_theta > 0:
            q = rope(q, P + i, rope_theta)
        n_q = q.shape[0]
        g = n_q // n_kv
        ks, vs = [], []
        for j in range(L):
            kj, vj = kv_of(walk_chain(fold, parent, b, j))
            ks.append(kj)
            vs.append(vj)
        keys = np.concatenate([np.asarray(prefK, F64), np.stack(ks)], axis=0)
        vals = np.concatenate([np.asarray(prefV, F64), np.stack(vs)], axis=0)
        o = np.zeros((n_q, hd))
        for hh in range(n_q):
            s = keys[:, hh // g, :] @ q[hh] / math.sqrt(hd)
            e = np.exp(s - s.max())
            o[hh] = (e / e.sum()) @ vals[:, hh // g, :]
        a = h + o.reshape(-1) @ _w(W, "w_o").T
        x2 = rmsnorm(a, W["g2"], eps)
        gg = silu(x2 @ _w(W, "w_gate").T) * (x2 @ _w(W, "w_up").T)
        cache[r] = a + gg @ _w(W, "w_down").T
        return cache[r]

    out = np.zeros((B, L, d))
    for b in range(B):
        for i in range(L):
            s = walk_chain(fold, parent, b, i)
            sb, si = divmod(s, L)
            if s == b * L + i:
                out[b, i] = computed_out(b, i)
            else:
                out[b, i] = computed_out(sb, si) + (H[b, i] - H[sb, si])
    return out


def near_tau_rows(rel: np.ndarray, tau: float, frac: float = 1e-4) -> np.ndarray:
    """Non-root rows whose relative difference lies within frac*tau of tau."""
    r = np.asarray(rel)
    m = np.abs(r - tau) <= frac * tau
    m[0, :] = False
    return m


# ---------------------------------------------------------------------------
# stack of layers (SpecFold explainer page, "mechanism" paragraph: automatic
# release; appendix D: how the recompute fraction evolves with depth)
# ---------------------------------------------------------------------------

def stack_forward(H, parent, layers, tau, eps, n_kv, hd, store=None, rope_theta: float = 0.0,
                  gate_ref: str = "parent") -> dict:
    """A stack of folded layers: layer l's output is layer l+1's input.

    ``layers`` is a sequence of (W, prefK, prefV), one per layer.  Each layer
    runs the gate again on its own input (the reading of "automatic release":
    a row folded at layer l is recomputed at layer l+1 once its difference to
    the parent's layer-(l+1) input is no longer below tau).  ``store``, when
    given, is applied to each layer's output before the next layer reads it
    (the storage precision of the hidden states between layers); without it
    the stack runs in float64 throughout.

    Returns the input of every layer ("inputs", [n_layers] arrays [B, L, d]),
    the final output "out", and per layer the gate decisions "fold", the
    relative differences "rel" and the packed-row count "n".
    """
    X = np.asarray(H, F64)
    B, L, d = X.shape
    inputs, folds, rels, ns = [], [], [], []
    for (W, pk, pv) in layers:
        inputs.append(X)
        res = layer_forward(X, parent, W, pk, pv, tau, eps, n_kv, hd, rope_theta=rope_theta, gate_ref=gate_ref)
        folds.append(res["fold"])
        rels.append(res["rel"])
        ns.append(int(res["n"]))
        X = res["out"].reshape(B, L, d)
        if store is not None:
            X = np.asarray(store(X), F64)
    return {"inputs": inputs, "out": X, "fold": folds, "rel": rels, "n": ns}
