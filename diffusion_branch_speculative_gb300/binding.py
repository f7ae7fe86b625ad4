"""Thin Python binding of libspecfold.so (include/specfold.h).

Argument marshalling only: torch tensors are passed by data pointer, the
stream is torch's current CUDA stream, and every step runs in the library's
CUDA kernels.  There is no CPU fallback: if the library is missing, loading
it raises.  Function names match the C entry points.
"""
from __future__ import annotations

import ctypes
import os
import re
from typing import Optional, Sequence

import torch

PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(PKG, "libspecfold.so")
HEADER = os.path.join(os.path.dirname(PKG), "include", "specfold.h")

OK, EINVAL, EALIGN, ECAPACITY, EUNSUPPORTED, ECUDA, EDEVICE = 0, -1, -2, -3, -4, -5, -6
DEV_TIMEOUT, DEV_BAD_PARENT, DEV_BAD_PAGE = 1, 2, 4
DEV_SITE_SHIFT = 8  # with DEV_TIMEOUT: bit DEV_SITE_SHIFT + site names the wait that ran out
DEV_SITES = ("attention loader: Q buffer free", "attention loader: K/V stage free", "attention softmax: S ready",
             "attention softmax: P V before a rescale", "attention softmax: P V before the last P",
             "attention softmax: last P V", "attention MMA: P ready", "attention MMA: Q loaded",
             "attention MMA: K/V loaded", "attention MMA: S buffer free", "attention MMA: accumulators free",
             "GEMM producer: stage free", "GEMM MMA: accumulator free", "GEMM MMA: stage loaded",
             "GEMM epilogue: accumulator ready", "gate/pack: row copies", "gate/pack: gains copy",
             "gate/pack: grid barrier", "timeout probe")


def timeout_sites(status: int) -> list:
    """The waits a device status word says ran out (empty without DEV_TIMEOUT)."""
    if not status & DEV_TIMEOUT:
        return []
    return [nm for i, nm in enumerate(DEV_SITES) if status >> (DEV_SITE_SHIFT + i) & 1]
BF16, F32 = 0, 1
STAGE_EVENTS = 9
STAGE_NAMES = ("gate", "select_pack", "qkv", "attention", "out_proj_norm", "gate_up", "down", "fold_fill")


class SpecfoldError(RuntimeError):
    def __init__(self, code: int, what: str):
        self.code = code
        super().__init__(f"{what}: {code} ({status_string(code)})")


class specfold_dims(ctypes.Structure):
    _fields_ = [("d_model", ctypes.c_int), ("n_q_heads", ctypes.c_int), ("n_kv_heads", ctypes.c_int),
                ("head_dim", ctypes.c_int), ("ffn_dim", ctypes.c_int), ("rms_eps", ctypes.c_float),
                ("dtype", ctypes.c_int), ("rope_theta", ctypes.c_float), ("gate_ref", ctypes.c_int),
                ("attn_rematch", ctypes.c_int), ("ffn_gate", ctypes.c_int)]


class specfold_weights(ctypes.Structure):
    _fields_ = [(k, ctypes.c_void_p) for k in
                ("g1", "w_q", "w_k", "w_v", "w_o", "g2", "w_gate", "w_up", "w_down")]


class specfold_kv_view(ctypes.Structure):
    _fields_ = [("ptr", ctypes.c_void_p), ("token_stride", ctypes.c_int64), ("head_stride", ctypes.c_int64),
                ("block_table", ctypes.c_void_p), ("page_size", ctypes.c_int32), ("num_pages", ctypes.c_int32)]


class specfold_ws_layout(ctypes.Structure):
    _fields_ = [(k, ctypes.c_size_t) for k in
                ("status", "n_packed", "fold", "rel", "src", "packed_idx", "slot_of_row", "dep_rng", "dep_rows", "sync", "x1", "q",
                 "block_k", "block_v", "attn_o", "a", "x2", "g", "q_all", "all_idx", "n_all", "a_all", "fold_ffn",
                 "rel_ffn", "src_ffn", "packed_ffn", "slot_ffn", "n_ffn", "dep_rng_ffn", "dep_rows_ffn",
                 "gemm_scratch", "attn_scratch", "total")]


class specfold_stack_trace(ctypes.Structure):
    _fields_ = [("hidden", ctypes.c_void_p), ("fold", ctypes.c_void_p), ("n_packed", ctypes.c_void_p)]


_P = ctypes.c_void_p
_I = ctypes.c_int
_SIG = {
    "specfold_gate": (_I, [_I, _P, _P, _I, _I, _I, ctypes.c_float, _P, _P, _P]),
    "specfold_gate_source": (_I, [_I, _P, _P, _I, _I, _I, ctypes.c_float, _P, _P, _P]),
    "specfold_resolve": (_I, [_P, _P, _I, _I, _P, _P, _P]),
    "specfold_pack": (_I, [_I, _P, _P, _P, ctypes.c_float, _I, _I, _I, _P, _P, _P, _P, _P]),
    "specfold_qkv": (_I, [_P, _P, _P, _P, _P, _I, _I, _P, _P, _P, _P, ctypes.c_size_t, _P]),
    "specfold_rope": (_I, [_P, _P, _P, _P, _P, _I, _I, _I, _P]),
    "specfold_attention": (_I, [_P, _P, specfold_kv_view, specfold_kv_view, _I, _P, _P, _P, _P, _P, _I, _I,
                                _P, _P, ctypes.c_size_t, _P]),
    "specfold_out_proj": (_I, [_P, _P, _P, _P, _P, _P, _I, _I, _P, _P, ctypes.c_size_t, _P]),
    "specfold_ffn": (_I, [_P, _P, _P, _P, _P, _P, _P, _P, _I, _I, _P, _P, ctypes.c_size_t, _P]),
    "specfold_layer_forward": (_I, [_P, _P, _P, _P, _I, _I, specfold_kv_view, specfold_kv_view, _I,
                                    ctypes.c_float, _P, _P, ctypes.c_size_t, _P, _P]),
    "specfold_linear": (_I, [_I, _P, _P, _I, _I, _I, _P, _P, ctypes.c_size_t, _P]),
    "specfold_linear_noalloc": (_I, [_I, _P, _P, _I, _I, _I, _P, _P]),
    "specfold_workspace_size": (ctypes.c_size_t, [_P, _I, _I]),
    "specfold_linear_workspace_size": (ctypes.c_size_t, [_I, _I]),
    "specfold_workspace_layout": (_I, [_P, _I, _I, _P]),
    "specfold_get_status": (_I, [_P, _P, _P]),
    "specfold_read_n_packed": (_I, [_P, _I, _I, _P, _P, _P]),
    "specfold_status_string": (ctypes.c_char_p, [_I]),
    "specfold_launch_count": (ctypes.c_uint64, []),
    "specfold_selftest_timeout": (_I, [_P, ctypes.c_uint64, _P]),
    "specfold_gate_pack": (_I, [_P, _P, _P, _P, ctypes.c_int, ctypes.c_int, ctypes.c_float, _P, ctypes.c_size_t, _P]),
    "specfold_layer_graph_create": (_I, [_P, _P, _P, _P, _I, _I, specfold_kv_view, specfold_kv_view, _I,
                                         ctypes.c_float, _P, _P, ctypes.c_size_t, _P, _P]),
    "specfold_stack_workspace_size": (ctypes.c_size_t, [_P, _I, _I]),
    "specfold_stack_forward": (_I, [_P, _I, _P, _P, _P, _I, _I, _P, _P, _I, ctypes.c_float, _P, _P, _P,
                                    ctypes.c_size_t, _P]),
    "specfold_stack_graph_create": (_I, [_P, _I, _P, _P, _P, _I, _I, _P, _P, _I, ctypes.c_float, _P, _P, _P,
                                         ctypes.c_size_t, _P]),
    "specfold_graph_launch": (_I, [_P, _P]),
    "specfold_graph_destroy": (_I, [_P]),
}

_lib = None


def lib(path: str = LIB_PATH):
    """Load libspecfold.so (raises if it has not been built)."""
    global _lib
    if _lib is None:
        if not os.path.exists(path):
            raise RuntimeError(f"{path} is missing: build it first (python -m diffusion_branch_speculative_gb300.build)")
        L = ctypes.CDLL(path)
        for name, (res, args) in _SIG.items():
            f = getattr(L, name)
            f.restype = res
            f.argtypes = args
        _lib = L
    return _lib


def header_functions(path: str = HEADER) -> list:
    """Names of the functions include/specfold.h declares."""
    txt = open(path).read()
    return sorted(set(re.findall(r"^\s*(?:int|size_t|uint64_t|const char\*)\s+(specfold_\w+)\s*\(", txt, re.M)))


def status_string(code: int) -> str:
    try:
        return lib().specfold_status_string(code).decode()
    except Exception:  # library not loadable: still give a message
        return "status"


def _check(rc: int, what: str):
    if rc != OK:
        raise SpecfoldError(rc, what)


def _ptr(t: Optional[torch.Tensor]):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream=None):
    s = stream if stream is not None else torch.cuda.current_stream()
    return ctypes.c_void_p(s.cuda_stream)


def dtype_code(t: torch.dtype) -> int:
    if t == torch.bfloat16:
        return BF16
    if t == torch.float32:
        return F32
    raise ValueError(f"unsupported dtype {t}")


def make_dims(d, n_q, n_kv, hd, F, eps=1e-6, dtype=BF16, rope_theta=0.0, gate_ref=0, attn_rematch=0,
              ffn_gate=0) -> specfold_dims:
    """gate_ref 0: the gate compares with the parent; 1: with the parent's
    computed source.  attn_rematch 1: folded rows run attention again (their
    source's query over their own branch's block).  ffn_gate 1: the FFN
    sublayer has a gate of its own on the attention sublayer's output."""
    return specfold_dims(d, n_q, n_kv, hd, F, eps, dtype, rope_theta, gate_ref, int(attn_rematch), int(ffn_gate))


def make_weights(w: dict) -> specfold_weights:
    return specfold_weights(*[ctypes.c_void_p(w[k].data_ptr()) for k in
                              ("g1", "w_q", "w_k", "w_v", "w_o", "g2", "w_gate", "w_up", "w_down")])


class PagedPrefix:
    """A paged prefix K or V: `pool` is [num_pages * page_size, n_kv, hd]
    (unit last stride), `block_table` int32 on the device, P the prefix
    length (the attention reads prefix token t from pool token
    block_table[t // page_size] * page_size + t % page_size)."""

    def __init__(self, pool: torch.Tensor, block_table: torch.Tensor, page_size: int, P: int):
        assert pool.dim() == 3 and pool.stride(2) == 1
        assert pool.shape[0] % page_size == 0
        self.pool, self.block_table, self.page_size, self.P = pool, block_table, int(page_size), int(P)
        self.shape = (self.P,) + tuple(pool.shape[1:])

    def view(self) -> "specfold_kv_view":
        p = self.pool
        return specfold_kv_view(p.data_ptr(), p.stride(0), p.stride(1), self.block_table.data_ptr(), self.page_size,
                                p.shape[0] // self.page_size)


def kv_view(t) -> specfold_kv_view:
    """A [P, n_kv, hd] strided view (last dim contiguous), passed without
    copy, or a PagedPrefix."""
    if isinstance(t, PagedPrefix):
        return t.view()
    if t is None or t.numel() == 0:
        return specfold_kv_view(None, 8, 8, None, 0, 0)
    assert t.dim() == 3 and t.stride(2) == 1, "prefix view must be [P, n_kv, hd] with unit last stride"
    return specfold_kv_view(t.data_ptr(), t.stride(0), t.stride(1), None, 0, 0)


def workspace_size(dims: specfold_dims, B: int, L: int) -> int:
    return int(lib().specfold_workspace_size(ctypes.byref(dims), B, L))


def workspace_layout(dims: specfold_dims, B: int, L: int) -> specfold_ws_layout:
    lo = specfold_ws_layout()
    _check(lib().specfold_workspace_layout(ctypes.byref(dims), B, L, ctypes.byref(lo)), "specfold_workspace_layout")
    return lo


def alloc_workspace(nbytes: int, device="cuda") -> torch.Tensor:
    """A zero-filled byte workspace (the library needs it zeroed once)."""
    return torch.zeros(nbytes + 256, dtype=torch.uint8, device=device)[: nbytes]


# ------------------------------------------------------------ entry points --

def specfold_gate(H: torch.Tensor, parent: torch.Tensor, tau: float, fold: torch.Tensor,
                  rel: Optional[torch.Tensor] = None, stream=None):
    B, L, d = H.shape
    _check(lib().specfold_gate(dtype_code(H.dtype), _ptr(H), _ptr(parent), B, L, d, float(tau), _ptr(fold),
                               _ptr(rel), _stream(stream)), "specfold_gate")


def specfold_gate_source(H: torch.Tensor, parent: torch.Tensor, tau: float, fold: torch.Tensor,
                         rel: Optional[torch.Tensor] = None, stream=None):
    B, L, d = H.shape
    _check(lib().specfold_gate_source(dtype_code(H.dtype), _ptr(H), _ptr(parent), B, L, d, float(tau), _ptr(fold),
                                      _ptr(rel), _stream(stream)), "specfold_gate_source")


def specfold_resolve(fold: torch.Tensor, parent: torch.Tensor, B: int, L: int, src: torch.Tensor,
                     status: Optional[torch.Tensor] = None, stream=None):
    _check(lib().specfold_resolve(_ptr(fold), _ptr(parent), B, L, _ptr(src), _ptr(status), _stream(stream)),
           "specfold_resolve")


def specfold_pack(fold, H, g1, eps, packed_idx, slot_of_row, n_dev, X1, stream=None):
    B, L, d = H.shape
    _check(lib().specfold_pack(dtype_code(H.dtype), _ptr(fold), _ptr(H), _ptr(g1), float(eps), B, L, d,
                               _ptr(packed_idx), _ptr(slot_of_row), _ptr(n_dev), _ptr(X1), _stream(stream)),
           "specfold_pack")


def specfold_qkv(dims, weights, X1, packed_idx, n_dev, B, L, Q, blockK, blockV, ws, stream=None):
    _check(lib().specfold_qkv(ctypes.byref(dims), ctypes.byref(weights), _ptr(X1), _ptr(packed_idx), _ptr(n_dev),
                              B, L, _ptr(Q), _ptr(blockK), _ptr(blockV), _ptr(ws), ws.numel(), _stream(stream)),
           "specfold_qkv")


def specfold_rope(dims, Q, blockK, packed_idx, n_dev, B, L, P, stream=None):
    _check(lib().specfold_rope(ctypes.byref(dims), _ptr(Q), _ptr(blockK), _ptr(packed_idx), _ptr(n_dev), B, L, P,
                               _stream(stream)), "specfold_rope")


def specfold_attention(dims, Q, prefK, prefV, P, blockK, blockV, src, packed_idx, n_dev, B, L, O, ws, stream=None):
    _check(lib().specfold_attention(ctypes.byref(dims), _ptr(Q), kv_view(prefK), kv_view(prefV), P, _ptr(blockK),
                                    _ptr(blockV), _ptr(src), _ptr(packed_idx), _ptr(n_dev), B, L, _ptr(O), _ptr(ws),
                                    ws.numel(), _stream(stream)), "specfold_attention")


def specfold_out_proj(dims, weights, O, packed_idx, n_dev, H_in, B, L, A, ws, stream=None):
    _check(lib().specfold_out_proj(ctypes.byref(dims), ctypes.byref(weights), _ptr(O), _ptr(packed_idx),
                                   _ptr(n_dev), _ptr(H_in), B, L, _ptr(A), _ptr(ws), ws.numel(), _stream(stream)),
           "specfold_out_proj")


def specfold_ffn(dims, weights, A, packed_idx, n_dev, H_in, src, fold, B, L, H_out, ws, stream=None):
    _check(lib().specfold_ffn(ctypes.byref(dims), ctypes.byref(weights), _ptr(A), _ptr(packed_idx), _ptr(n_dev),
                              _ptr(H_in), _ptr(src), _ptr(fold), B, L, _ptr(H_out), _ptr(ws), ws.numel(),
                              _stream(stream)), "specfold_ffn")


def specfold_layer_forward(dims, weights, H_in, parent, prefK, prefV, P, tau, H_out, ws,
                           events: Optional[Sequence] = None, stream=None):
    B, L, _ = H_in.shape
    ev = None
    if events is not None:
        assert len(events) == STAGE_EVENTS
        handles = [e.cuda_event for e in events]
        if not all(handles):
            raise ValueError("stage events must exist already (torch creates them at their first record())")
        ev = (ctypes.c_void_p * STAGE_EVENTS)(*handles)
    _check(lib().specfold_layer_forward(ctypes.byref(dims), ctypes.byref(weights), _ptr(H_in), _ptr(parent), B, L,
                                        kv_view(prefK), kv_view(prefV), P, float(tau), _ptr(H_out), _ptr(ws),
                                        ws.numel(), ev, _stream(stream)), "specfold_layer_forward")


def stack_workspace_size(dims: specfold_dims, B: int, L: int) -> int:
    return int(lib().specfold_stack_workspace_size(ctypes.byref(dims), B, L))


def _stack_args(weights: Sequence[specfold_weights], prefK: Sequence, prefV: Sequence):
    n = len(weights)
    if len(prefK) != n or len(prefV) != n:
        raise ValueError("one weight set and one prefix view per layer")
    W = (specfold_weights * n)(*weights)
    K = (specfold_kv_view * n)(*[kv_view(t) for t in prefK])
    V = (specfold_kv_view * n)(*[kv_view(t) for t in prefV])
    return n, W, K, V


def _trace_arg(hidden=None, fold=None, n_packed=None):
    if hidden is None and fold is None and n_packed is None:
        return None
    return specfold_stack_trace(None if hidden is None else hidden.data_ptr(),
                                None if fold is None else fold.data_ptr(),
                                None if n_packed is None else n_packed.data_ptr())


def specfold_stack_forward(dims, weights: Sequence[specfold_weights], H_in, parent, prefK: Sequence,
                           prefV: Sequence, P, tau, H_out, ws, hidden=None, fold=None, n_packed=None, stream=None):
    """weights / prefK / prefV: one entry per layer (specfold_weights structs,
    [P, n_kv, hd] views or None).  hidden / fold / n_packed: optional
    per-layer records (see specfold_stack_trace)."""
    B, L, _ = H_in.shape
    n, W, K, V = _stack_args(weights, prefK, prefV)
    tr = _trace_arg(hidden, fold, n_packed)
    _check(lib().specfold_stack_forward(ctypes.byref(dims), n, W, _ptr(H_in), _ptr(parent), B, L, K, V, P,
                                        float(tau), _ptr(H_out), None if tr is None else ctypes.byref(tr), _ptr(ws),
                                        ws.numel(), _stream(stream)), "specfold_stack_forward")


def specfold_linear(X: torch.Tensor, W: torch.Tensor, Y: torch.Tensor, ws: torch.Tensor, stream=None):
    M, K = X.shape
    N = W.shape[0]
    _check(lib().specfold_linear(dtype_code(X.dtype), _ptr(X), _ptr(W), M, N, K, _ptr(Y), _ptr(ws), ws.numel(),
                                 _stream(stream)), "specfold_linear")


def specfold_linear_noalloc(X: torch.Tensor, W: torch.Tensor, Y: torch.Tensor, stream=None):
    """Y = X W^T without a workspace (the library's static device scratch)."""
    M, K = X.shape
    N = W.shape[0]
    _check(lib().specfold_linear_noalloc(dtype_code(X.dtype), _ptr(X), _ptr(W), M, N, K, _ptr(Y), _stream(stream)),
           "specfold_linear_noalloc")


def linear_workspace_size(M: int, N: int) -> int:
    return int(lib().specfold_linear_workspace_size(M, N))


def specfold_get_status(ws: torch.Tensor, stream=None) -> int:
    v = ctypes.c_uint32(0)
    rc = lib().specfold_get_status(_ptr(ws), ctypes.byref(v), _stream(stream))
    if rc not in (OK, EDEVICE):
        raise SpecfoldError(rc, "specfold_get_status")
    return int(v.value)


def specfold_launch_count() -> int:
    return int(lib().specfold_launch_count())


def specfold_gate_pack(dims: specfold_dims, g1: torch.Tensor, H: torch.Tensor, parent: torch.Tensor, tau: float,
                       ws: torch.Tensor, stream=None):
    B, L, _ = H.shape
    _check(lib().specfold_gate_pack(ctypes.byref(dims), _ptr(g1), _ptr(H), _ptr(parent), B, L, float(tau), _ptr(ws),
                                    ws.numel(), _stream(stream)), "specfold_gate_pack")


def specfold_selftest_timeout(status: torch.Tensor, wait_ns: int, stream=None):
    _check(lib().specfold_selftest_timeout(_ptr(status), int(wait_ns), _stream(stream)), "specfold_selftest_timeout")


class _Graph:
    """A captured call: launch() replays all of its kernels with one graph
    launch.  Inputs are read from, and outputs written to, the buffers given
    at capture."""

    _h = None

    def launch(self, stream=None):
        _check(lib().specfold_graph_launch(self._h, _stream(stream)), "specfold_graph_launch")

    def close(self):
        if self._h:
            torch.cuda.synchronize()
            lib().specfold_graph_destroy(self._h)
            self._h = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


class LayerGraph(_Graph):
    """A captured specfold_layer_forward call (specfold_layer_graph_create)."""

    def __init__(self, dims, weights, H_in, parent, prefK, prefV, P, tau, H_out, ws,
                 events: Optional[Sequence] = None):
        B, L, _ = H_in.shape
        ev = None
        if events is not None:
            if len(events) != STAGE_EVENTS:
                raise ValueError("need SPECFOLD_STAGE_EVENTS entries (None skips a boundary)")
            handles = [None if e is None else e.cuda_event for e in events]
            if not all(h for e, h in zip(events, handles) if e is not None):
                raise ValueError("stage events must exist already (torch creates them at their first record())")
            ev = (ctypes.c_void_p * STAGE_EVENTS)(*handles)
        self._keep = (dims, weights, H_in, parent, prefK, prefV, H_out, ws, events, ev)
        h = ctypes.c_void_p()
        torch.cuda.synchronize()
        _check(lib().specfold_layer_graph_create(ctypes.byref(dims), ctypes.byref(weights), _ptr(H_in), _ptr(parent),
                                                 B, L, kv_view(prefK), kv_view(prefV), P, float(tau), _ptr(H_out),
                                                 _ptr(ws), ws.numel(), ev, ctypes.byref(h)),
               "specfold_layer_graph_create")
        self._h = h


class StackGraph(_Graph):
    """A captured specfold_stack_forward call (specfold_stack_graph_create)."""

    def __init__(self, dims, weights: Sequence[specfold_weights], H_in, parent, prefK: Sequence, prefV: Sequence,
                 P, tau, H_out, ws, hidden=None, fold=None, n_packed=None):
        B, L, _ = H_in.shape
        n, W, K, V = _stack_args(weights, prefK, prefV)
        tr = _trace_arg(hidden, fold, n_packed)
        self._keep = (dims, weights, H_in, parent, prefK, prefV, H_out, ws, hidden, fold, n_packed)
        h = ctypes.c_void_p()
        torch.cuda.synchronize()
        _check(lib().specfold_stack_graph_create(ctypes.byref(dims), n, W, _ptr(H_in), _ptr(parent), B, L, K, V, P,
                                                 float(tau), _ptr(H_out), None if tr is None else ctypes.byref(tr),
                                                 _ptr(ws), ws.numel(), ctypes.byref(h)),
               "specfold_stack_graph_create")
        self._h = h


# ------------------------------------------------------------ convenience --

class FoldedLayer:
    """One folded verification layer: weights on the device plus a workspace.

    forward(H_in, parent, tau) runs S1..S10 through specfold_layer_forward and
    returns H_out; intermediates can be read back with `view(name)`.
    """

    def __init__(self, dims: specfold_dims, weights: dict, B: int, L: int, prefK=None, prefV=None, device="cuda"):
        self.dims = dims
        self.w = weights
        self.cw = make_weights(weights)
        self.B, self.L = B, L
        self.prefK, self.prefV = prefK, prefV
        self.P = 0 if prefK is None else prefK.shape[0]
        self.lo = workspace_layout(dims, B, L)
        self.ws = alloc_workspace(self.lo.total, device)

    def forward(self, H_in, parent, tau, H_out=None, events=None, stream=None):
        if H_out is None:
            H_out = torch.empty_like(H_in)
        specfold_layer_forward(self.dims, self.cw, H_in, parent, self.prefK, self.prefV, self.P, tau, H_out,
                               self.ws, events=events, stream=stream)
        return H_out

    def view(self, name: str, dtype=None, shape=None) -> torch.Tensor:
        """A tensor view of one workspace section (see specfold_ws_layout)."""
        names = [f[0] for f in specfold_ws_layout._fields_]
        off = getattr(self.lo, name)
        nxt = min([getattr(self.lo, k) for k in names if getattr(self.lo, k) > off] + [self.lo.total])
        raw = self.ws[off:nxt]
        if dtype is not None:
            es = torch.empty((), dtype=dtype).element_size()
            raw = raw[: (raw.numel() // es) * es].view(dtype)
        if shape is not None:
            n = 1
            for s in shape:
                n *= s
            raw = raw[:n].view(*shape)
        return raw

    def graph(self, H_in, parent, tau, H_out, events=None) -> LayerGraph:
        """Capture forward(H_in, parent, tau, H_out) as one replayable graph."""
        return LayerGraph(self.dims, self.cw, H_in, parent, self.prefK, self.prefV, self.P, tau, H_out, self.ws,
                          events=events)

    def n_packed(self) -> int:
        return int(self.view("n_packed", torch.int32)[0].item())

    def status(self) -> int:
        return specfold_get_status(self.ws)


class FoldedStack:
    """A stack of folded layers: per-layer device weights and prefix views
    plus one workspace.  forward(H_in, parent, tau) runs every layer through
    specfold_stack_forward; with ``record=True`` the per-layer input states,
    decisions and packed counts are kept (self.hidden / self.fold /
    self.n_packed)."""

    def __init__(self, dims: specfold_dims, weights: Sequence[dict], B: int, L: int,
                 prefK: Sequence = None, prefV: Sequence = None, device="cuda"):
        self.dims = dims
        self.w = list(weights)
        self.cw = [make_weights(w) for w in self.w]
        self.n_layers = len(self.w)
        self.B, self.L = B, L
        self.prefK = list(prefK) if prefK is not None else [None] * self.n_layers
        self.prefV = list(prefV) if prefV is not None else [None] * self.n_layers
        Ps = {0 if k is None else k.shape[0] for k in self.prefK}
        if len(Ps) != 1:
            raise ValueError("every layer's prefix has the same length")
        self.P = Ps.pop()
        self.lo = workspace_layout(dims, B, L)
        self.ws = alloc_workspace(stack_workspace_size(dims, B, L), device)
        R = B * L
        self.fold = torch.zeros((self.n_layers, B, L), dtype=torch.uint8, device=device)
        self.n_packed = torch.zeros(self.n_layers, dtype=torch.int32, device=device)
        self.hidden = None
        self._device = device

    def _hidden(self, H_in):
        if self.hidden is None or self.hidden.dtype != H_in.dtype:
            self.hidden = torch.empty((max(self.n_layers - 1, 1),) + tuple(H_in.shape), dtype=H_in.dtype,
                                      device=self._device)
        return self.hidden

    def forward(self, H_in, parent, tau, H_out=None, record=False, stream=None):
        if H_out is None:
            H_out = torch.empty_like(H_in)
        hidden = self._hidden(H_in) if (record and self.n_layers > 1) else None
        specfold_stack_forward(self.dims, self.cw, H_in, parent, self.prefK, self.prefV, self.P, tau, H_out,
                               self.ws, hidden=hidden, fold=self.fold, n_packed=self.n_packed, stream=stream)
        return H_out

    def graph(self, H_in, parent, tau, H_out, record=False) -> StackGraph:
        """Capture forward(H_in, parent, tau, H_out) as one replayable graph."""
        hidden = self._hidden(H_in) if (record and self.n_layers > 1) else None
        return StackGraph(self.dims, self.cw, H_in, parent, self.prefK, self.prefV, self.P, tau, H_out, self.ws,
                          hidden=hidden, fold=self.fold, n_packed=self.n_packed)

    def layer_inputs(self, H_in) -> list:
        """Inputs of layers 0..n-1 of the last recorded forward."""
        return [H_in] + ([self.hidden[l] for l in range(self.n_layers - 1)] if self.n_layers > 1 else [])

    def status(self) -> int:
        return specfold_get_status(self.ws)
