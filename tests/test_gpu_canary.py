"""Out-of-bounds writes, caught without a device assert: the layer call gets
its output, its workspace and the caller's prefix cache inside larger
buffers whose guard regions hold a known byte pattern, and the host checks
after the call that every guard byte is intact, that the prefix cache was not
written, and that the output equals the one of an unguarded call bit for bit.
"""
import numpy as np
import pytest
import torch

from diffusion_branch_speculative_gb300 import binding, synth
from tests.gpu_cases import DeviceInputs

pytestmark = pytest.mark.gpu

GUARD = 64 << 10      # bytes of guard on each side (a multiple of 512: the inner views keep their alignment)
PATTERN = 0xA5


def _guarded(nbytes: int, fill=None):
    """A byte buffer [GUARD | nbytes | GUARD], guards set to PATTERN; the
    inner view zeroed, or a copy of `fill` (a byte tensor of nbytes)."""
    buf = torch.full((GUARD + nbytes + GUARD,), PATTERN, dtype=torch.uint8, device="cuda")
    inner = buf[GUARD:GUARD + nbytes]
    if fill is None:
        inner.zero_()
    else:
        inner.copy_(fill)
    return buf, inner


def _guards_intact(buf: torch.Tensor, nbytes: int) -> bool:
    return bool((buf[:GUARD] == PATTERN).all()) and bool((buf[GUARD + nbytes:] == PATTERN).all())


@pytest.mark.parametrize("name,frac,tau", [("7b_layer", None, 0.05), ("7b_layer", None, 0.0), ("stress", 0.25, 0.05),
                                           ("tiny", None, 0.05)])
def test_layer_guards_intact(name, frac, tau):
    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    inp = synth.make_layer_inputs(name, seed=3, dtype="bf16", forced_frac=frac)
    dev = DeviceInputs(inp)
    B, L, D = inp.H.shape
    # reference: the library's own workspace and output
    lay = binding.FoldedLayer(dev.dims, dev.W, B, L, dev.pk, dev.pv)
    ref = lay.forward(dev.H, dev.parent, tau).clone()
    # guarded output, workspace and prefix cache
    esz = dev.H.element_size()
    out_bytes = dev.H.numel() * esz
    obuf, oin = _guarded(out_bytes)
    H_out = oin.view(dev.H.dtype).view(B, L, D)
    ws_bytes = binding.workspace_size(dev.dims, B, L)
    wbuf, ws = _guarded(ws_bytes)
    cache = dev.cache
    cbytes = cache.numel() * cache.element_size()
    cbuf, cin = _guarded(cbytes, fill=cache.reshape(-1).view(torch.uint8))
    gcache = cin.view(cache.dtype).view(cache.shape)
    pre = inp.prefix
    pk = gcache[pre.offset:pre.offset + pre.P, 0] if pre.P else None
    pv = gcache[pre.offset:pre.offset + pre.P, 1] if pre.P else None
    cw = binding.make_weights(dev.W)
    for _ in range(2):   # twice: the second call runs on the first one's workspace
        binding.specfold_layer_forward(dev.dims, cw, dev.H, dev.parent, pk, pv, dev.P, tau, H_out, ws)
    torch.cuda.synchronize()
    assert binding.specfold_get_status(ws) == 0
    assert _guards_intact(obuf, out_bytes), "write outside H_out"
    assert _guards_intact(wbuf, ws_bytes), "write outside the workspace"
    assert _guards_intact(cbuf, cbytes), "write outside the prefix cache"
    assert torch.equal(cin, cache.reshape(-1).view(torch.uint8)), "the prefix cache was written"
    assert torch.equal(H_out, ref), "guarded call differs from the unguarded one"
