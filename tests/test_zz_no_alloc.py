"""specfold_linear_noalloc: the GEMM entry point for callers that cannot
allocate device memory (no workspace argument; the library's static device
scratch holds the split-K partials).  Checked through the C ABI against
specfold_linear, which takes a caller workspace, and against the float64
product of the same bf16 operands, on two calls in a row so the second call
runs on scratch left over from the first.

This file is collected last on purpose: if it fails, a run that stops at the
first failure has already run every other test.
"""
import numpy as np
import pytest
import torch

from diffusion_branch_speculative_gb300 import binding, synth

pytestmark = pytest.mark.gpu

TOL = 2e-2       # the relative-L2 bound the other GPU parity tests use
TOL_FP64 = 5e-3  # against the float64 product: the bound of the workspace GEMM's own test


def _rel_l2(a, b):
    a = a.double()
    b = b.double()
    return float((a - b).norm() / b.norm())


@pytest.mark.parametrize("M,N,K", [(64, 3584, 18944), (95, 4608, 3584), (300, 384, 1024), (2048, 1024, 4096),
                                   (2176, 2048, 1024),    # splits the tiles of a partial last wave
                                   (3072, 2048, 1024)])   # 192 tiles on 128 CTAs: 64 tail tiles x 2 splits fill
                                                          # all 128 partial slots of the scratch
def test_linear_noalloc_matches_workspace_linear(M, N, K):
    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    rng = np.random.default_rng(M * 7 + N + K)
    X = torch.from_numpy(synth.round_bf16(rng.standard_normal((M, K)).astype(np.float32))).cuda().to(torch.bfloat16)
    W = torch.from_numpy(synth.round_bf16((rng.standard_normal((N, K)) * 0.02).astype(np.float32))).cuda().to(torch.bfloat16)
    ref = torch.empty(M, N, dtype=torch.bfloat16, device="cuda")
    ws = binding.alloc_workspace(binding.linear_workspace_size(M, N))
    binding.specfold_linear(X, W, ref, ws)
    exact = X.double() @ W.double().T
    for _ in range(2):
        Y = torch.full((M, N), float("nan"), dtype=torch.bfloat16, device="cuda")
        binding.specfold_linear_noalloc(X, W, Y)
        torch.cuda.synchronize()
        assert torch.isfinite(Y.float()).all()
        assert _rel_l2(Y, ref) < TOL
        assert _rel_l2(Y, exact) < TOL_FP64
        # row by row too: one bad tile or partial slot cannot hide in the norm
        rows = ((Y.double() - exact).norm(dim=1) / exact.norm(dim=1).clamp_min(1e-30)).max().item()
        assert rows < TOL_FP64


def test_linear_noalloc_rejects_rows_beyond_its_limit():
    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    X = torch.zeros(16, 64, dtype=torch.bfloat16, device="cuda")
    W = torch.zeros(128, 64, dtype=torch.bfloat16, device="cuda")
    Y = torch.zeros(16, 128, dtype=torch.bfloat16, device="cuda")
    L = binding.lib()
    rc = L.specfold_linear_noalloc(binding.BF16, binding._ptr(X), binding._ptr(W), 16385, 128, 64, binding._ptr(Y),
                                   binding._stream())
    assert rc == binding.ECAPACITY
