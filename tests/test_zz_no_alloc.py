"""lce_forward_noalloc: the forward for callers that cannot allocate device
memory (their memory belongs to another allocator, or they must not call
cudaMalloc / cudaFree). It runs the same kernels on a fixed scratch array
inside the library, so its results must match lce_forward's with a
caller-provided workspace. Two calls in a row check that what the first call
leaves in the shared scratch does not leak into the second.

This file sorts last so a stop-at-first-failure run has done every other test
before it; it also passes on its own in a fresh process.
"""
import ctypes

import numpy as np
import pytest

from chunked_lm_head_linear_gb300 import inputs

pytestmark = pytest.mark.gpu

TOL_LOSS = 1e-3
TOL_LSE = 1e-4


def _case(seed, N=700, d=256, V=4096):
    w = inputs.Workload(f"noalloc{seed}", N=N, d=d, V=V, sigma_w=0.05, labels="uniform",
                        ignore="random", ignore_frac=0.1, seed=seed)
    inp = inputs.make_inputs(w)
    import torch
    H = torch.from_numpy(inp["H"].view(np.int16)).view(torch.bfloat16).cuda()
    W = torch.from_numpy(inp["W"].view(np.int16)).view(torch.bfloat16).cuda()
    y = torch.from_numpy(inp["y"]).cuda()
    return H, W, y


def _noalloc(lib, lce, H, W, y, **opt_kw):
    import torch
    N, d = H.shape
    V = W.shape[0]
    loss = torch.full((1,), float("nan"), dtype=torch.float32, device="cuda")
    lse = torch.full((N,), float("nan"), dtype=torch.float32, device="cuda")
    opts = lce.make_opts(**opt_kw)
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    rc = lib.lce_forward_noalloc(ctypes.c_void_p(H.data_ptr()), ctypes.c_void_p(W.data_ptr()),
                                 ctypes.c_void_p(y.data_ptr()), N, d, V, ctypes.c_void_p(loss.data_ptr()),
                                 ctypes.c_void_p(lse.data_ptr()), ctypes.byref(opts), stream)
    return rc, loss, lse


def test_noalloc_forward_matches_workspace_forward_twice(cuda_lib):
    import torch
    lib = cuda_lib.load()
    for seed, chunk in ((1, 256), (2, 0)):      # two calls in a row, different inputs and chunking
        H, W, y = _case(seed)
        ref_loss, ref_lse = cuda_lib.lce_forward(H, W, y, chunk_tokens=chunk, sync_check=True)
        rc, loss, lse = _noalloc(lib, cuda_lib, H, W, y, chunk_tokens=chunk, sync_check=True)
        torch.cuda.synchronize()
        assert rc == cuda_lib.LCE_OK, cuda_lib.status_string(rc)
        assert abs(loss.item() - ref_loss.item()) <= TOL_LOSS * abs(ref_loss.item())
        rel = ((lse - ref_lse).abs() / ref_lse.abs().clamp_min(1.0)).max().item()
        assert rel <= TOL_LSE


def test_noalloc_binding_writes_into_caller_tensors(cuda_lib):
    """The Python binding of the same name, with caller-owned outputs."""
    import torch
    H, W, y = _case(4, N=300, d=128, V=1000)
    ref_loss, ref_lse = cuda_lib.lce_forward(H, W, y, sync_check=True)
    loss = torch.full((1,), float("nan"), dtype=torch.float32, device="cuda")
    lse = torch.full((300,), float("nan"), dtype=torch.float32, device="cuda")
    out = cuda_lib.lce_forward_noalloc(H, W, y, loss=loss, lse=lse, sync_check=True)
    assert out[0] is loss and out[1] is lse
    assert abs(loss.item() - ref_loss.item()) <= TOL_LOSS * abs(ref_loss.item())
    assert ((lse - ref_lse).abs() / ref_lse.abs().clamp_min(1.0)).max().item() <= TOL_LSE


def test_noalloc_rejects_sizes_beyond_its_scratch(cuda_lib):
    lib = cuda_lib.load()
    H, W, y = _case(3, N=256, d=64, V=4096)
    # 8192-token chunks over a 151936-word vocabulary need ~39 MB of scratch (> 32 MiB)
    opts = cuda_lib.make_opts(chunk_tokens=8192)
    rc = lib.lce_forward_noalloc(ctypes.c_void_p(H.data_ptr()), ctypes.c_void_p(W.data_ptr()),
                                 ctypes.c_void_p(y.data_ptr()), 8192, 64, 151936, ctypes.c_void_p(H.data_ptr()),
                                 ctypes.c_void_p(H.data_ptr()), ctypes.byref(opts), None)
    assert rc == cuda_lib.LCE_ERR_WORKSPACE
