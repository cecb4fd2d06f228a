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


_CONTEXT_SCRIPT = r'''
import ctypes, sys
import numpy as np
sys.path.insert(0, sys.argv[1])
from chunked_lm_head_linear_gb300 import inputs, lce

cu = ctypes.CDLL("libcuda.so.1")


def ck(rc, what):
    if rc != 0:
        raise SystemExit(f"{what} returned {rc}")


def dalloc(n):
    p = ctypes.c_uint64()
    ck(cu.cuMemAlloc_v2(ctypes.byref(p), ctypes.c_size_t(max(n, 1))), "cuMemAlloc")
    return p.value


def h2d(a):
    p = dalloc(a.nbytes)
    ck(cu.cuMemcpyHtoD_v2(ctypes.c_uint64(p), a.ctypes.data_as(ctypes.c_void_p), ctypes.c_size_t(a.nbytes)), "HtoD")
    return p


def d2h(p, n, dtype):
    out = np.empty(n, dtype=dtype)
    ck(cu.cuMemcpyDtoH_v2(out.ctypes.data_as(ctypes.c_void_p), ctypes.c_uint64(p), ctypes.c_size_t(out.nbytes)), "DtoH")
    return out


def run_both(seed):
    """lce_forward with a workspace and lce_forward_noalloc, in the current context."""
    lib = lce.load()
    w = inputs.Workload(f"ctx{seed}", N=700, d=256, V=4096, sigma_w=0.05, labels="uniform", ignore="random",
                        ignore_frac=0.1, seed=seed)
    inp = inputs.make_inputs(w)
    N, d, V = 700, 256, 4096
    bufs = [h2d(np.ascontiguousarray(inp["H"])), h2d(np.ascontiguousarray(inp["W"])),
            h2d(np.ascontiguousarray(inp["y"]))]
    H, W, y = bufs
    opts = lce.make_opts(chunk_tokens=256, sync_check=True)
    need = lce.workspace_size(lce.LCE_OP_FORWARD, N, d, V, opts)
    ws, la, sa, lb, sb = dalloc(need), dalloc(4), dalloc(4 * N), dalloc(4), dalloc(4 * N)
    bufs += [ws, la, sa, lb, sb]
    rc = lib.lce_forward(H, W, y, N, d, V, la, sa, ctypes.byref(opts), ws, need, None)
    ck(rc, "lce_forward")
    rc = lib.lce_forward_noalloc(H, W, y, N, d, V, lb, sb, ctypes.byref(opts), None)
    ck(rc, "lce_forward_noalloc")
    ck(cu.cuCtxSynchronize(), "cuCtxSynchronize")
    loss_a, loss_b = d2h(la, 1, np.float32)[0], d2h(lb, 1, np.float32)[0]
    lse_a, lse_b = d2h(sa, N, np.float32), d2h(sb, N, np.float32)
    for p in bufs:
        ck(cu.cuMemFree_v2(ctypes.c_uint64(p)), "cuMemFree")
    assert abs(loss_b - loss_a) <= float(sys.argv[2]) * abs(loss_a), (loss_a, loss_b)
    rel = np.max(np.abs(lse_b - lse_a) / np.maximum(np.abs(lse_a), 1.0))
    assert rel <= float(sys.argv[3]), rel


ck(cu.cuInit(0), "cuInit")
dev = ctypes.c_int()
ck(cu.cuDeviceGet(ctypes.byref(dev), 0), "cuDeviceGet")
for seed in (11, 12):     # a context of its own, destroyed, then a new one: the library image moves
    ctx = ctypes.c_void_p()
    ck(cu.cuCtxCreate_v2(ctypes.byref(ctx), 0, dev), "cuCtxCreate")
    run_both(seed)
    ck(cu.cuCtxDestroy_v2(ctx), "cuCtxDestroy")
prim = ctypes.c_void_p()  # and the device's primary context after them
ck(cu.cuDevicePrimaryCtxRetain(ctypes.byref(prim), dev), "cuDevicePrimaryCtxRetain")
ck(cu.cuCtxSetCurrent(prim), "cuCtxSetCurrent")
run_both(13)
ck(cu.cuDevicePrimaryCtxRelease_v2(dev), "cuDevicePrimaryCtxRelease")
print("CONTEXTS_OK")
'''


def test_noalloc_in_contexts_the_caller_creates(cuda_lib, tmp_path):
    """A caller may run the library in a context it created with the driver
    API, destroy it and create another: each context holds its own copy of the
    library's device image, so the scratch array sits at a different device
    address in each, and lce_forward_noalloc must find the one of the current
    context (an address from a destroyed or a different context would be
    wrong memory). Runs in a child process without PyTorch, whose only
    contexts are the ones made here; each context's result is checked against
    lce_forward with a workspace in the same context."""
    import os
    import subprocess
    import sys
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    script = tmp_path / "contexts.py"
    script.write_text(_CONTEXT_SCRIPT)
    out = subprocess.run([sys.executable, str(script), root, str(TOL_LOSS), str(TOL_LSE)], capture_output=True,
                         text=True, timeout=300)
    assert out.returncode == 0 and "CONTEXTS_OK" in out.stdout, out.stdout[-2000:] + out.stderr[-2000:]
