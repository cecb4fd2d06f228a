"""The bounds-checking debug build (compiled with -DLCE_CHECKS), in place of a
memory sanitizer: every index the kernels compute into a plain global buffer
and every tile coordinate they hand to TMA is checked before use, and a bad
one sets the LCE_DEVICE_BOUNDS status bit instead of touching memory. Small
odd-sized cases (N = 1, 3, 129; V = 2, 37, 151655; row, column, K and
vocabulary tails) go through every kind of call of that build; each must leave
the bit clear and match the fp64 oracle within the parity tests' bounds.

The checked library runs in a child process (a process loads one liblce.so).
"""
import os
import subprocess
import sys

import numpy as np
import pytest

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HERE = os.path.dirname(os.path.abspath(__file__))

# N, d, V, chunk
CASES = [
    (1, 64, 37, 0),          # one token
    (3, 72, 2, 0),           # three tokens, two classes, K tail (72 = 64 + 8)
    (129, 136, 151655, 64),  # one row past a tile, the unpadded vocabulary, small chunks
    (129, 8, 37, 0),         # the smallest hidden size
    (300, 264, 4099, 128),   # row, column and vocabulary tails
    (513, 256, 1000, 200),   # chunks that are not a multiple of the tile
]


def _status_ok(lce, ws, what):
    flags = lce.read_device_status(ws)
    assert not flags & lce.LCE_DEVICE_BOUNDS, f"{what}: an index fell outside its buffer"


def _child():
    """Runs in the child process, with the checked library loaded first."""
    import torch

    from chunked_lm_head_linear_gb300 import build, lce
    lce.load(build.build(checks=True))
    import oracle
    from test_parity_gpu import check_against_oracle, small_inputs, to_dev, vshard_stored

    def ws_for(op, N, d, V, chunk):
        return torch.empty(lce.workspace_size(op, N, d, V, lce.make_opts(chunk_tokens=chunk)), dtype=torch.uint8,
                           device="cuda")

    for N, d, V, chunk in CASES:
        inp = small_inputs(N, d, V, seed=N + d + V, sigma_w=0.05)
        ref = oracle.lce_bf16(inp["H"], inp["W"], inp["y"])
        H, W, y = to_dev(inp)
        tag = f"N={N} d={d} V={V} chunk={chunk}"
        # the fused call
        ws = ws_for(lce.LCE_OP_FWD_BWD, N, d, V, chunk)
        loss, lse, dH, dW = lce.lce_fwd_bwd(H, W, y, workspace=ws, chunk_tokens=chunk)
        _status_ok(lce, ws, "lce_fwd_bwd " + tag)
        check_against_oracle(ref, inp["y"], loss.item(), lse.cpu().numpy(), dH.float().cpu().numpy(),
                             dW.cpu().numpy())
        # the split calls
        wf, wb = ws_for(lce.LCE_OP_FORWARD, N, d, V, chunk), ws_for(lce.LCE_OP_BACKWARD, N, d, V, chunk)
        loss, lse = lce.lce_forward(H, W, y, workspace=wf, chunk_tokens=chunk)
        dH, dW = lce.lce_backward(H, W, y, lse, workspace=wb, chunk_tokens=chunk)
        _status_ok(lce, wf, "lce_forward " + tag)
        _status_ok(lce, wb, "lce_backward " + tag)
        check_against_oracle(ref, inp["y"], loss.item(), lse.cpu().numpy(), dH.float().cpu().numpy(),
                             dW.cpu().numpy())
        # the sliced call
        ws = ws_for(lce.LCE_OP_FWD_BWD, N, d, V, chunk)
        loss, lse, dH, dW = lce.lce_fwd_bwd_sliced(H, W, y, bounds=lce.slice_bounds(V, 3), workspace=ws,
                                                   chunk_tokens=chunk)
        _status_ok(lce, ws, "lce_fwd_bwd_sliced " + tag)
        check_against_oracle(ref, inp["y"], loss.item(), lse.cpu().numpy(), dH.float().cpu().numpy(),
                             dW.cpu().numpy())
        # vocabulary shards (stored-tile schedule), three uneven shards
        if V >= 3:
            cuts = [0, V // 3 // 8 * 8 + 1, 2 * V // 3, V]
            # (with sync_check a bounds bit turns into LCE_ERR_BOUNDS, which the binding raises)
            loss, lse, dHs, dWs = vshard_stored(lce, H, W, y, cuts, chunk, sync_check=True)
            check_against_oracle(ref, inp["y"], loss.item(), lse.cpu().numpy(), dHs.cpu().numpy().astype(np.float64),
                                 dWs.cpu().numpy())
        torch.cuda.synchronize()
    # norm + head
    N, d, V = 129, 136, 4099
    inp = small_inputs(N, d, V, seed=7, sigma_w=0.05)
    rng = np.random.default_rng(7)
    wn = (rng.standard_normal(d) * 0.1).astype(np.float32)
    from chunked_lm_head_linear_gb300 import inputs
    xb = inputs.f64_to_bf16_bits(rng.standard_normal((N, d)) * 2)
    ref = oracle.norm_lce_bf16(xb, wn.astype(np.float64), inp["W"], inp["y"], 1e-6)
    x = torch.from_numpy(xb.view(np.int16)).view(torch.bfloat16).cuda()
    _, W, y = to_dev(inp)
    ws = torch.empty(lce.workspace_size(lce.LCE_OP_NORM_FWD_BWD, N, d, V, lce.make_opts(chunk_tokens=64)),
                     dtype=torch.uint8, device="cuda")
    loss, lse, dx, dw_norm, dW = lce.lce_norm_fwd_bwd(x, torch.from_numpy(wn).cuda(), W, y, workspace=ws,
                                                      chunk_tokens=64)
    _status_ok(lce, ws, "lce_norm_fwd_bwd")
    check_against_oracle(ref, inp["y"], loss.item(), lse.cpu().numpy(), None, dW.cpu().numpy())
    print("CHECKED_OK", flush=True)


def test_checked_build_small_odd_cases(cuda_lib):
    code = f"import sys; sys.path[:0] = [{ROOT!r}, {HERE!r}]; import test_checked_build_gpu as t; t._child()"
    out = subprocess.run([sys.executable, "-c", code], capture_output=True, text=True, timeout=900)
    assert out.returncode == 0 and "CHECKED_OK" in out.stdout, out.stdout[-3000:] + out.stderr[-3000:]
