"""The data-parallel and vocabulary-parallel host code (dp.py, tp.py) with
their default CUDA backend, on a one-rank NCCL group.

With one rank every collective is a copy, but the calls, the stream order of
kernels and collectives, the workspaces kept between the per-chunk shard calls
and the buffers the schedules allocate are the ones a multi-GPU run uses. The
results must equal the unsharded lce_fwd_bwd (bit for bit where the
arithmetic is the same) and the fp64 oracle."""
import os
import socket

import numpy as np
import pytest

import oracle

from test_parity_gpu import TOL_LSE, check_against_oracle, small_inputs, to_dev

pytestmark = pytest.mark.gpu


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


@pytest.fixture(scope="module")
def one_rank_nccl(cuda_lib):
    import torch.distributed as dist
    dist.init_process_group("nccl", init_method=f"tcp://127.0.0.1:{_free_port()}", rank=0, world_size=1)
    yield
    dist.destroy_process_group()


def test_dp_one_rank_equals_fused_call(cuda_lib, one_rank_nccl):
    import torch
    from chunked_lm_head_linear_gb300 import dp
    inp = small_inputs(700, 256, 4096, seed=81)
    H, W, y = to_dev(inp)
    n = dp.global_valid_count(y, V=4096)
    assert n == int((inp["y"] != oracle.IGNORE_INDEX).sum())
    loss, lse, dH, dW = dp.dp_fwd_bwd(H, W, y, n_global=n, chunk_tokens=256)
    ref = cuda_lib.lce_fwd_bwd(H, W, y, chunk_tokens=256)
    torch.cuda.synchronize()
    for a, b in zip((loss, lse, dH, dW), ref):
        assert torch.equal(a, b)


def test_dp_count_with_out_of_range_labels_matches_the_library(cuda_lib, one_rank_nccl):
    """Labels outside the vocabulary (an error the library reports and whose
    rows it treats as ignored) are not counted in the data-parallel
    denominator either: the DP step equals the one-rank call bit for bit, and
    the count equals the one the library itself took."""
    import torch
    from chunked_lm_head_linear_gb300 import dp
    inp = small_inputs(700, 256, 4096, seed=82)
    inp["y"][[3, 100, 555]] = [4096, -7, 10 ** 9]
    H, W, y = to_dev(inp)
    n = dp.global_valid_count(y, V=4096)
    valid = (inp["y"] != oracle.IGNORE_INDEX) & (inp["y"] >= 0) & (inp["y"] < 4096)
    assert n == int(valid.sum())
    ws = torch.empty(cuda_lib.workspace_size(cuda_lib.LCE_OP_FWD_BWD, 700, 256, 4096,
                                             cuda_lib.make_opts(chunk_tokens=256)), dtype=torch.uint8, device="cuda")
    loss, lse, dH, dW = dp.dp_fwd_bwd(H, W, y, n_global=n, chunk_tokens=256)
    ref = cuda_lib.lce_fwd_bwd(H, W, y, chunk_tokens=256, workspace=ws)
    flags = cuda_lib.read_device_status(ws)
    assert flags & cuda_lib.LCE_DEVICE_LABEL_RANGE
    # equal mean losses and gradients bit for bit: the two denominators agree
    for a, b in zip((loss, lse, dH, dW), ref):
        assert torch.equal(a, b)
    # the shards' own counts add up to the same denominator
    halves = [dp.global_valid_count(y[:350], V=4096), dp.global_valid_count(y[350:], V=4096)]
    assert sum(halves) == n


@pytest.mark.parametrize("method,chunk", [("stored", 256), ("stored", 0), ("recompute", 0)])
def test_tp_one_rank_matches_oracle(cuda_lib, one_rank_nccl, method, chunk):
    """vocab_parallel_fwd_bwd with the whole vocabulary as the one rank's shard."""
    import torch
    from chunked_lm_head_linear_gb300 import tp
    inp = small_inputs(700, 264, 4099, seed=83, sigma_w=0.05)
    ref = oracle.lce_bf16(inp["H"], inp["W"], inp["y"])
    H, W, y = to_dev(inp)
    loss, lse, dH, dW = tp.vocab_parallel_fwd_bwd(H, W, y, 0, 4099, method=method, chunk_tokens=chunk)
    torch.cuda.synchronize()
    check_against_oracle(ref, inp["y"], loss.item(), lse.cpu().numpy(), dH.cpu().numpy().astype(np.float64),
                         dW.cpu().numpy())
    _, lse_f, _, _ = cuda_lib.lce_fwd_bwd(H, W, y, chunk_tokens=chunk)
    assert ((lse - lse_f).abs() / lse_f.abs()).max().item() <= TOL_LSE
