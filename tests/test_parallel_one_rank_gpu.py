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
    n = dp.global_valid_count(y)
    assert n == int((inp["y"] != oracle.IGNORE_INDEX).sum())
    loss, lse, dH, dW = dp.dp_fwd_bwd(H, W, y, n_global=n, chunk_tokens=256)
    ref = cuda_lib.lce_fwd_bwd(H, W, y, chunk_tokens=256)
    torch.cuda.synchronize()
    for a, b in zip((loss, lse, dH, dW), ref):
        assert torch.equal(a, b)


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
