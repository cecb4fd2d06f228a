"""dW in vocabulary slices (lce_fwd_bwd_sliced) and the FSDP-style reduce to
the owners on a GPU.

The sliced call must give the same bits as lce_fwd_bwd (each output tile is
computed by the same arithmetic in whichever launch it falls), so these tests
compare the two CUDA calls for bitwise equality, and check the sliced result
against the fp64 oracle on a small case. The FSDP path runs with a one-rank
NCCL group: its reduces are then copies, but the streams, the per-slice
events and the owner bookkeeping are the ones a multi-GPU run uses."""
import os
import socket

import numpy as np
import pytest

import oracle
from chunked_lm_head_linear_gb300 import inputs

from test_parity_gpu import TOL_GRAD, bf16_to_np, check_against_oracle, small_inputs, to_dev

pytestmark = pytest.mark.gpu


def _same(a, b):
    import torch
    return a.shape == b.shape and torch.equal(a.view(torch.uint8) if a.dtype == torch.bfloat16 else a,
                                              b.view(torch.uint8) if b.dtype == torch.bfloat16 else b)


def _pair(lce, H, W, y, bounds, sm_limit=0, **kw):
    import torch
    ev = [torch.cuda.Event() for _ in range(len(bounds) - 1)]
    a = lce.lce_fwd_bwd(H, W, y, **kw)
    b = lce.lce_fwd_bwd_sliced(H, W, y, bounds=bounds, events=ev, sm_limit=sm_limit, **kw)
    torch.cuda.synchronize()
    assert all(e.query() for e in ev)
    return a, b


CASES = [
    # N, d, V, chunk, bounds (None: lce.slice_bounds(V, n) with n below), n, sm_limit
    (300, 136, 1000, 128, None, 3, 0),
    (300, 136, 1000, 0, [0, 1000], 1, 0),
    (513, 264, 4099, 200, [0, 0, 256, 256, 3840, 4099], 5, 16),
    (1000, 512, 4096, 256, None, 16, 7),
    (64, 2048, 151936, 0, None, 8, 0),
    # 1024-token chunks: the whole launches deal each dH block's four parts to one cluster, the last
    # slice's launch (an eighth of the dW tiles) deals them one by one; same arithmetic either way
    (2048, 2048, 151936, 1024, None, 8, 0),
]


@pytest.mark.parametrize("N,d,V,chunk,bounds,n,sm_limit", CASES)
def test_sliced_is_bitwise_the_fused_call(cuda_lib, N, d, V, chunk, bounds, n, sm_limit):
    inp = small_inputs(N, d, V, seed=N + V)
    H, W, y = to_dev(inp)
    bounds = bounds if bounds is not None else cuda_lib.slice_bounds(V, n)
    a, b = _pair(cuda_lib, H, W, y, bounds, sm_limit=sm_limit, chunk_tokens=chunk)
    for u, v in zip(a, b):
        assert _same(u, v)


def test_sliced_matches_oracle(cuda_lib):
    inp = small_inputs(513, 264, 4099, seed=3)
    H, W, y = to_dev(inp)
    ref = oracle.lce_bf16(inp["H"], inp["W"], inp["y"])
    loss, lse, dH, dW = cuda_lib.lce_fwd_bwd_sliced(H, W, y, bounds=cuda_lib.slice_bounds(4099, 4),
                                                    chunk_tokens=256)
    check_against_oracle(ref, inp["y"], loss.item(), lse.cpu().numpy(), bf16_to_np(dH), dW.cpu().numpy())


def test_sliced_accumulate_and_empty(cuda_lib):
    import torch
    inp = small_inputs(300, 136, 1000, seed=11)
    H, W, y = to_dev(inp)
    bounds = cuda_lib.slice_bounds(1000, 3)
    base = torch.randn(1000, 136, device="cuda")
    a = cuda_lib.lce_fwd_bwd(H, W, y, dW=base.clone(), accumulate_dW=1, chunk_tokens=128)
    b = cuda_lib.lce_fwd_bwd_sliced(H, W, y, bounds=bounds, dW=base.clone(), accumulate_dW=1, chunk_tokens=128)
    assert _same(a[3], b[3]) and _same(a[2], b[2])
    # no tokens: dW zeroed, every event still recorded
    ev = [torch.cuda.Event() for _ in range(3)]
    loss, _, _, dW = cuda_lib.lce_fwd_bwd_sliced(H[:0], W, y[:0], bounds=bounds, events=ev,
                                                 dW=torch.ones(1000, 136, device="cuda"))
    torch.cuda.synchronize()
    assert float(loss) == 0.0 and float(dW.abs().max()) == 0.0 and all(e.query() for e in ev)


def test_sliced_rejects_bad_bounds(cuda_lib):
    inp = small_inputs(64, 64, 1000, seed=1)
    H, W, y = to_dev(inp)
    for bad in ([0, 100, 1000], [0, 512, 256, 1000], [1, 1000], [0, 999], [0, 256]):
        with pytest.raises(RuntimeError):
            cuda_lib.lce_fwd_bwd_sliced(H, W, y, bounds=bad)


def test_full_qwen2b_sliced_bitwise(cuda_lib):
    """The bench workload (N=8192, d=2048, V=151936, chunk 4096) in 8 slices
    with a reduced SM count gives exactly lce_fwd_bwd's outputs."""
    inp = inputs.make_inputs("qwen2b_n8192_d2048_v151936")
    H, W, y = to_dev(inp)
    a, b = _pair(cuda_lib, H, W, y, cuda_lib.slice_bounds(151936, 8), sm_limit=136, chunk_tokens=4096)
    for u, v in zip(a, b):
        assert _same(u, v)


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def test_fsdp_one_rank_nccl(cuda_lib):
    """fsdp_fwd_bwd on a one-rank NCCL group: gather, sliced step, reduces on
    a side stream ordered by the slice events; equals lce_fwd_bwd."""
    import torch
    import torch.distributed as dist
    from chunked_lm_head_linear_gb300 import fsdp
    inp = small_inputs(700, 256, 4096, seed=5)
    H, W, y = to_dev(inp)
    dist.init_process_group("nccl", init_method=f"tcp://127.0.0.1:{_free_port()}", rank=0, world_size=1)
    try:
        owners = fsdp.owner_bounds(4096, 1)
        W_full = fsdp.gather_weight(W, owners)
        assert _same(W_full, W)
        loss, lse, dH, dW_own = fsdp.fsdp_fwd_bwd(H, W_full, y, owners=owners,
                                                  slices=cuda_lib.slice_bounds(4096, 4), chunk_tokens=256)
        ref = cuda_lib.lce_fwd_bwd(H, W, y, chunk_tokens=256)
        torch.cuda.synchronize()
        assert _same(loss, ref[0]) and _same(lse, ref[1]) and _same(dH, ref[2]) and _same(dW_own, ref[3])
        refo = oracle.lce_bf16(inp["H"], inp["W"], inp["y"])
        assert abs(loss.item() - refo["loss"]) <= 1e-3 * abs(refo["loss"])
        d = dW_own.cpu().numpy()
        assert np.linalg.norm(d - refo["dW"]) <= TOL_GRAD * np.linalg.norm(refo["dW"])
    finally:
        dist.destroy_process_group()
