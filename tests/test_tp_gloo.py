"""Host logic of the vocabulary-parallel path on CPU: two gloo ranks, each with
a slice of W's rows; statistics are all-gathered and merged, partial dH
all-reduced. The fp64 oracle stands in for the CUDA shard calls (test only)."""
import os
import socket

import numpy as np
import pytest

torch = pytest.importorskip("torch")
import torch.distributed as dist  # noqa: E402
import torch.multiprocessing as mp  # noqa: E402


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _problem():
    rng = np.random.default_rng(7)
    N, d, V = 45, 10, 33
    H = rng.standard_normal((N, d))
    W = rng.standard_normal((V, d)) * 0.7
    y = rng.integers(0, V, N)
    y[rng.random(N) < 0.2] = -100
    return H, W, y


class _OracleShards:
    @staticmethod
    def forward_stats(H, W_shard, y, off, V_total, **_):
        import oracle
        return torch.from_numpy(oracle.vshard_stats_f64(H.numpy(), W_shard.numpy(), y.numpy(), off, V_total))

    @staticmethod
    def combine(stats_all, y, V_total, **_):
        import oracle
        loss, lse = oracle.vshard_merge_f64(stats_all.numpy(), y.numpy(), V_total=V_total)
        return torch.tensor([loss], dtype=torch.float64), torch.from_numpy(lse)

    @staticmethod
    def backward(H, W_shard, y, off, V_total, lse, grad_loss=None, **_):
        import oracle
        scale, _ = oracle.grad_scale(y.numpy())
        dH, dW = oracle.vshard_backward_f64(H.numpy(), W_shard.numpy(), y.numpy(), off, lse.numpy(), scale)
        return torch.from_numpy(dH), torch.from_numpy(dW)


class _OracleChunks(_OracleShards):
    """The per-chunk calls of the stored-tile schedule, from the same oracle pieces."""

    @staticmethod
    def chunk_workspace(H, W_shard, y, **_):
        return None

    @staticmethod
    def chunk_stats(H, W_shard, y, off, V_total, c0, rows, *, workspace, **_):
        import oracle
        s = slice(c0, c0 + rows)
        return torch.from_numpy(oracle.vshard_stats_f64(H[s].numpy(), W_shard.numpy(), y[s].numpy(), off, V_total))

    @staticmethod
    def chunk_backward(H, W_shard, y, off, V_total, c0, rows, stats_all, *, workspace, lse, dH_partial, dW_shard,
                       grad_loss=None, **_):
        import oracle
        s = slice(c0, c0 + rows)
        _, lse_c = oracle.vshard_merge_f64(stats_all.numpy(), y[s].numpy(), V_total=V_total)
        scale, _ = oracle.grad_scale(y.numpy())          # n over all N labels
        dH_c, dW_c = oracle.vshard_backward_f64(H[s].numpy(), W_shard.numpy(), y[s].numpy(), off, lse_c, scale)
        lse[s] = torch.from_numpy(lse_c)
        dH_partial[s] = torch.from_numpy(dH_c)
        if c0 == 0:
            dW_shard.copy_(torch.from_numpy(dW_c))
        else:
            dW_shard.add_(torch.from_numpy(dW_c))


def _rank(rank, world, port, outdir):
    import sys
    sys.path.insert(0, os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
    from chunked_lm_head_linear_gb300 import tp
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    H, W, y = _problem()
    cuts = [0, 14, 33]                 # uneven vocabulary shards
    sl = slice(cuts[rank], cuts[rank + 1])
    for method, backend, chunk in (("recompute", _OracleShards, 0), ("stored", _OracleChunks, 16)):
        loss, lse, dH, dW = tp.vocab_parallel_fwd_bwd(torch.from_numpy(H), torch.from_numpy(W[sl]),
                                                      torch.from_numpy(y), cuts[rank], 33, backend=backend,
                                                      method=method, chunk_tokens=chunk)
        np.savez(os.path.join(outdir, f"{method}_rank{rank}.npz"), loss=loss.numpy(), lse=lse.numpy(),
                 dH=dH.numpy(), dW=dW.numpy())
    dist.barrier()
    dist.destroy_process_group()


def test_two_gloo_vocab_shards_equal_unsharded(tmp_path):
    import oracle
    mp.start_processes(_rank, args=(2, _free_port(), str(tmp_path)), nprocs=2, join=True, start_method="spawn")
    H, W, y = _problem()
    whole = oracle.lce_f64(H, W, y)
    for method in ("recompute", "stored"):      # stored: three chunks of 16, 16 and 13 tokens
        r = [np.load(tmp_path / f"{method}_rank{k}.npz") for k in range(2)]
        for k in range(2):
            assert float(r[k]["loss"][0]) == pytest.approx(whole["loss"], rel=1e-13)
            np.testing.assert_allclose(r[k]["lse"], whole["lse"], rtol=1e-14)
            np.testing.assert_allclose(r[k]["dH"], whole["dH"], rtol=1e-12, atol=1e-15)
        np.testing.assert_allclose(np.vstack([r[0]["dW"], r[1]["dW"]]), whole["dW"], rtol=1e-12, atol=1e-15)
