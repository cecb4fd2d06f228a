"""Host logic of the data-parallel path on CPU: two gloo ranks, each with a
token shard; the global valid count is all-reduced, each shard runs with it as
denominator, dW and the loss are summed. The fp64 oracle stands in for the
CUDA compute (test only) and the result must equal the unsharded oracle."""
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
    rng = np.random.default_rng(42)
    N, d, V = 97, 12, 31
    H = rng.standard_normal((N, d))
    W = rng.standard_normal((V, d)) * 0.5
    y = rng.integers(0, V, N)
    y[rng.random(N) < 0.2] = -100
    return H, W, y


def _oracle_compute(H, W, y, grad_loss=None, *, n_valid_override=-1, ignore_index=-100, **_):
    import oracle
    g = 1.0 if grad_loss is None else float(grad_loss)
    out = oracle.lce_f64(H.numpy(), W.numpy(), y.numpy(), n_valid_override=n_valid_override,
                         ignore_index=ignore_index, grad_loss=g)
    return (torch.tensor([out["loss"]], dtype=torch.float64), torch.from_numpy(out["lse"]),
            torch.from_numpy(out["dH"]), torch.from_numpy(out["dW"]))


def _rank(rank, world, port, outdir):
    import sys
    sys.path.insert(0, os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
    from chunked_lm_head_linear_gb300 import dp
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    H, W, y = _problem()
    cut = [0, 40, len(y)]                      # uneven shards
    sl = slice(cut[rank], cut[rank + 1])
    loss, lse, dH, dW = dp.dp_fwd_bwd(torch.from_numpy(H[sl]), torch.from_numpy(W), torch.from_numpy(y[sl]),
                                      compute=_oracle_compute)
    np.savez(os.path.join(outdir, f"rank{rank}.npz"), loss=loss.numpy(), lse=lse.numpy(), dH=dH.numpy(),
             dW=dW.numpy())
    dist.barrier()
    dist.destroy_process_group()


def test_two_gloo_ranks_equal_unsharded(tmp_path):
    import oracle
    port = _free_port()
    mp.start_processes(_rank, args=(2, port, str(tmp_path)), nprocs=2, join=True, start_method="spawn")
    H, W, y = _problem()
    whole = oracle.lce_f64(H, W, y)
    r0 = np.load(tmp_path / "rank0.npz")
    r1 = np.load(tmp_path / "rank1.npz")
    for r in (r0, r1):
        assert float(r["loss"][0]) == pytest.approx(whole["loss"], rel=1e-13)
        np.testing.assert_allclose(r["dW"], whole["dW"], rtol=1e-12, atol=1e-15)
    np.testing.assert_allclose(np.concatenate([r0["dH"], r1["dH"]]), whole["dH"], rtol=1e-12, atol=1e-15)
    np.testing.assert_allclose(np.concatenate([r0["lse"], r1["lse"]]), whole["lse"], rtol=1e-14)


def _count_rank(rank, world, port, outdir):
    import sys
    sys.path.insert(0, os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
    from chunked_lm_head_linear_gb300 import dp
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    y = torch.tensor([[5, -100, 31, -1, 0, 30], [7, 10 ** 9, -100, -100, 2, 3]][rank])
    n = dp.global_valid_count(y, V=31)
    np.save(os.path.join(outdir, f"count{rank}.npy"), np.array([n]))
    dist.barrier()
    dist.destroy_process_group()


def test_global_count_follows_the_library_rule(tmp_path):
    """The data-parallel denominator counts a label only if it is not
    ignore_index and lies in [0, V), as the library's own label scan does:
    31, -1 and 10**9 are out of range for V = 31 and are not counted."""
    port = _free_port()
    mp.start_processes(_count_rank, args=(2, port, str(tmp_path)), nprocs=2, join=True, start_method="spawn")
    for r in range(2):
        assert int(np.load(tmp_path / f"count{r}.npy")[0]) == 3 + 3   # {5, 0, 30} and {7, 2, 3}
