"""Host logic of the FSDP-style path on CPU: three gloo ranks with uneven token
shards; W stored by vocabulary rows (unequal owner ranges), gathered, the
local step computed by the fp64 oracle (test only) with the global count of
valid labels, and dW reduced to its owners slice by slice. Every rank's dW
rows, the loss and the concatenated lse / dH must equal the unsharded oracle."""
import os
import socket

import numpy as np
import pytest

torch = pytest.importorskip("torch")
import torch.distributed as dist  # noqa: E402
import torch.multiprocessing as mp  # noqa: E402

from chunked_lm_head_linear_gb300 import fsdp  # noqa: E402

WORLD = 3
ALIGN = 8          # a small tile height, so that 37 vocabulary rows give several owner ranges
CUTS = [0, 30, 41, 97]


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _problem():
    rng = np.random.default_rng(7)
    N, d, V = 97, 12, 37
    H = rng.standard_normal((N, d))
    W = rng.standard_normal((V, d)) * 0.5
    y = rng.integers(0, V, N)
    y[rng.random(N) < 0.2] = -100
    return H, W, y


def _oracle_backend(H, W, y, grad_loss, bounds, n_valid_override, ignore_index=-100, **_):
    import oracle
    g = 1.0 if grad_loss is None else float(grad_loss)
    out = oracle.lce_f64(H.numpy(), W.numpy(), y.numpy(), n_valid_override=n_valid_override,
                         ignore_index=ignore_index, grad_loss=g)
    return (torch.tensor([out["loss"]], dtype=torch.float64), torch.from_numpy(out["lse"]),
            torch.from_numpy(out["dH"]), torch.from_numpy(out["dW"]).clone(), [None] * (len(bounds) - 1))


def _rank(rank, world, port, outdir, slices):
    import sys
    sys.path.insert(0, os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
    from chunked_lm_head_linear_gb300 import fsdp as F
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    H, W, y = _problem()
    owners = F.owner_bounds(W.shape[0], world, align=ALIGN)
    W_shard = torch.from_numpy(W[owners[rank]:owners[rank + 1]].copy())
    W_full = F.gather_weight(W_shard, owners)
    sl = slice(CUTS[rank], CUTS[rank + 1])
    loss, lse, dH, dW_own = F.fsdp_fwd_bwd(torch.from_numpy(H[sl]), W_full, torch.from_numpy(y[sl]),
                                           owners=owners, slices=slices, backend=_oracle_backend)
    np.savez(os.path.join(outdir, f"rank{rank}.npz"), W_full=W_full.numpy(), loss=loss.numpy(), lse=lse.numpy(),
             dH=dH.numpy(), dW_own=dW_own.numpy())
    dist.barrier()
    dist.destroy_process_group()


def test_owner_bounds_and_pieces():
    assert fsdp.owner_bounds(151936, 8) == [0, 18944, 37888, 56832, 76032, 94976, 113920, 132864, 151936]
    b = fsdp.owner_bounds(37, 3, align=8)
    assert b == [0, 8, 24, 37]
    assert all(x % 8 == 0 for x in b[1:-1])
    assert fsdp.owner_bounds(100, 1) == [0, 100]
    assert fsdp.owner_bounds(5, 4, align=8) == [0, 0, 0, 0, 5]       # more ranks than tiles: empty ranges
    pieces = fsdp.slice_pieces([0, 16, 32, 37], b)
    assert pieces == [[(0, 0, 8), (1, 8, 16)], [(1, 16, 24), (2, 24, 32)], [(2, 32, 37)]]
    # every row of the vocabulary lands in exactly one piece
    rows = sorted(r for ps in pieces for _, a, z in ps for r in range(a, z))
    assert rows == list(range(37))


@pytest.mark.parametrize("slices", [None, [0, 16, 32, 37], [0, 8, 8, 16, 24, 32, 37]])
def test_three_gloo_ranks_equal_unsharded(tmp_path, slices):
    import oracle
    port = _free_port()
    mp.start_processes(_rank, args=(WORLD, port, str(tmp_path), slices), nprocs=WORLD, join=True,
                       start_method="spawn")
    H, W, y = _problem()
    whole = oracle.lce_f64(H, W, y)
    owners = fsdp.owner_bounds(W.shape[0], WORLD, align=ALIGN)
    rs = [np.load(tmp_path / f"rank{r}.npz") for r in range(WORLD)]
    for r, out in enumerate(rs):
        np.testing.assert_array_equal(out["W_full"], W)
        assert float(out["loss"][0]) == pytest.approx(whole["loss"], rel=1e-13)
        np.testing.assert_allclose(out["dW_own"], whole["dW"][owners[r]:owners[r + 1]], rtol=1e-12, atol=1e-15)
    np.testing.assert_allclose(np.concatenate([o["dH"] for o in rs]), whole["dH"], rtol=1e-12, atol=1e-15)
    np.testing.assert_allclose(np.concatenate([o["lse"] for o in rs]), whole["lse"], rtol=1e-14)
