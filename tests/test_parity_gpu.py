"""Parity of the CUDA path (through the C ABI) with the fp64 CPU oracle.

Tolerances (u = 2^-8, the unit roundoff of bf16 round-to-nearest-even):
  loss: relative error <= 1e-3;  dH, dW: relative Frobenius error <= 5e-3 over
  the whole tensor (the spec bar);
  lse: max relative error <= 1e-4 (fp32 logits and sum-exp; the fp64 oracle
  differs only by fp32 accumulation and exp rounding, ~1e-7 measured);
  the softmax-only rows of dW (vocabulary rows no valid label hits) are also
  held to 5e-3 on their own, because in the full dW the one-hot rows dominate
  the norm and would hide an error in the softmax part;
  the ragged tails (the last partial 256-row tile of tokens and of the
  vocabulary, the last partial 256-column tile of d) are held to 5e-3 on their
  own as well.

Local bounds, derived from the roundings the fused path makes. It rounds
twice to bf16 on the way to each gradient: every entry of the exp tile
bf16(exp(z - m)) (the label entry after the one-hot is folded in) and then
either the dH output (dH = alpha (g/n) P W, fp32 accumulate, bf16 store) or
the dW operand Ht = bf16(alpha H) (dW = (g/n) P^T Ht, fp32 throughout). Each
rounding errs by at most u relative, so
  * per row: a gradient row made of a few terms (a dH row, which its label's
    term dominates; a dW row hit by one or two labels) errs by at most 2u
    (1 + a small softmax share) relative; a row that sums many terms (dW rows
    of frequent labels or of the softmax only) averages independent roundings
    to ~sqrt(2/3) u ~ 3.2e-3 relative with little spread. TOL_ROW = 1e-2 bounds
    ||row_gpu - row_ref|| / ||row_ref|| for every row (rows whose reference
    norm is below 1e-6 of the largest are held to that floor instead: their
    probabilities underflow fp32 and they carry no weight);
  * per element: |x_gpu - x_ref| <= 2u |x_ref| + 10u rms(row): the two
    roundings relative to the element, plus room for elements near zero,
    where a sum of independently rounded terms of the row's size leaves an
    error of ~sqrt(2/3) u rms(row) per element (10u is ~8 of its standard
    deviations; terms that cancel within an element add at most u per term).
A localised fault (one wrong row, one wrong 32-column group, a tail tile)
breaks these local bounds even when it hides in the whole-tensor norm.
"""
import os

import numpy as np
import pytest

import oracle
from chunked_lm_head_linear_gb300 import inputs

pytestmark = pytest.mark.gpu

TOL_LOSS = 1e-3
TOL_GRAD = 5e-3
TOL_LSE = 1e-4
GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _torch():
    import torch
    return torch


def to_dev(inp):
    torch = _torch()
    H = torch.from_numpy(np.ascontiguousarray(inp["H"]).view(np.int16)).view(torch.bfloat16).cuda()
    W = torch.from_numpy(np.ascontiguousarray(inp["W"]).view(np.int16)).view(torch.bfloat16).cuda()
    y = torch.from_numpy(np.ascontiguousarray(inp["y"])).cuda()
    return H, W, y


def rel_fro(a, b):
    a = np.asarray(a, dtype=np.float64)
    b = np.asarray(b, dtype=np.float64)
    den = np.linalg.norm(b)
    return float(np.linalg.norm(a - b) / (den if den > 0 else 1.0))


def bf16_to_np(t):
    torch = _torch()
    return t.float().cpu().numpy().astype(np.float64) if t.dtype == torch.bfloat16 else t.cpu().numpy()


def small_inputs(N, d, V, seed=0, ignore_frac=0.1, sigma_w=0.02, labels="uniform"):
    w = inputs.Workload(f"n{N}_d{d}_v{V}", N=N, d=d, V=V, sigma_w=sigma_w, labels=labels,
                        ignore="random" if ignore_frac > 0 else "none", ignore_frac=ignore_frac, seed=seed)
    return inputs.make_inputs(w)


U_BF16 = 2.0 ** -8
TOL_ROW = 1e-2
EL_REL = 2 * U_BF16
EL_RMS = 10 * U_BF16
ROW_FLOOR = 1e-6
TILE = 256


def local_errors(gpu, ref):
    """Largest per-row relative error and largest per-element error over its
    bound (EL_REL |ref| + EL_RMS rms(row)) of a gradient [rows, d] against the
    oracle's; both must stay <= TOL_ROW and <= 1. Rows whose reference is
    exactly zero (ignored tokens) must be exactly zero."""
    gpu = np.asarray(gpu, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    if ref.size == 0:
        return 0.0, 0.0
    diff = np.abs(gpu - ref)
    rn = np.linalg.norm(ref, axis=1)
    dn = np.linalg.norm(gpu - ref, axis=1)
    zero = rn == 0
    assert not np.any(np.abs(gpu[zero]) > 0), "rows whose gradient is zero are not zero"
    floor = ROW_FLOOR * rn.max() if rn.max() > 0 else 1e-300
    row = float(np.max(dn / np.maximum(rn, floor)))
    rms = np.maximum(rn, floor)[:, None] / np.sqrt(ref.shape[1])
    elem = float(np.max(diff / (EL_REL * np.abs(ref) + EL_RMS * rms)))
    return row, elem


def _tails(n, tile=TILE):
    """Indices of the last partial tile of a dimension of size n (empty if none)."""
    return np.arange((n // tile) * tile, n) if n % tile else np.arange(0)


def check_grad(name, gpu, ref, errs, row_tail=None):
    """Whole-tensor, tail, per-row and per-element checks of one gradient.
    ``row_tail`` selects the rows of the last partial tile (default: the last
    partial 256-row tile of ``ref``'s rows)."""
    gpu = np.asarray(gpu, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    fro = rel_fro(gpu, ref)
    row, elem = local_errors(gpu, ref)
    errs.update({name: fro, name + "_row": row, name + "_elem": elem})
    assert fro <= TOL_GRAD, (name, fro)
    assert row <= TOL_ROW, (name + " per row", row)
    assert elem <= 1.0, (name + " per element", elem)
    rt, ct = (_tails(ref.shape[0]) if row_tail is None else np.asarray(row_tail)), _tails(ref.shape[1])
    if rt.size and np.linalg.norm(ref[rt]) > 0:
        assert rel_fro(gpu[rt], ref[rt]) <= TOL_GRAD, (name + " row tail", rel_fro(gpu[rt], ref[rt]))
    if ct.size and np.linalg.norm(ref[:, ct]) > 0:
        assert rel_fro(gpu[:, ct], ref[:, ct]) <= TOL_GRAD, (name + " column tail", rel_fro(gpu[:, ct], ref[:, ct]))


def check_against_oracle(ref, y, loss, lse, dH=None, dW=None, V=None):
    import _parity_log
    errs = {"loss": abs(float(loss) - ref["loss"]) / max(abs(ref["loss"]), 1e-30)}
    lse = np.asarray(lse, dtype=np.float64)
    errs["lse"] = float(np.max(np.abs(lse - ref["lse"]) / np.maximum(np.abs(ref["lse"]), 1.0))) if lse.size else 0.0
    try:
        assert abs(float(loss) - ref["loss"]) <= TOL_LOSS * max(abs(ref["loss"]), 1e-30) + 1e-7
        assert errs["lse"] <= TOL_LSE
        if dH is not None:
            check_grad("dH", dH, ref["dH"], errs)
        if dW is not None:
            check_grad("dW", dW, ref["dW"], errs)
            hit = np.zeros(ref["dW"].shape[0], dtype=bool)
            yv = np.asarray(y)
            hit[yv[(yv != oracle.IGNORE_INDEX) & (yv >= 0) & (yv < hit.size)]] = True
            if (~hit).any() and np.linalg.norm(ref["dW"][~hit]) > 0:
                errs["dW_softmax_rows"] = rel_fro(dW[~hit], ref["dW"][~hit])
                assert errs["dW_softmax_rows"] <= TOL_GRAD
    finally:
        _parity_log.report(**errs)


# ---------------------------------------------------------------------------
# Small cases: full oracle, element by element
# ---------------------------------------------------------------------------

def test_tiny_workload_fwd_bwd(cuda_lib):
    inp = inputs.make_inputs("tiny_n256_d256_v4096")
    ref = oracle.lce_bf16(inp["H"], inp["W"], inp["y"])
    H, W, y = to_dev(inp)
    loss, lse, dH, dW = cuda_lib.lce_fwd_bwd(H, W, y, sync_check=True)
    check_against_oracle(ref, inp["y"], loss.item(), lse.cpu().numpy(), bf16_to_np(dH), dW.cpu().numpy())


def test_tiny_workload_split_forward_backward(cuda_lib):
    torch = _torch()
    inp = inputs.make_inputs("tiny_n256_d256_v4096")
    g = 0.37
    ref = oracle.lce_bf16(inp["H"], inp["W"], inp["y"], grad_loss=g)
    H, W, y = to_dev(inp)
    loss, lse = cuda_lib.lce_forward(H, W, y, sync_check=True)
    gl = torch.tensor([g], dtype=torch.float32, device="cuda")
    dH, dW = cuda_lib.lce_backward(H, W, y, lse, gl, sync_check=True)
    check_against_oracle(ref, inp["y"], loss.item(), lse.cpu().numpy(), bf16_to_np(dH), dW.cpu().numpy())


RAGGED = [
    # N, d, V, chunk      what it exercises
    (300, 136, 1000, 128),   # row tail, K tail (136 = 2*64 + 8), partial d tile, vocab tail
    (129, 72, 517, 64),      # one row past a tile, chunks smaller than a tile
    (513, 264, 4099, 200),   # chunk not a multiple of the tile, 3-column vocab tail
    (1, 64, 300, 0),         # a single token
    (40, 8, 2, 0),           # two classes, d = 8 (smallest legal hidden size)
    (200, 512, 257, 0),      # vocabulary one past a tile
    (37, 16, 1, 0),          # a single class: loss 0, zero gradients
    (600, 16384, 5000, 256), # wide hidden size: 256 k-blocks per logits tile, 64 dW column blocks
    (300, 64, 1000003, 0),   # a million-word vocabulary: dH parts of 3907 k-blocks, 3-column tail
]


@pytest.mark.parametrize("N,d,V,chunk", RAGGED)
def test_ragged_shapes(cuda_lib, N, d, V, chunk):
    inp = small_inputs(N, d, V, seed=N + d + V, sigma_w=0.05)
    ref = oracle.lce_bf16(inp["H"], inp["W"], inp["y"])
    H, W, y = to_dev(inp)
    loss, lse, dH, dW = cuda_lib.lce_fwd_bwd(H, W, y, chunk_tokens=chunk, sync_check=True)
    check_against_oracle(ref, inp["y"], loss.item(), lse.cpu().numpy(), bf16_to_np(dH), dW.cpu().numpy())


def test_large_logits_and_zipf_labels(cuda_lib):
    """Logit spread of tens of nats (sigma_w = 1): exercises the max subtraction."""
    inp = small_inputs(384, 128, 3000, seed=5, sigma_w=1.0, labels="zipf")
    ref = oracle.lce_bf16(inp["H"], inp["W"], inp["y"])
    H, W, y = to_dev(inp)
    loss, lse, dH, dW = cuda_lib.lce_fwd_bwd(H, W, y, chunk_tokens=256, sync_check=True)
    check_against_oracle(ref, inp["y"], loss.item(), lse.cpu().numpy(), bf16_to_np(dH), dW.cpu().numpy())


def test_reference_guard_falls_back_to_exact_gradient(cuda_lib):
    """The fused call stores and sums exp(z - ref) with ref = the row's maximum
    over the first 128 words. A word outside them whose logits reach ~80 sigma
    above it overflows those sums and trips the guard; the chunk must then be
    redone exactly (statistics, combine, gradient tile) and match the oracle."""
    inp = small_inputs(300, 64, 1000, seed=17, sigma_w=0.05)
    W = inputs.bf16_bits_to_f32(inp["W"]).astype(np.float64)
    W[700] = 10.0                                  # z_{i,700} = 10 * sum_k H_ik ~ N(0, 80^2)
    inp["W"] = inputs.f64_to_bf16_bits(W)
    ref = oracle.lce_bf16(inp["H"], inp["W"], inp["y"])
    assert np.max(ref["lse"]) > 100
    H, Wd, y = to_dev(inp)
    for chunk in (0, 128):
        loss, lse, dH, dW = cuda_lib.lce_fwd_bwd(H, Wd, y, chunk_tokens=chunk, sync_check=True)
        check_against_oracle(ref, inp["y"], loss.item(), lse.cpu().numpy(), bf16_to_np(dH), dW.cpu().numpy())


def test_reduction_sum_grad_scale_and_override(cuda_lib):
    torch = _torch()
    inp = small_inputs(300, 128, 1500, seed=9)
    H, W, y = to_dev(inp)
    gl = torch.tensor([2.5], dtype=torch.float32, device="cuda")
    ref = oracle.lce_bf16(inp["H"], inp["W"], inp["y"], reduction=oracle.SUM, grad_loss=2.5)
    loss, lse, dH, dW = cuda_lib.lce_fwd_bwd(H, W, y, gl, reduction="sum", sync_check=True)
    check_against_oracle(ref, inp["y"], loss.item(), lse.cpu().numpy(), bf16_to_np(dH), dW.cpu().numpy())
    ref = oracle.lce_bf16(inp["H"], inp["W"], inp["y"], n_valid_override=1000, grad_loss=2.5)
    loss, lse, dH, dW = cuda_lib.lce_fwd_bwd(H, W, y, gl, n_valid_override=1000, sync_check=True)
    check_against_oracle(ref, inp["y"], loss.item(), lse.cpu().numpy(), bf16_to_np(dH), dW.cpu().numpy())


def test_accumulate_dW(cuda_lib):
    torch = _torch()
    inp = small_inputs(256, 64, 700, seed=11)
    ref = oracle.lce_bf16(inp["H"], inp["W"], inp["y"])
    H, W, y = to_dev(inp)
    base = torch.randn(700, 64, device="cuda", dtype=torch.float32)
    dW = base.clone()
    cuda_lib.lce_fwd_bwd(H, W, y, dW=dW, accumulate_dW=True, chunk_tokens=96, sync_check=True)
    assert rel_fro((dW - base).cpu().numpy(), ref["dW"]) <= TOL_GRAD


def test_gradient_accumulation_over_micro_batches(cuda_lib):
    """Micro-batches run one after the other with the denominator of the whole
    batch and dW accumulated in place equal one call on the whole batch."""
    torch = _torch()
    inp = small_inputs(600, 128, 2000, seed=31)
    ref = oracle.lce_bf16(inp["H"], inp["W"], inp["y"])
    H, W, y = to_dev(inp)
    n = int((inp["y"] != oracle.IGNORE_INDEX).sum())
    dW = torch.empty(2000, 128, dtype=torch.float32, device="cuda")
    losses, dHs = [], []
    for k, sl in enumerate((slice(0, 250), slice(250, 600))):
        loss, _, dH, _ = cuda_lib.lce_fwd_bwd(H[sl], W, y[sl], dW=dW, n_valid_override=n, accumulate_dW=k > 0,
                                              chunk_tokens=128, sync_check=True)
        losses.append(loss.item())
        dHs.append(dH)
    assert abs(sum(losses) - ref["loss"]) <= TOL_LOSS * ref["loss"]
    assert rel_fro(torch.cat(dHs).float().cpu().numpy(), ref["dH"]) <= TOL_GRAD
    assert rel_fro(dW.cpu().numpy(), ref["dW"]) <= TOL_GRAD


def test_data_parallel_simulated_on_one_gpu(cuda_lib):
    """Data parallelism over tokens on one GPU: three uneven shards run in turn
    with the global count of valid labels, their dW and losses summed on the
    device in rank order. lse and dH are row-local, so they equal the unsharded
    call bit for bit; loss and dW differ only by fp32 reassociation of the
    sums (bound TOL_DW_CHUNKING, derived below)."""
    torch = _torch()
    inp = small_inputs(700, 256, 4096, seed=41)
    H, W, y = to_dev(inp)
    whole = cuda_lib.lce_fwd_bwd(H, W, y, chunk_tokens=128, sync_check=True)
    n = int((inp["y"] != oracle.IGNORE_INDEX).sum())
    cuts = [0, 190, 431, 700]
    loss = torch.zeros(1, device="cuda")
    dW = torch.zeros_like(whole[3])
    lses, dHs = [], []
    for a, b in zip(cuts[:-1], cuts[1:]):
        l_r, lse_r, dH_r, dW_r = cuda_lib.lce_fwd_bwd(H[a:b], W, y[a:b], n_valid_override=n, chunk_tokens=128,
                                                      sync_check=True)
        loss += l_r
        dW += dW_r
        lses.append(lse_r)
        dHs.append(dH_r)
    assert torch.equal(torch.cat(lses), whole[1]) and torch.equal(torch.cat(dHs), whole[2])
    assert abs(loss.item() - whole[0].item()) <= TOL_DW_CHUNKING * abs(whole[0].item())
    assert ((dW - whole[3]).norm() / whole[3].norm()).item() <= TOL_DW_CHUNKING


def test_auto_chunk(cuda_lib):
    inp = small_inputs(700, 256, 4096, seed=33)
    ref = oracle.lce_bf16(inp["H"], inp["W"], inp["y"])
    H, W, y = to_dev(inp)
    loss, lse, dH, dW = cuda_lib.lce_fwd_bwd(H, W, y, chunk_tokens="auto", sync_check=True)
    check_against_oracle(ref, inp["y"], loss.item(), lse.cpu().numpy(), bf16_to_np(dH), dW.cpu().numpy())


@pytest.mark.parametrize("cuts,chunk", [((0, 1000, 2600, 4099), 0), ((0, 257, 4099), 200), ((0, 4000, 4099), 512)])
def test_vocab_shards_on_one_gpu(cuda_lib, cuts, chunk):
    """Vocabulary-parallel pieces run shard after shard on one GPU: merged
    statistics give the full lse and loss, partial dH sum to dH, and the
    shards' dW rows stack to dW (shards of ragged sizes, one with few labels)."""
    torch = _torch()
    inp = small_inputs(700, 264, 4099, seed=37, sigma_w=0.05)
    ref = oracle.lce_bf16(inp["H"], inp["W"], inp["y"])
    H, W, y = to_dev(inp)
    shards = list(zip(cuts[:-1], cuts[1:]))
    stats = [cuda_lib.lce_vshard_forward_stats(H, W[a:b], y, a, 4099, chunk_tokens=chunk, sync_check=True)
             for a, b in shards]
    loss, lse = cuda_lib.lce_vshard_combine(torch.stack(stats).contiguous(), y, 4099, sync_check=True)
    dH = torch.zeros(700, 264, dtype=torch.float32, device="cuda")
    dWs = []
    for a, b in shards:
        dHp, dWp = cuda_lib.lce_vshard_backward(H, W[a:b].contiguous(), y, a, 4099, lse, chunk_tokens=chunk,
                                                sync_check=True)
        dH += dHp
        dWs.append(dWp)
    check_against_oracle(ref, inp["y"], loss.item(), lse.cpu().numpy(), dH.cpu().numpy().astype(np.float64),
                         torch.cat(dWs).cpu().numpy())
    # the fused single-device call and the sharded route agree on lse
    _, lse_full, _, _ = cuda_lib.lce_fwd_bwd(H, W, y, sync_check=True)
    assert ((lse - lse_full).abs() / lse_full.abs()).max().item() <= TOL_LSE


def vshard_stored(cuda_lib, H, W, y, cuts, chunk, **kw):
    """The stored-tile vocabulary-parallel schedule with the shards run in turn
    on one GPU: per chunk every shard's statistics (each shard keeps its exp
    tile in its own workspace), their rank-order stack in place of the
    all-gather, then every shard's chunk backward; the loss from the merge of
    all chunks' statistics, the partial dH summed by torch in place of the
    all-reduce. Returns loss, lse, dH (fp32), dW (the shards' rows stacked)."""
    torch = _torch()
    N, d = H.shape
    V = W.shape[0]
    shards = list(zip(cuts[:-1], cuts[1:]))
    C = max(1, min(chunk or 4096, N))
    ws = [cuda_lib.vshard_chunk_workspace(H, W[a:b], y, chunk_tokens=C, **kw) for a, b in shards]
    lse = torch.empty(N, dtype=torch.float32, device="cuda")
    dHp = [torch.empty((N, d), dtype=torch.float32, device="cuda") for _ in shards]
    dW = torch.empty((V, d), dtype=torch.float32, device="cuda")
    per_chunk = []
    for c0 in range(0, N, C):
        rows = min(C, N - c0)
        st = torch.stack([cuda_lib.lce_vshard_chunk_stats(H, W[a:b], y, a, V, c0, rows, workspace=ws[k],
                                                          chunk_tokens=C, **kw)
                          for k, (a, b) in enumerate(shards)]).contiguous()
        for k, (a, b) in enumerate(shards):
            cuda_lib.lce_vshard_chunk_backward(H, W[a:b], y, a, V, c0, rows, st, workspace=ws[k], lse=lse,
                                               dH_partial=dHp[k], dW_shard=dW[a:b], chunk_tokens=C, **kw)
        per_chunk.append(st)
    loss, lse2 = cuda_lib.lce_vshard_combine(torch.cat(per_chunk, dim=1).contiguous(), y, V, **kw)
    assert torch.equal(lse, lse2)          # the chunk backward's merge is the combine's
    dH = dHp[0]
    for p in dHp[1:]:
        dH += p
    return loss, lse, dH, dW


@pytest.mark.parametrize("cuts,chunk", [((0, 1000, 2600, 4099), 0), ((0, 257, 4099), 200), ((0, 4000, 4099), 512)])
def test_vocab_shards_stored_tiles(cuda_lib, cuts, chunk):
    """The stored-tile shard calls (statistics and exp tile per chunk, backward
    from the kept tile) against the oracle and against the recomputing calls."""
    torch = _torch()
    inp = small_inputs(700, 264, 4099, seed=37, sigma_w=0.05)
    ref = oracle.lce_bf16(inp["H"], inp["W"], inp["y"])
    H, W, y = to_dev(inp)
    loss, lse, dH, dW = vshard_stored(cuda_lib, H, W, y, cuts, chunk, sync_check=True)
    check_against_oracle(ref, inp["y"], loss.item(), lse.cpu().numpy(), dH.cpu().numpy().astype(np.float64),
                         dW.cpu().numpy())
    stats = [cuda_lib.lce_vshard_forward_stats(H, W[a:b], y, a, 4099, chunk_tokens=chunk)
             for a, b in zip(cuts[:-1], cuts[1:])]
    loss_r, lse_r = cuda_lib.lce_vshard_combine(torch.stack(stats).contiguous(), y, 4099)
    assert torch.equal(lse, lse_r) and torch.equal(loss, loss_r)   # the same statistics, merged the same way


def test_vocab_shards_stored_tiles_guard(cuda_lib):
    """A word far above its shard's row reference (outside the shard's first
    128 words) trips that shard's guard: its chunk gets the exact gradient tile
    from the exchanged statistics; the other shard keeps its stored tile."""
    inp = small_inputs(300, 64, 1000, seed=17, sigma_w=0.05)
    W = inputs.bf16_bits_to_f32(inp["W"]).astype(np.float64)
    W[700] = 10.0                                  # z_{i,700} = 10 * sum_k H_ik ~ N(0, 80^2)
    inp["W"] = inputs.f64_to_bf16_bits(W)
    ref = oracle.lce_bf16(inp["H"], inp["W"], inp["y"])
    H, Wd, y = to_dev(inp)
    for chunk in (0, 128):
        loss, lse, dH, dW = vshard_stored(cuda_lib, H, Wd, y, (0, 500, 1000), chunk, sync_check=True)
        check_against_oracle(ref, inp["y"], loss.item(), lse.cpu().numpy(), dH.cpu().numpy().astype(np.float64),
                             dW.cpu().numpy())


@pytest.mark.parametrize("N,d", [(300, 64), (517, 2048), (130, 7168)])
def test_rmsnorm_forward_backward(cuda_lib, N, d):
    torch = _torch()
    rng = np.random.default_rng(N + d)
    xb = inputs.f64_to_bf16_bits(rng.standard_normal((N, d)) * 3)
    w = (rng.standard_normal(d) * 0.1).astype(np.float32)
    dHb = inputs.f64_to_bf16_bits(rng.standard_normal((N, d)) * 1e-3)
    x = torch.from_numpy(xb.view(np.int16)).view(torch.bfloat16).cuda()
    wt = torch.from_numpy(w).cuda()
    dH = torch.from_numpy(dHb.view(np.int16)).view(torch.bfloat16).cuda()
    H, rstd = cuda_lib.lce_rmsnorm_forward(x, wt, 1e-6)
    dx, dw = cuda_lib.lce_rmsnorm_backward(x, wt, rstd, dH)
    xo = oracle.decode_bf16(xb)
    h, r = oracle.rmsnorm_f64(xo, w.astype(np.float64), 1e-6)
    # one bf16 rounding of an fp32 product: within one bf16 ulp of the exact value
    assert np.max(np.abs(bf16_to_np(H) - h) / np.maximum(np.abs(h), 1e-30)) <= 2.0 ** -8
    np.testing.assert_allclose(rstd.cpu().numpy(), r, rtol=1e-5)
    dx_ref, dw_ref = oracle.rmsnorm_backward_f64(xo, w.astype(np.float64), r, oracle.decode_bf16(dHb))
    assert rel_fro(bf16_to_np(dx), dx_ref) <= TOL_GRAD
    assert rel_fro(dw.cpu().numpy(), dw_ref) <= 1e-4


def test_norm_fwd_bwd_matches_oracle(cuda_lib):
    """Norm -> fused linear cross-entropy -> norm backward in one call."""
    torch = _torch()
    inp = small_inputs(600, 256, 4096, seed=57, sigma_w=0.05)
    rng = np.random.default_rng(57)
    w = (rng.standard_normal(256) * 0.1).astype(np.float32)
    xb = inputs.f64_to_bf16_bits(rng.standard_normal((600, 256)) * 2)
    ref = oracle.norm_lce_bf16(xb, w.astype(np.float64), inp["W"], inp["y"], 1e-6)
    x = torch.from_numpy(xb.view(np.int16)).view(torch.bfloat16).cuda()
    _, W, y = to_dev(inp)
    loss, lse, dx, dw_norm, dW = cuda_lib.lce_norm_fwd_bwd(x, torch.from_numpy(w).cuda(), W, y, chunk_tokens=256,
                                                           sync_check=True)
    check_against_oracle(ref, inp["y"], loss.item(), lse.cpu().numpy(), None, dW.cpu().numpy())
    assert rel_fro(bf16_to_np(dx), ref["dx"]) <= TOL_GRAD
    assert rel_fro(dw_norm.cpu().numpy(), ref["dw_norm"]) <= TOL_GRAD


@pytest.mark.parametrize("recompute", [False, True])
def test_autograd_wrapper(cuda_lib, recompute):
    """loss.backward() through the torch.autograd wrapper, with an upstream
    gradient of 1 and of 2.5 (the loss scaled before backward)."""
    torch = _torch()
    from chunked_lm_head_linear_gb300.autograd import FusedLinearCrossEntropy
    inp = small_inputs(400, 128, 3000, seed=61)
    for scale in (1.0, 2.5):
        ref = oracle.lce_bf16(inp["H"], inp["W"], inp["y"], grad_loss=scale)
        H, W, y = to_dev(inp)
        H.requires_grad_(True)
        W.requires_grad_(True)
        loss = FusedLinearCrossEntropy(recompute=recompute, chunk_tokens=128)(H, W, y)
        (loss * scale).backward()
        assert abs(loss.item() - ref["loss"]) <= TOL_LOSS * ref["loss"]
        assert rel_fro(bf16_to_np(H.grad), ref["dH"]) <= TOL_GRAD
        assert rel_fro(W.grad.float().cpu().numpy(), ref["dW"]) <= TOL_GRAD


def test_binding_rejects_bad_caller_tensors(cuda_lib):
    """Outputs, saved lse, upstream gradient and workspace passed by the caller
    are checked before any launch, so a wrong one cannot send a kernel past it."""
    torch = _torch()
    inp = small_inputs(64, 64, 300, seed=9)
    H, W, y = to_dev(inp)
    bad = [dict(dW=torch.zeros(300, 64, dtype=torch.float64, device="cuda")),
           dict(dW=torch.zeros(299, 64, device="cuda")),
           dict(dW=torch.zeros(64, 300, device="cuda").t()),
           dict(lse=torch.zeros(63, device="cuda")),
           dict(grad_loss=torch.ones(1, dtype=torch.float64, device="cuda")),
           dict(workspace=torch.zeros(1 << 20, dtype=torch.float32, device="cuda"))]
    for kw in bad:
        with pytest.raises(ValueError):
            cuda_lib.lce_fwd_bwd(H, W, y, **kw)
    with pytest.raises(ValueError):
        cuda_lib.lce_backward(H, W, y, torch.zeros(64, dtype=torch.float16, device="cuda"))
    with pytest.raises(ValueError):
        cuda_lib.lce_scale_grads(None, torch.zeros(300, 64, device="cuda"), torch.ones(1, device="cuda").half())
    # accumulating needs the caller's dW to add into
    with pytest.raises(ValueError):
        cuda_lib.lce_fwd_bwd(H, W, y, accumulate_dW=True)
    with pytest.raises(ValueError):
        cuda_lib.lce_backward(H, W, y, torch.zeros(64, device="cuda"), accumulate_dW=True)


def test_all_ignored_and_empty(cuda_lib):
    torch = _torch()
    inp = small_inputs(130, 64, 600, seed=3)
    inp["y"][:] = oracle.IGNORE_INDEX
    ref = oracle.lce_bf16(inp["H"], inp["W"], inp["y"])
    H, W, y = to_dev(inp)
    loss, lse, dH, dW = cuda_lib.lce_fwd_bwd(H, W, y, sync_check=True)
    assert loss.item() == 0.0
    assert torch.count_nonzero(dH).item() == 0 and torch.count_nonzero(dW).item() == 0
    np.testing.assert_allclose(lse.cpu().numpy(), ref["lse"], rtol=TOL_LSE)
    # N = 0
    H0 = H[:0]
    y0 = y[:0]
    loss, lse, dH, dW = cuda_lib.lce_fwd_bwd(H0, W, y0, sync_check=True)
    assert loss.item() == 0.0 and lse.numel() == 0 and torch.count_nonzero(dW).item() == 0


def test_label_out_of_range_is_reported_and_ignored(cuda_lib):
    inp = small_inputs(200, 64, 500, seed=4)
    y_bad = inp["y"].copy()
    y_bad[[7, 150]] = [500, -3]
    H, W, _ = to_dev(inp)
    torch = _torch()
    y = torch.from_numpy(y_bad).cuda()
    with pytest.raises(cuda_lib.LCEError) as e:
        cuda_lib.lce_fwd_bwd(H, W, y, sync_check=True)
    assert e.value.code == cuda_lib.LCE_ERR_LABEL_RANGE
    # without sync_check the call returns OK, the status bit is set, and the
    # bad rows count as ignored
    ws = torch.empty(cuda_lib.workspace_size(cuda_lib.LCE_OP_FWD_BWD, 200, 64, 500), dtype=torch.uint8,
                     device="cuda")
    loss, lse, dH, dW = cuda_lib.lce_fwd_bwd(H, W, y, workspace=ws)
    assert cuda_lib.read_device_status(ws) & cuda_lib.LCE_DEVICE_LABEL_RANGE
    y_ign = y_bad.copy()
    y_ign[[7, 150]] = oracle.IGNORE_INDEX
    ref = oracle.lce_bf16(inp["H"], inp["W"], y_ign)
    check_against_oracle(ref, y_ign, loss.item(), lse.cpu().numpy(), bf16_to_np(dH), dW.cpu().numpy())


def test_cuda_graph_capture_and_replay(cuda_lib):
    """lce_fwd_bwd captured into a CUDA graph (its launches, tensor maps and
    workspace carve-up fixed at capture) and replayed on new inputs copied into
    the captured buffers gives the eager call's results bit for bit."""
    torch = _torch()
    N, d, V, chunk = 700, 256, 4096, 256
    H, W, y = to_dev(small_inputs(N, d, V, seed=71))
    ws = torch.empty(cuda_lib.workspace_size(cuda_lib.LCE_OP_FWD_BWD, N, d, V, cuda_lib.make_opts(chunk_tokens=chunk)),
                     dtype=torch.uint8, device="cuda")
    dW = torch.empty((V, d), dtype=torch.float32, device="cuda")
    lse = torch.empty(N, dtype=torch.float32, device="cuda")
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):                       # warm-up off the default stream, as torch asks
        cuda_lib.lce_fwd_bwd(H, W, y, dW=dW, lse=lse, workspace=ws, chunk_tokens=chunk)
    torch.cuda.current_stream().wait_stream(side)
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        loss, lse_g, dH, dW_g = cuda_lib.lce_fwd_bwd(H, W, y, dW=dW, lse=lse, workspace=ws, chunk_tokens=chunk)
    for seed in (72, 73):
        H2, W2, y2 = to_dev(small_inputs(N, d, V, seed=seed))
        H.copy_(H2)
        W.copy_(W2)
        y.copy_(y2)
        g.replay()
        ref = cuda_lib.lce_fwd_bwd(H2, W2, y2, chunk_tokens=chunk)
        torch.cuda.synchronize()
        for a, b in zip((loss, lse_g, dH, dW_g), ref):
            assert torch.equal(a, b)


def test_two_streams_at_once(cuda_lib):
    """Calls on two streams with their own workspaces, issued interleaved so that
    their kernels may run side by side: each gives what it gives alone."""
    torch = _torch()
    probs = [to_dev(small_inputs(700, 256, 4096, seed=s)) for s in (91, 92)]
    alone = [cuda_lib.lce_fwd_bwd(H, W, y, chunk_tokens=256) for H, W, y in probs]
    torch.cuda.synchronize()
    streams = [torch.cuda.Stream(), torch.cuda.Stream()]
    for s in streams:
        s.wait_stream(torch.cuda.current_stream())
    outs = [[], []]
    for _ in range(3):
        for k, (H, W, y) in enumerate(probs):
            outs[k].append(cuda_lib.lce_fwd_bwd(H, W, y, chunk_tokens=256, stream=streams[k]))
    torch.cuda.synchronize()
    for k in range(2):
        for o in outs[k]:
            for a, b in zip(o, alone[k]):
                assert torch.equal(a, b)


def test_stream_order_with_other_kernels_between_calls(cuda_lib):
    """The library launches its kernels so that each may start while the kernel
    before it in the stream finishes, and each waits at its start for that
    kernel to complete. Interleaved with PyTorch kernels on the same stream that
    rewrite the inputs and read and clear the outputs in between, every call
    still sees the inputs as the stream left them and leaves outputs the next
    kernel sees whole: each result equals the same call made alone."""
    torch = _torch()
    H, W, y = to_dev(small_inputs(700, 256, 4096, seed=95))
    Hn = -H
    ref_pos = cuda_lib.lce_fwd_bwd(H, W, y, chunk_tokens=256)
    ref_neg = cuda_lib.lce_fwd_bwd(Hn, W, y, chunk_tokens=256)
    torch.cuda.synchronize()
    ref_pos = [t.clone() for t in ref_pos]
    ref_neg = [t.clone() for t in ref_neg]
    Hx = H.clone()
    dW = torch.zeros_like(ref_pos[3])
    outs, dWs = [], []
    for k in range(4):                     # no host synchronisation inside the loop
        Hx.neg_()                          # a PyTorch kernel rewrites the input just before the call
        loss, lse, dH, _ = cuda_lib.lce_fwd_bwd(Hx, W, y, dW=dW, chunk_tokens=256)
        dWs.append(dW.clone())             # read the output at once
        dW.zero_()                         # and clear it right after
        outs.append((loss, lse, dH))
    torch.cuda.synchronize()
    for k, ((loss, lse, dH), dWk) in enumerate(zip(outs, dWs)):
        ref = ref_neg if k % 2 == 0 else ref_pos
        assert torch.equal(loss, ref[0]) and torch.equal(lse, ref[1]) and torch.equal(dH, ref[2]), k
        assert torch.equal(dWk, ref[3]), k


def test_chunk_size_invariance_and_determinism(cuda_lib):
    """loss, lse and dH are row-local with a fixed vocabulary order: bitwise
    equal for every chunk size; dW differs only by fp32 reassociation."""
    torch = _torch()
    inp = small_inputs(700, 256, 4096, seed=21)
    ref = oracle.lce_bf16(inp["H"], inp["W"], inp["y"])
    H, W, y = to_dev(inp)
    outs = {}
    for C in (64, 128, 256, 700, 1000):
        outs[C] = cuda_lib.lce_fwd_bwd(H, W, y, chunk_tokens=C, sync_check=True)
    base = outs[128]
    for C, o in outs.items():
        assert torch.equal(o[0], base[0]), C
        assert torch.equal(o[1], base[1]), C
        assert torch.equal(o[2], base[2]), C
        assert rel_fro(o[3].cpu().numpy(), base[3].cpu().numpy()) <= TOL_DW_CHUNKING, C
        check_against_oracle(ref, inp["y"], o[0].item(), o[1].cpu().numpy(), bf16_to_np(o[2]), o[3].cpu().numpy())
    again = cuda_lib.lce_fwd_bwd(H, W, y, chunk_tokens=128, sync_check=True)
    for a, b in zip(again, base):
        assert torch.equal(a, b)


# ---------------------------------------------------------------------------
# Full-size workloads: sampled rows against the oracle, properties on all of it
# ---------------------------------------------------------------------------

def _stratified_rows(y, N, rng, k=128):
    ign = np.nonzero(y == oracle.IGNORE_INDEX)[0]
    frequent = np.nonzero(y == 0)[0]
    picks = [np.arange(min(8, N)), np.arange(max(0, N - 8), N), ign[:8], frequent[:8],
             rng.choice(N, size=k, replace=False)]
    return np.unique(np.concatenate(picks))[:k + 40]


def _stratified_vocab(V, y, rng, k=128):
    labels, counts = np.unique(y[y != oracle.IGNORE_INDEX], return_counts=True)
    top = labels[np.argsort(-counts)[:8]]
    tail_tile = np.arange(max(0, V - 64), V)
    picks = [np.arange(10), top, tail_tile[:: max(1, tail_tile.size // 16)], [V - 1],
             rng.choice(V, size=k, replace=False)]
    return np.unique(np.concatenate(picks))


def sampled_full_check(cuda_lib, name, chunk_tokens=0, compute=None):
    """``compute(H, W, y) -> (loss, lse, dH, dW)`` on the device; by default the
    fused call ``lce_fwd_bwd`` with ``chunk_tokens``."""
    torch = _torch()
    gpath = os.path.join(GOLDEN, f"full_{name}.npz")
    if not os.path.exists(gpath):
        pytest.fail(f"missing cached oracle values {gpath} (tests/golden/make_full_golden.py writes them)")
    gold = np.load(gpath)
    inp = inputs.make_inputs(name)
    if str(gold["digest"]) != inputs.input_digest(inp):
        pytest.fail("input generator output differs from the one the cached oracle values were made for")
    w = inp["workload"]
    y_np = inp["y"]
    H, W, y = to_dev(inp)
    if compute is None:
        loss, lse, dH, dW = cuda_lib.lce_fwd_bwd(H, W, y, chunk_tokens=chunk_tokens, sync_check=True)
    else:
        loss, lse, dH, dW = compute(H, W, y)
    torch.cuda.synchronize()
    import _parity_log
    errs = {}
    try:
        # loss and every lse against the oracle
        errs["loss"] = abs(loss.item() - float(gold["loss"])) / abs(float(gold["loss"]))
        assert errs["loss"] <= TOL_LOSS
        lse_np = lse.cpu().numpy().astype(np.float64)
        errs["lse"] = float(np.max(np.abs(lse_np - gold["lse"]) / np.maximum(np.abs(gold["lse"]), 1.0)))
        assert errs["lse"] <= TOL_LSE
        # sampled rows of dH and vocabulary rows of dW: whole-sample, per-row and
        # per-element bounds, the rows of the last partial tiles on their own
        rng = np.random.default_rng(123)
        Hf = inputs.bf16_bits_to_f32(inp["H"])
        Wf = inputs.bf16_bits_to_f32(inp["W"])
        scale, _ = oracle.grad_scale(y_np)
        R = _stratified_rows(y_np, w.N, rng)
        dH_ref = oracle.dH_rows_f64(Hf, Wf, y_np, R, scale)
        dH_gpu = dH[torch.from_numpy(R).cuda()].float().cpu().numpy()
        check_grad("dH", dH_gpu, dH_ref, errs, row_tail=np.nonzero(np.isin(R, _tails(w.N)))[0])
        S = _stratified_vocab(w.V, y_np, rng)
        dW_ref = oracle.dW_rows_f64(Hf, Wf, y_np, gold["lse"], S, scale)
        dW_gpu = dW[torch.from_numpy(S).cuda()].cpu().numpy()
        check_grad("dW", dW_gpu, dW_ref, errs, row_tail=np.nonzero(np.isin(S, _tails(w.V)))[0])
        hit = np.isin(S, y_np[y_np != oracle.IGNORE_INDEX])
        if (~hit).sum() > 4:
            errs["dW_softmax_rows"] = rel_fro(dW_gpu[~hit], dW_ref[~hit])
            assert errs["dW_softmax_rows"] <= TOL_GRAD
        # properties on the whole outputs: sum_v dW_v = 0 and <dH, H> = <dW, W>
        colsum = dW.double().sum(dim=0)
        errs["sum_v_dW"] = (colsum.norm() / dW.double().norm()).item()
        assert errs["sum_v_dW"] <= TOL_GRAD
        a = (dH.double() * H.double()).sum().item()
        b = (dW.double() * W.double()).sum().item()
        errs["dH.H-dW.W"] = abs(a - b) / max(abs(a), abs(b))
        assert errs["dH.H-dW.W"] <= TOL_GRAD
    finally:
        _parity_log.report(**errs)
    return loss, lse, dH, dW


def test_full_qwen2b_workload(cuda_lib):
    sampled_full_check(cuda_lib, "qwen2b_n8192_d2048_v151936")


@pytest.mark.slow
@pytest.mark.parametrize("name", ["qwen2b_n8192_d2048_v151936", "packed_n32768_d2048_v151936"])
def test_full_tensor_parity(cuda_lib, name):
    """Every row and element of dH and dW at full size against the full fp64
    oracle, computed here on the host cores at test time (about a minute for
    the 8192-token head, about four for the 32768-token packed batch), in the
    launch configuration bench.py times: the fused call, 4096-token chunks.
    The loss, every lse and both gradients are held to the whole-tensor,
    tail, per-row and per-element bounds of check_against_oracle."""
    torch = _torch()
    inp = inputs.make_inputs(name)
    H, W, y = to_dev(inp)
    loss, lse, dH, dW = cuda_lib.lce_fwd_bwd(H, W, y, chunk_tokens=4096, sync_check=True)
    torch.cuda.synchronize()
    got = (loss.item(), lse.cpu().numpy(), bf16_to_np(dH), dW.cpu().numpy())
    del H, W, y, loss, lse, dH, dW
    torch.cuda.empty_cache()
    ref = oracle.lce_bf16(inp["H"], inp["W"], inp["y"])
    check_against_oracle(ref, inp["y"], *got)


def test_full_qwen2b_split_path(cuda_lib):
    """lce_forward then lce_backward (the backward recomputes the logits from the
    saved lse into the exact gradient tile) at the bench workload's size, in the
    launch configuration of bench.py --path split."""

    def split(H, W, y):
        loss, lse = cuda_lib.lce_forward(H, W, y, chunk_tokens=4096, sync_check=True)
        dH, dW = cuda_lib.lce_backward(H, W, y, lse, chunk_tokens=4096, sync_check=True)
        return loss, lse, dH, dW

    sampled_full_check(cuda_lib, "qwen2b_n8192_d2048_v151936", compute=split)


def test_full_qwen2b_vocab_shards(cuda_lib):
    """The vocabulary-parallel calls at the bench workload, four uneven shards
    run in turn on one GPU (the launch configuration of bench.py --path vshard):
    per-shard statistics, the rank-order merge, the shard backward; the partial
    dH summed by torch in place of the all-reduce."""
    torch = _torch()

    def shards(H, W, y):
        V = W.shape[0]
        cuts = [0, 37000, 76032, 114000, V]
        stats = [cuda_lib.lce_vshard_forward_stats(H, W[a:b], y, a, V, chunk_tokens=4096)
                 for a, b in zip(cuts[:-1], cuts[1:])]
        loss, lse = cuda_lib.lce_vshard_combine(torch.stack(stats), y, V)
        dW = torch.empty((V, W.shape[1]), dtype=torch.float32, device="cuda")
        dH = None
        for a, b in zip(cuts[:-1], cuts[1:]):
            part, _ = cuda_lib.lce_vshard_backward(H, W[a:b], y, a, V, lse, dW=dW[a:b], chunk_tokens=4096)
            dH = part if dH is None else dH.add_(part)
        return loss, lse, dH, dW

    sampled_full_check(cuda_lib, "qwen2b_n8192_d2048_v151936", compute=shards)


def test_full_qwen2b_vocab_shards_stored(cuda_lib):
    """The stored-tile shard calls at the bench workload (bench.py --path
    vshard): four uneven shards run in turn on one GPU, chunk 4096."""

    def stored(H, W, y):
        V = W.shape[0]
        return vshard_stored(cuda_lib, H, W, y, [0, 37000, 76032, 114000, V], 4096)

    sampled_full_check(cuda_lib, "qwen2b_n8192_d2048_v151936", compute=stored)


def test_full_qwen2b_norm_fwd_bwd(cuda_lib):
    """Final RMSNorm + head at the bench workload's size (x = the workload's
    hidden states, w ~ N(0, 0.1), eps 1e-6): lse and dx on sampled rows against
    the oracle (norm -> bf16 H -> rows of the cross-entropy -> norm backward),
    the loss from the GPU's lse and the oracle's label logits, dW on sampled
    vocabulary rows, and dw_norm through sum_k (1 + w_k) dw_k = <dH, H> = <dW, W>."""
    torch = _torch()
    name = "qwen2b_n8192_d2048_v151936"
    inp = inputs.make_inputs(name)
    wl = inp["workload"]
    y_np = inp["y"]
    wn = np.random.default_rng(99).normal(0.0, 0.1, wl.d).astype(np.float32)
    x, W, y = to_dev(inp)
    loss, lse, dx, dw_norm, dW = cuda_lib.lce_norm_fwd_bwd(x, torch.from_numpy(wn).cuda(), W, y, eps=1e-6,
                                                           chunk_tokens=4096, sync_check=True)
    torch.cuda.synchronize()
    xf = inputs.bf16_bits_to_f32(inp["H"]).astype(np.float64)
    Wf = inputs.bf16_bits_to_f32(inp["W"])
    h, r = oracle.rmsnorm_f64(xf, wn.astype(np.float64), 1e-6)
    Hb = oracle.decode_bf16(oracle.round_bf16_bits(h))
    scale, n = oracle.grad_scale(y_np)
    rng = np.random.default_rng(321)
    R = _stratified_rows(y_np, wl.N, rng)
    fw = oracle.forward_rows_f64(Hb, Wf, y_np, R)
    lse_gpu = lse.cpu().numpy().astype(np.float64)
    assert np.max(np.abs(lse_gpu[R] - fw["lse"]) / np.maximum(np.abs(fw["lse"]), 1.0)) <= TOL_LSE
    valid = y_np != oracle.IGNORE_INDEX
    z_y = np.einsum("ij,ij->i", Hb[valid], Wf.astype(np.float64)[y_np[valid]])
    loss_from_lse = float((lse_gpu[valid] - z_y).sum() / n)
    assert abs(loss.item() - loss_from_lse) <= TOL_LOSS * abs(loss_from_lse)
    dH_R = oracle.dH_rows_f64(Hb, Wf, y_np, R, scale)
    dx_R, _ = oracle.rmsnorm_backward_f64(xf[R], wn.astype(np.float64), r[R], dH_R)
    assert rel_fro(dx[torch.from_numpy(R).cuda()].float().cpu().numpy(), dx_R) <= TOL_GRAD
    S = _stratified_vocab(wl.V, y_np, rng)
    dW_ref = oracle.dW_rows_f64(Hb, Wf, y_np, lse_gpu, S, scale)
    assert rel_fro(dW[torch.from_numpy(S).cuda()].cpu().numpy(), dW_ref) <= TOL_GRAD
    a = float((torch.from_numpy(1.0 + wn.astype(np.float64)).cuda() * dw_norm.double()).sum().item())
    b = (dW.double() * W.double()).sum().item()
    assert abs(a - b) <= TOL_GRAD * max(abs(a), abs(b))


@pytest.mark.slow
def test_full_packed_workload(cuda_lib):
    sampled_full_check(cuda_lib, "packed_n32768_d2048_v151936")


@pytest.mark.slow
@pytest.mark.parametrize("name", ["moe_n16384_d7168_v129280", "moe_n16384_d7168_v151655"])
def test_full_moe_workloads(cuda_lib, name):
    sampled_full_check(cuda_lib, name)


# dW sums its N token terms in fp32, and the chunking decides the order of the
# additions: inside the dW GEMM a chunk's C tokens go into the fp32 accumulator
# in K steps of 16 (one rounding per MMA), then the chunks' partials are added
# one after another by the TMA reduce-adds. A chain of L fp32 additions errs by
# at most about L * 2^-24 * sum|addends| (first order), and the addends here (a
# chunk's running sum, the chunk partials) stay within about twice |dW| (their
# softmax and one-hot parts partly cancel). Two chunkings with chains
# L = ceil(C / 16) + ceil(N / C) therefore differ by at most
# (L1 + L2) * 2^-24 * 2 relative, a worst case: measured 1.5e-6 between chunks
# of 1024 and 8192 tokens of the 64k head (model: 7.7e-5), 1.6e-5 between 16384
# and 4096 on the 32768-token batch (model: 1.5e-4). The small cases (N = 700,
# chunks of 64 to 1000 tokens, model at most 7e-6) use the fixed 1e-5 below.
TOL_DW_CHUNKING = 1e-5


def tol_dw_chunking(N, *chunks):
    """The chain bound above for chunkings of N tokens into chunks of the given sizes (not below 1e-5)."""
    chain = sum(-(-min(C, N) // 16) + -(-N // min(C, N)) for C in chunks)
    return max(TOL_DW_CHUNKING, chain * 2.0 ** -24 * 2)


@pytest.mark.slow
def test_chunk_past_2_31_exp_tile_entries(cuda_lib):
    """32768-token packed batch in two chunks of 16384 tokens: each chunk's exp
    tile holds 16384 x 151936 = 2.49e9 entries, past 2^31, so any 32-bit
    element offset into it would wrap. Sampled rows against the oracle, and
    loss, lse and dH bitwise equal to the same call in 4096-token chunks (dW
    within the fp32 reassociation bound)."""
    torch = _torch()
    name = "packed_n32768_d2048_v151936"
    big = sampled_full_check(cuda_lib, name, chunk_tokens=16384)
    assert 16384 * 151936 > 2 ** 31
    inp = inputs.make_inputs(name)
    H, W, y = to_dev(inp)
    loss, lse, dH, dW = cuda_lib.lce_fwd_bwd(H, W, y, chunk_tokens=4096, sync_check=True)
    torch.cuda.synchronize()
    assert torch.equal(loss, big[0]) and torch.equal(lse, big[1]) and torch.equal(dH, big[2])
    assert ((dW - big[3]).norm() / dW.norm()).item() <= tol_dw_chunking(32768, 16384, 4096)
    del H, W, y, loss, lse, dH, dW, big
    torch.cuda.empty_cache()


@pytest.mark.slow
def test_full_seq64k_chunk_sweep(cuda_lib):
    """64k-token head, chunk sizes 512..8192: every chunk size within the oracle
    tolerance; loss, lse and dH bitwise equal across chunk sizes; dW within the
    fp32 reassociation bound tol_dw_chunking."""
    torch = _torch()
    name = "seq64k_n65536_d4096_v151936"
    first = None
    # 512 deals the dH parts one by one, 1024 and up a block at a time (the schedule differs, the
    # arithmetic of every output element does not)
    for C in (512, 1024, 2048, 4096, 8192):
        loss, lse, dH, dW = sampled_full_check(cuda_lib, name, chunk_tokens=C)
        if first is None:
            first = (loss.clone(), lse.clone(), dH.clone(), dW.clone())
        else:
            assert torch.equal(loss, first[0]) and torch.equal(lse, first[1]) and torch.equal(dH, first[2])
            assert ((dW - first[3]).norm() / first[3].norm()).item() <= tol_dw_chunking(65536, 512, C)
        del loss, lse, dH, dW
        torch.cuda.empty_cache()


def test_fused_path_is_the_documented_rounding(cuda_lib):
    """Beyond the oracle: the fused call's gradients against the fp64 oracle's
    own values with the fused path's two bf16 roundings applied (P =
    bf16(exp(z - m)) with the label entry folded in, then bf16 of the dH output
    or of the dW operand alpha H; tests/test_parity_bounds.py holds the
    simulation). What is left between the two is fp32 against fp64 arithmetic
    before each rounding: about 3e-6 relative in z, which moves an entry of P
    across a bf16 rounding boundary (2^-8 relative) now and then, and the
    final rounding of dH where its value sits near a boundary. Measured
    6.2e-5 (dW) and 9.7e-5 (dH), against 2.3e-3 from the oracle itself; bounds
    3e-4 and 5e-4. A change in the design (a rounding skipped, added or made
    differently) moves the result by ~1e-3 and fails them."""
    from test_parity_bounds import _case, _two_roundings
    torch = _torch()
    Hf, Wf, y, ref = _case(N=1000, d=256, V=4096, seed=7)
    dH_sim, dW_sim = _two_roundings(Hf, Wf, y, ref)
    to_bits = lambda a: np.ascontiguousarray(a.astype(np.float32)).view(np.uint32) >> 16
    H = torch.from_numpy(to_bits(Hf).astype(np.uint16).view(np.int16)).view(torch.bfloat16).cuda()
    W = torch.from_numpy(to_bits(Wf).astype(np.uint16).view(np.int16)).view(torch.bfloat16).cuda()
    yd = torch.from_numpy(np.ascontiguousarray(y)).cuda()
    loss, lse, dH, dW = cuda_lib.lce_fwd_bwd(H, W, yd, chunk_tokens=256, sync_check=True)
    e_dH = rel_fro(bf16_to_np(dH), dH_sim)
    e_dW = rel_fro(dW.cpu().numpy(), dW_sim)
    import _parity_log
    _parity_log.report(dH_vs_model=e_dH, dW_vs_model=e_dW, dH_vs_oracle=rel_fro(bf16_to_np(dH), ref["dH"]),
                       dW_vs_oracle=rel_fro(dW.cpu().numpy(), ref["dW"]))
    assert e_dW <= 3e-4, e_dW
    assert e_dH <= 5e-4, e_dH
