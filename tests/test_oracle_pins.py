"""Pins for the CPU oracle: closed forms, a library routine, finite differences,
invariants and an independent second implementation. CPU only.

Each test names the plausible oracle mistake it would catch.
"""
import json
import math
import os

import numpy as np
import pytest

import oracle
from chunked_lm_head_linear_gb300 import inputs

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _rand(rng, N, d, V, sw=0.5, ignore_frac=0.25):
    H = rng.standard_normal((N, d))
    W = rng.standard_normal((V, d)) * sw
    y = rng.integers(0, V, size=N)
    y[rng.random(N) < ignore_frac] = oracle.IGNORE_INDEX
    return H, W, y


def _rel(a, b):
    a, b = np.asarray(a, float), np.asarray(b, float)
    den = np.linalg.norm(b)
    return np.linalg.norm(a - b) / (den if den > 0 else 1.0)


# --------------------------------------------------------------------------
# Hand-worked closed forms (tests/golden/closed_forms.json)
# --------------------------------------------------------------------------

def _load_cases():
    with open(os.path.join(GOLDEN, "closed_forms.json")) as f:
        return json.load(f)["cases"]


@pytest.mark.parametrize("case", _load_cases(), ids=lambda c: c["name"])
def test_closed_form_cases(case):
    """Catches: wrong sign of the one-hot, a missing 1/n, transposed dW/dH,
    ignored rows leaking into loss or gradients."""
    sympy = pytest.importorskip("sympy")
    ev = lambda s: float(sympy.sympify(s, locals={"E": sympy.E}).evalf(30))
    H = np.array(case["H"], float)
    W = np.array(case["W"], float)
    y = np.array(case["y"])
    # inputs are exact in bf16: round-trip through the generator's rounding
    assert np.array_equal(oracle.decode_bf16(inputs.f64_to_bf16_bits(H)), H)
    out = oracle.lce_f64(H, W, y, grad_loss=case["g"])
    e = case["expect"]
    assert out["loss"] == pytest.approx(ev(e["loss"]), rel=1e-14, abs=1e-15)
    np.testing.assert_allclose(out["lse"], [ev(s) for s in e["lse"]], rtol=1e-14)
    np.testing.assert_allclose(out["dH"], [[ev(s) for s in r] for r in e["dH"]], rtol=1e-13, atol=1e-15)
    np.testing.assert_allclose(out["dW"], [[ev(s) for s in r] for r in e["dW"]], rtol=1e-13, atol=1e-15)
    c = oracle.lce_c(inputs.f64_to_bf16_bits(H), inputs.f64_to_bf16_bits(W), y, grad_loss=case["g"])
    assert c["loss"] == pytest.approx(ev(e["loss"]), rel=1e-14, abs=1e-15)
    np.testing.assert_allclose(c["dW"], [[ev(s) for s in r] for r in e["dW"]], rtol=1e-13, atol=1e-15)


# --------------------------------------------------------------------------
# A library routine: PyTorch's own cross_entropy + autograd in fp64 on CPU
# --------------------------------------------------------------------------

@pytest.mark.parametrize("reduction", [oracle.MEAN, oracle.SUM])
@pytest.mark.parametrize("shape", [(7, 5, 3), (33, 16, 37), (64, 24, 130)])
def test_matches_torch_cross_entropy(shape, reduction):
    """Catches any deviation from the textbook loss and its autograd gradients
    (wrong max subtraction, wrong normaliser, swapped dH/dW)."""
    torch = pytest.importorskip("torch")
    N, d, V = shape
    rng = np.random.default_rng(N * 1000 + d)
    H, W, y = _rand(rng, N, d, V)
    g = 1.7
    out = oracle.lce_f64(H, W, y, reduction=reduction, grad_loss=g)
    Ht = torch.tensor(H, dtype=torch.float64, requires_grad=True)
    Wt = torch.tensor(W, dtype=torch.float64, requires_grad=True)
    red = "mean" if reduction == oracle.MEAN else "sum"
    L = torch.nn.functional.cross_entropy(Ht @ Wt.T, torch.tensor(y), ignore_index=-100,
                                          reduction=red)
    (L * g).backward()
    assert out["loss"] == pytest.approx(L.item(), rel=1e-13)
    assert _rel(out["dH"], Ht.grad.numpy()) < 1e-12
    assert _rel(out["dW"], Wt.grad.numpy()) < 1e-12
    lse_t = torch.logsumexp(Ht.detach() @ Wt.detach().T, dim=1).numpy()
    np.testing.assert_allclose(out["lse"], lse_t, rtol=1e-14)


def test_ignore_index_inside_vocab_is_ignored():
    """Reading: a label equal to ignore_index is ignored even if in [0, V).
    PyTorch's cross_entropy treats it the same way."""
    torch = pytest.importorskip("torch")
    rng = np.random.default_rng(3)
    H, W, y = _rand(rng, 20, 6, 9, ignore_frac=0.0)
    y[::3] = 4
    out = oracle.lce_f64(H, W, y, ignore_index=4)
    Ht = torch.tensor(H, requires_grad=True)
    L = torch.nn.functional.cross_entropy(Ht @ torch.tensor(W).T, torch.tensor(y), ignore_index=4)
    L.backward()
    assert out["loss"] == pytest.approx(L.item(), rel=1e-13)
    assert _rel(out["dH"], Ht.grad.numpy()) < 1e-12
    assert out["n_valid"] == int((y != 4).sum())


def test_label_out_of_range_is_an_error():
    H, W, y = _rand(np.random.default_rng(0), 4, 3, 5)
    for bad in (5, -1, -101):
        yb = y.copy()
        yb[1] = bad
        with pytest.raises(oracle.LabelRangeError):
            oracle.lce_f64(H, W, yb)
        with pytest.raises(oracle.LabelRangeError):
            oracle.lce_c(inputs.f64_to_bf16_bits(H), inputs.f64_to_bf16_bits(W), yb)


# --------------------------------------------------------------------------
# Closed forms P1-P3
# --------------------------------------------------------------------------

def test_P1_zero_weight_gives_log_V():
    """W = 0: every logit is 0, L = ln V, dH = 0 and dW_v = g/n sum_valid (1/V - [v=y_i]) H_i.
    Catches a wrong lse constant or a dW that ignores the softmax part."""
    rng = np.random.default_rng(1)
    N, d, V = 40, 8, 11
    H, _, y = _rand(rng, N, d, V)
    W = np.zeros((V, d))
    g = 0.75
    out = oracle.lce_f64(H, W, y, grad_loss=g)
    valid = y != -100
    n = valid.sum()
    assert out["loss"] == pytest.approx(math.log(V), rel=1e-15)
    np.testing.assert_allclose(out["lse"], math.log(V), rtol=1e-15)
    assert np.abs(out["dH"]).max() == 0.0
    dW = np.zeros((V, d))
    for i in np.nonzero(valid)[0]:
        onehot = np.zeros(V)
        onehot[y[i]] = 1
        dW += np.outer(g / n * (1.0 / V - onehot), H[i])
    assert _rel(out["dW"], dW) < 1e-13


def test_P2_zero_hidden_gives_mean_minus_target_row():
    """H = 0: L = ln V, dW = 0, dH_i = g/n (mean_v W_v - W_{y_i}).
    Catches dH computed with W^T or without the softmax mean."""
    rng = np.random.default_rng(2)
    N, d, V = 30, 6, 13
    _, W, y = _rand(rng, N, d, V)
    H = np.zeros((N, d))
    out = oracle.lce_f64(H, W, y)
    valid = y != -100
    n = valid.sum()
    assert out["loss"] == pytest.approx(math.log(V), rel=1e-15)
    assert np.abs(out["dW"]).max() == 0.0
    exp = np.where(valid[:, None], (W.mean(axis=0)[None, :] - W[np.where(valid, y, 0)]) / n, 0.0)
    assert _rel(out["dH"], exp) < 1e-13


def test_P3_two_classes_is_binary_logistic():
    """V = 2: loss_i = softplus(-margin_i), d loss/d margin = -sigmoid(-margin).
    Catches an off-by-one in the target gather or a wrong softmax normaliser."""
    rng = np.random.default_rng(5)
    N, d = 50, 4
    H, W, y = _rand(rng, N, d, 2, sw=1.0)
    out = oracle.lce_f64(H, W, y, reduction=oracle.SUM)
    valid = y != -100
    z = H @ W.T
    yy = np.where(valid, y, 0)
    margin = z[np.arange(N), yy] - z[np.arange(N), 1 - yy]
    sp = np.log1p(np.exp(-margin))
    assert out["loss"] == pytest.approx(sp[valid].sum(), rel=1e-13)
    np.testing.assert_allclose(out["loss_i"][valid], sp[valid], rtol=1e-12)
    dmargin = -1.0 / (1.0 + np.exp(margin))
    dH = dmargin[:, None] * (W[yy] - W[1 - yy]) * valid[:, None]
    assert _rel(out["dH"], dH) < 1e-12


# --------------------------------------------------------------------------
# Finite differences P6
# --------------------------------------------------------------------------

@pytest.mark.parametrize("shape", [(5, 7, 2), (8, 16, 3), (6, 12, 37)])
def test_P6_finite_differences(shape):
    """Central differences of L in fp64 against dH and dW.
    Catches any scaling, sign or transposition error in the backward."""
    N, d, V = shape
    rng = np.random.default_rng(sum(shape))
    H, W, y = _rand(rng, N, d, V, sw=1.0, ignore_frac=0.2)
    y[0] = 0  # at least one valid row
    out = oracle.lce_f64(H, W, y)
    h = 1e-5
    fdH = np.zeros_like(H)
    for i in range(N):
        for k in range(d):
            Hp, Hm = H.copy(), H.copy()
            Hp[i, k] += h
            Hm[i, k] -= h
            fdH[i, k] = (oracle.lce_f64(Hp, W, y, grads=False)["loss"]
                         - oracle.lce_f64(Hm, W, y, grads=False)["loss"]) / (2 * h)
    fdW = np.zeros_like(W)
    for v in range(V):
        for k in range(d):
            Wp, Wm = W.copy(), W.copy()
            Wp[v, k] += h
            Wm[v, k] -= h
            fdW[v, k] = (oracle.lce_f64(H, Wp, y, grads=False)["loss"]
                         - oracle.lce_f64(H, Wm, y, grads=False)["loss"]) / (2 * h)
    assert _rel(out["dH"], fdH) < 1e-7
    assert _rel(out["dW"], fdW) < 1e-7


# --------------------------------------------------------------------------
# Invariants P4, P5, P7-P10
# --------------------------------------------------------------------------

def test_P4_gradient_rows_sum_to_zero():
    """sum_v G_iv = 0 per row, hence sum_v dW_v = 0 (a d-vector).
    Catches a one-hot subtracted with the wrong weight or lse off by a constant."""
    rng = np.random.default_rng(7)
    H, W, y = _rand(rng, 64, 10, 50)
    out = oracle.lce_f64(H, W, y)
    s = out["dW"].sum(axis=0)
    assert np.abs(s).max() < 1e-14 * max(1.0, np.abs(out["dW"]).max() * 50)


def test_P5_inner_products_match():
    """<dH, H>_F = <dW, W>_F (both equal sum_iv G_iv z_iv).
    Catches a mis-scaled dH relative to dW."""
    rng = np.random.default_rng(8)
    H, W, y = _rand(rng, 48, 12, 40)
    out = oracle.lce_f64(H, W, y)
    a = float((out["dH"] * H).sum())
    b = float((out["dW"] * W).sum())
    assert a == pytest.approx(b, rel=1e-12)


@pytest.mark.parametrize("chunk,vtile", [(1, 7), (16, 5), (64, 32), (100, 999)])
def test_P7_chunked_online_equals_unchunked(chunk, vtile):
    """Token chunks x vocab tiles with the streaming (m, s) update give the same
    result. Catches a wrong rescale exp(m - m') in the online update."""
    rng = np.random.default_rng(9)
    H, W, y = _rand(rng, 70, 9, 61, sw=2.0)
    a = oracle.lce_f64(H, W, y)
    b = oracle.lce_chunked_online(H, W, y, chunk=chunk, vtile=vtile)
    assert b["loss"] == pytest.approx(a["loss"], rel=1e-12)
    np.testing.assert_allclose(b["lse"], a["lse"], rtol=1e-12)
    assert _rel(b["dH"], a["dH"]) < 1e-12
    assert _rel(b["dW"], a["dW"]) < 1e-12


def test_P8_ignored_rows_do_not_contribute():
    """Changing an ignored row's H changes neither L nor dW; its dH row is 0."""
    rng = np.random.default_rng(10)
    H, W, y = _rand(rng, 30, 8, 20)
    y[3] = -100
    a = oracle.lce_f64(H, W, y)
    H2 = H.copy()
    H2[3] = rng.standard_normal(8) * 10
    b = oracle.lce_f64(H2, W, y)
    assert b["loss"] == a["loss"]
    assert np.abs(a["dH"][3]).max() == 0.0
    assert _rel(b["dW"], a["dW"]) < 1e-15


def test_P9_permutation_and_duplication():
    """Permuting tokens permutes dH; duplicating every token keeps L and dW and
    halves dH. Catches a normaliser that is not the count of valid tokens."""
    rng = np.random.default_rng(11)
    H, W, y = _rand(rng, 25, 6, 17)
    a = oracle.lce_f64(H, W, y)
    perm = rng.permutation(25)
    b = oracle.lce_f64(H[perm], W, y[perm])
    assert b["loss"] == pytest.approx(a["loss"], rel=1e-14)
    assert _rel(b["dH"], a["dH"][perm]) < 1e-14
    assert _rel(b["dW"], a["dW"]) < 1e-13
    c = oracle.lce_f64(np.vstack([H, H]), W, np.concatenate([y, y]))
    assert c["loss"] == pytest.approx(a["loss"], rel=1e-14)
    assert _rel(c["dW"], a["dW"]) < 1e-13
    assert _rel(c["dH"][:25], a["dH"] / 2) < 1e-14


def test_P10_logit_shift_invariance():
    """Adding the same vector c to every W row shifts each row's logits by a
    constant: L, dH and dW do not change. Catches a missing max subtraction
    or a gradient that depends on the absolute logit level."""
    rng = np.random.default_rng(12)
    H, W, y = _rand(rng, 20, 5, 15)
    a = oracle.lce_f64(H, W, y)
    c = rng.standard_normal(5) * 3
    b = oracle.lce_f64(H, W + c[None, :], y)
    assert b["loss"] == pytest.approx(a["loss"], rel=1e-12)
    assert _rel(b["dH"], a["dH"]) < 1e-11
    assert _rel(b["dW"], a["dW"]) < 1e-11


def test_P11_expected_loss_of_random_head():
    """For z ~ N(0, s^2) independent of the label, E[L] ~ ln V + s^2/2 with
    s^2 = d sigma_w^2 (tiny workload: 8.369). Statistical; catches gross errors."""
    inp = inputs.make_inputs("tiny_n256_d256_v4096")
    out = oracle.lce_bf16(inp["H"], inp["W"], inp["y"], grads=False)
    w = inp["workload"]
    expect = math.log(w.V) + w.d * w.sigma_w ** 2 / 2
    assert abs(out["loss"] - expect) < 0.05


# --------------------------------------------------------------------------
# Readings where the pages are silent
# --------------------------------------------------------------------------

def test_all_ignored_gives_zero_loss_and_grads():
    """Reading: n = 0 gives L = 0 and zero gradients (PyTorch's mean is NaN)."""
    rng = np.random.default_rng(13)
    H, W, _ = _rand(rng, 6, 4, 9)
    y = np.full(6, -100)
    out = oracle.lce_f64(H, W, y)
    assert out["loss"] == 0.0 and out["n_valid"] == 0
    assert np.abs(out["dH"]).max() == 0.0 and np.abs(out["dW"]).max() == 0.0
    assert np.all(np.isfinite(out["lse"]))
    c = oracle.lce_c(inputs.f64_to_bf16_bits(H), inputs.f64_to_bf16_bits(W), y)
    assert c["loss"] == 0.0 and np.abs(c["dW"]).max() == 0.0


def test_global_denominator_shards_sum_to_whole():
    """Data parallel over tokens: shards evaluated with the global valid count,
    then summed, equal the unsharded result."""
    rng = np.random.default_rng(14)
    H, W, y = _rand(rng, 90, 7, 23)
    whole = oracle.lce_f64(H, W, y)
    n = int((y != -100).sum())
    parts = [oracle.lce_f64(H[s], W, y[s], n_valid_override=n)
             for s in (slice(0, 31), slice(31, 60), slice(60, 90))]
    assert sum(p["loss"] for p in parts) == pytest.approx(whole["loss"], rel=1e-13)
    assert _rel(sum(p["dW"] for p in parts), whole["dW"]) < 1e-13
    assert _rel(np.vstack([p["dH"] for p in parts]), whole["dH"]) < 1e-14


# --------------------------------------------------------------------------
# P12: the two oracles agree
# --------------------------------------------------------------------------

@pytest.mark.parametrize("reduction", [oracle.MEAN, oracle.SUM])
def test_P12_c_oracle_matches_numpy_oracle(reduction):
    inp = inputs.make_inputs(inputs.WORKLOADS["tiny_n256_d256_v4096"].scaled(N=96, V=1000))
    a = oracle.lce_bf16(inp["H"], inp["W"], inp["y"], reduction=reduction, grad_loss=0.5)
    b = oracle.lce_c(inp["H"], inp["W"], inp["y"], reduction=reduction, grad_loss=0.5)
    assert b["loss"] == pytest.approx(a["loss"], rel=1e-12)
    np.testing.assert_allclose(b["lse"], a["lse"], rtol=1e-13)
    assert _rel(b["dH"], a["dH"]) < 1e-12
    assert _rel(b["dW"], a["dW"]) < 1e-12


def test_sampled_helpers_match_full_oracle():
    """The row / vocab-row samplers used at full size equal the full oracle."""
    inp = inputs.make_inputs(inputs.WORKLOADS["tiny_n256_d256_v4096"].scaled(N=80, V=700))
    H, W = oracle.decode_bf16(inp["H"]), oracle.decode_bf16(inp["W"])
    y = inp["y"]
    full = oracle.lce_f64(H, W, y, grad_loss=2.0)
    scale, n = oracle.grad_scale(y, grad_loss=2.0)
    rows = np.array([0, 5, 17, 79])
    f = oracle.forward_rows_f64(H, W.astype(np.float32), y, rows)
    np.testing.assert_allclose(f["lse"], full["lse"][rows], rtol=1e-14)
    np.testing.assert_allclose(f["loss_i"], full["loss_i"][rows], rtol=1e-13, atol=1e-15)
    assert _rel(oracle.dH_rows_f64(H, W, y, rows, scale), full["dH"][rows]) < 1e-13
    vrows = np.array([0, 1, 350, 699])
    assert _rel(oracle.dW_rows_f64(H, W, y, full["lse"], vrows, scale), full["dW"][vrows]) < 1e-13


@pytest.mark.parametrize("cuts", [(0, 13, 40), (0, 1, 2, 40), (0, 20, 33, 39, 40)])
def test_vocab_shards_merge_to_the_whole(cuts):
    """Per-shard (max, sum-exp, label logit) merged with the streaming rule, and
    per-shard backward pieces summed, equal the unsharded definition -- also for
    shards that hold no label at all."""
    rng = np.random.default_rng(sum(cuts))
    H, W, y = _rand(rng, 37, 9, 40, sw=1.5)
    whole = oracle.lce_f64(H, W, y)
    stats = np.stack([oracle.vshard_stats_f64(H, W[a:b], y, a, 40) for a, b in zip(cuts[:-1], cuts[1:])])
    loss, lse = oracle.vshard_merge_f64(stats, y, V_total=40)
    assert loss == pytest.approx(whole["loss"], rel=1e-13)
    np.testing.assert_allclose(lse, whole["lse"], rtol=1e-14)
    scale, _ = oracle.grad_scale(y)
    parts = [oracle.vshard_backward_f64(H, W[a:b], y, a, lse, scale) for a, b in zip(cuts[:-1], cuts[1:])]
    assert _rel(sum(p[0] for p in parts), whole["dH"]) < 1e-13
    assert _rel(np.vstack([p[1] for p in parts]), whole["dW"]) < 1e-13


# --------------------------------------------------------------------------
# The final zero-centred RMSNorm
# --------------------------------------------------------------------------

def test_rmsnorm_matches_torch_rms_norm_and_autograd():
    """PyTorch's rms_norm with weight (1 + w), fp64 autograd: out, dx and dw."""
    torch = pytest.importorskip("torch")
    rng = np.random.default_rng(51)
    x = rng.standard_normal((19, 24)) * 3
    w = rng.standard_normal(24) * 0.1
    dout = rng.standard_normal((19, 24))
    out, r = oracle.rmsnorm_f64(x, w, 1e-6)
    xt = torch.tensor(x, requires_grad=True)
    wt = torch.tensor(w, requires_grad=True)
    ot = torch.nn.functional.rms_norm(xt, (24,), weight=1.0 + wt, eps=1e-6)
    ot.backward(torch.tensor(dout))
    np.testing.assert_allclose(out, ot.detach().numpy(), rtol=1e-13)
    dx, dw = oracle.rmsnorm_backward_f64(x, w, r, dout)
    assert _rel(dx, xt.grad.numpy()) < 1e-12
    assert _rel(dw, wt.grad.numpy()) < 1e-12


def test_rmsnorm_closed_form_and_finite_differences():
    """A constant row c: r = 1/sqrt(c^2 + eps), out = c r (1 + w). Central
    differences of sum(out * dout) against dx and dw."""
    w = np.array([0.0, 0.5, -0.25, 1.0])
    out, r = oracle.rmsnorm_f64(np.full((1, 4), 2.0), w, 1e-6)
    assert r[0] == pytest.approx(1 / math.sqrt(4 + 1e-6), rel=1e-15)
    np.testing.assert_allclose(out[0], 2.0 * r[0] * (1 + w), rtol=1e-15)
    rng = np.random.default_rng(52)
    x = rng.standard_normal((3, 6))
    w = rng.standard_normal(6) * 0.2
    dout = rng.standard_normal((3, 6))
    f = lambda xx, ww: float((oracle.rmsnorm_f64(xx, ww, 1e-5)[0] * dout).sum())
    _, r = oracle.rmsnorm_f64(x, w, 1e-5)
    dx, dw = oracle.rmsnorm_backward_f64(x, w, r, dout)
    h = 1e-6
    fdx = np.zeros_like(x)
    for i in range(3):
        for k in range(6):
            xp, xm = x.copy(), x.copy()
            xp[i, k] += h
            xm[i, k] -= h
            fdx[i, k] = (f(xp, w) - f(xm, w)) / (2 * h)
    fdw = np.array([(f(x, w + h * np.eye(6)[k]) - f(x, w - h * np.eye(6)[k])) / (2 * h) for k in range(6)])
    assert _rel(dx, fdx) < 1e-8 and _rel(dw, fdw) < 1e-8


def test_norm_then_cross_entropy_chain_rule():
    """Norm + cross-entropy through the oracle equals PyTorch autograd through
    rms_norm, the bf16 rounding of H treated as the identity for gradients."""
    torch = pytest.importorskip("torch")
    rng = np.random.default_rng(53)
    N, d, V = 21, 16, 29
    xb = oracle.round_bf16_bits(rng.standard_normal((N, d)) * 2)
    Wb = oracle.round_bf16_bits(rng.standard_normal((V, d)) * 0.3)
    w = rng.standard_normal(d) * 0.1
    y = rng.integers(0, V, N)
    y[::5] = -100
    out = oracle.norm_lce_bf16(xb, w, Wb, y, 1e-6)
    x = oracle.decode_bf16(xb)
    xt = torch.tensor(x, requires_grad=True)
    wt = torch.tensor(w, requires_grad=True)
    Ht = torch.nn.functional.rms_norm(xt, (d,), weight=1.0 + wt, eps=1e-6)
    Hq = Ht + (torch.tensor(out["H"]) - Ht).detach()     # forward uses the rounded H
    L = torch.nn.functional.cross_entropy(Hq @ torch.tensor(oracle.decode_bf16(Wb)).T, torch.tensor(y))
    L.backward()
    assert out["loss"] == pytest.approx(L.item(), rel=1e-12)
    assert _rel(out["dx"], xt.grad.numpy()) < 1e-11
    assert _rel(out["dw_norm"], wt.grad.numpy()) < 1e-11


def _bf16_pin_vector():
    """Finite fp64 values that exercise every branch of fp32 -> bf16 rounding:
    random magnitudes over 24 decades, exact ties in both directions (1 + 2^-8
    rounds down to 1, 1 + 3 * 2^-8 rounds up to 1 + 2^-6), near-ties just above and below
    a tie, signed zeros, subnormals, the largest fp32 values (which round up to
    infinity in bf16) and negative copies of all of them."""
    rng = np.random.default_rng(0)
    base = rng.standard_normal(20000) * 10 ** rng.uniform(-12, 12, 20000)
    ties = np.array([1.00390625, 1.01171875, 1.005859375, 1.0 + 2 ** -8 + 2 ** -20, 1.0 + 2 ** -8 - 2 ** -20,
                     2.0 ** -126 * 1.00390625, 2.0 ** -140, 2.0 ** -149, 3.0e-39, 0.0, -0.0,
                     3.3895313892515355e38, 3.4e38, 3.4028234663852886e38, 65504.0, 1.0, 0.5])
    x = np.concatenate([base, ties])
    return np.concatenate([x, -x])


def bf16_rounding_pin_holds(round_fn) -> bool:
    """True if ``round_fn`` (fp64 values -> bf16 bit patterns) agrees with
    PyTorch's float32 -> bfloat16 cast on the pin vector and on the exact values
    whose answer is known without any library."""
    torch = pytest.importorskip("torch")
    x = _bf16_pin_vector()
    ours = np.asarray(round_fn(x))
    ref = torch.tensor(x).to(torch.float32).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    if not np.array_equal(ours, ref):
        return False
    known = {1.00390625: 0x3F80,             # tie: the even neighbour below
             1.01171875: 0x3F82,             # tie: the even neighbour above
             1.005859375: 0x3F81,            # three quarters of an ulp: up
             -1.00390625: 0xBF80,
             3.4028234663852886e38: 0x7F80}  # past the largest bf16: infinity
    return all(int(round_fn([v])[0]) == b for v, b in known.items())


def test_round_bf16_bits_matches_torch_cast():
    """The oracle's fp64 -> fp32 -> bf16 rounding of the norm output ("XTuner on
    Ascend 910C", section 3.1.1: one bf16 rounding of x r (1 + w)) is
    round-to-nearest-even, pinned against PyTorch's own float32 -> bfloat16
    cast on values it could plausibly get wrong (ties, overflow, subnormals)."""
    assert bf16_rounding_pin_holds(oracle.round_bf16_bits)
