"""The GPU parity bounds, checked on the CPU: they admit the error the fused
path is designed to make, and they catch a localised fault that the
whole-tensor norm would let through.

The fused path (the exp-tile design of lce_fwd_bwd) rounds twice to bf16 on
the way to each gradient: every entry of P = bf16(exp(z - m)) against a row
reference m (the label entry after the one-hot is folded in), then either the
dH output bf16(alpha (g/n) P W) or the dW operand Ht = bf16(alpha H), with
alpha = exp(m - lse). Here those roundings are applied to the fp64 oracle's
own quantities (a simulation of the error model, not of the kernels), and the
result is held to check_grad, the check every GPU parity test uses.
"""
import numpy as np
import pytest

import oracle
from chunked_lm_head_linear_gb300 import inputs
from test_parity_gpu import TOL_GRAD, check_grad, rel_fro


def _bf16(a):
    return oracle.decode_bf16(oracle.round_bf16_bits(a))


def _case(N=2000, d=264, V=8000, seed=5):
    w = inputs.Workload(f"bounds{seed}", N=N, d=d, V=V, sigma_w=0.05, labels="uniform", ignore="random",
                        ignore_frac=0.1, seed=seed)
    inp = inputs.make_inputs(w)
    H = oracle.decode_bf16(inp["H"])
    W = oracle.decode_bf16(inp["W"])
    y = np.asarray(inp["y"])
    ref = oracle.lce_bf16(inp["H"], inp["W"], y)
    return H, W, y, ref


def _two_roundings(H, W, y, ref):
    """dH and dW with the fused path's two bf16 roundings applied to exact values."""
    scale, _ = oracle.grad_scale(y)
    valid = y != oracle.IGNORE_INDEX
    z = H @ W.T
    m = z[:, :128].max(axis=1)                      # the row reference: the first 128 words
    lse = ref["lse"]
    P = _bf16(np.exp(z - m[:, None]))
    rows = np.nonzero(valid)[0]
    P[rows, y[rows]] = _bf16(np.exp(z[rows, y[rows]] - m[rows]) - np.exp(lse[rows] - m[rows]))
    alpha = np.where(valid, np.exp(m - lse), 0.0)
    dH = _bf16(scale * alpha[:, None] * (P @ W))
    dW = scale * (P.T @ _bf16(alpha[:, None] * H))
    return dH, dW


@pytest.fixture(scope="module")
def case():
    H, W, y, ref = _case()
    dH, dW = _two_roundings(H, W, y, ref)
    return y, ref, dH, dW


def test_designed_error_passes(case):
    y, ref, dH, dW = case
    errs = {}
    check_grad("dH", dH, ref["dH"], errs)
    check_grad("dW", dW, ref["dW"], errs)
    # the simulated errors sit where the GPU's measured ones do (2.2e-3 to 2.5e-3)
    assert 1e-3 < errs["dH"] < 4e-3 and 1e-3 < errs["dW"] < 4e-3, errs


def _fault_cases(grad, y):
    """(description, faulty copy) pairs: one row 10% off, one 32-column group of
    one row 10% off, one row of the last partial tile 10% off."""
    rows = np.nonzero(np.linalg.norm(grad, axis=1) > 0)[0]
    r = rows[len(rows) // 2]
    tail = rows[rows >= (grad.shape[0] // 256) * 256]
    out = []
    g = grad.copy()
    g[r] *= 1.1
    out.append(("one row", g))
    g = grad.copy()
    g[r, 32:64] *= 1.1
    out.append(("one 32-column group", g))
    if tail.size:
        g = grad.copy()
        g[tail[0]] *= 1.1
        out.append(("one tail row", g))
    return out


@pytest.mark.parametrize("which", ["dH", "dW"])
def test_localised_fault_is_caught(case, which):
    y, ref, dH, dW = case
    sim = dH if which == "dH" else dW
    for desc, faulty in _fault_cases(sim, y):
        # the whole-tensor norm alone lets the fault through ...
        assert rel_fro(faulty, ref[which]) <= TOL_GRAD, (which, desc)
        # ... the local bounds do not
        with pytest.raises(AssertionError):
            check_grad(which, faulty, ref[which], {})
