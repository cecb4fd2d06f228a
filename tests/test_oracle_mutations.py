"""Plant plausible mistakes in a copy of the numpy oracle and check that the
pins (closed forms, PyTorch's cross_entropy, the gradient-row-sum invariant)
catch every one of them. CPU only; the real oracle is never modified."""
import json
import math
import os
import types

import numpy as np
import pytest

import oracle

SRC = os.path.join(os.path.dirname(oracle.__file__), "lce_oracle.py")

MUTATIONS = {
    "one_hot_sign": ("p[(rows - r0)[v], yy[v]] -= 1.0", "p[(rows - r0)[v], yy[v]] += 1.0"),
    "dropped_1_over_n": ("G = p * (v * scale)[:, None]", "G = p * (v * 1.0)[:, None]"),
    "dropped_max_term": ("lse[r0:r1] = m + np.log(s)", "lse[r0:r1] = np.log(s)"),
    "target_off_by_one": ("z[rows - r0, yy]", "z[rows - r0, np.maximum(yy - 1, 0)]"),
    "loss_over_all_tokens": ("lscale = 0.0 if n == 0 else 1.0 / n", "lscale = 1.0 / len(y)"),
    "ignored_rows_in_grad": ("G = p * (v * scale)[:, None]", "G = p * scale"),
    "softmax_not_normalised": ("p = np.exp(z - lse[r0:r1, None])", "p = np.exp(z - m[:, None])"),
    "dW_from_wrong_chunk": ("dW += G.T @ H[r0:r1]", "dW += G.T @ H[:r1 - r0]"),
}


# Plausible mistakes in the fp64 -> bf16 rounding of the norm output, caught by
# the rounding pin (PyTorch's cast and hand-checked ties).
ROUNDING_MUTATIONS = {
    "bf16_truncation": ("return ((u + 0x7FFF + ((u >> 16) & 1)) >> 16).astype(np.uint16)",
                        "return (u >> 16).astype(np.uint16)"),
    "bf16_ties_away_from_zero": ("return ((u + 0x7FFF + ((u >> 16) & 1)) >> 16).astype(np.uint16)",
                                 "return ((u + 0x8000) >> 16).astype(np.uint16)"),
    "bf16_ties_to_odd": ("return ((u + 0x7FFF + ((u >> 16) & 1)) >> 16).astype(np.uint16)",
                         "return ((u + 0x8000 - ((u >> 16) & 1)) >> 16).astype(np.uint16)"),
}


def _mutant(name):
    old, new = {**MUTATIONS, **ROUNDING_MUTATIONS}[name]
    src = open(SRC).read()
    assert src.count(old) >= 1, f"mutation anchor for {name} not found"
    mod = types.ModuleType("mutant_" + name)
    exec(compile(src.replace(old, new, 1), SRC, "exec"), mod.__dict__)
    return mod


def _pins_pass(mod) -> bool:
    """True if the mutant survives every pin below."""
    torch = pytest.importorskip("torch")
    sympy = pytest.importorskip("sympy")
    with open(os.path.join(os.path.dirname(__file__), "golden", "closed_forms.json")) as f:
        cases = json.load(f)["cases"]
    ev = lambda s: float(sympy.sympify(s, locals={"E": sympy.E}).evalf(30))
    try:
        for c in cases:
            out = mod.lce_f64(np.array(c["H"], float), np.array(c["W"], float),
                              np.array(c["y"]), grad_loss=c["g"])
            if not math.isclose(out["loss"], ev(c["expect"]["loss"]), rel_tol=1e-12):
                return False
            exp_dW = np.array([[ev(s) for s in r] for r in c["expect"]["dW"]])
            if not np.allclose(out["dW"], exp_dW, rtol=1e-12, atol=1e-14):
                return False
        rng = np.random.default_rng(0)
        N, d, V = 300, 8, 19       # more than one 256-row block
        H = rng.standard_normal((N, d))
        W = rng.standard_normal((V, d))
        y = rng.integers(0, V, N)
        y[::7] = -100
        out = mod.lce_f64(H, W, y)
        Ht = torch.tensor(H, requires_grad=True)
        Wt = torch.tensor(W, requires_grad=True)
        L = torch.nn.functional.cross_entropy(Ht @ Wt.T, torch.tensor(y), ignore_index=-100)
        L.backward()
        if not math.isclose(out["loss"], L.item(), rel_tol=1e-12):
            return False
        if not np.allclose(out["dH"], Ht.grad.numpy(), rtol=1e-10, atol=1e-14):
            return False
        if not np.allclose(out["dW"], Wt.grad.numpy(), rtol=1e-10, atol=1e-14):
            return False
        if np.abs(out["dW"].sum(axis=0)).max() > 1e-12:
            return False
    except (IndexError, ValueError):
        return False
    return True


def test_unmutated_oracle_passes_the_pins():
    assert _pins_pass(oracle.lce_oracle)


@pytest.mark.parametrize("name", sorted(MUTATIONS))
def test_pins_catch_planted_mistake(name):
    assert not _pins_pass(_mutant(name)), f"pins did not catch mutation {name}"


@pytest.mark.parametrize("name", sorted(ROUNDING_MUTATIONS))
def test_rounding_pin_catches_planted_mistake(name):
    from test_oracle_pins import bf16_rounding_pin_holds
    assert bf16_rounding_pin_holds(oracle.round_bf16_bits)
    assert not bf16_rounding_pin_holds(_mutant(name).round_bf16_bits), f"rounding pin did not catch {name}"
