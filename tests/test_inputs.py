"""The seeded input generator: determinism, rounding and the workload recipe."""
import math

import numpy as np
import pytest

from chunked_lm_head_linear_gb300 import inputs


def test_bf16_rounding_is_round_to_nearest_even():
    torch = pytest.importorskip("torch")
    rng = np.random.default_rng(0)
    x = np.concatenate([rng.standard_normal(10000) * 10 ** rng.uniform(-6, 6, 10000),
                        [0.0, -0.0, 1.0, 1.00390625, 1.005859375, 3.4e38, -3.4e38]])
    ours = inputs.f64_to_bf16_bits(x)
    ref = torch.tensor(x.astype(np.float32)).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(ours, ref)
    back = inputs.bf16_bits_to_f32(ours)
    assert np.array_equal(inputs.f64_to_bf16_bits(back), ours)


def test_deterministic_and_blocking_independent():
    w = inputs.WORKLOADS["tiny_n256_d256_v4096"]
    a = inputs.make_inputs(w)
    b = inputs.make_inputs(w)
    assert np.array_equal(a["H"], b["H"]) and np.array_equal(a["W"], b["W"])
    assert np.array_equal(a["y"], b["y"])
    rng = np.random.Generator(np.random.PCG64(0))
    one = inputs.f64_to_bf16_bits(rng.standard_normal((300, 16)))
    blk = inputs._normal_bf16(np.random.Generator(np.random.PCG64(0)), 300, 16, 1.0, block_rows=7)
    assert np.array_equal(one, blk)
    c = inputs.make_inputs(w, with_W=False)
    assert np.array_equal(a["y"], c["y"]) and c["W"] is None


@pytest.mark.parametrize("name", list(inputs.WORKLOADS))
def test_workload_structure(name):
    w = inputs.WORKLOADS[name]
    small = w.scaled(N=min(w.N, 4096), d=8)  # labels/ignore structure at a cheap size
    inp = inputs.make_inputs(small)
    y = inp["y"]
    ign = y == inputs.IGNORE_INDEX
    assert np.all((y[~ign] >= 0) & (y[~ign] < w.V))
    if w.ignore in ("random", "doc_starts"):
        assert ign.sum() == round(w.ignore_frac * small.N)
    if w.ignore == "documents":
        st = inp["doc_starts"]
        assert st[0] == 0 and np.array_equal(np.nonzero(ign)[0], st)
        lens = np.diff(np.append(st, small.N))
        assert np.all(lens[:-1] >= w.doc_len_min) and np.all(lens[:-1] <= w.doc_len_max)


def test_zipf_head_mass():
    """P(id 0) = 1 / sum_{k=1}^{V} k^-1.1, about 13.2% at V = 151936."""
    rng = np.random.Generator(np.random.PCG64(1))
    lab = inputs.zipf_labels(rng, 200000, 151936, 1.1)
    Hn = float(np.sum(np.arange(1, 151937, dtype=np.float64) ** -1.1))
    assert abs((lab == 0).mean() - 1 / Hn) < 0.004
    assert abs(1 / Hn - 0.132) < 0.001
    assert lab.min() >= 0 and lab.max() < 151936


def test_value_distribution():
    inp = inputs.make_inputs(inputs.WORKLOADS["tiny_n256_d256_v4096"])
    H = inputs.bf16_bits_to_f32(inp["H"])
    W = inputs.bf16_bits_to_f32(inp["W"])
    assert abs(H.std() - 1.0) < 0.01 and abs(W.std() - 0.02) < 0.0005
    assert math.isclose(float(H.mean()), 0.0, abs_tol=0.01)
