"""Write the oracle's per-row log-sum-exp and loss for every full-size workload.

Calls only the CPU oracle (``oracle/``) and the seeded input generator. The
output, ``full_<workload>.npz``, holds the input digest, n_valid, the fp64
mean loss and the fp64 lse of every row; the GPU parity tests use it for the
loss check and as the lse the oracle needs for sampled dW rows. Usage:

    python tests/golden/make_full_golden.py [workload ...]
"""
import os
import sys
import time

import numpy as np

ROOT = os.path.dirname(os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
sys.path.insert(0, ROOT)

import oracle  # noqa: E402
from chunked_lm_head_linear_gb300 import inputs  # noqa: E402

OUT = os.path.dirname(os.path.abspath(__file__))
FULL = [k for k in inputs.WORKLOADS if not k.startswith("tiny")]


def make(name):
    t0 = time.time()
    inp = inputs.make_inputs(name)
    H = inputs.bf16_bits_to_f32(inp["H"])
    W = inputs.bf16_bits_to_f32(inp["W"])
    y = inp["y"]
    f = oracle.forward_rows_f64(H, W, y)
    valid = y != oracle.IGNORE_INDEX
    n = int(valid.sum())
    loss = float(np.sum(f["loss_i"], dtype=np.float64) / n)
    path = os.path.join(OUT, f"full_{name}.npz")
    np.savez(path, digest=inputs.input_digest(inp), n_valid=n, loss=loss, lse=f["lse"])
    print(f"{name}: loss={loss:.10f} n={n} ({time.time() - t0:.0f}s) -> {os.path.basename(path)}",
          flush=True)


if __name__ == "__main__":
    for name in sys.argv[1:] or FULL:
        make(name)
