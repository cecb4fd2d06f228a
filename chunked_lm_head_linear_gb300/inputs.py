"""Seeded synthetic inputs for the fused LM-head linear + cross-entropy path.

This module only draws numbers: hidden states H, LM-head weight W and labels y.
It holds none of the loss arithmetic, so the CPU oracle and the CUDA path can
both be fed from it without sharing any of the method's code.

Recipe (the same for every workload):
  * one ``numpy.random.Generator(PCG64(seed))`` per workload, drawn in a fixed
    order: H, then W, then the ignore mask / document layout, then labels;
  * floating draws are fp64, rounded to fp32 and then to bf16 with
    round-to-nearest-even; H ~ N(0, 1) (post-RMSNorm-like), W ~ N(0, sigma_w);
  * ignore positions: exactly round(p*N) distinct positions drawn without
    replacement, or, for packed documents, the first token of every document;
  * labels: uniform on [0, V), or a truncated Zipf law P(k) ~ (k+1)^-s on
    [0, V) sampled through its inverse CDF.

The workloads are the LM-head shapes of the chunked linear cross-entropy
described on "XTuner on Ascend 910C: Qwen3.5-2B training optimisation"
(section 3.1.4, the 154,880-wide vocabulary loss chain) and the 64k-token
sequences of "XTuner V1 introduction" (memory optimisation section); the
vocabulary sizes used here (151936, 129280, 151655) are those of the target
workloads, the page's 154,880 is context only.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field, replace

import numpy as np

IGNORE_INDEX = -100


@dataclass(frozen=True)
class Workload:
    """Shape and value distribution of one synthetic LM-head batch."""

    name: str
    N: int                     # tokens
    d: int                     # hidden size
    V: int                     # vocabulary size
    sigma_w: float = 0.02      # std of W entries
    labels: str = "uniform"    # "uniform" | "zipf"
    zipf_s: float = 1.1
    ignore: str = "random"     # "random" | "doc_starts" | "documents" | "none"
    ignore_frac: float = 0.10
    doc_len_min: int = 128     # log-uniform document lengths (ignore="documents")
    doc_len_max: int = 8192
    seed: int = 0
    notes: str = field(default="", compare=False)

    def scaled(self, **kw) -> "Workload":
        return replace(self, **kw)


# The five target workloads, named by what they are and their sizes.
WORKLOADS = {
    "tiny_n256_d256_v4096": Workload(
        "tiny_n256_d256_v4096", N=256, d=256, V=4096, sigma_w=0.02,
        labels="uniform", ignore="random", ignore_frac=0.10,
        notes="small case the oracle finishes in well under a second"),
    "qwen2b_n8192_d2048_v151936": Workload(
        "qwen2b_n8192_d2048_v151936", N=8192, d=2048, V=151936, sigma_w=0.02,
        labels="uniform", ignore="doc_starts", ignore_frac=0.05,
        notes="Qwen3.5-2B-like LM head, one packed 8192-token sequence"),
    "packed_n32768_d2048_v151936": Workload(
        "packed_n32768_d2048_v151936", N=32768, d=2048, V=151936, sigma_w=0.02,
        labels="zipf", ignore="documents",
        notes="long packed batch of log-uniform 128..8192-token documents"),
    "seq64k_n65536_d4096_v151936": Workload(
        "seq64k_n65536_d4096_v151936", N=65536, d=4096, V=151936, sigma_w=0.015,
        labels="zipf", ignore="random", ignore_frac=0.02,
        notes="64k-token sequence head; chunk size swept 1024..8192"),
    "moe_n16384_d7168_v129280": Workload(
        "moe_n16384_d7168_v129280", N=16384, d=7168, V=129280, sigma_w=0.01,
        labels="uniform", ignore="random", ignore_frac=0.05,
        notes="wide MoE-style head"),
    "moe_n16384_d7168_v151655": Workload(
        "moe_n16384_d7168_v151655", N=16384, d=7168, V=151655, sigma_w=0.01,
        labels="uniform", ignore="random", ignore_frac=0.05,
        notes="wide MoE-style head, unpadded vocabulary (ragged tile tail)"),
}

BENCH_WORKLOAD = "qwen2b_n8192_d2048_v151936"


def f64_to_bf16_bits(x) -> np.ndarray:
    """Round fp64 values to fp32, then to bf16 (round-to-nearest-even).

    Returns the bf16 bit patterns as uint16. NaNs never occur in the draws.
    """
    f = np.ascontiguousarray(np.asarray(x, dtype=np.float64).astype(np.float32))
    u = f.view(np.uint32).astype(np.uint64)
    u = (u + 0x7FFF + ((u >> 16) & 1)) >> 16
    return u.astype(np.uint16)


def bf16_bits_to_f32(bits) -> np.ndarray:
    """Exact widening of bf16 bit patterns to fp32 (used to build test tensors)."""
    b = np.ascontiguousarray(np.asarray(bits, dtype=np.uint16))
    return (b.astype(np.uint32) << 16).view(np.float32)


def _normal_bf16(rng: np.random.Generator, rows: int, cols: int, sigma: float,
                 block_rows: int = 4096) -> np.ndarray:
    """rows x cols bf16 draws of N(0, sigma^2), generated in row blocks.

    Drawing in blocks consumes the generator in exactly the same order as one
    large call, so the result does not depend on ``block_rows``; it only bounds
    the fp64 scratch to block_rows*cols*8 bytes.
    """
    out = np.empty((rows, cols), dtype=np.uint16)
    for r0 in range(0, rows, block_rows):
        r1 = min(rows, r0 + block_rows)
        blk = rng.standard_normal((r1 - r0, cols))
        if sigma != 1.0:
            blk *= sigma
        out[r0:r1] = f64_to_bf16_bits(blk)
    return out


def zipf_labels(rng: np.random.Generator, n: int, V: int, s: float) -> np.ndarray:
    """Truncated Zipf draws on [0, V): P(k) proportional to (k+1)^-s."""
    w = np.arange(1, V + 1, dtype=np.float64) ** (-s)
    cdf = np.cumsum(w)
    cdf /= cdf[-1]
    u = rng.random(n)
    lab = np.searchsorted(cdf, u, side="right")
    return np.minimum(lab, V - 1).astype(np.int64)


def document_starts(rng: np.random.Generator, N: int, lmin: int, lmax: int):
    """Concatenate documents of length round(exp(U(ln lmin, ln lmax))) until
    they cover N tokens; the last one is truncated. Returns start offsets."""
    starts, pos = [], 0
    lo, hi = math.log(lmin), math.log(lmax)
    while pos < N:
        starts.append(pos)
        pos += int(round(math.exp(rng.uniform(lo, hi))))
    return np.asarray(starts, dtype=np.int64)


def make_inputs(w: Workload | str, seed: int | None = None, with_W: bool = True):
    """Draw (H, W, y) for a workload.

    Returns a dict with ``H`` (uint16 bf16 bits, [N, d]), ``W`` (uint16 bf16
    bits, [V, d], or None if ``with_W`` is False -- W is still drawn so the
    labels do not change), ``y`` (int64 [N]) and ``doc_starts`` where relevant.
    """
    if isinstance(w, str):
        w = WORKLOADS[w]
    if seed is not None:
        w = w.scaled(seed=seed)
    rng = np.random.Generator(np.random.PCG64(w.seed))
    H = _normal_bf16(rng, w.N, w.d, 1.0)
    if with_W:
        W = _normal_bf16(rng, w.V, w.d, w.sigma_w)
    else:  # consume the same draws without keeping them
        for r0 in range(0, w.V, 4096):
            rng.standard_normal((min(w.V, r0 + 4096) - r0, w.d))
        W = None

    starts = None
    ignore_pos = np.zeros(0, dtype=np.int64)
    if w.ignore in ("random", "doc_starts"):
        k = int(round(w.ignore_frac * w.N))
        ignore_pos = np.sort(rng.choice(w.N, size=k, replace=False)).astype(np.int64)
        if w.ignore == "doc_starts":
            starts = ignore_pos
    elif w.ignore == "documents":
        starts = document_starts(rng, w.N, w.doc_len_min, w.doc_len_max)
        ignore_pos = starts
    elif w.ignore != "none":
        raise ValueError(f"unknown ignore mode {w.ignore!r}")

    if w.labels == "uniform":
        y = rng.integers(0, w.V, size=w.N, dtype=np.int64)
    elif w.labels == "zipf":
        y = zipf_labels(rng, w.N, w.V, w.zipf_s)
    else:
        raise ValueError(f"unknown label law {w.labels!r}")
    y[ignore_pos] = IGNORE_INDEX
    return {"H": H, "W": W, "y": y, "doc_starts": starts, "workload": w}


def input_digest(inp) -> str:
    """Short content hash of a drawn input set (guards cached expected values
    against a change of the generator between numpy versions)."""
    import hashlib
    h = hashlib.sha256()
    for key in ("H", "W", "y"):
        a = inp[key]
        if a is None:
            continue
        a = np.ascontiguousarray(a)
        # hashing the whole of W at full size takes a few seconds; rows are
        # strided so the digest still touches every part of the tensor
        if a.ndim == 2 and a.shape[0] > 4096:
            a = np.ascontiguousarray(a[:: max(1, a.shape[0] // 4096)])
        h.update(a.tobytes())
    return h.hexdigest()[:16]
