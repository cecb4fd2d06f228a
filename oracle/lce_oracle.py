"""fp64 CPU oracle for the fused LM-head linear + cross-entropy (TEST INFRASTRUCTURE).

This is the plain, slow, obviously correct definition of what the CUDA path
computes. Only the tests, the smoke check and the benchmark's CPU-baseline leg
may import it; the product path never does. It shares no code with the CUDA
path (the two only share the seeded input generator, which does no loss
arithmetic).

What is computed (the definition, written out):
  "XTuner on Ascend 910C: Qwen3.5-2B training optimisation", section 3.1.4
  (Liger chunked cross-entropy, Fig. 12): the loss chain turns the LM-head
  logits of an mbs x seq x vocab batch into a token-level cross-entropy and
  back-propagates it to d_input and d_weight; the fused kernel never keeps the
  full d_logits. The formula itself is the standard token-level
  cross-entropy with ignore_index and a mean over valid tokens:

    z      = H W^T                               [N, V]   (fp64, exact products)
    lse_i  = m_i + log sum_v exp(z_iv - m_i),    m_i = max_v z_iv
    loss_i = valid_i * (lse_i - z_{i, y_i})
    L      = sum_i loss_i / n        (mean)   or   sum_i loss_i   (sum)
    G_iv   = valid_i * g * (exp(z_iv - lse_i) - [v = y_i]) / n   (mean; no /n for sum)
    dH     = G W                                 [N, d]
    dW     = G^T H                               [V, d]

with valid_i = [y_i != ignore_index] and n = sum_i valid_i (or a caller-given
global count, the data-parallel denominator). Readings where the pages are
silent: n = 0 gives L = 0 and G = 0; lse is computed for every row, ignored
ones included; a label equal to ignore_index is ignored even inside [0, V);
any other label outside [0, V) is an error.

The row-block loop below is the token chunking the method itself prescribes
("XTuner V1 introduction", memory optimisation section: the loss graph is
computed in chunks); ``lce_chunked_online`` additionally splits the
vocabulary into tiles with the streaming max/sum-exp update of
"MindSpeed fusion optimisation: principles and practice", section 3.2
(blockwise softmax without the full score matrix), and must agree with the
unchunked result to rounding.

Matrix products use numpy's fp64 matmul as a library step. Inputs are bf16
bit patterns (uint16) decoded exactly to fp64.
"""
from __future__ import annotations

import math

import numpy as np

IGNORE_INDEX = -100
MEAN, SUM = 0, 1


class LabelRangeError(ValueError):
    """A label is neither ignore_index nor inside [0, V)."""


def decode_bf16(bits) -> np.ndarray:
    """bf16 bit patterns -> fp64, exactly (bits << 16 is the fp32 pattern)."""
    b = np.ascontiguousarray(np.asarray(bits, dtype=np.uint16))
    return (b.astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def _prepare(y, V, ignore_index, reduction, n_valid_override, grad_loss):
    y = np.asarray(y, dtype=np.int64)
    valid = y != ignore_index
    bad = valid & ((y < 0) | (y >= V))
    if bad.any():
        raise LabelRangeError(f"{int(bad.sum())} labels outside [0, {V}) and != {ignore_index}")
    n = int(valid.sum()) if n_valid_override is None or n_valid_override < 0 else int(n_valid_override)
    if reduction == MEAN:
        scale = 0.0 if n == 0 else float(grad_loss) / n
        lscale = 0.0 if n == 0 else 1.0 / n
    elif reduction == SUM:
        scale, lscale = float(grad_loss), 1.0
    else:
        raise ValueError("reduction must be MEAN (0) or SUM (1)")
    return y, valid, n, scale, lscale


def lce_f64(H, W, y, *, ignore_index=IGNORE_INDEX, reduction=MEAN,
            n_valid_override=-1, grad_loss=1.0, row_block=256, grads=True):
    """The definition on fp64 arrays H [N, d], W [V, d], labels y [N].

    Returns dict(loss, lse, loss_i, zt, n_valid, dH, dW) (dH/dW only if grads).
    """
    H = np.asarray(H, dtype=np.float64)
    W = np.asarray(W, dtype=np.float64)
    N, d = H.shape
    V = W.shape[0]
    y, valid, n, scale, lscale = _prepare(y, V, ignore_index, reduction,
                                          n_valid_override, grad_loss)
    lse = np.empty(N)
    loss_i = np.zeros(N)
    zt = np.zeros(N)
    dH = np.zeros((N, d)) if grads else None
    dW = np.zeros((V, d)) if grads else None
    for r0 in range(0, N, row_block):
        r1 = min(N, r0 + row_block)
        rows = np.arange(r0, r1)
        z = H[r0:r1] @ W.T                                  # logits of this chunk
        m = z.max(axis=1)
        s = np.exp(z - m[:, None]).sum(axis=1)
        lse[r0:r1] = m + np.log(s)
        v = valid[r0:r1]
        yy = np.where(v, y[r0:r1], 0)
        zt[r0:r1] = np.where(v, z[rows - r0, yy], 0.0)
        loss_i[r0:r1] = np.where(v, lse[r0:r1] - zt[r0:r1], 0.0)
        if grads:
            p = np.exp(z - lse[r0:r1, None])                # softmax
            p[(rows - r0)[v], yy[v]] -= 1.0                 # minus one-hot
            G = p * (v * scale)[:, None]
            dH[r0:r1] = G @ W
            dW += G.T @ H[r0:r1]
    loss = math.fsum(loss_i.tolist()) * lscale
    out = {"loss": loss, "lse": lse, "loss_i": loss_i, "zt": zt, "n_valid": n}
    if grads:
        out["dH"], out["dW"] = dH, dW
    return out


def lce_bf16(Hbits, Wbits, y, **kw):
    """``lce_f64`` on bf16 bit-pattern inputs (the CUDA path's input format)."""
    return lce_f64(decode_bf16(Hbits), decode_bf16(Wbits), y, **kw)


def lce_chunked_online(H, W, y, *, chunk=64, vtile=32, ignore_index=IGNORE_INDEX,
                       reduction=MEAN, n_valid_override=-1, grad_loss=1.0):
    """Chunked tokens x tiled vocabulary with the streaming (m, s) update.

    For each token chunk, the vocabulary is visited tile by tile and each row
    keeps a running max m and a running sum s of exp(z - m):
        m' = max(m, max_T z),  s' = s * exp(m - m') + sum_T exp(z - m').
    The gradient is formed per (chunk, tile) once lse is known and summed into
    dH (over tiles) and dW (over chunks). Must equal ``lce_f64`` to rounding.
    """
    H = np.asarray(H, dtype=np.float64)
    W = np.asarray(W, dtype=np.float64)
    N, d = H.shape
    V = W.shape[0]
    y, valid, n, scale, lscale = _prepare(y, V, ignore_index, reduction,
                                          n_valid_override, grad_loss)
    lse = np.empty(N)
    loss_i = np.zeros(N)
    dH = np.zeros((N, d))
    dW = np.zeros((V, d))
    for c0 in range(0, N, chunk):
        c1 = min(N, c0 + chunk)
        Hc = H[c0:c1]
        m = np.full(c1 - c0, -np.inf)
        s = np.zeros(c1 - c0)
        zt = np.zeros(c1 - c0)
        for t0 in range(0, V, vtile):
            t1 = min(V, t0 + vtile)
            z = Hc @ W[t0:t1].T
            m_new = np.maximum(m, z.max(axis=1))
            s = s * np.exp(m - m_new) + np.exp(z - m_new[:, None]).sum(axis=1)
            m = m_new
            for r in range(c1 - c0):
                yi = y[c0 + r]
                if valid[c0 + r] and t0 <= yi < t1:
                    zt[r] = z[r, yi - t0]
        lse_c = m + np.log(s)
        lse[c0:c1] = lse_c
        v = valid[c0:c1]
        loss_i[c0:c1] = np.where(v, lse_c - zt, 0.0)
        for t0 in range(0, V, vtile):
            t1 = min(V, t0 + vtile)
            z = Hc @ W[t0:t1].T
            p = np.exp(z - lse_c[:, None])
            for r in range(c1 - c0):
                yi = y[c0 + r]
                if v[r] and t0 <= yi < t1:
                    p[r, yi - t0] -= 1.0
            G = p * (v * scale)[:, None]
            dH[c0:c1] += G @ W[t0:t1]
            dW[t0:t1] += G.T @ Hc
    loss = math.fsum(loss_i.tolist()) * lscale
    return {"loss": loss, "lse": lse, "loss_i": loss_i, "n_valid": n, "dH": dH, "dW": dW}


# ---------------------------------------------------------------------------
# Sampled evaluation for full-size workloads: each function computes exactly
# the same quantities as ``lce_f64`` for a subset of outputs.
# ---------------------------------------------------------------------------

def forward_rows_f64(H, W, y, rows=None, *, ignore_index=IGNORE_INDEX, row_block=128):
    """lse_i, loss_i (unscaled) and z_{i,y_i} for the given rows (all by default).

    ``W`` may be fp32 (exact for bf16 inputs); every product is done in fp64.
    """
    N = H.shape[0]
    rows = np.arange(N) if rows is None else np.asarray(rows, dtype=np.int64)
    y = np.asarray(y, dtype=np.int64)
    W64 = np.asarray(W, dtype=np.float64)
    lse = np.empty(rows.size)
    zt = np.zeros(rows.size)
    for b0 in range(0, rows.size, row_block):
        rb = rows[b0:b0 + row_block]
        z = np.asarray(H[rb], dtype=np.float64) @ W64.T
        m = z.max(axis=1)
        lse[b0:b0 + rb.size] = m + np.log(np.exp(z - m[:, None]).sum(axis=1))
        yy = y[rb]
        v = yy != ignore_index
        zt[b0:b0 + rb.size] = np.where(v, z[np.arange(rb.size), np.where(v, yy, 0)], 0.0)
    valid = y[rows] != ignore_index
    loss_i = np.where(valid, lse - zt, 0.0)
    return {"rows": rows, "lse": lse, "zt": zt, "loss_i": loss_i}


def grad_scale(y, *, ignore_index=IGNORE_INDEX, reduction=MEAN, n_valid_override=-1,
               grad_loss=1.0):
    """The factor g/n (mean) or g (sum) that multiplies softmax - one-hot."""
    y = np.asarray(y)
    n = int((y != ignore_index).sum()) if n_valid_override < 0 else int(n_valid_override)
    if reduction == SUM:
        return float(grad_loss), n
    return (0.0 if n == 0 else float(grad_loss) / n), n


def dH_rows_f64(H, W, y, rows, scale, *, ignore_index=IGNORE_INDEX):
    """dH_i = sum_v G_iv W_v for the given rows (lse recomputed per row)."""
    rows = np.asarray(rows, dtype=np.int64)
    y = np.asarray(y, dtype=np.int64)
    W64 = np.asarray(W, dtype=np.float64)
    yr = y[rows]
    valid = yr != ignore_index
    z = np.asarray(H[rows], dtype=np.float64) @ W64.T          # logits of the sampled rows
    m = z.max(axis=1)
    lse = m + np.log(np.exp(z - m[:, None]).sum(axis=1))
    p = np.exp(z - lse[:, None])
    p[np.nonzero(valid)[0], yr[valid]] -= 1.0
    G = p * (valid * scale)[:, None]
    return G @ W64


def dW_rows_f64(H, W, y, lse, vrows, scale, *, ignore_index=IGNORE_INDEX):
    """dW_v = sum_i G_iv H_i for the given vocabulary rows.

    ``lse`` must be the oracle's own per-row log-sum-exp for all N rows.
    """
    vrows = np.asarray(vrows, dtype=np.int64)
    y = np.asarray(y, dtype=np.int64)
    H64 = np.asarray(H, dtype=np.float64)
    Wv = np.asarray(W[vrows], dtype=np.float64)
    z = H64 @ Wv.T                                # [N, |S|]
    p = np.exp(z - np.asarray(lse)[:, None])
    valid = y != ignore_index
    for j, v in enumerate(vrows):
        p[valid & (y == v), j] -= 1.0
    G = p * (valid * scale)[:, None]
    return G.T @ H64


# ---------------------------------------------------------------------------
# Vocabulary shards: the per-shard statistics and their merge, written from
# the streaming max / sum-exp rule ("MindSpeed fusion optimisation: principles
# and practice", section 3.2), with the shards playing the role of blocks.
# ---------------------------------------------------------------------------

def vshard_stats_f64(H, W_shard, y, vocab_offset, V_total, *, ignore_index=IGNORE_INDEX):
    """Per row of this shard: m = max_v z, s = sum_v exp(z - m), the label's logit
    if the label lies in the shard, and 1/0 for whether it does. [N, 4] fp64."""
    H = np.asarray(H, dtype=np.float64)
    Ws = np.asarray(W_shard, dtype=np.float64)
    y = np.asarray(y, dtype=np.int64)
    z = H @ Ws.T
    m = z.max(axis=1)
    s = np.exp(z - m[:, None]).sum(axis=1)
    valid = (y != ignore_index) & (y >= 0) & (y < V_total)
    col = y - vocab_offset
    here = valid & (col >= 0) & (col < Ws.shape[0])
    zt = np.where(here, z[np.arange(len(y)), np.where(here, col, 0)], 0.0)
    return np.stack([m, s, zt, here.astype(np.float64)], axis=1)


def vshard_merge_f64(stats_all, y, *, ignore_index=IGNORE_INDEX, V_total=None, n_valid_override=-1):
    """Merge [R, N, 4] shard statistics: M = max_r m_r, S = sum_r s_r exp(m_r - M),
    lse = M + log S, z_y from the shard that has the label. Returns (loss, lse)."""
    st = np.asarray(stats_all, dtype=np.float64)
    y = np.asarray(y, dtype=np.int64)
    M = st[:, :, 0].max(axis=0)
    S = (st[:, :, 1] * np.exp(st[:, :, 0] - M[None, :])).sum(axis=0)
    lse = M + np.log(S)
    zt = (st[:, :, 2] * st[:, :, 3]).sum(axis=0)
    valid = y != ignore_index
    if V_total is not None:
        valid &= (y >= 0) & (y < V_total)
    n = int(valid.sum()) if n_valid_override < 0 else int(n_valid_override)
    loss_i = np.where(valid, lse - zt, 0.0)
    return (math.fsum(loss_i.tolist()) / n if n else 0.0), lse


def vshard_backward_f64(H, W_shard, y, vocab_offset, lse, scale, *, ignore_index=IGNORE_INDEX):
    """This shard's dW rows and its part of dH, from the full-vocabulary lse."""
    H = np.asarray(H, dtype=np.float64)
    Ws = np.asarray(W_shard, dtype=np.float64)
    y = np.asarray(y, dtype=np.int64)
    z = H @ Ws.T
    p = np.exp(z - np.asarray(lse)[:, None])
    valid = y != ignore_index
    col = y - vocab_offset
    here = valid & (col >= 0) & (col < Ws.shape[0])
    p[np.nonzero(here)[0], col[here]] -= 1.0
    G = p * (valid * scale)[:, None]
    return G @ Ws, G.T @ H


# ---------------------------------------------------------------------------
# The final zero-centred RMSNorm in front of the LM head ("XTuner on Ascend
# 910C: Qwen3.5-2B training optimisation", section 3.1.1: x / rms(x) scaled by
# (1 + w), one bf16 rounding of the output), and its backward, from the
# definition.
# ---------------------------------------------------------------------------

def round_bf16_bits(a) -> np.ndarray:
    """fp64 -> fp32 -> bf16 bit patterns, round to nearest even."""
    f = np.ascontiguousarray(np.asarray(a, dtype=np.float64).astype(np.float32))
    u = f.view(np.uint32).astype(np.uint64)
    return ((u + 0x7FFF + ((u >> 16) & 1)) >> 16).astype(np.uint16)


def rmsnorm_f64(x, w, eps):
    """out = x r (1 + w), r_i = 1 / sqrt(mean_k x_ik^2 + eps). Returns (out, r)."""
    x = np.asarray(x, dtype=np.float64)
    r = 1.0 / np.sqrt((x * x).mean(axis=1) + eps)
    return x * r[:, None] * (1.0 + np.asarray(w, dtype=np.float64))[None, :], r


def rmsnorm_backward_f64(x, w, r, dout):
    """dx_ik = r_i ((1 + w_k) dout_ik - x_ik r_i^2 c_i / d), c_i = sum_k dout_ik (1 + w_k) x_ik;
    dw_k = sum_i dout_ik x_ik r_i."""
    x = np.asarray(x, dtype=np.float64)
    g = 1.0 + np.asarray(w, dtype=np.float64)
    dout = np.asarray(dout, dtype=np.float64)
    r = np.asarray(r, dtype=np.float64)
    c = (dout * g[None, :] * x).sum(axis=1)
    dx = r[:, None] * (g[None, :] * dout - x * (r * r * c / x.shape[1])[:, None])
    dw = (dout * x * r[:, None]).sum(axis=0)
    return dx, dw


def norm_lce_bf16(xbits, w, Wbits, y, eps, **kw):
    """Norm -> bf16 H -> token cross-entropy -> back through the norm.
    Returns the lce_f64 dict plus dx, dw_norm (fp64)."""
    x = decode_bf16(xbits)
    h, r = rmsnorm_f64(x, w, eps)
    Hb = decode_bf16(round_bf16_bits(h))
    out = lce_f64(Hb, decode_bf16(Wbits), y, **kw)
    out["dx"], out["dw_norm"] = rmsnorm_backward_f64(x, w, r, out["dH"])
    out["H"] = Hb
    return out
