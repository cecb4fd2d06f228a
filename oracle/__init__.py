"""CPU oracle for the fused LM-head linear + cross-entropy (TEST INFRASTRUCTURE).

Two independent fp64 implementations of the same definition:
  * ``lce_oracle.py`` -- numpy, library matmul as a step;
  * ``lce_oracle.c``  -- plain C loops over the definition, loaded with ctypes.

Only ``tests/``, ``__graft_entry__.smoke()`` and ``bench.py``'s CPU-baseline
leg may import this package. The product path (``chunked_lm_head_linear_gb300``)
never imports it, and this package never imports the product path.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

from .lce_oracle import (  # noqa: F401
    IGNORE_INDEX, MEAN, SUM, LabelRangeError, decode_bf16, dH_rows_f64,
    dW_rows_f64, forward_rows_f64, grad_scale, lce_bf16, lce_chunked_online,
    lce_f64, norm_lce_bf16, rmsnorm_backward_f64, rmsnorm_f64, round_bf16_bits,
    vshard_backward_f64, vshard_merge_f64, vshard_stats_f64,
)

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "lce_oracle.c")
_LIB = os.path.join(_HERE, "_build", "liblce_oracle.so")
_lock = threading.Lock()
_lib = None


def build_c_oracle(force: bool = False) -> str:
    """Compile the plain-C oracle with gcc (no fast-math: libm exp/log, IEEE fp64)."""
    os.makedirs(os.path.dirname(_LIB), exist_ok=True)
    if (not force and os.path.exists(_LIB)
            and os.path.getmtime(_LIB) >= os.path.getmtime(_SRC)):
        return _LIB
    tmp = _LIB + f".{os.getpid()}.tmp"
    subprocess.run(["gcc", "-O2", "-fno-fast-math", "-ffp-contract=off", "-std=c11",
                    "-shared", "-fPIC", "-pthread", "-o", tmp, _SRC, "-lm"], check=True)
    os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    with _lock:
        if _lib is None:
            lib = ctypes.CDLL(build_c_oracle())
            f = lib.lce_oracle_f64
            P = ctypes.c_void_p
            f.argtypes = [P, P, P, ctypes.c_int64, ctypes.c_int64, ctypes.c_int64,
                          ctypes.c_int64, ctypes.c_int, ctypes.c_int64, ctypes.c_double,
                          ctypes.c_int, P, P, P, P, P]
            f.restype = ctypes.c_int
            _lib = lib
    return _lib


def lce_c(Hbits, Wbits, y, *, ignore_index=IGNORE_INDEX, reduction=MEAN,
          n_valid_override=-1, grad_loss=1.0, grads=True, nthreads=None):
    """Run the plain-C oracle. Same outputs as ``lce_bf16`` (fp64)."""
    lib = _load()
    H = np.ascontiguousarray(Hbits, dtype=np.uint16)
    W = np.ascontiguousarray(Wbits, dtype=np.uint16)
    y = np.ascontiguousarray(y, dtype=np.int64)
    N, d = H.shape
    V = W.shape[0]
    loss = np.zeros(1)
    lse = np.zeros(N)
    loss_i = np.zeros(N)
    dH = np.zeros((N, d)) if grads else None
    dW = np.zeros((V, d)) if grads else None
    ptr = lambda a: None if a is None else a.ctypes.data
    nthreads = nthreads or os.cpu_count() or 1
    rc = lib.lce_oracle_f64(ptr(H), ptr(W), ptr(y), N, d, V, ignore_index, reduction,
                            n_valid_override, float(grad_loss), int(nthreads),
                            ptr(loss), ptr(lse), ptr(loss_i), ptr(dH), ptr(dW))
    if rc == 2:
        raise LabelRangeError("label outside [0, V) and != ignore_index")
    if rc != 0:
        raise RuntimeError(f"C oracle failed with code {rc}")
    out = {"loss": float(loss[0]), "lse": lse, "loss_i": loss_i}
    if grads:
        out["dH"], out["dW"] = dH, dW
    return out
