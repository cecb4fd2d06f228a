"""Python binding of liblce.so (the C ABI declared in include/lce.h).

Argument marshalling only: PyTorch allocates outputs and the workspace and
supplies the current CUDA stream; every step of the computation runs in the
library's CUDA kernels. There is no CPU fallback: if the library is missing,
``load()`` raises.

Entry points (same names as the C ABI):
  lce_forward(H, W, y)                   -> loss [1], lse [N]
  lce_backward(H, W, y, lse, g)          -> dH [N, d] bf16, dW [V, d] fp32
  lce_fwd_bwd(H, W, y, g)                -> loss, lse, dH, dW
  lce_fwd_bwd_sliced(H, W, y, bounds=..) -> the same, dW finished in vocabulary slices with an event each
  lce_forward_noalloc(H, W, y)           -> loss, lse without a workspace
  lce_vshard_forward_stats / lce_vshard_combine / lce_vshard_backward   W split by vocabulary rows
  lce_vshard_chunk_stats / lce_vshard_chunk_backward   the same per chunk, the exp tile kept between them
  lce_rmsnorm_forward / lce_rmsnorm_backward / lce_norm_fwd_bwd         the final RMSNorm, alone or fused
  lce_scale_grads, auto_chunk (lce_auto_chunk), workspace_size, read_device_status, profile_begin/end
"""
from __future__ import annotations

import ctypes
import os
import threading

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "_build", "liblce.so")

LCE_OK = 0
LCE_ERR_INVALID_ARG = 1
LCE_ERR_ALIGNMENT = 2
LCE_ERR_WORKSPACE = 3
LCE_ERR_UNSUPPORTED_DEVICE = 4
LCE_ERR_CUDA = 5
LCE_ERR_LABEL_RANGE = 6
LCE_ERR_TIMEOUT = 7
LCE_ERR_BOUNDS = 8

LCE_MEAN, LCE_SUM = 0, 1
LCE_OP_FORWARD, LCE_OP_BACKWARD, LCE_OP_FWD_BWD, LCE_OP_VSHARD_COMBINE, LCE_OP_NORM_FWD_BWD = 0, 1, 2, 3, 4
LCE_OP_VSHARD_CHUNK = 5
LCE_DEVICE_LABEL_RANGE, LCE_DEVICE_TIMEOUT, LCE_DEVICE_BOUNDS = 1, 2, 4
LCE_TEST_FORCE_TIMEOUT = 0x7E57

# Every symbol include/lce.h declares.
EXPORTED = ("lce_opts_init", "lce_workspace_size", "lce_forward", "lce_backward", "lce_fwd_bwd",
            "lce_read_device_status", "lce_status_string", "lce_version", "lce_profile_begin",
            "lce_profile_end", "lce_kernel_name", "lce_forward_noalloc", "lce_auto_chunk",
            "lce_vshard_forward_stats", "lce_vshard_combine", "lce_vshard_backward",
            "lce_rmsnorm_workspace_size", "lce_rmsnorm_forward", "lce_rmsnorm_backward", "lce_norm_fwd_bwd",
            "lce_scale_grads", "lce_fwd_bwd_sliced", "lce_vshard_chunk_stats", "lce_vshard_chunk_backward")
LCE_KERNEL_KINDS = 11
# Kernel kinds whose profiled work is flops (tensor-core GEMMs); the others count bytes.
GEMM_KINDS = ("logits_stats", "logits_grad", "gemm_dH_dW", "logits_ref")
# HBM-bound kernels whose profiled work is bytes and which bench.py reports on their own.
HBM_KINDS = ("rmsnorm_fwd", "rmsnorm_bwd")


class LceOpts(ctypes.Structure):
    _fields_ = [("chunk_tokens", ctypes.c_int64), ("ignore_index", ctypes.c_int64),
                ("n_valid_override", ctypes.c_int64), ("reduction", ctypes.c_int32),
                ("accumulate_dW", ctypes.c_int32), ("sync_check", ctypes.c_int32),
                ("reserved", ctypes.c_int32)]


class LceProfile(ctypes.Structure):
    _fields_ = [("launches", ctypes.c_int32 * LCE_KERNEL_KINDS), ("ms", ctypes.c_double * LCE_KERNEL_KINDS),
                ("work", ctypes.c_double * LCE_KERNEL_KINDS)]


class LCEError(RuntimeError):
    def __init__(self, code: int, where: str):
        self.code = code
        super().__init__(f"{where}: {status_string(code)} (status {code})")


_lock = threading.Lock()
_lib = None


def load(path: str | None = None):
    """Load liblce.so (built by ``chunked_lm_head_linear_gb300.build``)."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        p = path or LIB_PATH
        if not os.path.exists(p):
            raise RuntimeError(f"liblce.so not found at {p}: build it with "
                               "`python -m chunked_lm_head_linear_gb300.build` (there is no CPU fallback)")
        lib = ctypes.CDLL(p)
        P, I64, I32 = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int
        OPT = ctypes.POINTER(LceOpts)
        lib.lce_opts_init.argtypes = [OPT]
        lib.lce_opts_init.restype = None
        lib.lce_workspace_size.argtypes = [I32, I64, I64, I64, OPT]
        lib.lce_workspace_size.restype = ctypes.c_size_t
        lib.lce_forward.argtypes = [P, P, P, I64, I64, I64, P, P, OPT, P, ctypes.c_size_t, P]
        lib.lce_forward.restype = I32
        lib.lce_backward.argtypes = [P, P, P, I64, I64, I64, P, P, P, P, OPT, P, ctypes.c_size_t, P]
        lib.lce_backward.restype = I32
        lib.lce_fwd_bwd.argtypes = [P, P, P, I64, I64, I64, P, P, P, P, P, OPT, P, ctypes.c_size_t, P]
        lib.lce_fwd_bwd_sliced.restype = I32
        lib.lce_fwd_bwd_sliced.argtypes = [P, P, P, I64, I64, I64, P, P, P, P, P, I32, ctypes.POINTER(I64),
                                           ctypes.POINTER(P), I32, OPT, P, ctypes.c_size_t, P]
        lib.lce_fwd_bwd.restype = I32
        lib.lce_read_device_status.argtypes = [P, P, ctypes.POINTER(I32)]
        lib.lce_read_device_status.restype = I32
        lib.lce_status_string.argtypes = [I32]
        lib.lce_status_string.restype = ctypes.c_char_p
        lib.lce_version.argtypes = []
        lib.lce_version.restype = I32
        lib.lce_profile_begin.argtypes = []
        lib.lce_profile_begin.restype = I32
        lib.lce_profile_end.argtypes = [ctypes.POINTER(LceProfile)]
        lib.lce_profile_end.restype = I32
        lib.lce_vshard_forward_stats.argtypes = [P, P, P, I64, I64, I64, I64, I64, P, OPT, P, ctypes.c_size_t, P]
        lib.lce_vshard_forward_stats.restype = I32
        lib.lce_vshard_combine.argtypes = [P, I64, P, I64, I64, P, P, OPT, P, ctypes.c_size_t, P]
        lib.lce_vshard_combine.restype = I32
        lib.lce_vshard_backward.argtypes = [P, P, P, I64, I64, I64, I64, I64, P, P, P, P, OPT, P, ctypes.c_size_t, P]
        lib.lce_vshard_backward.restype = I32
        lib.lce_vshard_chunk_stats.argtypes = [P, P, P, I64, I64, I64, I64, I64, I64, I64, P, OPT, P, ctypes.c_size_t,
                                               P]
        lib.lce_vshard_chunk_stats.restype = I32
        lib.lce_vshard_chunk_backward.argtypes = [P, P, P, I64, I64, I64, I64, I64, I64, I64, P, I64, P, P, P, P, OPT,
                                                  P, ctypes.c_size_t, P]
        lib.lce_vshard_chunk_backward.restype = I32
        F32 = ctypes.c_float
        lib.lce_rmsnorm_workspace_size.argtypes = [I64, I64]
        lib.lce_rmsnorm_workspace_size.restype = ctypes.c_size_t
        lib.lce_rmsnorm_forward.argtypes = [P, P, I64, I64, F32, P, P, P]
        lib.lce_rmsnorm_forward.restype = I32
        lib.lce_rmsnorm_backward.argtypes = [P, P, P, P, I64, I64, P, P, P, ctypes.c_size_t, P]
        lib.lce_rmsnorm_backward.restype = I32
        lib.lce_norm_fwd_bwd.argtypes = [P, P, F32, P, P, I64, I64, I64, P, P, P, P, P, P, OPT, P, ctypes.c_size_t, P]
        lib.lce_norm_fwd_bwd.restype = I32
        lib.lce_scale_grads.argtypes = [P, P, I64, I64, I64, P, P]
        lib.lce_scale_grads.restype = I32
        lib.lce_auto_chunk.argtypes = [I64, I64, I64, ctypes.c_size_t, OPT]
        lib.lce_auto_chunk.restype = I64
        lib.lce_forward_noalloc.argtypes = [P, P, P, I64, I64, I64, P, P, OPT, P]
        lib.lce_forward_noalloc.restype = I32
        lib.lce_kernel_name.argtypes = [I32]
        lib.lce_kernel_name.restype = ctypes.c_char_p
        _lib = lib
        return lib


def status_string(code: int) -> str:
    return load().lce_status_string(int(code)).decode()


def auto_chunk(N: int, d: int, V: int, budget_bytes: int, opts: LceOpts | None = None) -> int:
    """Largest chunk (multiple of 256 tokens, <= 4096) whose workspace fits the budget; 0 if none."""
    return int(load().lce_auto_chunk(N, d, V, int(budget_bytes), ctypes.byref(opts) if opts is not None else None))


def _resolve_chunk(chunk_tokens, N, d, V, device):
    """chunk_tokens="auto": half of the device's free memory is the workspace budget."""
    if chunk_tokens != "auto":
        return chunk_tokens
    import torch
    free, _ = torch.cuda.mem_get_info(device)
    c = auto_chunk(N, d, V, free // 2)
    if c == 0:
        raise LCEError(LCE_ERR_WORKSPACE, "auto_chunk: not even a 256-token chunk fits in half the free memory")
    return c


def make_opts(chunk_tokens=0, ignore_index=-100, reduction="mean", n_valid_override=-1,
              accumulate_dW=False, sync_check=False, reserved=0) -> LceOpts:
    o = LceOpts()
    load().lce_opts_init(ctypes.byref(o))
    o.chunk_tokens = int(chunk_tokens)
    o.ignore_index = int(ignore_index)
    o.n_valid_override = int(n_valid_override)
    o.reduction = {"mean": LCE_MEAN, "sum": LCE_SUM}[reduction] if isinstance(reduction, str) else int(reduction)
    o.accumulate_dW = int(bool(accumulate_dW))
    o.sync_check = int(bool(sync_check))
    o.reserved = int(reserved)
    return o


def workspace_size(op: int, N: int, d: int, V: int, opts: LceOpts | None = None) -> int:
    return int(load().lce_workspace_size(op, N, d, V, ctypes.byref(opts) if opts is not None else None))


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream=None):
    import torch
    s = stream if stream is not None else torch.cuda.current_stream()
    return ctypes.c_void_p(s.cuda_stream)


def _check_inputs(H, W, y):
    import torch
    if not (H.is_cuda and W.is_cuda and y.is_cuda):
        raise ValueError("H, W and y must be CUDA tensors (there is no CPU path)")
    if H.dtype != torch.bfloat16 or W.dtype != torch.bfloat16 or y.dtype != torch.int64:
        raise ValueError("H and W must be bfloat16, y int64")
    if H.dim() != 2 or W.dim() != 2 or y.dim() != 1 or H.shape[1] != W.shape[1] or y.shape[0] != H.shape[0]:
        raise ValueError("shapes must be H [N, d], W [V, d], y [N]")
    if not (H.is_contiguous() and W.is_contiguous() and y.is_contiguous()):
        raise ValueError("H, W and y must be contiguous")
    if not (H.device == W.device == y.device):
        raise ValueError("H, W and y must be on the same device")
    if H.device.index != torch.cuda.current_device():
        raise ValueError(f"the inputs are on {H.device}; make it the current device (torch.cuda.set_device)")
    return H.shape[0], H.shape[1], W.shape[0]


def _check_grads(H, N, d, V, *, lse=None, grad_loss=None, dW=None, lse_needs_n=True):
    import torch
    _check_dev(lse, "lse", torch.float32, numel=N if lse_needs_n else None, device=H.device)
    _check_dev(grad_loss, "grad_loss", torch.float32, numel=1, device=H.device)
    _check_dev(dW, "dW", torch.float32, shape=(V, d), device=H.device)


def _check_dev(t, name, dtype, numel=None, shape=None, device=None):
    """A caller-supplied tensor the kernels read or write: CUDA, the given dtype,
    contiguous, on ``device``, and with the shape (or at least ``numel``
    elements) the call needs, so that no kernel touches memory past it."""
    import torch
    if t is None:
        return
    if not isinstance(t, torch.Tensor) or not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if t.dtype != dtype:
        raise ValueError(f"{name} must be {dtype}, got {t.dtype}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if device is not None and t.device != device:
        raise ValueError(f"{name} is on {t.device}, the inputs on {device}")
    if shape is not None and tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name} must have shape {tuple(shape)}, got {tuple(t.shape)}")
    if numel is not None and t.numel() < numel:
        raise ValueError(f"{name} needs at least {numel} elements, has {t.numel()}")


def _workspace(op, N, d, V, opts, device, workspace=None):
    """The caller's workspace if it is large enough (else LCE_ERR_WORKSPACE, as
    the C ABI answers: a caller that sized its own workspace, to bound memory or
    for graph capture, must not get a hidden allocation); a new one only when
    the caller passed none."""
    import torch
    need = workspace_size(op, N, d, V, opts)
    if need == 0:
        raise LCEError(LCE_ERR_INVALID_ARG, "lce_workspace_size")
    if workspace is not None:
        _check_dev(workspace, "workspace", torch.uint8, device=device)
        if workspace.numel() < need:
            raise LCEError(LCE_ERR_WORKSPACE, f"workspace of {workspace.numel()} bytes, the call needs {need}")
        return workspace
    # torch's allocator returns 512-byte aligned blocks
    return torch.empty(need, dtype=torch.uint8, device=device)


def _no_accumulate_without_dW(opts):
    """accumulate_dW adds into the caller's dW: without one there is nothing to add to."""
    if opts.accumulate_dW:
        raise ValueError("accumulate_dW=True needs the dW tensor to accumulate into")


def _keep(stream, *tensors):
    """Tensors a call used on a stream other than the current one: tell the
    caching allocator, so that their memory is not handed out again while that
    stream's kernels may still use it (the workspace is freed as the wrapper
    returns)."""
    if stream is None:
        return
    for t in tensors:
        if t is not None:
            t.record_stream(stream)


def _raise(rc, where):
    if rc != LCE_OK:
        raise LCEError(rc, where)


def lce_forward(H, W, y, *, workspace=None, stream=None, **opt_kw):
    """loss (fp32 [1]) and lse (fp32 [N]) of the token-level cross-entropy."""
    import torch
    N, d, V = _check_inputs(H, W, y)
    if "chunk_tokens" in opt_kw:
        opt_kw["chunk_tokens"] = _resolve_chunk(opt_kw["chunk_tokens"], N, d, V, H.device)
    opts = make_opts(**opt_kw)
    ws = _workspace(LCE_OP_FORWARD, N, d, V, opts, H.device, workspace)
    loss = torch.empty(1, dtype=torch.float32, device=H.device)
    lse = torch.empty(max(N, 1), dtype=torch.float32, device=H.device)[:N]
    rc = load().lce_forward(_ptr(H), _ptr(W), _ptr(y), N, d, V, _ptr(loss), _ptr(lse), ctypes.byref(opts),
                            _ptr(ws), ws.numel(), _stream(stream))
    _raise(rc, "lce_forward")
    _keep(stream, ws, loss, lse)
    return loss, lse


def lce_backward(H, W, y, lse, grad_loss=None, *, dW=None, workspace=None, stream=None, **opt_kw):
    """dH (bf16 [N, d]) and dW (fp32 [V, d]) from a saved lse; grad_loss is a
    device fp32 scalar tensor or None (1.0)."""
    import torch
    N, d, V = _check_inputs(H, W, y)
    _check_grads(H, N, d, V, lse=lse, grad_loss=grad_loss, dW=dW)
    if N > 0 and lse is None:
        raise ValueError("lse is required")
    if "chunk_tokens" in opt_kw:
        opt_kw["chunk_tokens"] = _resolve_chunk(opt_kw["chunk_tokens"], N, d, V, H.device)
    opts = make_opts(**opt_kw)
    ws = _workspace(LCE_OP_BACKWARD, N, d, V, opts, H.device, workspace)
    dH = torch.empty_like(H)
    if dW is None:
        _no_accumulate_without_dW(opts)
        dW = torch.empty((V, d), dtype=torch.float32, device=H.device)
    rc = load().lce_backward(_ptr(H), _ptr(W), _ptr(y), N, d, V, _ptr(lse), _ptr(grad_loss), _ptr(dH), _ptr(dW),
                             ctypes.byref(opts), _ptr(ws), ws.numel(), _stream(stream))
    _raise(rc, "lce_backward")
    _keep(stream, ws, dH, dW, lse, grad_loss)
    return dH, dW


def lce_fwd_bwd(H, W, y, grad_loss=None, *, dW=None, lse=None, workspace=None, stream=None, **opt_kw):
    """loss, lse, dH, dW in one call."""
    import torch
    N, d, V = _check_inputs(H, W, y)
    _check_grads(H, N, d, V, lse=lse, grad_loss=grad_loss, dW=dW)
    if "chunk_tokens" in opt_kw:
        opt_kw["chunk_tokens"] = _resolve_chunk(opt_kw["chunk_tokens"], N, d, V, H.device)
    opts = make_opts(**opt_kw)
    ws = _workspace(LCE_OP_FWD_BWD, N, d, V, opts, H.device, workspace)
    loss = torch.empty(1, dtype=torch.float32, device=H.device)
    if lse is None:
        lse = torch.empty(max(N, 1), dtype=torch.float32, device=H.device)[:N]
    dH = torch.empty_like(H)
    if dW is None:
        _no_accumulate_without_dW(opts)
        dW = torch.empty((V, d), dtype=torch.float32, device=H.device)
    rc = load().lce_fwd_bwd(_ptr(H), _ptr(W), _ptr(y), N, d, V, _ptr(grad_loss), _ptr(loss), _ptr(lse), _ptr(dH),
                            _ptr(dW), ctypes.byref(opts), _ptr(ws), ws.numel(), _stream(stream))
    _raise(rc, "lce_fwd_bwd")
    _keep(stream, ws, loss, lse, dH, dW, grad_loss)
    return loss, lse, dH, dW


def lce_forward_noalloc(H, W, y, *, loss=None, lse=None, stream=None, **opt_kw):
    """loss and lse like lce_forward, but the library uses its fixed device
    scratch array instead of a workspace (nothing is allocated by the library;
    ``loss`` / ``lse`` may be passed in so that this call allocates nothing
    either). Calls that overlap on the GPU share the scratch and must be
    serialised by the caller."""
    import torch
    N, d, V = _check_inputs(H, W, y)
    _check_dev(loss, "loss", torch.float32, numel=1, device=H.device)
    _check_dev(lse, "lse", torch.float32, numel=N, device=H.device)
    if "chunk_tokens" in opt_kw and opt_kw["chunk_tokens"] == "auto":
        raise ValueError('lce_forward_noalloc: chunk_tokens="auto" sizes a workspace; give a number')
    opts = make_opts(**opt_kw)
    if loss is None:
        loss = torch.empty(1, dtype=torch.float32, device=H.device)
    if lse is None:
        lse = torch.empty(max(N, 1), dtype=torch.float32, device=H.device)[:N]
    rc = load().lce_forward_noalloc(_ptr(H), _ptr(W), _ptr(y), N, d, V, _ptr(loss), _ptr(lse), ctypes.byref(opts),
                                    _stream(stream))
    _raise(rc, "lce_forward_noalloc")
    _keep(stream, loss, lse)
    return loss, lse


LCE_MAX_SLICES = 4096
LCE_SLICE_ALIGN = 256


def slice_bounds(V: int, n_slices: int) -> list:
    """Vocabulary cut into n_slices contiguous row ranges of (nearly) equal
    numbers of 256-row dW tiles: [0, b_1, ..., V], interior bounds multiples of 256."""
    if n_slices < 1:
        raise ValueError("n_slices must be >= 1")
    tiles = (V + LCE_SLICE_ALIGN - 1) // LCE_SLICE_ALIGN
    n = min(n_slices, max(tiles, 1))
    b = [min(V, LCE_SLICE_ALIGN * ((k * tiles) // n)) for k in range(n + 1)]
    b[-1] = V
    return b


def lce_fwd_bwd_sliced(H, W, y, grad_loss=None, *, bounds, events=None, sm_limit: int = 0, dW=None, lse=None,
                       workspace=None, stream=None, **opt_kw):
    """lce_fwd_bwd whose dW is finished slice by slice: ``events[s]`` (torch.cuda.Event,
    or None for no events) is recorded on the stream once dW rows
    [bounds[s], bounds[s+1]) are final. Same outputs as lce_fwd_bwd, bit for bit."""
    import torch
    N, d, V = _check_inputs(H, W, y)
    _check_grads(H, N, d, V, lse=lse, grad_loss=grad_loss, dW=dW)
    if "chunk_tokens" in opt_kw:
        opt_kw["chunk_tokens"] = _resolve_chunk(opt_kw["chunk_tokens"], N, d, V, H.device)
    opts = make_opts(**opt_kw)
    n = len(bounds) - 1
    if n < 1:
        raise ValueError("bounds must hold at least two entries")
    ws = _workspace(LCE_OP_FWD_BWD, N, d, V, opts, H.device, workspace)
    loss = torch.empty(1, dtype=torch.float32, device=H.device)
    if lse is None:
        lse = torch.empty(max(N, 1), dtype=torch.float32, device=H.device)[:N]
    dH = torch.empty_like(H)
    if dW is None:
        _no_accumulate_without_dW(opts)
        dW = torch.empty((V, d), dtype=torch.float32, device=H.device)
    b = (ctypes.c_int64 * (n + 1))(*[int(x) for x in bounds])
    ev = None
    if events is not None:
        if len(events) != n:
            raise ValueError("one event per slice")
        st = stream if stream is not None else torch.cuda.current_stream(H.device)
        for e in events:          # creates the underlying CUDA event if it does not exist yet
            e.record(st)
        ev = (ctypes.c_void_p * n)(*[ctypes.c_void_p(e.cuda_event) for e in events])
    rc = load().lce_fwd_bwd_sliced(_ptr(H), _ptr(W), _ptr(y), N, d, V, _ptr(grad_loss), _ptr(loss), _ptr(lse),
                                   _ptr(dH), _ptr(dW), n, b, ev, int(sm_limit), ctypes.byref(opts), _ptr(ws),
                                   ws.numel(), _stream(stream))
    _raise(rc, "lce_fwd_bwd_sliced")
    _keep(stream, ws, loss, lse, dH, dW, grad_loss)
    return loss, lse, dH, dW


def read_device_status(workspace, stream=None) -> int:
    """Device status bits (LCE_DEVICE_*) left in a workspace by the last call."""
    flags = ctypes.c_int(0)
    _raise(load().lce_read_device_status(_ptr(workspace), _stream(stream), ctypes.byref(flags)),
           "lce_read_device_status")
    return flags.value


def profile_begin():
    """Start bracketing every library launch with CUDA events on its stream."""
    _raise(load().lce_profile_begin(), "lce_profile_begin")


def profile_end() -> dict:
    """Stop profiling; per kernel kind: launches, summed device ms, summed work."""
    p = LceProfile()
    _raise(load().lce_profile_end(ctypes.byref(p)), "lce_profile_end")
    out = {}
    for k in range(LCE_KERNEL_KINDS):
        name = load().lce_kernel_name(k).decode()
        out[name] = {"launches": p.launches[k], "ms": p.ms[k], "work": p.work[k]}
    return out


# The C ABI's helper calls under their own names (the wrappers above use shorter ones).
def lce_opts_init(**opt_kw) -> LceOpts:
    """Defaults of the C ABI (chunk chosen by the library, ignore_index -100,
    mean), then the given fields."""
    return make_opts(**opt_kw)


def lce_workspace_size(op: int, N: int, d: int, V: int, opts: LceOpts | None = None) -> int:
    return workspace_size(op, N, d, V, opts)


def lce_auto_chunk(N: int, d: int, V: int, budget_bytes: int, opts: LceOpts | None = None) -> int:
    return auto_chunk(N, d, V, budget_bytes, opts)


def lce_read_device_status(workspace, stream=None) -> int:
    return read_device_status(workspace, stream)


def lce_status_string(code: int) -> str:
    return status_string(code)


def lce_version() -> int:
    return int(load().lce_version())


def lce_profile_begin():
    profile_begin()


def lce_profile_end() -> dict:
    return profile_end()


def lce_kernel_name(kind: int) -> str:
    return load().lce_kernel_name(int(kind)).decode()


def lce_rmsnorm_workspace_size(N: int, d: int) -> int:
    return int(load().lce_rmsnorm_workspace_size(int(N), int(d)))


# ---------------------------------------------------------------------------
# Vocabulary-parallel pieces (W split by rows; see include/lce.h)
# ---------------------------------------------------------------------------
def lce_vshard_forward_stats(H, W_shard, y, vocab_offset: int, V_total: int, *, workspace=None, stream=None,
                             **opt_kw):
    """Per-row (max, sum-exp, label logit, has-label) of this vocabulary shard: fp32 [N, 4]."""
    import torch
    N, d, Vs = _check_inputs(H, W_shard, y)
    opts = make_opts(**opt_kw)
    ws = _workspace(LCE_OP_FORWARD, N, d, Vs, opts, H.device, workspace)
    stats = torch.empty((max(N, 1), 4), dtype=torch.float32, device=H.device)[:N]
    rc = load().lce_vshard_forward_stats(_ptr(H), _ptr(W_shard), _ptr(y), N, d, Vs, int(vocab_offset), int(V_total),
                                         _ptr(stats), ctypes.byref(opts), _ptr(ws), ws.numel(), _stream(stream))
    _raise(rc, "lce_vshard_forward_stats")
    _keep(stream, ws, stats)
    return stats


def lce_vshard_combine(stats_all, y, V_total: int, *, workspace=None, stream=None, **opt_kw):
    """Merge the shards' statistics [R, N, 4] (rank order) into lse [N] and the loss [1]."""
    import torch
    if not (isinstance(stats_all, torch.Tensor) and stats_all.dim() == 3 and stats_all.shape[2] == 4):
        raise ValueError("stats_all must be an fp32 CUDA tensor [R, N, 4]")
    R, N = int(stats_all.shape[0]), int(stats_all.shape[1])
    _check_dev(stats_all, "stats_all", torch.float32)
    _check_dev(y, "y", torch.int64, shape=(N,), device=stats_all.device)
    opts = make_opts(**opt_kw)
    ws = _workspace(LCE_OP_VSHARD_COMBINE, N, 8, V_total, opts, stats_all.device, workspace)
    lse = torch.empty(max(N, 1), dtype=torch.float32, device=stats_all.device)[:N]
    loss = torch.empty(1, dtype=torch.float32, device=stats_all.device)
    rc = load().lce_vshard_combine(_ptr(stats_all), R, _ptr(y), N, int(V_total), _ptr(lse), _ptr(loss),
                                   ctypes.byref(opts), _ptr(ws), ws.numel(), _stream(stream))
    _raise(rc, "lce_vshard_combine")
    _keep(stream, ws, loss, lse)
    return loss, lse


def lce_vshard_backward(H, W_shard, y, vocab_offset: int, V_total: int, lse, grad_loss=None, *, dW=None,
                        workspace=None, stream=None, **opt_kw):
    """This shard's dW [V_shard, d] and its fp32 partial dH [N, d] (sum over shards = dH)."""
    import torch
    N, d, Vs = _check_inputs(H, W_shard, y)
    _check_grads(H, N, d, Vs, lse=lse, grad_loss=grad_loss, dW=dW)
    if N > 0 and lse is None:
        raise ValueError("lse is required")
    opts = make_opts(**opt_kw)
    ws = _workspace(LCE_OP_BACKWARD, N, d, Vs, opts, H.device, workspace)
    dH = torch.empty((N, d), dtype=torch.float32, device=H.device)
    if dW is None:
        _no_accumulate_without_dW(opts)
        dW = torch.empty((Vs, d), dtype=torch.float32, device=H.device)
    rc = load().lce_vshard_backward(_ptr(H), _ptr(W_shard), _ptr(y), N, d, Vs, int(vocab_offset), int(V_total),
                                    _ptr(lse), _ptr(grad_loss), _ptr(dH), _ptr(dW), ctypes.byref(opts), _ptr(ws),
                                    ws.numel(), _stream(stream))
    _raise(rc, "lce_vshard_backward")
    _keep(stream, ws, dH, dW, lse, grad_loss)
    return dH, dW


def vshard_chunk_workspace(H, W_shard, y, **opt_kw):
    """Workspace for lce_vshard_chunk_stats / lce_vshard_chunk_backward (one chunk's exp tile)."""
    N, d, Vs = _check_inputs(H, W_shard, y)
    return _workspace(LCE_OP_VSHARD_CHUNK, N, d, Vs, make_opts(**opt_kw), H.device)


def _chunk_ws(workspace, N, d, Vs, opts, device):
    import torch
    _check_dev(workspace, "workspace", torch.uint8, device=device)
    if workspace is None or workspace.numel() < workspace_size(LCE_OP_VSHARD_CHUNK, N, d, Vs, opts):
        raise LCEError(LCE_ERR_WORKSPACE, "vshard chunk calls need vshard_chunk_workspace(...)")
    return workspace


def lce_vshard_chunk_stats(H, W_shard, y, vocab_offset: int, V_total: int, c0: int, rows: int, *, workspace,
                           stream=None, **opt_kw):
    """Statistics [rows, 4] of chunk rows [c0, c0 + rows) of this shard (as
    lce_vshard_forward_stats); the chunk's exp tile stays in ``workspace``."""
    import torch
    N, d, Vs = _check_inputs(H, W_shard, y)
    opts = make_opts(**opt_kw)
    ws = _chunk_ws(workspace, N, d, Vs, opts, H.device)
    stats = torch.empty((max(int(rows), 1), 4), dtype=torch.float32, device=H.device)[:int(rows)]
    rc = load().lce_vshard_chunk_stats(_ptr(H), _ptr(W_shard), _ptr(y), N, d, Vs, int(vocab_offset), int(V_total),
                                       int(c0), int(rows), _ptr(stats), ctypes.byref(opts), _ptr(ws), ws.numel(),
                                       _stream(stream))
    _raise(rc, "lce_vshard_chunk_stats")
    _keep(stream, ws, stats)
    return stats


def lce_vshard_chunk_backward(H, W_shard, y, vocab_offset: int, V_total: int, c0: int, rows: int, stats_all, *,
                              workspace, lse, dH_partial, dW_shard, grad_loss=None, stream=None, **opt_kw):
    """With the R ranks' statistics of the chunk (stats_all [R, rows, 4], rank
    order) and the workspace of the stats call: writes lse and dH_partial rows
    [c0, c0 + rows) and writes (c0 == 0) or adds to dW_shard [V_shard, d]."""
    import torch
    N, d, Vs = _check_inputs(H, W_shard, y)
    opts = make_opts(**opt_kw)
    ws = _chunk_ws(workspace, N, d, Vs, opts, H.device)
    _check_grads(H, N, d, Vs, lse=lse, grad_loss=grad_loss, dW=dW_shard)
    _check_dev(dH_partial, "dH_partial", torch.float32, shape=(N, d), device=H.device)
    _check_dev(stats_all, "stats_all", torch.float32, device=H.device)
    if stats_all is None or stats_all.dim() != 3 or stats_all.shape[1:] != (int(rows), 4):
        raise ValueError(f"stats_all must have shape [R, {int(rows)}, 4]")
    if lse is None or dH_partial is None or dW_shard is None:
        raise ValueError("lse, dH_partial and dW_shard are required")
    rc = load().lce_vshard_chunk_backward(_ptr(H), _ptr(W_shard), _ptr(y), N, d, Vs, int(vocab_offset), int(V_total),
                                          int(c0), int(rows), _ptr(stats_all), int(stats_all.shape[0]),
                                          _ptr(grad_loss), _ptr(lse), _ptr(dH_partial), _ptr(dW_shard),
                                          ctypes.byref(opts), _ptr(ws), ws.numel(), _stream(stream))
    _raise(rc, "lce_vshard_chunk_backward")
    _keep(stream, ws, stats_all, lse, dH_partial, dW_shard, grad_loss)


# ---------------------------------------------------------------------------
# Final zero-centred RMSNorm (see include/lce.h)
# ---------------------------------------------------------------------------
def _check_norm(x, w):
    import torch
    if not (x.is_cuda and w.is_cuda) or x.dtype != torch.bfloat16 or w.dtype != torch.float32:
        raise ValueError("x must be a bf16 CUDA tensor [N, d], w an fp32 CUDA tensor [d]")
    if x.dim() != 2 or w.dim() != 1 or w.shape[0] != x.shape[1] or not (x.is_contiguous() and w.is_contiguous()):
        raise ValueError("shapes must be x [N, d], w [d], contiguous")
    if x.device != w.device or x.device.index != torch.cuda.current_device():
        raise ValueError("x and w must be on the current CUDA device")
    return x.shape[0], x.shape[1]


def lce_rmsnorm_forward(x, w, eps=1e-6, *, stream=None):
    """H = bf16(x / rms(x) * (1 + w)) and the per-row 1/rms (fp32)."""
    import torch
    N, d = _check_norm(x, w)
    H = torch.empty_like(x)
    rstd = torch.empty(max(N, 1), dtype=torch.float32, device=x.device)[:N]
    _raise(load().lce_rmsnorm_forward(_ptr(x), _ptr(w), N, d, float(eps), _ptr(H), _ptr(rstd), _stream(stream)),
           "lce_rmsnorm_forward")
    _keep(stream, H, rstd)
    return H, rstd


def lce_rmsnorm_backward(x, w, rstd, dH, *, stream=None):
    """dx (bf16 [N, d]) and dw (fp32 [d]) of the zero-centred RMSNorm."""
    import torch
    N, d = _check_norm(x, w)
    _check_dev(rstd, "rstd", torch.float32, numel=N, device=x.device)
    _check_dev(dH, "dH", torch.bfloat16, shape=(N, d), device=x.device)
    dx = torch.empty_like(x)
    dw = torch.empty(d, dtype=torch.float32, device=x.device)
    need = int(load().lce_rmsnorm_workspace_size(N, d))
    if need == 0:
        raise LCEError(LCE_ERR_INVALID_ARG, "lce_rmsnorm_workspace_size")
    ws = torch.empty(need, dtype=torch.uint8, device=x.device)
    _raise(load().lce_rmsnorm_backward(_ptr(x), _ptr(w), _ptr(rstd), _ptr(dH), N, d, _ptr(dx), _ptr(dw), _ptr(ws),
                                       ws.numel(), _stream(stream)), "lce_rmsnorm_backward")
    _keep(stream, ws, dx, dw)
    return dx, dw


def lce_norm_fwd_bwd(x, w_norm, W, y, grad_loss=None, eps=1e-6, *, dW=None, workspace=None, stream=None, **opt_kw):
    """Final norm + LM head + cross-entropy, forward and backward:
    returns loss, lse, dx, dw_norm, dW."""
    import torch
    N, d = _check_norm(x, w_norm)
    if W.dim() != 2 or W.shape[1] != d or W.dtype != torch.bfloat16 or not W.is_contiguous():
        raise ValueError("W must be a contiguous bf16 [V, d] tensor")
    V = W.shape[0]
    _check_dev(W, "W", torch.bfloat16, device=x.device)
    _check_dev(y, "y", torch.int64, shape=(N,), device=x.device)
    _check_grads(x, N, d, V, grad_loss=grad_loss, dW=dW)
    opts = make_opts(**opt_kw)
    ws = _workspace(LCE_OP_NORM_FWD_BWD, N, d, V, opts, x.device, workspace)
    loss = torch.empty(1, dtype=torch.float32, device=x.device)
    lse = torch.empty(max(N, 1), dtype=torch.float32, device=x.device)[:N]
    dx = torch.empty_like(x)
    dw_norm = torch.empty(d, dtype=torch.float32, device=x.device)
    if dW is None:
        _no_accumulate_without_dW(opts)
        dW = torch.empty((V, d), dtype=torch.float32, device=x.device)
    rc = load().lce_norm_fwd_bwd(_ptr(x), _ptr(w_norm), float(eps), _ptr(W), _ptr(y), N, d, V, _ptr(grad_loss),
                                 _ptr(loss), _ptr(lse), _ptr(dx), _ptr(dw_norm), _ptr(dW), ctypes.byref(opts),
                                 _ptr(ws), ws.numel(), _stream(stream))
    _raise(rc, "lce_norm_fwd_bwd")
    _keep(stream, ws, loss, lse, dx, dw_norm, dW, grad_loss)
    return loss, lse, dx, dw_norm, dW


def lce_scale_grads(dH, dW, grad_loss, *, stream=None):
    """In place: dH *= g, dW *= g with g = grad_loss[0] read on the device (no-op when g == 1)."""
    import torch
    if dH is None and dW is None:
        return
    _check_dev(dH, "dH", torch.bfloat16)
    _check_dev(dW, "dW", torch.float32)
    _check_dev(grad_loss, "grad_loss", torch.float32, numel=1)
    if (dH is not None and dH.dim() != 2) or (dW is not None and dW.dim() != 2) or \
            (dH is not None and dW is not None and dH.shape[1] != dW.shape[1]):
        raise ValueError("dH must be [N, d] and dW [V, d]")
    N, d = (dH.shape if dH is not None else (0, dW.shape[1]))
    V = dW.shape[0] if dW is not None else 0
    _raise(load().lce_scale_grads(_ptr(dH), _ptr(dW), N, d, V, _ptr(grad_loss), _stream(stream)), "lce_scale_grads")
