"""The C-ABI library: it builds, loads, exports every symbol include/lce.h
declares, and rejects bad arguments on the host before touching a device.
CPU only (no compute calls)."""
import ctypes
import os
import re

import pytest

from chunked_lm_head_linear_gb300 import build, lce

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "lce.h")


@pytest.fixture(scope="module")
def lib():
    build.build()
    return lce.load()


def _declared_functions():
    src = open(HEADER).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(lce_[a-z_]+)\s*\(", src)))


def test_header_and_binding_agree():
    assert _declared_functions() == sorted(lce.EXPORTED)


def test_binding_has_every_entry_point_by_name():
    """The Python binding offers each C entry point under the same name."""
    for name in lce.EXPORTED:
        assert callable(getattr(lce, name, None)), name


def test_every_declared_symbol_is_exported(lib):
    for name in _declared_functions():
        assert hasattr(lib, name), name
    out = os.popen(f"nm -D --defined-only {lce.LIB_PATH}").read()
    for name in _declared_functions():
        assert re.search(rf"\bT {name}$", out, flags=re.M), name


def test_version_and_status_strings(lib):
    assert lib.lce_version() == 1
    for code in range(9):
        s = lce.status_string(code)
        assert s and s != "unknown status"
    assert lce.status_string(99) == "unknown status"


def test_opts_defaults(lib):
    o = lce.LceOpts()
    lib.lce_opts_init(ctypes.byref(o))
    assert (o.chunk_tokens, o.ignore_index, o.n_valid_override, o.reduction,
            o.accumulate_dW, o.sync_check, o.reserved) == (0, -100, -1, 0, 0, 0, 0)
    assert ctypes.sizeof(lce.LceOpts) == 40


def test_workspace_size(lib):
    V, d = 151936, 2048
    fwd = lce.workspace_size(lce.LCE_OP_FORWARD, 8192, d, V)
    bwd = lce.workspace_size(lce.LCE_OP_BACKWARD, 8192, d, V)
    both = lce.workspace_size(lce.LCE_OP_FWD_BWD, 8192, d, V)
    assert 0 < fwd < bwd < both
    # extra memory grows with the chunk, not with N
    o = lce.make_opts(chunk_tokens=1024)
    a = lce.workspace_size(lce.LCE_OP_FWD_BWD, 65536, 4096, V, o)
    b = lce.workspace_size(lce.LCE_OP_FWD_BWD, 8 * 65536, 4096, V, o)
    assert b - a < 8 * 65536 * 16          # only per-token vectors scale with N
    assert a < 65536 * V * 4 / 8           # far below the unfused fp32 logits
    assert lce.workspace_size(lce.LCE_OP_FWD_BWD, 8192, 7, V) == 0      # d % 8 != 0
    assert lce.workspace_size(lce.LCE_OP_FWD_BWD, -1, 8, V) == 0
    assert lce.workspace_size(7, 8, 8, 8) == 0


FAKE = 0x100000  # an aligned non-null address; never dereferenced by host-side checks


def _call_fwd(lib, H=FAKE, W=FAKE, y=FAKE, N=256, d=256, V=4096, loss=FAKE, lse=FAKE, opts=None,
              ws=FAKE, ws_bytes=1 << 40):
    o = opts if opts is not None else lce.make_opts()
    return lib.lce_forward(H, W, y, N, d, V, loss, lse, ctypes.byref(o), ws, ws_bytes, None)


def test_host_side_argument_errors(lib):
    E = lce
    assert _call_fwd(lib, W=None) == E.LCE_ERR_INVALID_ARG
    assert _call_fwd(lib, H=None) == E.LCE_ERR_INVALID_ARG
    assert _call_fwd(lib, y=None) == E.LCE_ERR_INVALID_ARG
    assert _call_fwd(lib, d=12) == E.LCE_ERR_INVALID_ARG
    assert _call_fwd(lib, d=0) == E.LCE_ERR_INVALID_ARG
    assert _call_fwd(lib, V=0) == E.LCE_ERR_INVALID_ARG
    assert _call_fwd(lib, N=-5) == E.LCE_ERR_INVALID_ARG
    assert _call_fwd(lib, H=FAKE + 8) == E.LCE_ERR_ALIGNMENT
    assert _call_fwd(lib, y=FAKE + 4) == E.LCE_ERR_ALIGNMENT           # int64 labels: 8-byte alignment
    assert _call_fwd(lib, lse=FAKE + 2) == E.LCE_ERR_ALIGNMENT
    assert _call_fwd(lib, ws=FAKE + 64) == E.LCE_ERR_ALIGNMENT
    assert _call_fwd(lib, ws_bytes=16) == E.LCE_ERR_WORKSPACE
    bad = lce.make_opts()
    bad.reduction = 7
    assert _call_fwd(lib, opts=bad) == E.LCE_ERR_INVALID_ARG
    bad = lce.make_opts()
    bad.reserved = 1
    assert _call_fwd(lib, opts=bad) == E.LCE_ERR_INVALID_ARG
    o = lce.make_opts()
    P = FAKE
    assert lib.lce_backward(P, P, P, 16, 8, 8, None, None, P, P, ctypes.byref(o), P, 1 << 30, None) \
        == E.LCE_ERR_INVALID_ARG                      # lse missing
    assert lib.lce_fwd_bwd(P, P, P, 16, 8, 8, None, P, None, None, P, ctypes.byref(o), P, 1 << 30, None) \
        == E.LCE_ERR_INVALID_ARG                      # dH missing
    flags = ctypes.c_int()
    assert lib.lce_read_device_status(None, None, ctypes.byref(flags)) == E.LCE_ERR_INVALID_ARG


def test_valid_call_without_a_gpu_fails_cleanly(lib):
    torch = pytest.importorskip("torch")
    if torch.cuda.is_available():
        pytest.skip("a GPU is present")
    rc = _call_fwd(lib)
    assert rc in (lce.LCE_ERR_CUDA, lce.LCE_ERR_UNSUPPORTED_DEVICE)
    # labels at an odd row offset (8-byte aligned) and lse at any 4-byte boundary are accepted
    assert _call_fwd(lib, y=FAKE + 8, lse=FAKE + 4) in (lce.LCE_ERR_CUDA, lce.LCE_ERR_UNSUPPORTED_DEVICE)


def test_binding_refuses_cpu_tensors():
    torch = pytest.importorskip("torch")
    H = torch.zeros(4, 8, dtype=torch.bfloat16)
    W = torch.zeros(3, 8, dtype=torch.bfloat16)
    y = torch.zeros(4, dtype=torch.int64)
    with pytest.raises(ValueError):
        lce.lce_forward(H, W, y)


def test_missing_library_fails_loudly(tmp_path):
    import importlib
    mod = importlib.import_module("chunked_lm_head_linear_gb300.lce")
    with pytest.raises(RuntimeError, match="no CPU fallback"):
        saved = mod._lib
        mod._lib = None
        try:
            mod.load(str(tmp_path / "missing.so"))
        finally:
            mod._lib = saved


def test_auto_chunk_policy(lib):
    """The automatic chunk: largest multiple of 256 (<= 4096, <= N rounded up)
    whose fused workspace fits the budget."""
    V, d = 151936, 2048
    big = 1 << 40
    assert lce.auto_chunk(8192, d, V, big) == 4096
    assert lce.auto_chunk(1000, d, V, big) == 1024
    assert lce.auto_chunk(100, d, V, big) == 256
    for budget_gb in (0.2, 0.5, 1.0, 2.0):
        budget = int(budget_gb * 2**30)
        C = lce.auto_chunk(65536, 4096, V, budget)
        assert C % 256 == 0 and 0 < C <= 4096
        ws = lce.workspace_size(lce.LCE_OP_FWD_BWD, 65536, 4096, V, lce.make_opts(chunk_tokens=C))
        assert ws <= budget
        if C < 4096:   # the next size up would not fit
            assert lce.workspace_size(lce.LCE_OP_FWD_BWD, 65536, 4096, V,
                                      lce.make_opts(chunk_tokens=C + 256)) > budget
    assert lce.auto_chunk(65536, 4096, V, 1 << 20) == 0          # nothing fits in 1 MiB
    assert lce.auto_chunk(8192, 7, V, big) == 0                  # invalid d


def test_profiler_kind_names(lib):
    names = [lib.lce_kernel_name(k).decode() for k in range(lce.LCE_KERNEL_KINDS)]
    assert len(set(names)) == lce.LCE_KERNEL_KINDS
    assert set(lce.GEMM_KINDS) <= set(names)
    assert lib.lce_kernel_name(lce.LCE_KERNEL_KINDS) is None
    assert "memset" in names   # the one kind that is not a library kernel (bench.py leaves it out of gpu_launches)


def test_sliced_bounds_checked_on_host(lib):
    o = lce.make_opts()
    P = FAKE

    def call(bounds, n=None, events=None, sm=0, V=1000):
        n = len(bounds) - 1 if n is None else n
        b = (ctypes.c_int64 * len(bounds))(*bounds)
        return lib.lce_fwd_bwd_sliced(P, P, P, 64, 64, V, None, P, P, P, P, n, b, events, sm,
                                      ctypes.byref(o), P, 1 << 40, None)

    E = lce
    assert call([0, 100, 1000]) == E.LCE_ERR_INVALID_ARG          # interior bound not a multiple of 256
    assert call([0, 512, 256, 1000]) == E.LCE_ERR_INVALID_ARG     # decreasing
    assert call([1, 1000]) == E.LCE_ERR_INVALID_ARG               # does not start at 0
    assert call([0, 999]) == E.LCE_ERR_INVALID_ARG                # does not end at V
    assert call([0, 1000], n=0) == E.LCE_ERR_INVALID_ARG
    assert call([0] * (lce.LCE_MAX_SLICES + 1) + [1000], n=lce.LCE_MAX_SLICES + 1) == E.LCE_ERR_INVALID_ARG
    assert call([0, 1000], sm=1) == E.LCE_ERR_INVALID_ARG
    assert call([0, 1000], sm=-2) == E.LCE_ERR_INVALID_ARG
    null_ev = (ctypes.c_void_p * 2)(None, None)
    assert call([0, 256, 1000], events=null_ev) == E.LCE_ERR_INVALID_ARG
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():      # valid bounds get as far as the device check
        assert call([0, 0, 256, 1000]) in (E.LCE_ERR_CUDA, E.LCE_ERR_UNSUPPORTED_DEVICE)


def test_vshard_chunk_calls_checked_on_host(lib):
    o = lce.make_opts(chunk_tokens=256)
    P = FAKE
    N, d, Vs, Vt = 700, 64, 1000, 4000

    def stats(c0=0, rows=256, st=P, off=1000, opts=o):
        return lib.lce_vshard_chunk_stats(P, P, P, N, d, Vs, off, Vt, c0, rows, st, ctypes.byref(opts), P, 1 << 40,
                                          None)

    def back(c0=0, rows=256, st=P, R=4, lse=P, dH=P, dW=P):
        return lib.lce_vshard_chunk_backward(P, P, P, N, d, Vs, 1000, Vt, c0, rows, st, R, None, lse, dH, dW,
                                             ctypes.byref(o), P, 1 << 40, None)

    E = lce
    assert stats(rows=257) == E.LCE_ERR_INVALID_ARG          # more rows than the chunk
    assert stats(c0=600, rows=101) == E.LCE_ERR_INVALID_ARG   # past N
    assert stats(c0=-1) == E.LCE_ERR_INVALID_ARG
    assert stats(off=3500) == E.LCE_ERR_INVALID_ARG           # shard past V_total
    assert stats(st=None) == E.LCE_ERR_INVALID_ARG
    assert stats(st=P + 8) == E.LCE_ERR_ALIGNMENT
    assert stats(rows=0, st=None) == E.LCE_OK                 # nothing to do
    assert back(R=0) == E.LCE_ERR_INVALID_ARG
    assert back(R=4097) == E.LCE_ERR_INVALID_ARG
    assert back(dW=None) == E.LCE_ERR_INVALID_ARG
    assert back(lse=None) == E.LCE_ERR_INVALID_ARG
    assert back(dH=P + 4) == E.LCE_ERR_ALIGNMENT
    assert back(st=P + 4) == E.LCE_ERR_ALIGNMENT
    assert back(rows=0, st=None, lse=None, dH=None) == E.LCE_OK
    small = lce.workspace_size(lce.LCE_OP_VSHARD_CHUNK, N, d, Vs, o)
    assert 0 < small < lce.workspace_size(lce.LCE_OP_FWD_BWD, N, d, Vs, o)
    assert lib.lce_vshard_chunk_stats(P, P, P, N, d, Vs, 1000, Vt, 0, 256, P, ctypes.byref(o), P, small - 1,
                                      None) == E.LCE_ERR_WORKSPACE
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():      # valid calls get as far as the device check
        assert stats() in (E.LCE_ERR_CUDA, E.LCE_ERR_UNSUPPORTED_DEVICE)
        assert back() in (E.LCE_ERR_CUDA, E.LCE_ERR_UNSUPPORTED_DEVICE)


def test_slice_bounds_helper():
    b = lce.slice_bounds(151936, 8)
    assert b[0] == 0 and b[-1] == 151936 and len(b) == 9
    assert all(x % lce.LCE_SLICE_ALIGN == 0 for x in b[1:-1])
    assert all(b[k] < b[k + 1] for k in range(8))
    tiles = [(b[k + 1] - b[k] + 255) // 256 for k in range(8)]
    assert max(tiles) - min(tiles) <= 1
    assert lce.slice_bounds(1000, 1) == [0, 1000]
    assert lce.slice_bounds(300, 5) == [0, 256, 300]            # no more slices than dW tiles
    with pytest.raises(ValueError):
        lce.slice_bounds(1000, 0)


def test_binding_validates_caller_tensors():
    """A caller's tensor that is not on the GPU is refused before any launch
    (the dtype / shape / contiguity checks run in the GPU tests)."""
    torch = pytest.importorskip("torch")
    with pytest.raises(ValueError, match="CUDA tensor"):
        lce._check_dev(torch.zeros(4, 8), "dW", torch.float32)


def test_binding_refuses_undersized_caller_workspace(lib, monkeypatch):
    """A workspace the caller passes is used as it is or refused with
    LCE_ERR_WORKSPACE (the C ABI's answer), never silently replaced by a larger
    hidden allocation; only a call without one gets a new workspace."""
    torch = pytest.importorskip("torch")
    monkeypatch.setattr(lce, "_check_dev", lambda *a, **k: None)   # CPU tensors stand in for device ones
    need = lce.workspace_size(lce.LCE_OP_FWD_BWD, 700, 64, 1000)
    small = torch.zeros(need - 1, dtype=torch.uint8)
    with pytest.raises(lce.LCEError) as err:
        lce._workspace(lce.LCE_OP_FWD_BWD, 700, 64, 1000, None, torch.device("cpu"), small)
    assert err.value.code == lce.LCE_ERR_WORKSPACE
    exact = torch.zeros(need, dtype=torch.uint8)
    assert lce._workspace(lce.LCE_OP_FWD_BWD, 700, 64, 1000, None, torch.device("cpu"), exact) is exact
    fresh = lce._workspace(lce.LCE_OP_FWD_BWD, 700, 64, 1000, None, torch.device("cpu"), None)
    assert fresh.numel() == need
