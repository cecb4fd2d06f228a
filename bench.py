"""Benchmark of the fused chunked LM-head linear + cross-entropy (forward + backward).

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                    [--workload NAME] [--chunk C]

One step = one lce_fwd_bwd call over the whole batch: logits GEMMs with the
streaming log-sum-exp epilogue, gradient tiles, dH and dW GEMMs, loss
reduction, on synthetic inputs of the Qwen3.5-2B-like LM-head workload
(N = 8192 tokens, d = 2048, V = 151936; H ~ N(0,1) bf16, W ~ N(0, 0.02) bf16,
uniform labels, 5% ignored at packed-document starts, seed 0).

Prints ONE JSON line (rank 0). Metric: tokens/s of the fused fwd+bwd, with
TFLOP/s counted as 6*N*V*d per step and its fraction of the dense bf16 peak.
``roofline`` holds the dominant kernel (events around every library launch on
its stream) against the measured burst peak when the timed region is under a
second and the sustained one otherwise; ``gemm_kernels`` gives both GEMM
kinds' fractions of both peaks and, for regions of a second or more, of the
tensor-core limit at the sampled SM clock (``frac_per_clock``).
``value`` is device-resident throughput; ``e2e`` repeats it through the same
public call with every step's inputs copied from pinned host memory (the next
step's copy overlapping the current step's compute) and the loss read back
every step. Inputs (W 0.62 GB, dW 1.24 GB, gradient tiles
> 1 GB) are larger than the 129 MB L2, so no separate L2 flush is done.

Multi-GPU (torchrun, one rank per GPU): data parallel over tokens, weak
scaling. Each rank holds its own 8192-token shard; the global count of valid
tokens is all-reduced once, every step runs lce_fwd_bwd with that global
denominator and all-reduces dW (sum) and the loss (sum) over NCCL.

``--impl reference`` times the fp64 CPU oracle on the host cores instead
(rank 0 only), each step a bounded sample of the same workload.
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from chunked_lm_head_linear_gb300 import inputs  # noqa: E402

METRIC = "tokens/s fused linear-CE fwd+bwd (d=2048,V=151936); % of BF16 tensor peak"
UNIT = "tokens/s"
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return d, "measured"
    return dict(FALLBACK_PEAKS), "fallback"


# ---------------------------------------------------------------------------
# clocks during the timed region
# ---------------------------------------------------------------------------
class ClockSampler:
    FIELDS = ("timestamp,uuid,index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, uuid: str | None):
        self.uuid = uuid
        self.proc = None
        self.lines = []
        self.thread = None
        self.window = None   # (start, end) host time of the timed region

    def mark(self, start: float, end: float):
        """The timed region, in host seconds since the epoch: only samples taken
        inside it count."""
        self.window = (start, end)

    def start(self):
        try:
            self.proc = subprocess.Popen(["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader",
                                          "-lms", "50"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL,
                                         text=True)
        except OSError:
            self.proc = None
            return
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        if self.thread:
            self.thread.join(timeout=5)
        import datetime
        sm, smax, power, reasons = [], [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        outside = 0
        for ln in self.lines:
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) < 11:
                continue
            if self.uuid and self.uuid not in parts[1]:
                continue
            if self.window is not None:
                try:
                    t = datetime.datetime.strptime(parts[0], "%Y/%m/%d %H:%M:%S.%f").timestamp()
                except ValueError:
                    t = None
                if t is not None and not (self.window[0] <= t <= self.window[1]):
                    outside += 1
                    continue
            try:
                sm.append(float(parts[3].split()[0]))
                smax.append(float(parts[4].split()[0]))
                power.append(float(parts[5].split()[0]))
            except (ValueError, IndexError):
                continue
            for nm, v in zip(names, parts[7:11]):
                if v.lower().startswith("active"):
                    reasons.add(nm)
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(smax) if smax else None,
                "power_w_max": max(power) if power else None,
                "samples": len(sm), "samples_outside_timed_region": outside, "reasons": sorted(reasons)}


def gpu_uuid(torch):
    try:
        u = str(torch.cuda.get_device_properties(torch.cuda.current_device()).uuid)
        return u.replace("GPU-", "")
    except Exception:
        return None


# ---------------------------------------------------------------------------
# CPU oracle timing (reported baseline)
# ---------------------------------------------------------------------------
def cpu_model() -> str:
    """The host CPU's model name (lscpu, else /proc/cpuinfo)."""
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        fields = dict(ln.split(":", 1) for ln in out.splitlines() if ":" in ln)
        vendor = fields.get("Vendor ID", "").strip()
        model = fields.get("Model name", "").strip()
        if model:
            return f"{vendor} {model}".strip()
    except (OSError, subprocess.SubprocessError, ValueError):
        pass
    try:
        with open("/proc/cpuinfo") as f:
            for ln in f:
                if ln.lower().startswith(("model name", "cpu part")):
                    return ln.split(":", 1)[1].strip()
    except OSError:
        pass
    return "unknown"


def _rows_for(run, target_s, min_rows, max_rows, step=1):
    """Number of rows for which ``run(rows) -> seconds`` takes about
    ``target_s``: a warm-up run (one-time costs), then two runs of min_rows
    and 2 min_rows rows separate the fixed part of a call (e.g. writing the
    fp64 dW [V, d]) from the part per row."""
    run(min_rows)
    t1, t2 = run(min_rows), run(2 * min_rows)
    per_row = max((t2 - t1) / min_rows, 1e-6)
    fixed = max(t1 - min_rows * per_row, 0.0)
    rows = int(min(max_rows, max(min_rows, (target_s - fixed) / per_row)))
    return max(min_rows, rows // step * step)


def _time_numpy(inp, rows, Wd=None):
    import oracle
    Wd = oracle.decode_bf16(inp["W"]) if Wd is None else Wd
    Hd = oracle.decode_bf16(inp["H"][:rows])
    t0 = time.perf_counter()
    oracle.lce_f64(Hd, Wd, inp["y"][:rows])
    return time.perf_counter() - t0


def _time_c(inp, rows, nthreads):
    import oracle
    t0 = time.perf_counter()
    oracle.lce_c(inp["H"][:rows], inp["W"], inp["y"][:rows], nthreads=nthreads)
    return time.perf_counter() - t0


_ONE_CORE_NUMPY = r"""
import json, sys, time
sys.path.insert(0, sys.argv[1])
import bench
from chunked_lm_head_linear_gb300 import inputs
w = inputs.WORKLOADS[sys.argv[2]]
N = int(sys.argv[3])
inp = inputs.make_inputs(w if N == w.N else w.scaled(N=N, name=f"{w.name}_tokens{N}"))
import oracle
Wd = oracle.decode_bf16(inp["W"])
target = float(sys.argv[4])
rows = bench._rows_for(lambda r: bench._time_numpy(inp, r, Wd), target, 8, N, step=8)
t = bench._time_numpy(inp, rows, Wd)
print(json.dumps({"rows": rows, "s": t}))
"""


def _numpy_one_core(base_name, N, target_s):
    """The numpy oracle with one BLAS thread (a child process: BLAS reads its
    thread count when numpy loads)."""
    env = dict(os.environ, OPENBLAS_NUM_THREADS="1", OMP_NUM_THREADS="1", MKL_NUM_THREADS="1",
               BLIS_NUM_THREADS="1")
    try:
        out = subprocess.run([sys.executable, "-c", _ONE_CORE_NUMPY, ROOT, base_name, str(N), str(target_s)],
                             env=env, capture_output=True, text=True, timeout=600)
    except subprocess.TimeoutExpired:
        return None
    if out.returncode != 0:
        return None
    return json.loads(out.stdout.strip().splitlines()[-1])


def cpu_baseline(inp, base_name, target_s=5.0):
    """The oracle as it stands, timed on the host cores (a reported baseline,
    not the target): the numpy fp64 oracle and the plain-C fp64 oracle, each on
    all cores and on one core, over the first rows of the workload at full d
    and V (a bounded sample), plus the whole tiny workload. ``value`` is the
    numpy oracle on all cores; full-workload times are extrapolated from the
    samples at constant work per token (8 V d fp64 flop per token) and are
    labelled as extrapolations."""
    import oracle
    w = inp["workload"]
    cores = os.cpu_count() or 1
    Wd = oracle.decode_bf16(inp["W"])
    rows = _rows_for(lambda r: _time_numpy(inp, r, Wd), 2 * target_s, 32, min(4096, w.N), step=32)
    t = _time_numpy(inp, rows, Wd)
    res = {"value": rows / t, "unit": UNIT, "cores": cores, "kind": "oracle", "cpu_model": cpu_model(),
           "sample": f"first {rows} tokens of the workload at full d and V, numpy fp64 oracle "
                     f"(forward + backward), {t:.1f} s; BLAS threads = all {cores} host cores"}
    samples = {"numpy_all_cores": {"tokens_per_s": rows / t, "rows": rows, "s": t, "threads": cores}}
    one = _numpy_one_core(base_name, w.N, target_s)
    if one:
        samples["numpy_one_core"] = {"tokens_per_s": one["rows"] / one["s"], "rows": one["rows"], "s": one["s"],
                                     "threads": 1}
    oracle.build_c_oracle()
    # the plain-C oracle is slow (scalar fp64 loops, about 1 s per token on one core): a few
    # tokens per thread, one timed run each
    for label, nth in (("c_all_cores", cores), ("c_one_core", 1)):
        r = min(4 * nth, w.N)
        tc = _time_c(inp, r, nth)
        samples[label] = {"tokens_per_s": r / tc, "rows": r, "s": tc, "threads": nth}
    res["samples"] = samples
    res["full_workload_s_extrapolated"] = {k: w.N / v["tokens_per_s"] for k, v in samples.items()}
    tiny = inputs.make_inputs("tiny_n256_d256_v4096")
    tiny_s = {}
    for label, fn in (("numpy_all_cores", lambda: oracle.lce_bf16(tiny["H"], tiny["W"], tiny["y"])),
                      ("c_all_cores", lambda: oracle.lce_c(tiny["H"], tiny["W"], tiny["y"], nthreads=cores)),
                      ("c_one_core", lambda: oracle.lce_c(tiny["H"], tiny["W"], tiny["y"], nthreads=1))):
        fn()
        t0 = time.perf_counter()
        fn()
        tiny_s[label] = time.perf_counter() - t0
    res["tiny_whole_workload_s"] = tiny_s
    return res


def run_reference(args, w):
    """--impl reference: the CPU oracle, each step a bounded sample of the workload."""
    import oracle
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return
    inp = inputs.make_inputs(w)
    Hd = oracle.decode_bf16(inp["H"])
    Wd = oracle.decode_bf16(inp["W"])
    y = inp["y"]
    def timed_call(rows):
        t = time.perf_counter()
        oracle.lce_f64(Hd[:rows], Wd, y[:rows])
        return time.perf_counter() - t

    timed_call(16)                               # first call pays page faults: calibrate on warm ones
    t16, t80 = timed_call(16), timed_call(80)
    per_row = max((t80 - t16) / 64.0, 1e-6)      # each call: a fixed part (the fp64 dW) + a part per row
    fixed = max(t16 - 16 * per_row, 0.0)
    budget = 150.0 / max(1, args.steps + args.warmup)     # whole run within a few minutes
    rows = int(max(16, min(w.N, (budget - fixed) / per_row)) // 16 * 16)
    for s in range(args.warmup):
        oracle.lce_f64(Hd[:rows], Wd, y[:rows])
    t0 = time.perf_counter()
    for s in range(args.steps):
        r0 = (s * rows) % max(1, w.N - rows + 1)
        oracle.lce_f64(Hd[r0:r0 + rows], Wd, y[r0:r0 + rows])
    dt = time.perf_counter() - t0
    value = rows * args.steps / dt
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * dt / args.steps,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic", "config": config_of(w, min(args.chunk, w.N) if args.chunk > 0 else 0, args),
            "cpu_baseline": {"value": value, "unit": UNIT, "cores": os.cpu_count(), "kind": "oracle",
                             "cpu_model": cpu_model(),
                             "sample": f"{rows} tokens per step at full d and V (numpy fp64 oracle, fwd+bwd)"},
            "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def config_of(w, chunk, args):
    cfg = {"workload": w.name, "N_tokens_per_gpu": w.N, "d": w.d, "V": w.V, "chunk_tokens": chunk,
            "labels": w.labels, "ignore": w.ignore, "seed": w.seed,
            "global_batch_tokens": w.N * args.gpus, "parallelism": f"dp{args.gpus}",
            "l2": "inputs larger than L2 (W 0.62 GB, dW 1.24 GB, gradient tiles > 1 GB); no flush"}
    if getattr(args, "path", "fused") != "fused":
        cfg["path"] = args.path
        if args.path == "vshard":
            cfg["vocab_shards"] = args.shards
            cfg["vshard_method"] = args.vshard_method
            cfg["flops_executed_per_token"] = ("6*V*d (exp tile kept per chunk)" if args.vshard_method == "stored"
                                               else "8*V*d (logits recomputed in the shard backward)")
        if args.path == "norm":
            cfg["norm"] = "zero-centred RMSNorm of x [N, d] in front of the head (eps 1e-6)"
        if args.path == "split":
            cfg["flops_executed_per_token"] = "8*V*d (lce_forward, then lce_backward recomputing the logits)"
    if getattr(args, "slices", 0) > 0:
        cfg["dw_slices"] = args.slices
        cfg["sm_limit"] = args.sm_limit
        if args.gpus > 1:
            cfg["parallelism"] = f"fsdp{args.gpus} (dW reduced to vocabulary-row owners)"
            cfg["weight_gather"] = "outside the step (FSDP gathers it while the layer before computes)"
    return cfg


# ---------------------------------------------------------------------------
# GPU arm
# ---------------------------------------------------------------------------
def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--workload", default=inputs.BENCH_WORKLOAD, choices=sorted(inputs.WORKLOADS))
    ap.add_argument("--chunk", type=int, default=4096)
    ap.add_argument("--tokens", type=int, default=0,
                    help="override the workload's token count (same d, V and label law); for small profiling runs")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--slices", type=int, default=0,
                    help="finish dW in this many vocabulary slices (lce_fwd_bwd_sliced); with --gpus > 1 the "
                         "FSDP-style step: dW reduced to its row owners slice by slice on a side stream")
    ap.add_argument("--sm-limit", type=int, default=0, help="with --slices: SMs the GEMM launches may use (0 = all)")
    ap.add_argument("--path", default="fused", choices=["fused", "norm", "vshard", "split"],
                    help="fused: lce_fwd_bwd (the metric's step); norm: final RMSNorm + LM head + CE "
                         "(lce_norm_fwd_bwd, x in place of H); vshard: the vocabulary-parallel calls with "
                         "--shards shards run in turn on one GPU (partial dH summed by torch in place of the "
                         "all-reduce); split: lce_forward then lce_backward (the recompute path behind "
                         "FusedLinearCrossEntropy(recompute=True), 8*N*V*d executed)")
    ap.add_argument("--shards", type=int, default=4, help="with --path vshard: number of vocabulary shards")
    ap.add_argument("--graph", action="store_true",
                    help="also time the step captured once into a CUDA graph and replayed (one GPU; reported as "
                         "'graph' beside the eager value)")
    ap.add_argument("--vshard-method", default="stored", choices=["stored", "recompute"],
                    help="with --path vshard: the per-chunk calls keeping the exp tile (lce_vshard_chunk_*), or the "
                         "three calls that recompute the logits in the backward")
    ap.add_argument("--cublas-logits", action="store_true",
                    help="also time cuBLAS (torch.matmul, bf16 output) on one chunk's logits GEMM, C x V x d, "
                         "for comparison with the exp-tile pass; reported as cublas_logits_gemm")
    args = ap.parse_args()
    args.warmup = max(args.warmup, 3)

    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    w = inputs.WORKLOADS[args.workload]
    if args.tokens > 0:
        w = w.scaled(N=args.tokens, name=f"{w.name}_tokens{args.tokens}")
    if args.impl == "reference":
        run_reference(args, w)
        return

    import torch
    import torch.distributed as dist
    from chunked_lm_head_linear_gb300 import dp, fsdp, lce

    torch.cuda.set_device(local)
    if world > 1:
        dist.init_process_group("nccl")
    lce.load()
    dev = torch.device("cuda", local)

    # weak scaling: each rank draws its own shard (seed = rank)
    inp = inputs.make_inputs(w, seed=w.seed + rank)
    N, d, V = w.N, w.d, w.V
    H_host = torch.from_numpy(inp["H"].view(np.int16)).view(torch.bfloat16).pin_memory()
    y_host = torch.from_numpy(inp["y"]).pin_memory()
    W = torch.from_numpy(inp["W"].view(np.int16)).view(torch.bfloat16).to(dev)
    H = H_host.to(dev)
    y = y_host.to(dev)
    n_global = dp.global_valid_count(y, V=V) if world > 1 else -1

    chunk = min(args.chunk, N) if args.chunk > 0 else 0
    opts = dict(chunk_tokens=chunk, n_valid_override=n_global)
    ws = torch.empty(lce.workspace_size(lce.LCE_OP_FWD_BWD, N, d, V, lce.make_opts(**opts)), dtype=torch.uint8,
                     device=dev)
    dW = torch.empty((V, d), dtype=torch.float32, device=dev)
    lse = torch.empty(N, dtype=torch.float32, device=dev)
    stream = torch.cuda.current_stream()

    bounds = lce.slice_bounds(V, args.slices) if args.slices > 0 else None
    owners = fsdp.owner_bounds(V, world)
    slice_events = [torch.cuda.Event() for _ in range(len(bounds) - 1)] if bounds else None
    comm = torch.cuda.Stream(dev) if (bounds and world > 1) else None

    if args.path != "fused" and (world > 1 or bounds):
        raise SystemExit("--path norm / vshard run on one GPU without --slices")
    if args.path == "norm":
        w_norm = torch.from_numpy(np.random.default_rng(w.seed + 1).normal(0.0, 0.1, d).astype(np.float32)).to(dev)
        ws_norm = torch.empty(lce.workspace_size(lce.LCE_OP_NORM_FWD_BWD, N, d, V, lce.make_opts(**opts)),
                              dtype=torch.uint8, device=dev)
    shard_cuts = [V * r // args.shards // 8 * 8 for r in range(args.shards)] + [V]
    if args.path == "vshard" and args.vshard_method == "stored":
        vs_chunk = max(1, min(chunk or 4096, N))
        vs_ws = [lce.vshard_chunk_workspace(H, W[shard_cuts[r]:shard_cuts[r + 1]], y, chunk_tokens=vs_chunk)
                 for r in range(args.shards)]
        vs_dH = [torch.empty((N, d), dtype=torch.float32, device=dev) for _ in range(args.shards)]

    if args.path == "split":
        ws_f = torch.empty(lce.workspace_size(lce.LCE_OP_FORWARD, N, d, V, lce.make_opts(**opts)), dtype=torch.uint8,
                           device=dev)
        ws_b = torch.empty(lce.workspace_size(lce.LCE_OP_BACKWARD, N, d, V, lce.make_opts(**opts)),
                           dtype=torch.uint8, device=dev)

    def step(Hx, yx):
        if args.path == "split":
            loss, lse_s = lce.lce_forward(Hx, W, yx, workspace=ws_f, **opts)
            dH, _ = lce.lce_backward(Hx, W, yx, lse_s, dW=dW, workspace=ws_b, **opts)
            return loss, dH
        if args.path == "norm":
            loss, _, dx, _, _ = lce.lce_norm_fwd_bwd(Hx, w_norm, W, yx, dW=dW, workspace=ws_norm, **opts)
            return loss, dx
        if args.path == "vshard" and args.vshard_method == "stored":
            cuts = shard_cuts
            per_chunk = []
            for c0 in range(0, N, vs_chunk):
                rows = min(vs_chunk, N - c0)
                st = torch.stack([lce.lce_vshard_chunk_stats(Hx, W[cuts[r]:cuts[r + 1]], yx, cuts[r], V, c0, rows,
                                                             workspace=vs_ws[r], chunk_tokens=vs_chunk)
                                  for r in range(args.shards)])
                for r in range(args.shards):
                    lce.lce_vshard_chunk_backward(Hx, W[cuts[r]:cuts[r + 1]], yx, cuts[r], V, c0, rows, st,
                                                  workspace=vs_ws[r], lse=lse, dH_partial=vs_dH[r],
                                                  dW_shard=dW[cuts[r]:cuts[r + 1]], chunk_tokens=vs_chunk)
                per_chunk.append(st)
            loss, _ = lce.lce_vshard_combine(torch.cat(per_chunk, dim=1), yx, V)
            dH = vs_dH[0]
            for r in range(1, args.shards):
                dH.add_(vs_dH[r])
            return loss, dH
        if args.path == "vshard":
            cuts = shard_cuts
            stats = [lce.lce_vshard_forward_stats(Hx, W[cuts[r]:cuts[r + 1]], yx, cuts[r], V, chunk_tokens=chunk)
                     for r in range(args.shards)]
            loss, lse_v = lce.lce_vshard_combine(torch.stack(stats), yx, V)
            dH = None
            for r in range(args.shards):
                part, _ = lce.lce_vshard_backward(Hx, W[cuts[r]:cuts[r + 1]], yx, cuts[r], V, lse_v,
                                                  dW=dW[cuts[r]:cuts[r + 1]], chunk_tokens=chunk)
                dH = part if dH is None else dH.add_(part)
            return loss, dH
        if bounds and world > 1:
            loss, _, dH, _ = fsdp.fsdp_fwd_bwd(Hx, W, yx, owners=owners, slices=bounds, comm_stream=comm,
                                               sm_limit=args.sm_limit, dW=dW, lse=lse, workspace=ws,
                                               chunk_tokens=chunk)
        elif bounds:
            loss, _, dH, _ = lce.lce_fwd_bwd_sliced(Hx, W, yx, bounds=bounds, events=slice_events,
                                                    sm_limit=args.sm_limit, dW=dW, lse=lse, workspace=ws, **opts)
        elif world > 1:
            loss, _, dH, _ = dp.dp_fwd_bwd(Hx, W, yx, n_global=n_global, dW=dW, lse=lse, workspace=ws,
                                           chunk_tokens=chunk)
        else:
            loss, _, dH, _ = lce.lce_fwd_bwd(Hx, W, yx, dW=dW, lse=lse, workspace=ws, **opts)
        return loss, dH

    def barrier():
        if world > 1:
            dist.barrier()
        torch.cuda.synchronize()

    # ---- device-resident throughput, kernels timed by events on their stream
    for _ in range(args.warmup):
        step(H, y)
    barrier()
    clocks = ClockSampler(gpu_uuid(torch))
    clocks.start()
    time.sleep(0.3)
    lce.profile_begin()
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    barrier()
    t_start = time.time()
    ev0.record(stream)
    for _ in range(args.steps):
        step(H, y)
    ev1.record(stream)
    barrier()
    t_end = time.time()
    prof = lce.profile_end()
    time.sleep(0.2)            # the sampler's last in-region lines
    clocks.mark(t_start, t_end)
    clk = clocks.stop()
    ms = ev0.elapsed_time(ev1)
    if world > 1:
        t = torch.tensor([ms], dtype=torch.float64, device=dev)
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
        ms = float(t.item())
    ms_per_step = ms / args.steps
    value = N * world * args.steps / (ms * 1e-3)

    # ---- the same device-resident loop without the per-kernel events. The library launches its
    # kernels with programmatic stream serialization, so a kernel's launch overlaps the end of
    # the one before it; an event recorded between two kernels makes the second wait for the
    # whole of the first and takes that overlap away. This region is what the plain call does.
    # An event at each step boundary (not between kernels) also gives the median and the fastest step.
    step_ev = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps + 1)]
    barrier()
    step_ev[0].record(stream)
    for k in range(args.steps):
        step(H, y)
        step_ev[k + 1].record(stream)
    barrier()
    ms_plain = step_ev[0].elapsed_time(step_ev[-1])
    per_step = sorted(step_ev[k].elapsed_time(step_ev[k + 1]) for k in range(args.steps))
    if world > 1:
        t = torch.tensor([ms_plain], dtype=torch.float64, device=dev)
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
        ms_plain = float(t.item())
    no_events = {"value": N * world * args.steps / (ms_plain * 1e-3), "unit": UNIT,
                 "ms_per_step": ms_plain / args.steps,
                 "ms_per_step_median": per_step[len(per_step) // 2], "ms_per_step_min": per_step[0],
                 "how": "the timed loop again, device-resident inputs, without the event pair around each "
                        "kernel launch (those events serialise the kernels' programmatic launch overlap); "
                        "one event per step boundary gives the median and minimum step (this rank)"}

    # ---- end to end through the same public call, host buffers: every step's H and y are copied
    # from pinned host memory and every step's loss is read back into pinned host memory. The
    # inputs are double-buffered: step k+1's copy runs on a copy stream while step k computes (a
    # training loop's prefetch); the first copy starts after the region's start event and the
    # last step ends before its stop event, so every copy is inside the timed region.
    loss_host = torch.empty(1, dtype=torch.float32).pin_memory()
    Hb = [H, torch.empty_like(H)]
    yb = [y, torch.empty_like(y)]
    copy_stream = torch.cuda.Stream(dev)
    copied = [torch.cuda.Event(), torch.cuda.Event()]
    used = [torch.cuda.Event(), torch.cuda.Event()]

    def prefetch(b, after_use):
        with torch.cuda.stream(copy_stream):
            if after_use:
                copy_stream.wait_event(used[b])    # the step that read this buffer last is done
            Hb[b].copy_(H_host, non_blocking=True)
            yb[b].copy_(y_host, non_blocking=True)
            copied[b].record(copy_stream)

    def run_e2e(steps):
        copy_stream.wait_stream(stream)
        prefetch(0, False)
        for k in range(steps):
            b = k % 2
            stream.wait_event(copied[b])
            if k + 1 < steps:
                prefetch(1 - b, k >= 1)
            loss, _ = step(Hb[b], yb[b])
            used[b].record(stream)
            loss_host.copy_(loss, non_blocking=True)

    run_e2e(2)
    barrier()
    ev0.record(stream)
    run_e2e(args.steps)
    ev1.record(stream)
    barrier()
    ms_e2e = ev0.elapsed_time(ev1)
    if world > 1:
        t = torch.tensor([ms_e2e], dtype=torch.float64, device=dev)
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
        ms_e2e = float(t.item())
    e2e = {"value": N * world * args.steps / (ms_e2e * 1e-3), "unit": UNIT,
           "h2d_bytes_per_step": H_host.numel() * 2 + y_host.numel() * 8, "d2h_bytes_per_step": 4,
           "loss_last_step": float(loss_host.item()),
           "how": "each step's H and y copied from pinned host memory (double-buffered: the next step's "
                  "copy on a copy stream while the current step computes), each step's loss copied "
                  "back to pinned host memory; all inside the timed region"}

    # ---- the same step captured into a CUDA graph and replayed (launch cost off the host path)
    graph = None
    if args.graph and world == 1:
        side = torch.cuda.Stream(dev)
        side.wait_stream(stream)
        with torch.cuda.stream(side):
            step(H, y)
        stream.wait_stream(side)
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            step(H, y)
        for _ in range(3):
            g.replay()
        barrier()
        ev0.record(stream)
        for _ in range(args.steps):
            g.replay()
        ev1.record(stream)
        barrier()
        ms_g = ev0.elapsed_time(ev1)
        graph = {"value": N * args.steps / (ms_g * 1e-3), "unit": UNIT, "ms_per_step": ms_g / args.steps,
                 "how": "one step captured with torch.cuda.graph and replayed; device-resident inputs"}
        del g

    cublas = None
    if args.cublas_logits:
        C = chunk if chunk > 0 else N
        out = torch.empty((C, V), dtype=torch.bfloat16, device=dev)
        Hc = H[:C]
        for _ in range(3):
            torch.matmul(Hc, W.t(), out=out)
        iters = max(10, args.steps)
        barrier()
        ev0.record(stream)
        for _ in range(iters):
            torch.matmul(Hc, W.t(), out=out)
        ev1.record(stream)
        barrier()
        ms_c = ev0.elapsed_time(ev1) / iters
        lg = prof.get("logits_stats", {})
        ours = lg["ms"] / lg["launches"] if lg.get("launches") else None
        cublas = {"shape": f"{C} x {V} x {d}", "ms": ms_c, "tflops": 2.0 * C * V * d / (ms_c * 1e-3) / 1e12,
                  "exp_tile_pass_ms": ours,
                  "note": "cuBLAS writes the bf16 logits; the exp-tile pass writes bf16 exp(z - ref) and the "
                          "per-tile sums; both measured in this run, the cuBLAS loop after the fused steps"}
        del out

    if rank != 0:
        if world > 1:
            dist.destroy_process_group()
        return

    peaks, peak_src = load_peaks()
    flops_step = 6.0 * N * V * d
    tflops = flops_step * args.steps / (ms * 1e-3) / 1e12
    # The peak a kernel is held to depends on how long it runs: a timed region under
    # about a second runs at the burst clock (the board has not reached its power
    # limit yet), a longer one settles at the power-capped, sustained clock.
    region_s = ms * 1e-3
    regime = "burst" if region_s < 1.0 else "sustained"
    peak_key = "bf16_tflops" if regime == "burst" else "bf16_tflops_sustained"
    num_sms = torch.cuda.get_device_properties(dev).multi_processor_count
    # per-clock fractions need the clock the region ran at: at least three samples inside a region
    # of at least a second (in shorter regions nvidia-smi's clock and power readings lag the
    # board: power.draw averages over about a second)
    sm_mhz = clk.get("sm_mhz") if (clk.get("samples") or 0) >= 3 and region_s >= 1.0 else None
    # tensor-core limit at the clock the region ran at: SMs x 8192 dense bf16 flop per SM per clock
    per_clock_tflops = num_sms * 8192 * sm_mhz * 1e6 / 1e12 if sm_mhz else None

    def gemm_roof(kind):
        v = prof[kind]
        ms_l = v["ms"] / max(1, v["launches"])
        work_l = v["work"] / max(1, v["launches"])
        ach = work_l / (ms_l * 1e-3) / 1e12
        return {"achieved": ach, "ms_per_launch": ms_l, "work_per_launch": work_l, "launches": v["launches"],
                "frac_burst": ach / peaks["bf16_tflops"], "frac_sustained": ach / peaks["bf16_tflops_sustained"],
                "frac_per_clock": ach / per_clock_tflops if per_clock_tflops else None}

    gemm_kinds = set(lce.GEMM_KINDS)
    gemm_kernels = {k: gemm_roof(k) for k in lce.GEMM_KINDS
                    if k in prof and prof[k]["launches"] and prof[k]["ms"] > 0 and prof[k]["work"] > 0}
    # dominant kernel of the timed region
    dom = max(prof, key=lambda k: prof[k]["ms"])
    p = prof[dom]
    per_launch_ms = p["ms"] / max(1, p["launches"])
    per_launch_work = p["work"] / max(1, p["launches"])
    if dom in gemm_kinds:
        g = gemm_kernels[dom]
        peak = peaks[peak_key]
        roof = {"kernel": dom, "bound": "tensor", "achieved": g["achieved"], "peak": peak, "unit": "TFLOP/s",
                "frac": g["achieved"] / peak, "peak_source": f"{peak_key} ({peak_src}; {regime}: timed region "
                                                              f"{region_s:.2f} s)",
                "frac_burst": g["frac_burst"], "frac_sustained": g["frac_sustained"],
                "frac_per_clock": g["frac_per_clock"],
                "work_per_launch": per_launch_work,
                "work_unit": "flop (4*C*V*d: dH + dW of a chunk)" if dom == "gemm_dH_dW" else "flop (2*C*V*d)",
                "ms_per_launch": per_launch_ms}
    else:
        achieved = per_launch_work / (per_launch_ms * 1e-3) / 1e9
        peak = peaks["hbm_gbs"]
        roof = {"kernel": dom, "bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s",
                "frac": achieved / peak, "peak_source": f"hbm_gbs ({peak_src})",
                "work_per_launch": per_launch_work, "work_unit": "bytes", "ms_per_launch": per_launch_ms}
    roof["traffic"] = traffic_for(dom)
    total_ms = sum(v["ms"] for v in prof.values())
    kernels = {k: {"launches": v["launches"], "ms": round(v["ms"], 3),
                   "share": round(v["ms"] / total_ms, 4) if total_ms else 0.0}
               for k, v in prof.items() if v["launches"]}
    gpu_launches = sum(v["launches"] for k, v in prof.items() if k != "memset")  # every library kernel
    hbm_kernels = {}
    for k in lce.HBM_KINDS:
        v = prof.get(k)
        if v and v["launches"] and v["ms"] > 0:
            gbs = v["work"] / (v["ms"] * 1e-3) / 1e9
            hbm_kernels[k] = {"achieved": gbs, "peak": peaks["hbm_gbs"], "unit": "GB/s",
                              "frac": gbs / peaks["hbm_gbs"], "bytes_per_launch": v["work"] / v["launches"],
                              "ms_per_launch": v["ms"] / v["launches"]}

    line = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms_per_step, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16", "data": "synthetic", "config": config_of(w, chunk, args),
        "tflops": tflops, "pct_of_bf16_peak": tflops / peaks["bf16_tflops"],
        "pct_of_bf16_peak_sustained": tflops / peaks["bf16_tflops_sustained"],
        "pct_of_bf16_peak_per_clock": tflops / per_clock_tflops if per_clock_tflops else None,
        "peak_source": peak_src, "peak_regime": regime, "flops_per_step": flops_step,
        "roofline": roof, "gemm_kernels": gemm_kernels, "kernels": kernels, "gpu_launches": gpu_launches,
        "value_without_kernel_events": no_events, "e2e": e2e, "clocks": clk,
        **({"hbm_kernels": hbm_kernels} if hbm_kernels else {}),
        **({"cublas_logits_gemm": cublas} if cublas else {}),
        **({"graph": graph} if graph else {}),
        "extra_device_bytes": int(ws_f.numel() + ws_b.numel()) if args.path == "split" else int(ws.numel()),
        "unfused_logits_bytes": N * V * 4,
    }
    if world == 1 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(inp, args.workload)
    print(json.dumps(line), flush=True)
    if world > 1:
        dist.destroy_process_group()


def traffic_for(kernel: str):
    """DRAM bytes per launch of ``kernel`` from the committed ncu summary, if it
    was taken on the kernels as they are now (same source stamp), else None."""
    path = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(path):
        return None
    try:
        from chunked_lm_head_linear_gb300 import build
        with open(path) as f:
            d = json.load(f)
        if d.get("source_stamp") != build.source_stamp():
            return None
        return d.get("per_launch_bytes", {}).get(kernel)
    except Exception:
        return None


if __name__ == "__main__":
    main()
