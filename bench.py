"""Benchmark: exact masked attention, forward + reverse, on GB300.

One step = attn_fwd + attn_bwd (every step of the path: forward kernel,
delta, reverse kernel, dQ conversion) over one batch of the workload,
default B=4, H=32, n=4096, d=v=128, bf16, causal (the training-shaped
attention problem; inputs 4 x 134 MB, larger than the 129 MB L2, so no flush
is needed between steps).

Flop convention: forward 4 n^2 d per head (2 n^2 (d+v) when d != v), reverse
2.5x the forward, both halved under the causal mask; for window and bitmask
masks the algorithmic 2 |A| (d+v) is used instead (|A| = allowed pairs).

Prints ONE JSON line (rank 0).  ``--impl reference`` times the float64 CPU
oracle instead, on a bounded sample of the same workload.

``--decode`` times the split-KV forward instead: nq (default 1) queries at the
end of nk=16384 keys, B=8, H=32, d=v=128, bf16, causal; the metric is the
algorithmic HBM bytes (read Q, K, V, write Y, L) per second against the
measured copy bandwidth.
"""
from __future__ import annotations

import argparse
import json
import math
import os
import statistics
import subprocess
import sys
import threading
import time

import numpy as np
import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import workloads  # noqa: E402

FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            return json.load(f), "measured"
    return dict(FALLBACK_PEAKS), "fallback"


def max_over_ranks(val, dist_mod=None, device=None):
    """Largest value of a float over all ranks of the default process group
    (the value itself without one).  Times are max-reduced: the job is as
    slow as its slowest rank."""
    if dist_mod is None or not dist_mod.is_available() or not dist_mod.is_initialized():
        return float(val)
    t = torch.tensor([float(val)], dtype=torch.float64, device=device)
    dist_mod.all_reduce(t, op=dist_mod.ReduceOp.MAX)
    return float(t.item())


def whole_job_tflops(flops_per_rank_step, steps, world, ms_max):
    """Whole-job throughput: every rank processes its own batch (weak scaling),
    timed by the slowest rank."""
    return world * flops_per_rank_step * steps / (ms_max * 1e-3) / 1e12


def flops(w: workloads.Workload, allowed_pairs=None):
    """(forward, reverse) flop counts of one step of workload ``w``."""
    heads = w.B * w.H
    if w.n_keys != w.n and w.mask != "bitmask":
        f = 2.0 * w.allowed_pairs_per_head() * (w.d + w.v) * heads
    elif w.mask in ("none", "causal"):
        f = 2.0 * w.n * w.n * (w.d + w.v) * heads
        if w.mask == "causal":
            f /= 2.0
    else:
        pairs = allowed_pairs if allowed_pairs is not None else w.allowed_pairs_per_head()
        f = 2.0 * pairs * (w.d + w.v) * heads
    return f, 2.5 * f


# --------------------------------------------------------------------------- #
# Clock sampling during the timed region
# --------------------------------------------------------------------------- #

class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.lines = []

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "50"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.thread = threading.Thread(target=self._read, daemon=True)
            self.thread.start()
        except (OSError, FileNotFoundError):
            self.proc = None
        return self

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def __exit__(self, *exc):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
            self.thread.join(timeout=2)

    def summary(self):
        sm, smax, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in self.lines:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                smax = float(parts[2])
            except ValueError:
                continue
            for name, val in zip(names, parts[5:9]):
                if val.lower() == "active":
                    reasons.add(name)
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": smax, "reasons": sorted(reasons),
                "samples": len(sm)}


# --------------------------------------------------------------------------- #
# The oracle on the host cores (cpu_baseline and the reference arm)
# --------------------------------------------------------------------------- #

def oracle_sample_step(w, Q, K, V, G, rows, dropout=None, bits=None):
    """Oracle forward + reverse over the last ``rows`` query rows of head 0.
    ``dropout`` = (keep mask of those rows, keep scale) for the dropout forms;
    ``bits`` = the workload's bit rows for the bitmask mask.

    Returns the algorithmic flops of that sample (same convention as the GPU
    metric: 2 |A| (d+v) forward, 2.5x that reverse)."""
    from oracle import dense, masks
    n = w.n
    r0 = n - rows
    if w.n_keys != w.n:  # the last rows of a cross-attention problem are one too
        dense.forward_rect(Q[None, None, r0:], K[None, None], V[None, None], w.scale,
                           w.mask_kind, w.window)
        dense.backward_rect(Q[None, None, r0:], K[None, None], V[None, None],
                            G[None, None, r0:], w.scale, w.mask_kind, w.window)
        off = w.n_keys - n
        pairs = sum(max(0, min(w.n_keys, i + off + 1)) if w.mask == "causal" else w.n_keys
                    for i in range(r0, n))
        return 3.5 * 2.0 * pairs * (w.d + w.v)
    allowed = masks.allowed_matrix(n, w.mask_kind, w.window, bits)[r0:]
    if dropout is None:
        dense.head_forward(Q[r0:], K, V, w.scale, allowed)
        dense.head_backward(Q[r0:], K, V, G[r0:], w.scale, allowed)
    else:
        keep, ks = dropout
        dense.head_forward_dropout(Q[r0:], K, V, w.scale, allowed, keep, ks)
        dense.head_backward_dropout(Q[r0:], K, V, G[r0:], w.scale, allowed, keep, ks)
    f = 2.0 * float(allowed.sum()) * (w.d + w.v)
    return 3.5 * f


def oracle_inputs(w, x):
    return tuple(t[0, 0].to(torch.float64).numpy() for t in (x.Q, x.K, x.V, x.dY))


def oracle_dropout(w, rows, q, seed):
    """Keep mask of the last ``rows`` rows of head 0, and the keep scale."""
    if not q:
        return None
    from oracle import philox
    keep = philox.keep_mask(0, w.n, w.n, q, seed)[w.n - rows:]
    return keep, philox.keep_scale(q)


_BLAS_ENV = ("OPENBLAS_NUM_THREADS", "OMP_NUM_THREADS", "MKL_NUM_THREADS")


def _oracle_worker(w, arrays, bits, rows, drop, budget_s, barrier, out):
    """One process of the CPU baseline: the oracle sample on one BLAS thread,
    started with the others at the barrier, for ``budget_s`` seconds.  A failure
    is reported on the queue (and breaks the barrier) instead of hanging it."""
    try:
        Q, K, V, G = arrays
        oracle_sample_step(w, Q, K, V, G, min(rows, 32),
                           drop and (drop[0][-32:], drop[1]), bits)  # warm-up
        barrier.wait()
        done, samples, t0 = 0.0, 0, time.perf_counter()
        while True:
            done += oracle_sample_step(w, Q, K, V, G, rows, drop, bits)
            samples += 1
            if time.perf_counter() - t0 >= budget_s:
                break
        out.put((done, samples, time.perf_counter() - t0))
    except BaseException as e:  # noqa: BLE001 -- reported to the parent
        barrier.abort()
        out.put(("error", repr(e)))


def cpu_baseline(w, x, budget_s=12.0, rows=512, q=0.0, seed=0):
    """The oracle as it stands, timed on the host cores: one process per core in
    os.sched_getaffinity (spawned, each with one BLAS thread), all running the
    same bounded sample (forward and reverse pass of the last ``rows`` query
    rows of head 0) for ``budget_s`` seconds after a common start."""
    import multiprocessing as mp
    Q, K, V, G = oracle_inputs(w, x)
    rows = min(rows, w.n)
    drop = oracle_dropout(w, rows, q, seed)
    procs_n = max(1, host_cores())
    ctx = mp.get_context("spawn")
    saved = {k: os.environ.get(k) for k in _BLAS_ENV}
    for k in _BLAS_ENV:
        os.environ[k] = "1"
    try:
        barrier, out = ctx.Barrier(procs_n), ctx.Queue()
        procs = [ctx.Process(target=_oracle_worker,
                             args=(w, (Q, K, V, G), x.bitmask, rows, drop, budget_s, barrier,
                                   out))
                 for _ in range(procs_n)]
        for pr in procs:
            pr.start()
        res = []
        for _ in procs:
            r = out.get(timeout=budget_s + 300)
            if r[0] == "error":
                for pr in procs:
                    pr.terminate()
                raise RuntimeError(f"CPU baseline worker failed: {r[1]}")
            res.append(r)
        for pr in procs:
            pr.join()
    finally:
        for k, v in saved.items():
            if v is None:
                os.environ.pop(k, None)
            else:
                os.environ[k] = v
    flops = sum(r[0] for r in res)
    samples = sum(r[1] for r in res)
    el = max(r[2] for r in res)
    return {"value": flops / el / 1e12, "unit": "TFLOP/s", "cores": procs_n,
            "processes": procs_n, "blas_threads_per_process": 1, "kind": "oracle",
            "sample": f"{samples} x (fwd+bwd of the last {rows} query rows of head 0, float64 "
                      f"dense NumPy) over {procs_n} processes, {el:.1f} s"}


def host_cores():
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:
        return os.cpu_count()


def run_reference(args, w):
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return
    x = workloads.make_inputs(w, heads=1)
    Q, K, V, G = oracle_inputs(w, x)
    rows = min(args.ref_rows, w.n)
    drop = oracle_dropout(w, rows, args.dropout, args.seed)
    for _ in range(args.warmup):
        oracle_sample_step(w, Q, K, V, G, rows, drop, x.bitmask)
    t0 = time.perf_counter()
    total = 0.0
    for _ in range(args.steps):
        total += oracle_sample_step(w, Q, K, V, G, rows, drop, x.bitmask)
    el = time.perf_counter() - t0
    value = total / el / 1e12
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "TFLOP/s",
        "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": el / args.steps * 1e3, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": w.name, "B": w.B, "H": w.H, "n": w.n, "d": w.d, "v": w.v,
                   "mask": w.mask, "input_dtype": w.dtype, "dropout_p": args.dropout,
                   "step": f"oracle fwd+bwd of the last {rows} query rows of head 0"},
        "cpu_baseline": {"value": value, "unit": "TFLOP/s", "cores": host_cores(),
                         "kind": "oracle",
                         "sample": f"{args.steps} x fwd+bwd of the last {rows} query rows of "
                                   f"head 0 (float64 dense NumPy)"},
        "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


# --------------------------------------------------------------------------- #
# The GPU arm
# --------------------------------------------------------------------------- #

METRIC = "attention TFLOP/s fwd+bwd (fwd alone in fwd_tflops) at 1 GB300; % of dense BF16 peak"


def read_traffic(kernel_tag, workload):
    """DRAM bytes per launch from the committed ncu summary, if it was taken for
    this workload's launch and still matches the current kernel source (null
    otherwise)."""
    import hashlib
    path = os.path.join(ROOT, "profiles", "ncu_traffic.txt")
    if not os.path.exists(path):
        return None
    entries = {}
    with open(path) as f:
        lines = f.read().splitlines()
    for line in lines:
        line = line.strip()
        if not line or line.startswith("#"):
            continue
        kv = dict(p.split("=", 1) for p in line.split() if "=" in p)
        entries[kv.get("kernel")] = kv
    e = entries.get(kernel_tag)
    if e is None or e.get("launch") != workload:
        return None
    src = os.path.join(ROOT, "exact_tiled_softmax_gb300", "csrc", e.get("source", ""))
    if not os.path.exists(src):
        return None
    with open(src, "rb") as f:
        sha = hashlib.sha256(f.read()).hexdigest()[:16]
    if sha != e.get("source_sha"):
        return None
    return float(e["bytes_per_launch"])


# Peaks beyond the measured bf16 figure (derived, stated in the roofline):
# tf32 dense = measured bf16 burst x 1.1 / 2.25 (nominal per-GPU ratio); fp32
# FMA = 152 SMs x 128 lanes x 2 flop x the maximum SM clock.
TF32_OVER_BF16 = 1.1 / 2.25


def kernel_roofline(args, w, which, achieved, peaks, peak_kind):
    """Roofline object for the forward ("fwd") or reverse ("bwd") kernel(s)."""
    eligible = args.path != "simt" and w.d == w.v and w.d in (64, 128)
    # bf16 widths up to 128 in steps of 8 run on the tensor-core kernels of width 64
    # or 128 (zero-padded); the atomic reverse form takes only d = v in {64, 128}.
    padded = not eligible
    tc_bf16 = (args.path != "simt" and w.d % 8 == 0 and w.v % 8 == 0 and w.d <= 128
               and w.v <= 128 and not (which == "bwd" and args.path == "atomic_dq" and padded))
    bf16_peak = float(peaks["bf16_tflops"])
    if w.dtype == "bf16" and tc_bf16:
        tag = f"tc_{which}"
        if which == "bwd":
            tag += "_atomic" if args.path == "atomic_dq" else "_split"
        out = {"kernel": tag, "bound": "tensor", "achieved": achieved, "peak": bf16_peak,
               "unit": "TFLOP/s", "frac": achieved / bf16_peak,
               "peak_kind": f"bf16 dense burst, of {peak_kind}",
               "traffic": None if padded else read_traffic(tag, w.name)}
        if padded:
            out["padded_to"] = 64 if w.d <= 64 and w.v <= 64 else 128
        return out
    if w.dtype == "f32" and eligible and which == "fwd" and not args.dropout:
        peak = bf16_peak * TF32_OVER_BF16
        return {"kernel": "tc32_fwd", "bound": "tensor", "achieved": achieved, "peak": peak,
                "unit": "TFLOP/s", "frac": achieved / peak,
                "peak_kind": f"tf32 dense = bf16 burst of {peak_kind} x 1.1/2.25 (nominal ratio)",
                "tensor_work_frac": 3 * achieved / peak,
                "note": "3xTF32: the tensor pipe runs three tf32 products per product",
                "traffic": read_traffic("tc32_fwd", w.name)}
    if (w.dtype == "f32" and which == "bwd" and args.path == "auto" and not args.dropout
            and w.d == 64 and w.v == 64):
        peak = bf16_peak * TF32_OVER_BF16
        return {"kernel": "tc32_bwd", "bound": "tensor", "achieved": achieved, "peak": peak,
                "unit": "TFLOP/s", "frac": achieved / peak,
                "peak_kind": f"tf32 dense = bf16 burst of {peak_kind} x 1.1/2.25 (nominal ratio)",
                "tensor_work_frac": 21 / 5 * achieved / peak,
                "note": "3xTF32 reverse: 7 products per tile (S, dP twice; dV, dK, dQ), "
                        "three tf32 products each, against the convention's 5",
                "traffic": read_traffic("tc32_bwd", w.name)}
    mhz = float(peaks.get("sm_max_mhz", 2070.0))
    peak = 152 * 128 * 2 * mhz * 1e6 / 1e12
    return {"kernel": f"simt_{which}", "bound": "alu", "achieved": achieved, "peak": peak,
            "unit": "TFLOP/s", "frac": achieved / peak,
            "peak_kind": f"fp32 FMA: 152 SMs x 128 lanes x 2 flop x {mhz:.0f} MHz",
            "traffic": read_traffic(f"simt_{which}", w.name)}


def host_link(stream, h_in, d_in, h_out, d_out, reps=5):
    """The host link as the end-to-end step sees it, after its timed region: the
    step's own input copies alone, its result copies alone, and both at once on
    two streams, with the lower bound they put on a step that moves those bytes.
    Each figure is the best of `reps` timed runs: the link is shared with other
    work on the machine, and a run that met such traffic says nothing about the
    link itself."""
    side = torch.cuda.Stream()
    bi = sum(t.numel() * t.element_size() for t in h_in)
    bo = sum(t.numel() * t.element_size() for t in h_out)

    def copy_in(s):
        with torch.cuda.stream(s):
            for dst, src in zip(d_in, h_in):
                dst.copy_(src, non_blocking=True)

    def copy_out(s):
        with torch.cuda.stream(s):
            for dst, src in zip(h_out, d_out):
                dst.copy_(src, non_blocking=True)

    def both(_s):
        copy_in(stream)
        copy_out(side)

    def ms(fn):
        fn(stream)
        torch.cuda.synchronize()
        best = float("inf")
        for _ in range(reps):
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record(stream)
            side.wait_event(a)
            fn(stream)
            side_done = torch.cuda.Event()
            side_done.record(side)
            stream.wait_event(side_done)
            b.record(stream)
            torch.cuda.synchronize()
            best = min(best, a.elapsed_time(b))
        return best

    t_in, t_out, t_both = ms(copy_in), ms(copy_out), ms(both)
    return {"h2d_gbs": bi / t_in / 1e6, "d2h_gbs": bo / t_out / 1e6,
            "duplex_gbs": (bi + bo) / t_both / 1e6,
            "copy_bound_ms": max(t_in, t_out, t_both)}


def run_gpu(args, w):
    import exact_tiled_softmax_gb300 as ex
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    dist = None
    if world > 1:
        import torch.distributed as dist
        torch.cuda.set_device(local)
        dist.init_process_group("nccl")
    dev = torch.device(f"cuda:{local}")
    torch.cuda.set_device(dev)
    if args.path != "auto":
        ex.set_path(args.path)

    x = workloads.make_inputs(w)
    q, k, v, dy = (t.to(dev) for t in (x.Q, x.K, x.V, x.dY))
    bm = None if x.bitmask is None else torch.from_numpy(x.bitmask.view(np.int32)).to(dev)
    if w.n_keys != w.n:
        import ctypes
        shape = ex.QKShape(w.B, w.H, w.n, w.n_keys, w.d, w.v, 0 if w.dtype == "f32" else 1)
        lib = ex.load_library()
        ws_f = ex.workspace(lib.exattn_fwd_qk_workspace_size(ctypes.byref(shape),
                                                             w.mask_kind), dev)
        ws_b = ex.workspace(lib.exattn_bwd_qk_workspace_size(ctypes.byref(shape),
                                                             w.mask_kind), dev)
    else:
        shape = ex.Shape(w.B, w.H, w.n, w.d, w.v, 0 if w.dtype == "f32" else 1)
        ws_f = ex.workspace(ex.fwd_workspace_size(shape, w.mask), dev)
        ws_b = ex.workspace(ex.bwd_workspace_size(shape, w.mask), dev)
    y = torch.empty(q.shape[:-1] + (w.v,), dtype=q.dtype, device=dev)
    L = torch.empty(q.shape[:-1], dtype=torch.float32, device=dev)
    dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
    stream = torch.cuda.current_stream(dev)

    drop = dict(dropout_p=args.dropout, seed=args.seed)

    def step():
        ex.fwd(q, k, v, w.scale, w.mask, w.window, bm, y=y, L=L, ws=ws_f, stream=stream, **drop)
        ex.bwd(q, k, v, y, dy, L, w.scale, w.mask, w.window, bm, dq=dq, dk=dk, dv=dv, ws=ws_b,
               stream=stream, **drop)

    def fwd_only():
        ex.fwd(q, k, v, w.scale, w.mask, w.window, bm, y=y, L=L, ws=ws_f, stream=stream, **drop)

    def barrier():
        if dist is not None:
            dist.barrier()
        torch.cuda.synchronize(dev)

    def rank_max(val):
        return max_over_ranks(val, dist, dev)

    pairs = None
    if w.mask == "bitmask":
        from_words = np.unpackbits(x.bitmask.view(np.uint8)).sum()
        pairs = int(from_words)
    f_fwd, f_bwd = flops(w, pairs)

    clocks = ClockSampler(dev.index)
    clocks.__enter__()  # sampled from the warm-up through the end-to-end runs
    for _ in range(args.warmup):
        step()
    barrier()

    # Timed region: K full steps; the forward and reverse kernels of every step
    # are also bracketed by events recorded on this stream by the library.
    K = args.steps
    # The split tensor-core reverse pass (bf16, d = v in {64, 128}) also brackets
    # its dQ kernel, so the dK/dV kernel's time is the difference; its dQ kernel
    # forms delta itself (no delta launch).
    split_bwd = (w.dtype == "bf16" and w.d % 8 == 0 and w.v % 8 == 0 and w.d <= 128
                 and w.v <= 128 and args.path == "auto"
                 and (w.mask != "bitmask" or max(w.n, w.n_keys) <= 256 * 128))
    roles = ((ex.KERNEL_FWD, ex.KERNEL_BWD, ex.KERNEL_BWD_Q) if split_bwd
             else (ex.KERNEL_FWD, ex.KERNEL_BWD, ex.KERNEL_DELTA))
    ev = {role: [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
                 for _ in range(K)] for role in roles}
    for pairs_ in ev.values():
        for a, b in pairs_:
            a.record(stream)
            b.record(stream)
    barrier()
    launches0 = ex.launch_count()
    start, stop = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    barrier()
    start.record(stream)
    for i in range(K):
        for role in ev:
            ex.record_kernel_events(role, *ev[role][i])
        step()
    stop.record(stream)
    barrier()
    launches = ex.launch_count() - launches0
    ms = rank_max(start.elapsed_time(stop))
    kern_ms = {role: sum(a.elapsed_time(b) for a, b in ev[role]) / K for role in ev}
    delta_ms = kern_ms.pop(ex.KERNEL_DELTA, None)
    bwd_q_ms = kern_ms.pop(ex.KERNEL_BWD_Q, None)

    # Forward alone.
    for _ in range(args.warmup):
        fwd_only()
    barrier()
    s2, e2 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    s2.record(stream)
    for _ in range(K):
        fwd_only()
    e2.record(stream)
    barrier()
    ms_fwd = rank_max(s2.elapsed_time(e2))

    # End to end through the public API: pinned host inputs in, results out.
    e2e = None
    if not args.no_e2e:
        pin = [t.pin_memory() for t in (x.Q, x.K, x.V, x.dY)]
        outs = [torch.empty(t.shape, dtype=t.dtype, pin_memory=True) for t in (y, L, dq, dk, dv)]
        h2d = sum(t.numel() * t.element_size() for t in pin)
        d2h = sum(t.numel() * t.element_size() for t in outs)

        # attn_step_host: the C-ABI call on host buffers, which overlaps the copies
        # of neighbouring chunks of slices with the kernels.  Dropout and nq != nk
        # shapes copy around the device calls instead.
        host_step = not args.dropout and w.n_keys == w.n
        if host_step:
            import ctypes
            lib = ex.load_library()
            ws_h = ex.workspace(lib.exattn_host_step_workspace_size(
                ctypes.byref(ex._shape(q, v)), ex._mask_kind(w.mask)), dev)
            bm_h = None if x.bitmask is None else torch.from_numpy(x.bitmask.view(np.int32))

            def e2e_step():
                ex.step_host(*pin, w.scale, w.mask, w.window, bm_h, out=outs, ws=ws_h,
                             stream=stream, device=dev)
        else:
            def e2e_step():
                for dst, src in zip((q, k, v, dy), pin):
                    dst.copy_(src, non_blocking=True)
                step()
                for dst, src in zip(outs, (y, L, dq, dk, dv)):
                    dst.copy_(src, non_blocking=True)

        for _ in range(max(1, args.warmup)):
            e2e_step()
        barrier()
        # One event per step boundary on the call's stream (the call joins its
        # internal streams back to it), so the spread of the steps shows too.
        marks = [torch.cuda.Event(enable_timing=True) for _ in range(K + 1)]
        marks[0].record(stream)
        for j in range(K):
            e2e_step()
            marks[j + 1].record(stream)
        barrier()
        ms_e2e = rank_max(marks[0].elapsed_time(marks[K]))
        steps_ms = sorted(marks[j].elapsed_time(marks[j + 1]) for j in range(K))
        e2e = {"value": whole_job_tflops(f_fwd + f_bwd, K, world, ms_e2e), "unit": "TFLOP/s",
               "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
               "ms_per_step": ms_e2e / K,
               "call": "attn_step_host" if host_step else "copies + attn_fwd + attn_bwd",
               "step_ms": {"min": steps_ms[0], "median": steps_ms[K // 2], "max": steps_ms[-1]},
               "link": host_link(stream, pin, (q, k, v, dy), outs, (y, L, dq, dk, dv))}

    clocks.__exit__(None, None, None)
    peaks, peak_kind = load_peaks()
    peak = float(peaks["bf16_tflops"])
    tflops = whole_job_tflops(f_fwd + f_bwd, K, world, ms)
    tflops_fwd = whole_job_tflops(f_fwd, K, world, ms_fwd)
    # Dominant kernel by measured time.
    dom = max(kern_ms, key=kern_ms.get)
    dom_flops = f_fwd if dom == ex.KERNEL_FWD else f_bwd
    dom_name = "fwd" if dom == ex.KERNEL_FWD else "bwd"
    achieved = dom_flops / (kern_ms[dom] * 1e-3) / 1e12
    roofline = kernel_roofline(args, w, dom_name, achieved, peaks, peak_kind)
    roofline["kernel_ms"] = {"fwd": kern_ms[ex.KERNEL_FWD], "bwd": kern_ms[ex.KERNEL_BWD]}
    if bwd_q_ms is not None:
        roofline["kernel_ms"]["bwd_kv"] = kern_ms[ex.KERNEL_BWD] - bwd_q_ms
        roofline["kernel_ms"]["bwd_q"] = bwd_q_ms
    roofline_fwd = kernel_roofline(args, w, "fwd", f_fwd / (kern_ms[ex.KERNEL_FWD] * 1e-3) / 1e12,
                                   peaks, peak_kind)
    # delta_i = dY_i . Y_i: reads Y and dY, writes delta and L log2(e) (both padded to 128 rows).
    e = 4 if w.dtype == "f32" else 2
    npad = (w.n + 127) // 128 * 128
    delta_bytes = w.B * w.H * (2 * w.n * w.v * e + 4 * w.n + 8 * npad)
    hbm = float(peaks["hbm_gbs"])
    if delta_ms is None:
        roofline_delta = {"kernel": "delta", "fused_into": "tc_bwd_q_kernel", "bytes": delta_bytes}
    else:
        roofline_delta = {"kernel": "delta", "bound": "hbm",
                          "achieved": delta_bytes / (delta_ms * 1e-3) / 1e9, "peak": hbm,
                          "unit": "GB/s", "frac": delta_bytes / (delta_ms * 1e-3) / 1e9 / hbm,
                          "peak_kind": f"copy bandwidth, of {peak_kind}", "bytes": delta_bytes,
                          "ms": delta_ms}
    line = {
        "metric": METRIC, "value": tflops, "unit": "TFLOP/s", "n_gpus": world,
        "steps": K, "warmup": args.warmup, "ms_per_step": ms / K, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": w.dtype, "data": "synthetic",
        "config": {"workload": w.name, "B": w.B, "H": w.H, "n": w.n, "nk": w.n_keys, "d": w.d,
                   "v": w.v, "mask": w.mask, "window": w.window, "scale": w.scale,
                   "kernel_path": args.path, "dropout_p": args.dropout,
                   "l2": ("inputs larger than L2 (%d MB of Q, K, V, dY vs 129 MB), no flush"
                          % (sum(t.numel() * t.element_size() for t in (q, k, v, dy)) >> 20)),
                   "flops_per_step": f_fwd + f_bwd},
        "fwd_tflops": tflops_fwd, "fwd_frac_of_peak": tflops_fwd / peak,
        "fwd_bwd_frac_of_peak": tflops / peak, "ms_fwd": ms_fwd / K,
        "gpu_launches": launches,
        "roofline": roofline,
        "roofline_fwd": roofline_fwd,
        "roofline_delta": roofline_delta,
        "e2e": e2e,
        "clocks": clocks.summary(),
    }
    if rank == 0 and not args.no_cpu:
        line["cpu_baseline"] = cpu_baseline(w, x, budget_s=args.cpu_budget, q=args.dropout,
                                            seed=args.seed)
    if rank == 0:
        print(json.dumps(line), flush=True)
    if dist is not None:
        dist.barrier()
        dist.destroy_process_group()


# --------------------------------------------------------------------------- #
# Decode mode: the split-KV forward (a few queries against a long key sequence)
# --------------------------------------------------------------------------- #

DECODE_METRIC = ("decode attention HBM GB/s (split-KV forward + star merge) at 1 GB300; "
                 "% of measured copy bandwidth")


def decode_inputs(w, heads=None):
    B, H = (w.B, w.H) if heads is None else (1, heads)
    return workloads.make_decode_inputs(B, H, w.nq, w.nk, w.d, w.v, w.dtype, w.mask,
                                        seed=w.seed)


def oracle_decode_sample(w, Q, K, V):
    """Oracle forward of every query of one (batch, head) slice; returns the
    algorithmic bytes of that slice (same convention as the GPU metric)."""
    from oracle import dense
    dense.forward_rect(Q, K, V, w.scale, workloads.MASK_KINDS[w.mask], w.window)
    return w.bytes_moved() / (w.B * w.H)


def decode_cpu_run(w, steps=None, budget_s=12.0, warmup=0):
    """Oracle over single slices (drawn once, float64): a bounded sample."""
    Q, K, V, _ = decode_inputs(w, heads=1)
    Q, K, V = (t.to(torch.float64).numpy() for t in (Q, K, V))
    for _ in range(warmup):
        oracle_decode_sample(w, Q, K, V)
    t0, done, n = time.perf_counter(), 0.0, 0
    while True:
        done += oracle_decode_sample(w, Q, K, V)
        n += 1
        el = time.perf_counter() - t0
        if (steps is not None and n >= steps) or (steps is None and el >= budget_s):
            break
    return done / el / 1e9, n, el


def run_reference_decode(args, w):
    if int(os.environ.get("RANK", "0")) != 0:
        return
    value, n, el = decode_cpu_run(w, steps=args.steps, warmup=args.warmup)
    sample = f"{n} x (all {w.nq} queries of one batch*head slice, nk={w.nk}, float64 NumPy)"
    line = {
        "impl": "reference", "metric": DECODE_METRIC, "value": value, "unit": "GB/s",
        "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": el / n * 1e3, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": w.name, "step": "oracle forward of one batch*head slice"},
        "cpu_baseline": {"value": value, "unit": "GB/s", "cores": host_cores(), "kind": "oracle",
                         "sample": sample},
        "e2e": {"value": value, "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def decode_kernels(w):
    """The split-KV kernels the library runs for a decode workload (kernel path
    "auto", positive scale): bf16 with d = v in {64, 128} and nq >= 2 takes the
    tensor-core chunks and a merge launch ("tc"); otherwise nq <= 4 takes the
    register kernel, which merges in its last CTA per slice ("reg"), and larger nq
    the shared-memory chunk kernel and a merge launch ("smem")."""
    if w.dtype == "bf16" and w.d == w.v and w.d in (64, 128) and w.nq > 1:
        return "tc"
    return "reg" if w.nq <= 4 else "smem"


def run_gpu_decode(args, w):
    import exact_tiled_softmax_gb300 as ex
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    dist = None
    if world > 1:
        import torch.distributed as dist
        torch.cuda.set_device(local)
        dist.init_process_group("nccl")
    dev = torch.device(f"cuda:{local}")
    torch.cuda.set_device(dev)
    Qh, Kh, Vh, _ = decode_inputs(w)
    q, k, v = (t.to(dev) for t in (Qh, Kh, Vh))
    stream = torch.cuda.current_stream(dev)
    y = torch.empty((w.B, w.H, w.nq, w.v), dtype=q.dtype, device=dev)
    L = torch.empty((w.B, w.H, w.nq), dtype=torch.float32, device=dev)
    shape = ex.QKShape(w.B, w.H, w.nq, w.nk, w.d, w.v, 0 if w.dtype == "f32" else 1)
    ws = ex.workspace(ex.load_library().exattn_splitkv_workspace_size(
        __import__("ctypes").byref(shape), args.splits), dev)

    def step():
        ex.fwd_splitkv(q, k, v, w.scale, w.mask, w.window, None, num_splits=args.splits, y=y,
                       L=L, ws=ws, stream=stream)

    def barrier():
        if dist is not None:
            dist.barrier()
        torch.cuda.synchronize(dev)

    clocks = ClockSampler(dev.index)
    clocks.__enter__()
    for _ in range(args.warmup):
        step()
    barrier()
    K = args.steps
    kind = decode_kernels(w)
    fused = kind == "reg"  # the register kernel merges in its last CTA per slice
    roles = (ex.KERNEL_SPLIT_PARTIAL,) if fused else (ex.KERNEL_SPLIT_PARTIAL,
                                                     ex.KERNEL_SPLIT_MERGE)
    ev = {r: [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
              for _ in range(K)] for r in roles}
    for pairs_ in ev.values():
        for a, b in pairs_:
            a.record(stream)
            b.record(stream)
    barrier()
    launches0 = ex.launch_count()
    start, stop = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    start.record(stream)
    for i in range(K):
        for r in roles:
            ex.record_kernel_events(r, *ev[r][i])
        step()
    stop.record(stream)
    barrier()
    launches = ex.launch_count() - launches0
    ms = max_over_ranks(start.elapsed_time(stop), dist, dev)
    kern_ms = {r: sum(a.elapsed_time(b) for a, b in ev[r]) / K for r in roles}
    total_bytes = w.bytes_moved()
    value = total_bytes * world * K / (ms * 1e-3) / 1e9

    e2e = None
    if not args.no_e2e:
        pin = [t.pin_memory() for t in (Qh, Kh, Vh)]
        outs = [torch.empty(t.shape, dtype=t.dtype, pin_memory=True) for t in (y, L)]
        h2d = sum(t.numel() * t.element_size() for t in pin)
        d2h = sum(t.numel() * t.element_size() for t in outs)

        def e2e_step():
            for dst, src in zip((q, k, v), pin):
                dst.copy_(src, non_blocking=True)
            step()
            for dst, src in zip(outs, (y, L)):
                dst.copy_(src, non_blocking=True)

        for _ in range(max(1, args.warmup)):
            e2e_step()
        barrier()
        s3, e3 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        s3.record(stream)
        for _ in range(K):
            e2e_step()
        e3.record(stream)
        barrier()
        ms_e2e = max_over_ranks(s3.elapsed_time(e3), dist, dev)
        e2e = {"value": total_bytes * world * K / (ms_e2e * 1e-3) / 1e9, "unit": "GB/s",
               "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "ms_per_step": ms_e2e / K}
    clocks.__exit__(None, None, None)

    peaks, peak_kind = load_peaks()
    peak = float(peaks["hbm_gbs"])
    e = 4 if w.dtype == "f32" else 2
    partial_bytes = w.B * w.H * (w.nq * w.d * e + w.nk * (w.d + w.v) * e)
    achieved = partial_bytes / (kern_ms[ex.KERNEL_SPLIT_PARTIAL] * 1e-3) / 1e9
    roofline = {"kernel": f"splitkv_partial_{kind}", "bound": "hbm", "achieved": achieved,
                "peak": peak, "unit": "GB/s", "frac": achieved / peak,
                "peak_kind": f"copy bandwidth, of {peak_kind}",
                "traffic": read_traffic(f"splitkv_partial_{kind}", w.name),
                "kernel_ms": {"partial": kern_ms[ex.KERNEL_SPLIT_PARTIAL],
                              "merge": "in the chunk kernel" if fused
                              else kern_ms[ex.KERNEL_SPLIT_MERGE]}}
    line = {
        "metric": DECODE_METRIC, "value": value, "unit": "GB/s", "n_gpus": world, "steps": K,
        "warmup": args.warmup, "ms_per_step": ms / K, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": w.dtype, "data": "synthetic",
        "config": {"workload": w.name, "B": w.B, "H": w.H, "nq": w.nq, "nk": w.nk, "d": w.d,
                   "v": w.v, "mask": w.mask, "num_splits": args.splits,
                   "bytes_per_step": total_bytes,
                   "l2": "inputs larger than L2 (%d MB of K and V vs 129 MB), no flush"
                         % ((k.numel() * k.element_size() + v.numel() * v.element_size()) >> 20)},
        "frac_of_hbm": value / peak,
        "gpu_launches": launches,
        "roofline": roofline,
        "e2e": e2e,
        "clocks": clocks.summary(),
    }
    if rank == 0 and not args.no_cpu:
        cv, n, el = decode_cpu_run(w, budget_s=args.cpu_budget)
        line["cpu_baseline"] = {"value": cv, "unit": "GB/s", "cores": host_cores(),
                                "kind": "oracle",
                                "sample": f"{n} x (all {w.nq} queries of one batch*head slice, "
                                          f"nk={w.nk}, float64 NumPy), {el:.1f} s"}
    if rank == 0:
        print(json.dumps(line), flush=True)
    if dist is not None:
        dist.barrier()
        dist.destroy_process_group()


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", type=int, default=3)
    ap.add_argument("--variant", default="")
    ap.add_argument("--path", choices=["auto", "simt", "atomic_dq"], default="auto")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu", action="store_true")
    ap.add_argument("--cpu-budget", type=float, default=12.0)
    ap.add_argument("--ref-rows", type=int, default=256)
    ap.add_argument("--batch", type=int, default=None,
                    help="override the batch size (a smaller case of the same workload)")
    ap.add_argument("--heads", type=int, default=None, help="override the head count")
    ap.add_argument("--dtype", choices=["bf16", "f32"], default=None,
                    help="override the workload's input dtype")
    ap.add_argument("--nk", type=int, default=0,
                    help="keys per slice (cross-attention: the n queries sit at the end)")
    ap.add_argument("--dropout", type=float, default=0.0,
                    help="drop probability (dropout with a replayed mask), default none")
    ap.add_argument("--seed", type=int, default=1234, help="dropout seed")
    ap.add_argument("--decode", action="store_true",
                    help="time the split-KV decode forward instead (B=8, H=32, nk=16384)")
    ap.add_argument("--nq", type=int, default=1, help="queries per slice in --decode mode")
    ap.add_argument("--splits", type=int, default=0,
                    help="key chunks in --decode mode (0: the library chooses)")
    args = ap.parse_args()
    if args.warmup < 3:
        args.warmup = 3
    if args.decode:
        dw = workloads.decode_workload(args.nq)
        if args.batch is not None or args.heads is not None:
            import dataclasses
            B = args.batch if args.batch is not None else dw.B
            H = args.heads if args.heads is not None else dw.H
            dw = dataclasses.replace(dw, B=B, H=H, name=f"{dw.name}-as-b{B}h{H}")
        (run_reference_decode if args.impl == "reference" else run_gpu_decode)(args, dw)
        return
    w = workloads.workload(args.workload, args.variant)
    if args.dtype and args.dtype != w.dtype:
        import dataclasses
        w = dataclasses.replace(w, dtype=args.dtype, name=f"{w.name}-as-{args.dtype}")
    if args.nk and args.nk != w.n:
        import dataclasses
        w = dataclasses.replace(w, nk=args.nk, name=f"{w.name}-nk{args.nk}")
    if args.batch is not None or args.heads is not None:
        import dataclasses
        B = args.batch if args.batch is not None else w.B
        H = args.heads if args.heads is not None else w.H
        w = dataclasses.replace(w, B=B, H=H, name=f"{w.name}-as-b{B}h{H}")
    if args.impl == "reference":
        run_reference(args, w)
    else:
        run_gpu(args, w)


if __name__ == "__main__":
    main()
