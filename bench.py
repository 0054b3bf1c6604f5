"""Throughput of diffuser_forward: edge-hops per second on one GB300.

A step is one whole forward (scores + masked softmax + K diffusion hops +
output) of the configured workload, inputs resident in HBM.  Default
workload: batch 2, 12 heads, n = 4096, d = 64, bf16 I/O, window radius 256,
16 globals, 32 random edges per row, K = 5, alpha = 0.1.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                    [--workload NAME]

Prints one JSON line.  `value` = edge-hops/s = units * nnz * hops / step time,
summed over ranks (weak scaling: every rank runs its own copy of the
workload), time from CUDA events around each forward, L2 flushed between
steps outside the events.  `e2e` runs the same forward through the host-buffer
entry point, host<->device copies inside the timed region.  The library
replays a repeated forward as a captured CUDA graph.  `roofline` is for the
dominant kernel (the diffusion hop): algorithmic bytes per launch over its mean
device time from per-kernel CUDA events (a second pass of the same steps,
kernels launched directly), against the measured HBM copy bandwidth.
`--impl reference` times the fp64 CPU oracle instead (the reference arm).
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from sparse_long_sequence_gb300 import synthetic, workloads  # noqa: E402

METRIC = "edge-hops/sec for diffuser_forward (n=4096, K=5); % of GB300 HBM roofline"
# the arithmetic of each kernel family (diffuser_kernels_for: CSR, band, block)
ARITH = ("fp32 SIMT (CSR path)",
         "A and Z_k as bf16 hi + lo pairs on the tensor cores (window, globals), fp32 gathers and accumulation",
         "A and Z_k as bf16 hi + lo pairs on the tensor cores (every 64 x 64 block)")
UNIT = "edge-hops/s"
L2_FLUSH_BYTES = 256 << 20          # > 129 MB of L2
FALLBACK_HBM_GBS = 6800.0


# ---------------------------------------------------------------- byte model
def algorithmic_bytes(w: workloads.Workload, nnz: int) -> dict:
    """"Score once, store A, read it K times" model, per forward.

    Per unit: Q, K, V read and out written once (4 n d s), A written once and
    read K times (4 E (K+1)), the fp32 hop state Z_k written and read between
    hops with V re-read per hop ((K-1)(8 n d + n d s)); plus the graph (once).
    The hop kernels' share per unit: 4 E K + 2 n d s + (K-1)(8 n d + n d s).
    """
    s = 2 if w.dtype == "bf16" else 4
    n, d, K, E, U = w.n, w.d, w.hops, nnz, w.units
    per_unit_total = 4 * n * d * s + (1 + K) * E * 4 + (K - 1) * (2 * n * d * 4 + n * d * s)
    per_unit_hops = 4 * E * K + 2 * n * d * s + (K - 1) * (8 * n * d + n * d * s)
    return dict(total=U * per_unit_total + (n + 1) * 8 + E * 4,
                hops_total=U * per_unit_hops,
                per_hop_launch=U * per_unit_hops / max(K, 1))


def measured_peaks() -> tuple[float, str]:
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(p) as f:
            return float(json.load(f)["hbm_gbs"]), "measured"
    except Exception:
        return FALLBACK_HBM_GBS, "fallback"


FALLBACK_BF16_TFLOPS = 1900.0


def measured_bf16_peak() -> tuple[float, str]:
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(p) as f:
            return float(json.load(f)["bf16_tflops"]), "measured"
    except Exception:
        return FALLBACK_BF16_TFLOPS, "fallback"


def time_events(fn, steps: int, stream, flush) -> list[float]:
    """Device milliseconds of fn() per step: CUDA events on `stream`, L2 flushed
    between steps outside the events."""
    import torch
    ms = []
    for k in range(steps):
        flush.fill_(k & 0xFF)
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        fn()
        b.record(stream)
        torch.cuda.synchronize()
        ms.append(a.elapsed_time(b))
    return ms


def measure_layer(dl, w, g, steps: int, stream, flush) -> dict:
    """The module's projections at the workload's sizes (model width D = 64 H):
    each GEMM's TFLOP/s (2 M N K flops over its median device time) against the
    measured bf16 peak, and the whole module (projections + forward) per step."""
    import torch
    B, n, H = w.B, w.n, w.H
    D = 64 * H
    X, Wqkv, Wo = (torch.from_numpy(t).view(torch.bfloat16).cuda()
                   for t in synthetic.layer_inputs(B, n, D, H, seed=w.seed))
    Q, K, V = (torch.empty((B, H, n, 64), dtype=torch.bfloat16, device="cuda") for _ in range(3))
    Y = torch.empty_like(X)
    ws = dl.alloc_workspace(dl.diffuser_layer_workspace_size(g, B, D, H))
    for _ in range(3):
        dl.diffuser_qkv_projection(X, Wqkv, H, Q=Q, K=K, V=V, stream=stream)
        dl.diffuser_output_projection(Q, Wo, Y=Y, stream=stream)
        dl.diffuser_layer_forward(X, Wqkv, Wo, g, H, w.hops, w.alpha, Y=Y, workspace=ws, stream=stream)
    torch.cuda.synchronize()
    t_qkv = statistics.median(time_events(
        lambda: dl.diffuser_qkv_projection(X, Wqkv, H, Q=Q, K=K, V=V, stream=stream), steps, stream, flush))
    t_out = statistics.median(time_events(
        lambda: dl.diffuser_output_projection(Q, Wo, Y=Y, stream=stream), steps, stream, flush))
    t_mod = statistics.median(time_events(
        lambda: dl.diffuser_layer_forward(X, Wqkv, Wo, g, H, w.hops, w.alpha, Y=Y, workspace=ws,
                                          stream=stream), steps, stream, flush))
    peak, kind = measured_bf16_peak()
    M = B * n
    f_qkv, f_out = 2.0 * M * (3 * D) * D, 2.0 * M * D * D
    tf_qkv, tf_out = f_qkv / (t_qkv / 1e3) / 1e12, f_out / (t_out / 1e3) / 1e12
    return {"model_width": D, "tokens": M,
            "qkv_projection": {"ms": t_qkv, "tflops": tf_qkv, "frac": tf_qkv / peak},
            "output_projection": {"ms": t_out, "tflops": tf_out, "frac": tf_out / peak},
            "module_ms": t_mod, "peak_tflops": peak, "peak_kind": kind,
            "bound": "tensor", "timing": "median device time of the steps, L2 flushed between them"}


def measure_backward(dl, w, g, Q, K, V, steps: int, stream, flush) -> dict:
    """The backward pass (gradients of <dOut, forward>) on the workload: median
    device time per step and edge-hops per second of the hops it reverses."""
    import torch
    dO = V.flip(-1).contiguous()
    code = dl.DIFFUSER_DTYPE_BF16 if w.dtype == "bf16" else dl.DIFFUSER_DTYPE_FP32
    ws = dl.alloc_workspace(dl.diffuser_backward_workspace_size(g, w.B, w.H, w.d, code, w.hops))
    grads = [torch.empty_like(Q) for _ in range(3)]
    for _ in range(2):
        dl.diffuser_backward(Q, K, V, dO, g, w.hops, w.alpha, *grads, workspace=ws, stream=stream)
    torch.cuda.synchronize()
    t = statistics.median(time_events(
        lambda: dl.diffuser_backward(Q, K, V, dO, g, w.hops, w.alpha, *grads, workspace=ws, stream=stream),
        steps, stream, flush))
    kernels = ("SIMT: the window's edges as 64 x 64 shared-memory tiles, the other edges on CSR "
               "kernels (recompute, reversed hops over the transposed edge list)"
               if w.kind in ("token", "causal") else
               "CSR SIMT (recompute, reversed hops over the transposed edge list)")
    return {"ms": t, "value": w.units * g.nnz * w.hops / (t / 1e3), "unit": UNIT, "kernels": kernels}


# the source files of each path's hop kernels (and what they include): a traffic
# record holds while these are unchanged
BAND_FILES = ("band_hop.cu", "band_score.cu", "band_common.cuh", "sm100_ptx.cuh", "internal.h")
BLOCK_FILES = ("block_path.cu", "band_common.cuh", "sm100_ptx.cuh", "internal.h")
CSR_FILES = ("simt_path.cu", "internal.h")


def path_files(kernels: str) -> tuple:
    return {"band": BAND_FILES, "block": BLOCK_FILES}.get(kernels, CSR_FILES)


def hop_kernel_traffic(workload: str, kernels: str) -> float | None:
    """ncu DRAM bytes of one middle hop (all its launches), if recorded for the
    current source of that path's kernels (profiles/traffic.json)."""
    p = os.path.join(ROOT, "profiles", "traffic.json")
    try:
        with open(p) as f:
            rec = json.load(f).get(workload)
    except Exception:
        return None
    if not rec or rec.get("source_sha") != kernel_source_sha(path_files(kernels)):
        return None
    return float(rec["bytes_per_hop"])


def kernel_source_sha(files: tuple | None = None) -> str:
    """sha256 prefix over the named files of sparse_long_sequence_gb300/csrc (all of
    its sources when None)."""
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "sparse_long_sequence_gb300", "csrc")
    names = sorted(files) if files else sorted(n for n in os.listdir(csrc) if n.endswith((".cu", ".h", ".cuh")))
    for name in names:
        with open(os.path.join(csrc, name), "rb") as f:
            h.update(name.encode() + f.read())
    return h.hexdigest()[:16]


# ---------------------------------------------------------------- clocks
class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, device_index: int):
        self.idx = device_index
        self.proc = None
        self.path = os.path.join("/tmp", f"bench_clocks_{os.getpid()}.csv")

    def start(self):
        try:
            self.fh = open(self.path, "w")
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.idx}", f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "200"],
                stdout=self.fh, stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None

    def stop(self) -> dict | None:
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        self.fh.close()
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        with open(self.path) as f:
            for line in f:
                p = [x.strip() for x in line.split(",")]
                if len(p) < 9:
                    continue
                try:
                    sm.append(float(p[1]))
                    smax.append(float(p[2]))
                except ValueError:
                    continue
                for name, val in zip(names, p[5:9]):
                    if val.lower() == "active":
                        reasons.add(name)
        os.unlink(self.path)
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(smax),
                "reasons": sorted(reasons), "samples": len(sm)}


# ---------------------------------------------------------------- shared pieces
def bench_config(w: workloads.Workload, world: int) -> dict:
    """The `config` object of the JSON line, identical for both arms."""
    return {**w.describe(), "parallelism": f"dp{world}" if world > 1 else "single GPU",
            "l2": "GPU arm: flushed between steps (256 MB write outside the timed events)"}


def cpu_model() -> str:
    """The host CPU's model name (lscpu, else /proc/cpuinfo), for the CPU legs."""
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        for line in out.splitlines():
            if line.startswith("Model name:"):
                return line.split(":", 1)[1].strip()
    except Exception:
        pass
    try:
        with open("/proc/cpuinfo") as f:
            for line in f:
                if line.lower().startswith(("model name", "cpu model")):
                    return line.split(":", 1)[1].strip()
    except Exception:
        pass
    return "unknown"


class BenchCheckFailed(RuntimeError):
    """A timed forward did not complete correctly: the line must not be printed."""


def check_graph_status(dl, g, where: str) -> None:
    """Fail when a kernel on graph g reported a failure (a bounded wait that gave
    up): every result since the last reset, timed ones included, is invalid."""
    st = dl.diffuser_graph_status(g)
    if st != 0:
        raise BenchCheckFailed(f"device status word {st:#x} set after {where}")


def check_sampled_unit(w: workloads.Workload, out_unit, Qh, Kh, Vh, unit: int) -> dict:
    """Compare one (batch, head) unit of a timed forward's output with the fp64
    oracle on the same inputs: fp32 max-abs <= 1e-5, bf16 per-row max error over
    the row's max-norm <= 4e-3."""
    import oracle
    b, h = divmod(unit, w.H)
    gargs = w.graph_args()
    if w.kind == "block":
        row_ptr, col = oracle.block_graph(**gargs)
    else:
        row_ptr, col = oracle.token_graph(**gargs, causal=w.kind == "causal")
    one = [oracle.widen(x[b:b + 1, h:h + 1], w.dtype) for x in (Qh, Kh, Vh)]
    ref = oracle.forward(*one, row_ptr, col, w.hops, w.alpha, nthreads=os.cpu_count() or 1)[0, 0]
    got = np.asarray(out_unit, dtype=np.float64)
    if w.dtype == "fp32":
        err, tol = float(np.abs(got - ref).max()), 1e-5
    else:
        den = np.abs(ref).max(axis=-1)
        err = float((np.abs(got - ref).max(axis=-1) / np.where(den > 0, den, 1.0)).max())
        tol = 4e-3
    if not err <= tol:
        raise BenchCheckFailed(f"unit {unit} differs from the oracle: error {err:.3e} > {tol}")
    return {"unit": unit, "error": err, "tolerance": tol,
            "metric": "max-abs" if w.dtype == "fp32" else "per-row max error / row max-norm"}


# ---------------------------------------------------------------- CPU oracle arm
def oracle_sample(w: workloads.Workload, units: int, nthreads: int) -> tuple[float, int, int]:
    """Run the fp64 oracle on `units` units of the workload; returns (seconds,
    edge-hops, nnz)."""
    import oracle
    gargs = w.graph_args()
    if w.kind == "block":
        row_ptr, col = oracle.block_graph(**gargs)
    else:
        row_ptr, col = oracle.token_graph(**gargs, causal=w.kind == "causal")
    nnz = int(row_ptr[-1])
    Q, K, V = synthetic.qkv(1, units, w.n, w.d, w.dtype, seed=w.seed)
    Qw, Kw, Vw = (oracle.widen(x, w.dtype) for x in (Q, K, V))
    t0 = time.perf_counter()
    oracle.forward(Qw, Kw, Vw, row_ptr, col, w.hops, w.alpha, nthreads=nthreads)
    dt = time.perf_counter() - t0
    return dt, units * nnz * w.hops, nnz


def cpu_sample_units(w) -> tuple[int, int]:
    """All units of the workload (the oracle takes well under a minute for any of
    them on a 16-core host), threads over units."""
    cores = os.cpu_count() or 1
    return w.units, cores


def run_reference(args, w) -> None:
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return
    units, cores = cpu_sample_units(w)
    for _ in range(args.warmup):        # warm-up steps: one unit each (loads, page-ins)
        oracle_sample(w, 1, 1)
    times, eh = [], 0
    for _ in range(args.steps):
        dt, eh, nnz = oracle_sample(w, units, cores)
        times.append(dt)
    value = eh / statistics.mean(times)
    sample = (f"{units} of {w.units} (batch, head) units of {w.name} per step, "
              f"fp64 oracle, {cores} threads over units")
    world = int(os.environ.get("WORLD_SIZE", "1"))
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": 0,
        "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": 1e3 * statistics.mean(times), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": bench_config(w, world),
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": cores, "kind": "oracle",
                         "sample": sample, "cpu_model": cpu_model()},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


# ---------------------------------------------------------------- ranks
def max_over_ranks(x: float, device=None) -> float:
    """The maximum of x over the ranks of the default process group (x itself
    with no group or one rank): every rank's replica must have finished."""
    import torch
    import torch.distributed as dist
    if not dist.is_available() or not dist.is_initialized() or dist.get_world_size() == 1:
        return x
    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def whole_job_rate(units_per_rank: int, nnz: int, hops: int, world: int, ms: float) -> float:
    """Edge-hops per second over all ranks: each rank runs its own replica of the
    workload (weak scaling), and the job takes the slowest rank's time."""
    return world * units_per_rank * nnz * hops / (ms / 1e3)


def step_stats(ms: list[float]) -> dict:
    """Median, 10th and 90th percentile of the per-step times (any count >= 1)."""
    a = np.asarray(ms, dtype=np.float64)
    return {"median": float(np.median(a)), "p10": float(np.percentile(a, 10)),
            "p90": float(np.percentile(a, 90)), "n": int(a.size)}


# ---------------------------------------------------------------- GPU arm
def run_ours(args, w) -> None:
    import torch
    import torch.distributed as dist

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if not torch.cuda.is_available():
        raise SystemExit("bench.py needs a CUDA device for --impl ours")
    torch.cuda.set_device(local)
    if world > 1:
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))

    from sparse_long_sequence_gb300 import binding as dl

    # graph + inputs (each rank its own copy of the workload: weak scaling)
    if w.kind in ("token", "causal"):
        build = dl.diffuser_build_causal_graph if w.kind == "causal" else dl.diffuser_build_graph
        g = build(w.n, w.r, w.n_globals, rand_per_row=w.rand_per_row, seed=w.seed)
    else:
        g = dl.diffuser_build_block_graph(w.n, w.block, w.window_blocks, w.rand_blocks,
                                          w.global_blocks, seed=w.seed)
    Qh, Kh, Vh = synthetic.qkv(w.B, w.H, w.n, w.d, w.dtype, seed=w.seed)
    tdt = torch.bfloat16 if w.dtype == "bf16" else torch.float32

    def host(x):
        t = torch.from_numpy(x)
        return (t.view(torch.bfloat16) if w.dtype == "bf16" else t).pin_memory()

    Qp, Kp, Vp = host(Qh), host(Kh), host(Vh)
    Q, K, V = Qp.cuda(), Kp.cuda(), Vp.cuda()
    out = torch.empty_like(V)
    code = dl.DIFFUSER_DTYPE_BF16 if w.dtype == "bf16" else dl.DIFFUSER_DTYPE_FP32
    ws = dl.alloc_workspace(dl.diffuser_workspace_size(g, w.B, w.H, w.d, code))
    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device="cuda")
    stream = torch.cuda.current_stream()

    def step():
        dl.diffuser_forward(Q, K, V, g, w.hops, w.alpha, out=out, workspace=ws, stream=stream)

    dl.diffuser_graph_status(g, reset=True)     # every later check covers all of this run
    for _ in range(max(args.warmup, 0)):
        flush.fill_(1)
        step()
    torch.cuda.synchronize()

    # ---- timed region: K steps, CUDA events around each forward
    starts = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    clocks = ClockSampler(local)
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize()
    clocks.start()
    time.sleep(0.3)
    launches0, _ = dl.diffuser_launch_count()
    for k in range(args.steps):
        flush.fill_(k & 0xFF)
        starts[k].record(stream)
        step()
        ends[k].record(stream)
    torch.cuda.synchronize()
    launches1, _ = dl.diffuser_launch_count()
    if world > 1:
        dist.barrier()
    clock_info = clocks.stop()
    step_ms = [s.elapsed_time(e) for s, e in zip(starts, ends)]
    check_graph_status(dl, g, "the warm-up and timed steps")
    # the last timed forward's output, one sampled (batch, head) unit against the oracle
    # (outside the timed region; the unit differs per rank)
    sample_unit = (w.units - 1 - rank) % w.units
    sb, sh = divmod(sample_unit, w.H)
    checked = check_sampled_unit(w, out[sb, sh].float().cpu().numpy(), Qh, Kh, Vh, sample_unit)

    # ---- the same K steps again with per-kernel CUDA events (the library
    # launches each kernel directly while its profile is open): the device time
    # of every kernel, for the roofline of the dominant one
    prof_ms = []
    torch.cuda.synchronize()
    dl.diffuser_profile_begin()
    for k in range(args.steps):
        flush.fill_(k & 0xFF)
        starts[k].record(stream)
        step()
        ends[k].record(stream)
    torch.cuda.synchronize()
    prof = dl.diffuser_profile_end()
    prof_ms = [s.elapsed_time(e) for s, e in zip(starts, ends)]
    t_step = max_over_ranks(statistics.mean(step_ms), device="cuda")

    if args.forward_only:
        # profiling runs: the timed and kernel-timing passes only
        check_graph_status(dl, g, "the kernel-timing pass")
        print(json.dumps({"metric": METRIC, "value": whole_job_rate(w.units, g.nnz, w.hops, world, t_step),
                          "unit": UNIT, "ms_per_step": t_step, "forward_only": True,
                          "kernel_ms_per_step": {k: v[0] / args.steps for k, v in prof.items() if v[1]}}),
              flush=True)
        return
    # ---- end to end through the host-buffer entry point
    Oh = torch.empty_like(Vp).pin_memory()
    ws_h = dl.alloc_workspace(dl.diffuser_host_workspace_size(g, w.B, w.H, w.d, code))
    for _ in range(2):
        dl.diffuser_forward_host(Qp, Kp, Vp, g, w.hops, w.alpha, Oh, ws_h, stream=stream)
    torch.cuda.synchronize()
    e2e_ms = []
    for k in range(args.steps):
        flush.fill_(k & 0xFF)
        torch.cuda.synchronize()
        t0 = time.perf_counter()
        dl.diffuser_forward_host(Qp, Kp, Vp, g, w.hops, w.alpha, Oh, ws_h, stream=stream)
        stream.synchronize()
        e2e_ms.append(1e3 * (time.perf_counter() - t0))
    t_e2e = max_over_ranks(statistics.mean(e2e_ms), device="cuda")
    check_graph_status(dl, g, "the kernel-timing and end-to-end passes")
    if not torch.equal(Oh, out.cpu()):
        raise BenchCheckFailed("end-to-end output differs from the device forward")

    check_graph_status(dl, g, "the kernel-timing and end-to-end passes")
    extra_steps = max(3, min(args.steps, 10))
    layer = measure_layer(dl, w, g, extra_steps, stream, flush) if w.dtype == "bf16" else None
    backward = measure_backward(dl, w, g, Q, K, V, extra_steps, stream, flush)
    check_graph_status(dl, g, "the module and backward passes")

    value = whole_job_rate(w.units, g.nnz, w.hops, world, t_step)
    io_bytes = w.units * w.n * w.d * (2 if w.dtype == "bf16" else 4)
    model = algorithmic_bytes(w, g.nnz)
    # the dominant kernel is the diffusion hop; on the band path one hop is two
    # launches (the tensor-core window kernel and the gather kernel), so the
    # hop's device time is their sum, per hop
    hop_ms = prof["hop"][0] + prof.get("gather", (0.0, 0))[0]
    band = prof.get("gather", (0.0, 0))[1] > 0
    n_hops = args.steps * w.hops
    peak, peak_kind = measured_peaks()
    roofline = None
    if n_hops and prof["hop"][1]:
        per_hop_s = hop_ms / n_hops / 1e3
        achieved = model["per_hop_launch"] / per_hop_s / 1e9
        traffic = hop_kernel_traffic(w.name, ["CSR", "band", "block"][dl.diffuser_kernels_for(g, code) - 1])
        measured_frac = traffic / per_hop_s / 1e9 / peak if traffic else None
        roofline = {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s",
                    "frac": achieved / peak, "traffic": traffic, "measured_frac": measured_frac,
                    "kernel": ("diffusion hop (window tcgen05 kernel + gather kernel)" if band
                               else "diffusion hop (block-sparse tcgen05 kernel)"
                               if dl.diffuser_kernels_for(g, code) == dl.DIFFUSER_KERNELS_BLOCK
                               else "diffusion hop (CSR SIMT kernel)"),
                    "peak_kind": peak_kind,
                    "algorithmic_bytes_per_hop": model["per_hop_launch"],
                    "mean_hop_ms": hop_ms / n_hops}
    whole_frac = model["total"] / (t_step / 1e3) / 1e9 / peak

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        units, cores = cpu_sample_units(w)
        dt, eh, _ = oracle_sample(w, units, cores)
        dt1, eh1, _ = oracle_sample(w, 1, 1)
        cpu = {"value": eh / dt, "unit": UNIT, "cores": cores, "kind": "oracle",
               "sample": f"{units} of {w.units} (batch, head) units of {w.name}, fp64 oracle, "
                         f"{cores} threads over units, {dt:.1f} s",
               "cpu_model": cpu_model(),
               "single_thread": {"value": eh1 / dt1, "unit": UNIT, "cores": 1,
                                 "sample": f"1 (batch, head) unit of {w.name}, {dt1:.1f} s"}}

    if rank == 0:
        line = {
            "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": t_step,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "step_ms": step_stats(step_ms),
            "dtype": "bf16" if w.dtype == "bf16" else "fp32", "data": "synthetic",
            "config": bench_config(w, world),
            "details": {"nnz": g.nnz, "units_per_gpu": w.units,
                        "arith": ARITH[dl.diffuser_kernels_for(g, code) - 1]},
            "checked": {**checked, "device_status": 0,
                        "what": "graph status word read after the warm-up + timed steps and after the "
                                "later passes (a bounded wait that gave up would set it); one sampled "
                                "unit of the last timed forward against the fp64 oracle"},
            "e2e": {"value": whole_job_rate(w.units, g.nnz, w.hops, world, t_e2e), "unit": UNIT,
                    "h2d_bytes_per_step": 3 * io_bytes, "d2h_bytes_per_step": io_bytes},
            "roofline": roofline,
            "whole_forward_hbm_frac": whole_frac,
            "kernel_ms_per_step": {k: v[0] / args.steps for k, v in prof.items() if v[1]},
            "kernel_timing": "a second pass of the same steps with per-kernel CUDA events "
                             f"(direct launches; {statistics.mean(prof_ms):.4f} ms per step there); "
                             "the timed steps replay the forward as a captured CUDA graph",
            "kernel_launches_per_step": {k: v[1] / args.steps for k, v in prof.items() if v[1]},
            "gpu_launches": int(launches1 - launches0),
            "kernels": ["CSR", "band", "block"][dl.diffuser_kernels_for(g, code) - 1],
            "layer": layer,
            "backward": backward,
            "clocks": clock_info,
            "cpu_baseline": cpu,
        }
        print(json.dumps(line), flush=True)
    if world > 1:
        dist.destroy_process_group()


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default=workloads.TEXT.name, choices=sorted(workloads.BY_NAME))
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--forward-only", action="store_true",
                    help="time the forward only (no end-to-end, module or backward passes); for profiling")
    args = ap.parse_args()
    args.warmup = max(args.warmup, 3)   # at least three untimed warm-up steps
    w = workloads.BY_NAME[args.workload]
    if args.impl == "reference":
        run_reference(args, w)
    else:
        try:
            run_ours(args, w)
        except BenchCheckFailed as e:
            print(json.dumps({"metric": METRIC, "value": None, "unit": UNIT, "error": str(e)}),
                  flush=True)
            raise SystemExit(3)


if __name__ == "__main__":
    main()
