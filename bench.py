"""Benchmark of the W4A16 fused dequant-GEMM on GB300.

One step = one pass of the decode sweep: the fused GEMM for M in {1,2,4,8,16},
K = 4096, N in {4096, 11008}, group 128, fp16 activations, asymmetric int4 weights
(10 launches).  The repack is offline and not timed.  The headline metric is achieved
HBM TB/s over algorithmic bytes (packed weights + scales + zeros + A + Y).  A default run
also times, with the same step count, the 70B-shaped decode FFN (HBM TB/s), the batch
transition sweep and the prefill GEMM (tensor TFLOP/s), the W4A8 decode path and the MX
block-scaled decode path (HBM TB/s), each with its own roofline, under the line's
"per_workload" key.  `--w4a8-only` / `--mx-only` time just those two.

Prints ONE JSON line (rank 0).  `--impl reference` times the CPU oracle instead, with the
same metric string, unit and workload.
Usage: python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                       [--workload NAME] [--no-extra-workloads] [--w4a8-only | --mx-only]
"""
from __future__ import annotations

import argparse
import hashlib
import glob
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

import synth_inputs as si  # noqa: E402

DEFAULT_WORKLOAD = "decode_k4096_n4096_n11008"
L2_BYTES = 129 * 1024 * 1024


class CudaRuntime:
    """Stream-ordered copies and events through the CUDA runtime library this process has
    already loaded (the one PyTorch uses), called directly: about a microsecond of host
    time per call, against several for the tensor-level equivalents, so that a serving
    loop's host side keeps ahead of the GPU even for 5 us GEMMs."""

    H2D, D2H = 1, 2  # cudaMemcpyKind

    def __init__(self):
        import ctypes
        path = None
        with open("/proc/self/maps") as f:
            for line in f:
                if "libcudart.so" in line:
                    path = line.split()[-1]
                    break
        for cand in ([path] if path else []) + ["libcudart.so.13", "libcudart.so.12",
                                                 "/usr/local/cuda/lib64/libcudart.so"]:
            try:
                L = ctypes.CDLL(cand)
                break
            except OSError:
                continue
        else:
            raise RuntimeError("no CUDA runtime library found")
        P, I, U, Z = ctypes.c_void_p, ctypes.c_int, ctypes.c_uint, ctypes.c_size_t
        L.cudaMemcpyAsync.argtypes = [P, P, Z, I, P]
        L.cudaMemcpyAsync.restype = I
        L.cudaEventCreateWithFlags.argtypes = [ctypes.POINTER(P), U]
        L.cudaEventCreateWithFlags.restype = I
        L.cudaEventRecord.argtypes = [P, P]
        L.cudaEventRecord.restype = I
        L.cudaStreamWaitEvent.argtypes = [P, P, U]
        L.cudaStreamWaitEvent.restype = I
        L.cudaEventDestroy.argtypes = [P]
        L.cudaEventDestroy.restype = I
        self.L, self.ctypes = L, ctypes

    def _ok(self, rc, what):
        if rc != 0:
            raise RuntimeError(f"{what} failed: CUDA error {rc}")

    def event(self):
        ev = self.ctypes.c_void_p()
        self._ok(self.L.cudaEventCreateWithFlags(self.ctypes.byref(ev), 2), "cudaEventCreate")
        return ev.value  # cudaEventDisableTiming

    def destroy(self, ev):
        self.L.cudaEventDestroy(ev)

    def copy(self, dst, src, nbytes, kind, stream):
        self._ok(self.L.cudaMemcpyAsync(dst, src, nbytes, kind, stream), "cudaMemcpyAsync")

    def record(self, ev, stream):
        self._ok(self.L.cudaEventRecord(ev, stream), "cudaEventRecord")

    def wait(self, stream, ev):
        self._ok(self.L.cudaStreamWaitEvent(stream, ev, 0), "cudaStreamWaitEvent")


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD, choices=sorted(si.WORKLOADS))
    ap.add_argument("--graph-steps", type=int, default=10,
                    help="steps captured per CUDA graph (replayed to reach --steps)")
    ap.add_argument("--e2e-steps", type=int, default=200)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--kernel", type=int, default=0, help="0 auto, 1 tcgen05, 2 SIMT")
    ap.add_argument("--split-k", type=int, default=0)
    ap.add_argument("--tile-m", type=int, default=0)
    ap.add_argument("--stages", type=int, default=0)
    ap.add_argument("--epilogue", default="none",
                    choices=["none", "bias", "bias_relu", "bias_silu", "bias_residual",
                             "bias_silu_residual"],
                    help="fuse a bias / activation / residual epilogue into every GEMM")
    ap.add_argument("--dequant", default="magic", choices=["magic", "lut", "int"],
                    help="weight unpack of the tensor-core decode tiles: exponent injection "
                         "(default), the 16-entry shared-memory table (same results), or "
                         "the integer operand with fp32 group rescale (16-row tiles, "
                         "groups of 128; unrounded weights)")
    ap.add_argument("--shape", action="append", default=[],
                    help="restrict the workload to this shape tag (repeatable; profiling)")
    ap.add_argument("--mx-only", action="store_true",
                    help="time only the MX block-scaled decode workload (mx_ffn70b_decode)")
    ap.add_argument("--w4a8-only", action="store_true",
                    help="time only the W4A8 decode workload (w4a8_ffn70b_decode_bf16) and "
                         "print its line")
    ap.add_argument("--no-extra-workloads", dest="extra_workloads", action="store_false",
                    help="time only --workload (by default the 70B-shaped decode, the batch "
                         "transition and the prefill workloads are timed beside it)")
    return ap.parse_args()


def workload_shapes(a):
    shapes = si.WORKLOADS[a.workload]
    if a.shape:
        shapes = [p for p in shapes if si.shape_tag(p) in a.shape]
        if not shapes:
            raise SystemExit(f"no shape of {a.workload} matches {a.shape}")
    return shapes


# ---- distributed plumbing (one process per GPU; replicas, no data-path collective) ---

def dist_info():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


def dist_init(backend):
    import torch.distributed as dist
    ws, rank, _ = dist_info()
    if ws > 1 and not dist.is_initialized():
        os.environ.setdefault("MASTER_ADDR", "127.0.0.1")
        dist.init_process_group(backend=backend, rank=rank, world_size=ws)
    return ws, rank


def barrier(device=None):
    import torch.distributed as dist
    if dist.is_available() and dist.is_initialized():
        if device is not None and dist.get_backend() == "nccl":
            dist.barrier(device_ids=[device.index])
        else:
            dist.barrier()


def max_over_ranks(x: float, device=None) -> float:
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()):
        return x
    t = torch.tensor([x], dtype=torch.float64,
                     device=device if dist.get_backend() == "nccl" else "cpu")
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


# ---- measured peaks, clocks, profile traffic ------------------------------------------

def measured_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        d = json.load(open(p))
        return d, "measured"
    return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}, "fallback"


class ClockSampler:
    """nvidia-smi clocks / throttle reasons sampled every 200 ms while running."""
    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.lines = []
        self.t = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.Q}",
                 "--format=csv,noheader,nounits", "-lms", "200"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
            return
        self.t = threading.Thread(target=self._read, daemon=True)
        self.t.start()

    def _read(self):
        for ln in self.proc.stdout:
            self.lines.append((time.time(), ln.strip()))

    def stop(self):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=2)
            except subprocess.TimeoutExpired:
                self.proc.kill()
            if self.t is not None:
                self.t.join(timeout=2)

    def summary(self, t0=None, t1=None):
        rows = []
        for ts, ln in self.lines:
            f = [x.strip() for x in ln.split(",")]
            if len(f) < 9:
                continue
            try:
                rows.append((ts, float(f[1]), float(f[2]), f[5:9]))
            except ValueError:
                continue
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"], "samples": 0}
        sel = [r for r in rows if t0 is None or (t0 - 0.25 <= r[0] <= t1 + 0.25)] or rows
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in sel for i, v in enumerate(r[3]) if v == "Active"})
        return {"sm_mhz": statistics.median(r[1] for r in sel),
                "sm_max_mhz": max(r[2] for r in sel), "reasons": reasons, "samples": len(sel)}


# Device-code sources of each kernel family: a traffic record applies only while these
# are byte-for-byte the ones it was captured with.
_KERNEL_SOURCES = {
    "w4a8_gemm_kernel": ["w4a8.cu", "ptx.cuh"],
}
_W4A16_SOURCES = ["gemm_tc.cu", "gemv_simt.cu", "repack.cu", "dequant.cuh", "epilogue.cuh",
                  "format.cuh", "ptx.cuh"]


def kernel_source_hash(kernel="w4a16_tc_kernel"):
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "weight_only_int4_tma_gb300", "csrc")
    for name in _KERNEL_SOURCES.get(kernel, _W4A16_SOURCES):
        h.update(open(os.path.join(csrc, name), "rb").read())
    return h.hexdigest()[:16]


def profiled_traffic(workload, kernel):
    """DRAM bytes per launch of `kernel` from the committed ncu summary, if the kernel
    sources are unchanged since it was taken."""
    p = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(p):
        return None
    d = json.load(open(p)).get(workload)
    if not d or d.get("kernel_source_hash") != kernel_source_hash(kernel) or d.get("kernel") != kernel:
        return None
    return d.get("dram_bytes_per_launch")


# ---- what a workload is measured in (shared by both arms) ----------------------------

def compute_bound(shapes) -> bool:
    """Prefill and batch-transition workloads (M >= 64 everywhere) are bound by the tensor
    pipe and measured in TFLOP/s; decode-sized ones by HBM, in TB/s."""
    return min(p["M"] for p in shapes) >= 64


def metric_name(workload: str, shapes) -> str:
    """The line's metric string: identical for the GPU arm and the reference arm of one
    workload, so that their values divide."""
    kind = "tensor TFLOP/s" if compute_bound(shapes) else "HBM TB/s"
    return f"W4A16 GEMM achieved {kind} ({workload})"


def metric_unit(shapes) -> str:
    return "TFLOP/s" if compute_bound(shapes) else "TB/s"


# ---- the reference arm: the CPU oracle ----------------------------------------------

def oracle_slice(orc, c, n0, nc):
    """Oracle dequant + GEMM for output channels [n0, n0 + nc) of a case."""
    qw = c.qweight[n0:n0 + nc]
    sc = np.ascontiguousarray(c.scales[:, n0:n0 + nc])
    qz = None if c.qzeros is None else np.ascontiguousarray(c.qzeros[:, n0 // 8:(n0 + nc) // 8])
    wd = orc.dequant(qw, sc, qz, nc, c.K, c.group, c.dtype)
    orc.gemm(c.A, wd, c.M, nc, c.K, c.dtype)


def shape_bytes(p, epilogue="none"):
    b = si.algorithmic_bytes(p["M"], p["N"], p["K"], p["group"], p.get("asym", True))
    if epilogue != "none":
        b += 2 * p["N"]             # bias
    if epilogue.endswith("residual"):
        b += 2 * p["M"] * p["N"]    # residual read
    return b


def shape_work(p, tflops: bool, epilogue="none"):
    """Work of one GEMM in the workload's unit: flops, or algorithmic bytes."""
    return si.flops(p["M"], p["N"], p["K"]) if tflops else shape_bytes(p, epilogue)


def cpu_oracle_rate(cases, shapes, budget_s):
    """Times the oracle over slices of the workload's shapes for about budget_s seconds.
    Returns (work units/s in the workload's unit, sample description, threads, seconds)."""
    import oracle as orc
    orc.build()
    tfl = compute_bound(shapes)
    total = 0.0
    t_used = 0.0
    done = []
    nc = 256
    i = 0
    while t_used < budget_s and i < 100000:
        c, p = cases[i % len(cases)], shapes[i % len(cases)]
        n0 = (i // len(cases)) * nc % c.N
        n = min(nc, c.N - n0)
        t0 = time.perf_counter()
        oracle_slice(orc, c, n0, n)
        dt = time.perf_counter() - t0
        t_used += dt
        total += shape_work(p, tfl) * n / c.N
        done.append(f"{si.shape_tag(p)}[n {n0}:{n0 + n}]")
        i += 1
    desc = (f"{len(done)} slices of up to {nc} output channels (dequant + fp64 GEMM), e.g. "
            + ", ".join(done[:3]))
    return total / t_used, desc, orc.num_threads(), t_used


def run_reference(a):
    ws, rank, _ = dist_info()
    if ws > 1:
        dist_init("gloo")
        if rank != 0:
            return
    shapes = workload_shapes(a)
    cases = [si.make_case(**p) for p in shapes]
    tfl = compute_bound(shapes)
    import oracle as orc
    orc.build()
    # Each step: one slice of output channels of one shape (the shapes in turn), sized so
    # that the whole run stays within about two minutes.
    budget = 120.0 / max(1, a.steps + a.warmup)
    probe_c = max(cases, key=lambda c: c.M * c.K)
    t0 = time.perf_counter()
    oracle_slice(orc, probe_c, 0, 8)
    per_ch = (time.perf_counter() - t0) / 8
    nc = int(max(8, min(max(c.N for c in cases), (budget / max(per_ch, 1e-9)) // 8 * 8)))
    for i in range(a.warmup):
        c = cases[i % len(cases)]
        oracle_slice(orc, c, 0, min(nc, c.N))
    tot = 0.0
    t0 = time.perf_counter()
    for i in range(a.steps):
        c, p = cases[i % len(cases)], shapes[i % len(cases)]
        n = min(nc, c.N)
        n0 = (i * n) % c.N
        n = min(n, c.N - n0)
        oracle_slice(orc, c, n0, n)
        tot += shape_work(p, tfl) * n / c.N
    el = time.perf_counter() - t0
    v = tot / el / 1e12
    unit = metric_unit(shapes)
    sample = (f"per step: up to {nc} output channels of one shape of the workload, the shapes "
              f"in turn (dequant + fp64 GEMM)")
    line = {
        "impl": "reference", "metric": metric_name(a.workload, shapes),
        "value": v, "unit": unit, "n_gpus": a.gpus, "steps": a.steps, "warmup": a.warmup,
        "ms_per_step": el / max(1, a.steps) * 1e3, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": a.workload, "shapes": len(shapes),
                   "step_bytes": sum(shape_bytes(p) for p in shapes),
                   "step_flops": sum(si.flops(p["M"], p["N"], p["K"]) for p in shapes)},
        "cpu_baseline": {"value": v, "unit": unit, "cores": orc.num_threads(),
                         "kind": "oracle", "sample": sample},
        "e2e": {"value": v, "unit": unit, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


# ---- our arm ------------------------------------------------------------------------

def tensor_peak(peaks, region_s: float):
    """The dense bf16 (= fp16) tensor peak that matches a timed region: the burst figure
    for a region under a second, the sustained (power-capped) one for longer regions."""
    burst = float(peaks.get("bf16_tflops", 1900.0))
    sustained = float(peaks.get("bf16_tflops_sustained", burst))
    return (burst, "burst") if region_s < 1.0 else (sustained, "sustained")


class Measured:
    """Everything one workload's measurement produces (the JSON line's parts)."""


def measure_workload(a, w4, device, stream, sampler, workload, shapes, ex, steps,
                     warmup, epilogue="none"):
    import torch

    ws, rank, _ = dist_info()
    cases = [si.make_case(**p) for p in shapes]
    tfl = compute_bound(shapes)
    step_bytes = sum(shape_bytes(p, epilogue) for p in shapes)
    step_flops = sum(si.flops(p["M"], p["N"], p["K"]) for p in shapes)
    step_work = step_flops if tfl else step_bytes

    def dev(x):
        if x is None:
            return None
        v = x.view(np.int16) if x.dtype == np.uint16 else x.view(np.int32)
        return torch.from_numpy(np.ascontiguousarray(v)).to(device)

    # Weights rotate over enough copies that each launch reads them from HBM, not L2.
    shape_packed = [w4.w4a16_packed_bytes(c.N, c.K, c.group, c.qzeros is not None)
                    for c in cases]
    packed_per_step = sum(shape_packed)
    copies = max(2, -(-3 * L2_BYTES // max(1, packed_per_step)))
    bufs = []
    for c in cases:
        first = w4.repack(dev(c.qweight), dev(c.scales), dev(c.qzeros), c.N, c.K, c.group,
                          c.dtype)
        reps = [first] + [first.clone() for _ in range(copies - 1)]
        A = dev(c.A)
        Y = torch.empty((c.M, c.N), dtype=torch.int16, device=device)
        bufs.append((c, reps, A, Y))
    torch.cuda.synchronize()
    # the plain public call when every launch option is the library's default
    default_launch = not any(ex.values())
    act = {"relu": w4.W4A16_ACT_RELU, "silu": w4.W4A16_ACT_SILU}
    epi_act = next((v for k, v in act.items() if k in epilogue), w4.W4A16_ACT_NONE)
    # optional fused epilogue: a seeded bias per shape (resident, like the weights) and a
    # device-resident residual (the previous layer's output in a real forward pass)
    epi = []
    for c, _, _, _ in bufs:
        tdt = torch.float16 if c.dtype == 0 else torch.bfloat16
        g = torch.Generator().manual_seed(c.M * 100003 + c.N)
        bias = (torch.randn(c.N, generator=g).to(tdt).view(torch.int16).to(device)
                if epilogue != "none" else None)
        res = (torch.randn((c.M, c.N), generator=g).to(tdt).view(torch.int16).to(device)
               if epilogue.endswith("residual") else None)
        epi.append((bias, res))

    def gemm_call(j, A, packed, Y, stream_, public=False):
        c = bufs[j][0]
        if epilogue == "none":
            if public and default_launch:
                w4.w4a16_gemm(A, packed, c.M, c.N, c.K, c.group, c.dtype, Y, stream_)
            else:
                w4.w4a16_gemm_ex(A, packed, c.M, c.N, c.K, c.group, c.dtype, Y, stream=stream_,
                                 **ex)
        else:
            bias, res = epi[j]
            w4.w4a16_gemm_epilogue(A, packed, c.M, c.N, c.K, c.group, c.dtype, bias, res,
                                   epi_act, Y, stream=stream_,
                                   **({} if public and default_launch else ex))

    # which of the two kernels each shape runs on (the library's own launch choice)
    kname = {w4.W4A16_KERNEL_TC: "w4a16_tc_kernel", w4.W4A16_KERNEL_SIMT: "w4a16_gemv_kernel"}
    shape_kernel = [kname[w4.w4a16_gemm_plan(c.M, c.N, c.K, c.group, c.dtype, **ex)["kernel"]]
                    for c in cases]

    def launch_step(step_idx):
        for j, (c, reps, A, Y) in enumerate(bufs):
            gemm_call(j, A, reps[step_idx % copies], Y, stream)

    with torch.cuda.stream(stream):
        for i in range(max(3, warmup)):
            launch_step(i)
    stream.synchronize()
    st = w4.w4a16_get_device_status(stream)
    if st != 0:
        raise SystemExit(f"{workload}: device status after warm-up: {w4.status_string(st)}")

    # Per-shape pass (before the timed region, so that it runs at the clocks of a short
    # burst even when the timed region is long enough to reach the power cap): back-to-
    # back launches of one shape in a graph, rotating over at least 3 x L2 of that shape's
    # own weight copies.
    per_shape_ms = []
    per_shape_region_s = []
    for j, (c, reps, A, Y) in enumerate(bufs):
        cs = max(3, -(-3 * L2_BYTES // max(1, shape_packed[j])))
        own = list(reps[:cs]) + [reps[0].clone() for _ in range(cs - len(reps))]
        nl = max(20, cs)
        gj = torch.cuda.CUDAGraph()
        with torch.cuda.stream(stream):
            with torch.cuda.graph(gj, stream=stream):
                for i in range(nl):
                    gemm_call(j, A, own[i % cs], Y, stream)
            gj.replay()
            f0, f1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            f0.record(stream)
            for _ in range(3):
                gj.replay()
            f1.record(stream)
        stream.synchronize()
        ms = f0.elapsed_time(f1)
        per_shape_ms.append(ms / (3 * nl))
        per_shape_region_s.append(ms * 1e-3)
        del gj, own
    torch.cuda.synchronize(device)
    st = w4.w4a16_get_device_status(stream)
    if st != 0:
        raise SystemExit(f"{workload}: device status after per-shape pass: {w4.status_string(st)}")

    # Capture G steps into one CUDA graph (no events inside: consecutive GEMMs overlap
    # their prologues through programmatic dependent launch).
    G = max(1, min(a.graph_steps, steps))
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.stream(stream):
        with torch.cuda.graph(graph, stream=stream):
            for g in range(G):
                launch_step(g)
    stream.synchronize()
    full_replays = steps // G
    eager_tail = steps - full_replays * G
    with torch.cuda.stream(stream):
        for _ in range(2):
            graph.replay()
    stream.synchronize()

    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    barrier(device)
    torch.cuda.synchronize(device)
    t_wall0 = time.time()
    with torch.cuda.stream(stream):
        e0.record(stream)
        for _ in range(full_replays):
            graph.replay()
        for i in range(eager_tail):
            launch_step(i)
        e1.record(stream)
    stream.synchronize()
    torch.cuda.synchronize(device)
    barrier(device)
    t_wall1 = time.time()
    elapsed_ms = e0.elapsed_time(e1)
    st = w4.w4a16_get_device_status(stream)
    if st != 0:
        raise SystemExit(f"{workload}: device status after timed region: {w4.status_string(st)}")
    elapsed_ms = max_over_ranks(elapsed_ms, device)
    del graph

    peaks, peak_kind = measured_peaks()
    hbm_peak = float(peaks["hbm_gbs"])
    launch_bytes = [shape_bytes(p, epilogue) for p in shapes]
    launch_flops = [si.flops(p["M"], p["N"], p["K"]) for p in shapes]
    # The roofline is that of the dominant kernel (the one most launches of a step run
    # on): its algorithmic bytes (or flops) per launch over its average launch duration,
    # both over its own shapes, the durations from the per-shape pass (CUDA events on the
    # launch stream, back-to-back launches of one shape).
    counts = {k: shape_kernel.count(k) for k in sorted(set(shape_kernel))}
    dominant = max(sorted(counts), key=lambda k: (counts[k], k == "w4a16_tc_kernel"))
    dom = [j for j, k in enumerate(shape_kernel) if k == dominant]
    dom_launch_s = sum(per_shape_ms[j] for j in dom) * 1e-3 / len(dom)
    # the recorded counters describe the default launch of the whole workload only
    traffic = (profiled_traffic(workload, dominant)
               if default_launch and epilogue == "none" and not a.shape else None)
    if tfl:
        dom_flops = sum(launch_flops[j] for j in dom) / len(dom)
        achieved = dom_flops / dom_launch_s / 1e12
        tpeak, tkind = tensor_peak(peaks, max(per_shape_region_s[j] for j in dom))
        roofline = {"bound": "tensor", "achieved": achieved, "peak": tpeak,
                    "unit": "TFLOP/s", "frac": achieved / tpeak, "traffic": traffic,
                    "peak_kind": f"{peak_kind} bf16 dense, {tkind} (the fp16 dense rate is "
                                 f"the same)",
                    "kernel": dominant, "launches_per_step": counts[dominant],
                    "algorithmic_flops_per_launch": dom_flops}
        value = step_flops * steps * ws / (elapsed_ms * 1e-3) / 1e12
    else:
        dom_bytes = sum(launch_bytes[j] for j in dom) / len(dom)
        achieved = dom_bytes / dom_launch_s / 1e9
        roofline = {"bound": "hbm", "achieved": achieved, "peak": hbm_peak,
                    "unit": "GB/s", "frac": achieved / hbm_peak, "traffic": traffic,
                    "peak_kind": peak_kind, "kernel": dominant,
                    "launches_per_step": counts[dominant],
                    "algorithmic_bytes_per_launch": dom_bytes}
        value = step_bytes * steps * ws / (elapsed_ms * 1e-3) / 1e12
    tpeak_shape, _ = tensor_peak(peaks, 0.0)

    # End to end through the public API, as a serving loop runs it: every step copies that
    # step's activations (all shapes, one copy) from pinned host memory, calls w4a16_gemm
    # once per shape, and copies all of the step's outputs back (one copy).  Two buffer
    # sets and separate copy-in / copy-out streams let step i+1's input copy and step
    # i-1's output copy run while step i's GEMMs do.  The loop's host side is kept lean
    # (runtime calls for copies and events, the C entry point called directly) so that it
    # stays ahead of the GPU.
    def offsets(sizes):  # int16 element offsets, 256-byte aligned
        offs, o = [], 0
        for n in sizes:
            offs.append(o)
            o += -(-n // 128) * 128
        return offs, o
    a_sizes = [c.M * c.K for c in cases]
    y_sizes = [c.M * c.N for c in cases]
    a_offs, a_tot = offsets(a_sizes)
    y_offs, y_tot = offsets(y_sizes)
    hostA = torch.zeros(a_tot, dtype=torch.int16).pin_memory()
    for c, o, n in zip(cases, a_offs, a_sizes):
        hostA[o:o + n] = torch.from_numpy(np.ascontiguousarray(c.A.view(np.int16)).ravel())
    hostY = [torch.empty(y_tot, dtype=torch.int16).pin_memory() for _ in range(2)]
    devA = [torch.empty(a_tot, dtype=torch.int16, device=device) for _ in range(2)]
    devY = [torch.empty(y_tot, dtype=torch.int16, device=device) for _ in range(2)]
    h2d, d2h = 2 * a_tot, 2 * y_tot
    in_stream = torch.cuda.Stream(device=device)
    out_stream = torch.cuda.Stream(device=device)
    rt = CudaRuntime()
    in_done = [rt.event() for _ in range(2)]
    gemm_done = [rt.event() for _ in range(2)]
    out_done = [rt.event() for _ in range(2)]
    s_in, s_out = in_stream.cuda_stream, out_stream.cuda_stream

    # device addresses of every shape's A and Y in both buffer sets, taken once
    a_ptr = [[devA[b][o:o + n].data_ptr() for o, n in zip(a_offs, a_sizes)] for b in range(2)]
    y_ptr = [[devY[b][o:o + n].data_ptr() for o, n in zip(y_offs, y_sizes)] for b in range(2)]
    p_ptr = [[r.data_ptr() for r in reps] for _, reps, _, _ in bufs]
    s_ptr = stream.cuda_stream
    hA, hY = hostA.data_ptr(), [h.data_ptr() for h in hostY]
    dA, dY = [d.data_ptr() for d in devA], [d.data_ptr() for d in devY]
    # the public C entry points, called directly (the binding adds only marshalling)
    L = w4.lib()
    plain = epilogue == "none" and default_launch

    def e2e_step(i):
        b = i & 1
        if i >= 2:
            rt.wait(s_in, gemm_done[b])  # step i-2 has finished reading devA[b]
        rt.copy(dA[b], hA, h2d, rt.H2D, s_in)
        rt.record(in_done[b], s_in)
        rt.wait(s_ptr, in_done[b])
        if i >= 2:
            rt.wait(s_ptr, out_done[b])  # step i-2's outputs have left devY[b]
        for j, c in enumerate(cases):
            if plain:
                rc = L.w4a16_gemm(a_ptr[b][j], p_ptr[j][i % copies], c.M, c.N, c.K, c.group,
                                  c.dtype, y_ptr[b][j], s_ptr)
                if rc != 0:
                    raise w4.W4A16Error(rc, "w4a16_gemm")
            else:
                gemm_call(j, a_ptr[b][j], p_ptr[j][i % copies], y_ptr[b][j], s_ptr,
                          public=True)
        rt.record(gemm_done[b], s_ptr)
        rt.wait(s_out, gemm_done[b])
        rt.copy(hY[b], dY[b], d2h, rt.D2H, s_out)
        rt.record(out_done[b], s_out)

    e2e_steps = max(1, min(a.e2e_steps, steps))
    e2e_steps = max(1, min(e2e_steps, int(8e9 // (h2d + d2h))))
    for i in range(3):
        e2e_step(i)
    torch.cuda.synchronize(device)
    barrier(device)
    f0, f1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    f0.record(in_stream)
    for i in range(e2e_steps):
        e2e_step(i)
    out_stream.wait_stream(stream)
    out_stream.wait_stream(in_stream)
    f1.record(out_stream)
    torch.cuda.synchronize(device)
    for ev in in_done + gemm_done + out_done:
        rt.destroy(ev)
    st = w4.w4a16_get_device_status(stream)
    if st != 0:
        raise SystemExit(f"{workload}: device status after end-to-end region: "
                         f"{w4.status_string(st)}")
    e2e_ms = max_over_ranks(f0.elapsed_time(f1), device)
    e2e_val = step_work * e2e_steps * ws / (e2e_ms * 1e-3) / 1e12

    per_shape = []
    for j, (p, ms, b, fl) in enumerate(zip(shapes, per_shape_ms, launch_bytes, launch_flops)):
        per_shape.append({"shape": si.shape_tag(p), "kernel": shape_kernel[j],
                          "us": round(ms * 1e3, 3),
                          "gbs": round(b / (ms * 1e-3) / 1e9, 1),
                          "hbm_frac": round(b / (ms * 1e-3) / 1e9 / hbm_peak, 4),
                          "tflops": round(fl / (ms * 1e-3) / 1e12, 1),
                          "tensor_frac": round(fl / (ms * 1e-3) / 1e12 / tpeak_shape, 4)})
    m = Measured()
    m.cases, m.shapes, m.tfl = cases, shapes, tfl
    m.value, m.unit = value, metric_unit(shapes)
    m.elapsed_ms, m.steps = elapsed_ms, steps
    m.step_bytes, m.step_flops = step_bytes, step_flops
    m.copies, m.packed_per_step, m.G = copies, packed_per_step, G
    m.roofline, m.per_shape = roofline, per_shape
    m.e2e = {"value": e2e_val, "unit": m.unit, "h2d_bytes_per_step": h2d,
             "d2h_bytes_per_step": d2h, "steps": e2e_steps,
             "note": "per step: one pinned-host copy of all shapes' A in, one w4a16_gemm "
                     "call per shape, one copy of all Y out; two buffer sets, copy-in and "
                     "copy-out streams overlapping the neighbouring steps' GEMMs; packed "
                     "weights resident (uploaded once, as in serving)"}
    m.dominant, m.counts = dominant, counts
    m.gpu_launches = steps * len(shapes)
    m.clocks = sampler.summary(t_wall0, t_wall1)
    del bufs, devA, devY, hostA, hostY
    torch.cuda.synchronize(device)
    torch.cuda.empty_cache()
    return m


def measure_w4a8(a, w4, device, stream, sampler, workload, steps, warmup):
    """The W4A8 (LiquidQuant) decode path: per shape one w4a8_quantize_act and one
    w4a8_gemm per step.  The step's value is its algorithmic bytes (the GEMM's: codes,
    steps and offsets, channel scales, int8 A with its row scales, Y; plus the quantiser's
    read of A and write of the int8 A and row scales) over the step time; the roofline is
    that of the GEMM kernel over its own algorithmic bytes and launch time."""
    import torch

    ws, rank, _ = dist_info()
    shapes = si.W4A8_WORKLOADS[workload]
    cases = [si.make_w4a8_case(**p) for p in shapes]

    def dev(x):
        v = x.view(np.int16) if x.dtype == np.uint16 else (
            x.view(np.int32) if x.dtype == np.uint32 else x)
        return torch.from_numpy(np.ascontiguousarray(v)).to(device)

    gemm_bytes = [si.w4a8_algorithmic_bytes(c.M, c.N, c.K) for c in cases]
    quant_bytes = [2 * c.M * c.K + c.M * c.K + 4 * c.M for c in cases]
    step_bytes = sum(gemm_bytes) + sum(quant_bytes)
    shape_packed = [w4.w4a8_packed_bytes(c.N, c.K) for c in cases]
    copies = max(2, -(-3 * L2_BYTES // max(1, sum(shape_packed))))
    bufs = []
    for c, nb in zip(cases, shape_packed):
        first = torch.empty(nb, dtype=torch.uint8, device=device)
        w4.w4a8_repack(dev(c.qweight), dev(c.s_u8), dev(c.a), dev(c.s_w), c.N, c.K, first)
        reps = [first] + [first.clone() for _ in range(copies - 1)]
        A = dev(c.A)
        A_i8 = torch.empty((c.M, c.K), dtype=torch.int8, device=device)
        s_a = torch.empty(c.M, dtype=torch.float32, device=device)
        Y = torch.empty((c.M, c.N), dtype=torch.int16, device=device)
        bufs.append((c, reps, A, A_i8, s_a, Y))
    st = w4.w4a16_get_device_status(stream)
    if st != 0:
        raise SystemExit(f"{workload}: device status after repack: {w4.status_string(st)}")

    def launch_step(i):
        for c, reps, A, A_i8, s_a, Y in bufs:
            w4.w4a8_quantize_act(A, c.M, c.K, c.dtype, A_i8, s_a, stream)
            w4.w4a8_gemm(A_i8, s_a, reps[i % copies], c.M, c.N, c.K, c.dtype, Y, stream)

    with torch.cuda.stream(stream):
        for i in range(max(3, warmup)):
            launch_step(i)
    st = w4.w4a16_get_device_status(stream)
    if st != 0:
        raise SystemExit(f"{workload}: device status after warm-up: {w4.status_string(st)}")

    # per-shape pass: back-to-back GEMM launches of one shape in a graph, rotating over at
    # least 3 x L2 of that shape's own weight copies
    per_shape_us = []
    for j, (c, reps, A, A_i8, s_a, Y) in enumerate(bufs):
        cs = max(3, -(-3 * L2_BYTES // max(1, shape_packed[j])))
        own = list(reps[:cs]) + [reps[0].clone() for _ in range(cs - len(reps))]
        nl = max(20, cs)
        gj = torch.cuda.CUDAGraph()
        with torch.cuda.stream(stream):
            with torch.cuda.graph(gj, stream=stream):
                for i in range(nl):
                    w4.w4a8_gemm(A_i8, s_a, own[i % cs], c.M, c.N, c.K, c.dtype, Y, stream)
            gj.replay()
            f0, f1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            f0.record(stream)
            for _ in range(3):
                gj.replay()
            f1.record(stream)
        stream.synchronize()
        per_shape_us.append(f0.elapsed_time(f1) * 1e3 / (3 * nl))
        del gj, own

    G = max(1, min(a.graph_steps, steps))
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.stream(stream):
        with torch.cuda.graph(graph, stream=stream):
            for g in range(G):
                launch_step(g)
        graph.replay()
    stream.synchronize()
    full_replays, tail = steps // G, steps % G
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    barrier(device)
    torch.cuda.synchronize(device)
    t_wall0 = time.time()
    with torch.cuda.stream(stream):
        e0.record(stream)
        for _ in range(full_replays):
            graph.replay()
        for i in range(tail):
            launch_step(i)
        e1.record(stream)
    stream.synchronize()
    barrier(device)
    t_wall1 = time.time()
    st = w4.w4a16_get_device_status(stream)
    if st != 0:
        raise SystemExit(f"{workload}: device status after timed region: {w4.status_string(st)}")
    elapsed_ms = max_over_ranks(e0.elapsed_time(e1), device)
    del graph

    peaks, peak_kind = measured_peaks()
    hbm_peak = float(peaks["hbm_gbs"])
    dom_bytes = sum(gemm_bytes) / len(gemm_bytes)
    dom_s = sum(per_shape_us) * 1e-6 / len(per_shape_us)
    achieved = dom_bytes / dom_s / 1e9
    roofline = {"bound": "hbm", "achieved": achieved, "peak": hbm_peak, "unit": "GB/s",
                "frac": achieved / hbm_peak,
                "traffic": profiled_traffic(workload, "w4a8_gemm_kernel"), "peak_kind": peak_kind,
                "kernel": "w4a8_gemm_kernel", "launches_per_step": len(cases),
                "algorithmic_bytes_per_launch": dom_bytes}
    value = step_bytes * steps * ws / (elapsed_ms * 1e-3) / 1e12

    # end to end through the public calls: per step one pinned-host copy of all shapes' A
    # in, the quantiser and the GEMM per shape, one copy of all Y out, on one stream
    a_sizes = [c.M * c.K for c in cases]
    y_sizes = [c.M * c.N for c in cases]
    hostA = torch.cat([torch.from_numpy(np.ascontiguousarray(c.A.view(np.int16)).ravel())
                       for c in cases]).pin_memory()
    hostY = torch.empty(sum(y_sizes), dtype=torch.int16).pin_memory()
    devA = torch.empty(sum(a_sizes), dtype=torch.int16, device=device)
    devY = torch.empty(sum(y_sizes), dtype=torch.int16, device=device)
    a_views, y_views, oa, oy = [], [], 0, 0
    for na, ny in zip(a_sizes, y_sizes):
        a_views.append(devA[oa:oa + na])
        y_views.append(devY[oy:oy + ny])
        oa, oy = oa + na, oy + ny

    def e2e_step(i):
        devA.copy_(hostA, non_blocking=True)
        for j, (c, reps, _, A_i8, s_a, _) in enumerate(bufs):
            w4.w4a8_quantize_act(a_views[j], c.M, c.K, c.dtype, A_i8, s_a, stream)
            w4.w4a8_gemm(A_i8, s_a, reps[i % copies], c.M, c.N, c.K, c.dtype, y_views[j],
                         stream)
        hostY.copy_(devY, non_blocking=True)

    e2e_steps = max(1, min(a.e2e_steps, steps))
    with torch.cuda.stream(stream):
        for i in range(3):
            e2e_step(i)
        stream.synchronize()
        f0, f1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        f0.record(stream)
        for i in range(e2e_steps):
            e2e_step(i)
        f1.record(stream)
    stream.synchronize()
    st = w4.w4a16_get_device_status(stream)
    if st != 0:
        raise SystemExit(f"{workload}: device status after end-to-end region: "
                         f"{w4.status_string(st)}")
    e2e_ms = max_over_ranks(f0.elapsed_time(f1), device)
    unit = "TB/s"
    per_shape = [{"shape": si.w4a8_shape_tag(p), "kernel": "w4a8_gemm_kernel",
                  "us": round(us, 3), "gbs": round(b / (us * 1e-6) / 1e9, 1),
                  "hbm_frac": round(b / (us * 1e-6) / 1e9 / hbm_peak, 4)}
                 for p, us, b in zip(shapes, per_shape_us, gemm_bytes)]
    out = {
        "workload": workload, "metric": f"W4A8 GEMM achieved HBM TB/s ({workload})",
        "value": value, "unit": unit, "ms_per_step": elapsed_ms / steps, "steps": steps,
        "shapes": len(shapes), "step_bytes": step_bytes, "step_flops": sum(
            si.flops(c.M, c.N, c.K) for c in cases),
        "l2": f"inputs larger than L2: {copies} rotating copies of the packed weights "
              f"({copies * sum(shape_packed) / 2**20:.0f} MiB per rotation)",
        "roofline": roofline, "per_shape": per_shape,
        "e2e": {"value": step_bytes * e2e_steps * ws / (e2e_ms * 1e-3) / 1e12, "unit": unit,
                "h2d_bytes_per_step": 2 * sum(a_sizes), "d2h_bytes_per_step": 2 * sum(y_sizes),
                "steps": e2e_steps,
                "note": "per step: one pinned-host copy of all shapes' A in, "
                        "w4a8_quantize_act + w4a8_gemm per shape, one copy of all Y out, "
                        "one stream; packed weights resident"},
        "kernels_per_step": {"w4a8_quantize_kernel": len(cases), "w4a8_gemm_kernel": len(cases)},
        "gpu_launches": 2 * len(cases) * steps,
        "clocks": sampler.summary(t_wall0, t_wall1),
        "dtype": "int8 products, int32 sums, fp32 scaling",
        "note": "dp4a on the CUDA cores: sm_103a has no int8 tensor-core MMA"}
    del bufs, devA, devY, hostA, hostY
    torch.cuda.synchronize(device)
    torch.cuda.empty_cache()
    return out


def measure_mx(a, w4, device, stream, sampler, workload, steps, warmup):
    """The MX block-scaled decode GEMM (MXFP4 weights x MXFP8 activations): per shape one
    mx_gemm per step, activations given as codes.  Value and roofline over the GEMM's
    algorithmic bytes (codes, scales, activations, Y)."""
    import torch

    ws, rank, _ = dist_info()
    shapes = si.MX_WORKLOADS[workload]
    cases = [si.make_mx_case(**p) for p in shapes]
    gemm_bytes = [si.mx_algorithmic_bytes(c.M, c.N, c.K) for c in cases]
    shape_packed = [w4.mx_packed_bytes(c.N, c.K) for c in cases]
    copies = max(2, -(-3 * L2_BYTES // max(1, sum(shape_packed))))
    bufs = []
    for c, nb in zip(cases, shape_packed):
        first = torch.empty(nb, dtype=torch.uint8, device=device)
        w4.mx_repack(torch.from_numpy(c.w_codes).to(device), torch.from_numpy(c.w_scales).to(device),
                     c.N, c.K, first)
        reps = [first] + [first.clone() for _ in range(copies - 1)]
        ac = torch.from_numpy(c.a_codes).to(device)
        asc = torch.from_numpy(c.a_scales).to(device)
        Y = torch.empty((c.M, c.N), dtype=torch.int16, device=device)
        bufs.append((c, reps, ac, asc, Y))
    st = w4.w4a16_get_device_status(stream)
    if st != 0:
        raise SystemExit(f"{workload}: device status after repack: {w4.status_string(st)}")

    def launch_step(i):
        for c, reps, ac, asc, Y in bufs:
            w4.mx_gemm(ac, asc, reps[i % copies], c.M, c.N, c.K, c.dtype, Y, stream)

    with torch.cuda.stream(stream):
        for i in range(max(3, warmup)):
            launch_step(i)
    per_shape_us = []
    for j, (c, reps, ac, asc, Y) in enumerate(bufs):
        cs = max(3, -(-3 * L2_BYTES // max(1, shape_packed[j])))
        own = list(reps[:cs]) + [reps[0].clone() for _ in range(cs - len(reps))]
        nl = max(20, cs)
        gj = torch.cuda.CUDAGraph()
        with torch.cuda.stream(stream):
            with torch.cuda.graph(gj, stream=stream):
                for i in range(nl):
                    w4.mx_gemm(ac, asc, own[i % cs], c.M, c.N, c.K, c.dtype, Y, stream)
            gj.replay()
            f0, f1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            f0.record(stream)
            for _ in range(3):
                gj.replay()
            f1.record(stream)
        stream.synchronize()
        per_shape_us.append(f0.elapsed_time(f1) * 1e3 / (3 * nl))
        del gj, own
    G = max(1, min(a.graph_steps, steps))
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.stream(stream):
        with torch.cuda.graph(graph, stream=stream):
            for g in range(G):
                launch_step(g)
        graph.replay()
    stream.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    barrier(device)
    torch.cuda.synchronize(device)
    t_wall0 = time.time()
    with torch.cuda.stream(stream):
        e0.record(stream)
        for _ in range(steps // G):
            graph.replay()
        for i in range(steps % G):
            launch_step(i)
        e1.record(stream)
    stream.synchronize()
    t_wall1 = time.time()
    st = w4.w4a16_get_device_status(stream)
    if st != 0:
        raise SystemExit(f"{workload}: device status after timed region: {w4.status_string(st)}")
    elapsed_ms = max_over_ranks(e0.elapsed_time(e1), device)
    del graph
    peaks, peak_kind = measured_peaks()
    hbm_peak = float(peaks["hbm_gbs"])
    dom_bytes = sum(gemm_bytes) / len(gemm_bytes)
    achieved = dom_bytes / (sum(per_shape_us) * 1e-6 / len(per_shape_us)) / 1e9
    step_bytes = sum(gemm_bytes)
    # end to end: per step one pinned-host copy of all shapes' activation codes and scales
    # in, one mx_gemm per shape, one copy of all Y out, on one stream
    host_in = [(torch.from_numpy(c.a_codes).pin_memory(), torch.from_numpy(c.a_scales).pin_memory())
               for c in cases]
    host_y = [torch.empty((c.M, c.N), dtype=torch.int16).pin_memory() for c in cases]
    h2d = sum(x.numel() + y.numel() for x, y in host_in)
    d2h = sum(2 * y.numel() for y in host_y)

    def e2e_step(i):
        for (c, reps, ac, asc, Y), (hx, hs), hy in zip(bufs, host_in, host_y):
            ac.copy_(hx, non_blocking=True)
            asc.copy_(hs, non_blocking=True)
            w4.mx_gemm(ac, asc, reps[i % copies], c.M, c.N, c.K, c.dtype, Y, stream)
            hy.copy_(Y, non_blocking=True)

    e2e_steps = max(1, min(a.e2e_steps, steps))
    with torch.cuda.stream(stream):
        for i in range(3):
            e2e_step(i)
        stream.synchronize()
        f0, f1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        f0.record(stream)
        for i in range(e2e_steps):
            e2e_step(i)
        f1.record(stream)
    stream.synchronize()
    e2e_ms = max_over_ranks(f0.elapsed_time(f1), device)
    out = {
        "workload": workload, "metric": f"MX block-scaled GEMM achieved HBM TB/s ({workload})",
        "value": step_bytes * steps * ws / (elapsed_ms * 1e-3) / 1e12, "unit": "TB/s",
        "ms_per_step": elapsed_ms / steps, "steps": steps, "shapes": len(shapes),
        "step_bytes": step_bytes,
        "l2": f"inputs larger than L2: {copies} rotating copies of the packed weights "
              f"({copies * sum(shape_packed) / 2**20:.0f} MiB per rotation)",
        "roofline": {"bound": "hbm", "achieved": achieved, "peak": hbm_peak, "unit": "GB/s",
                     "frac": achieved / hbm_peak, "traffic": None, "peak_kind": peak_kind,
                     "kernel": "mx_gemm_kernel", "launches_per_step": len(cases),
                     "algorithmic_bytes_per_launch": dom_bytes},
        "per_shape": [{"shape": si.mx_shape_tag(p), "kernel": "mx_gemm_kernel",
                       "us": round(us, 3), "gbs": round(b / (us * 1e-6) / 1e9, 1),
                       "hbm_frac": round(b / (us * 1e-6) / 1e9 / hbm_peak, 4)}
                      for p, us, b in zip(shapes, per_shape_us, gemm_bytes)],
        "e2e": {"value": step_bytes * e2e_steps * ws / (e2e_ms * 1e-3) / 1e12, "unit": "TB/s",
                "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "steps": e2e_steps},
        "kernels_per_step": {"mx_gemm_kernel": len(cases)},
        "gpu_launches": len(cases) * steps,
        "clocks": sampler.summary(t_wall0, t_wall1),
        "note": "E2M1 / E4M3 decoded by cvt into the f16 mma.sync, E8M0 block scales on each "
                "32-value partial sum; not the native block-scaled MMA"}
    del bufs
    torch.cuda.synchronize(device)
    torch.cuda.empty_cache()
    return out


# Workloads timed beside the headline in a default run (M <= 16 decode at 70B scale, the
# batch transition and prefill: the rest of the metric), each with its own roofline.
EXTRA_WORKLOADS = ["ffn70b_decode_bf16", "transition_k8192_n8192",
                   "prefill_m4096_k4096_n11008"]


def run_ours(a):
    import torch

    ws, rank, local = dist_info()
    if not torch.cuda.is_available():
        raise SystemExit("bench.py needs a CUDA device (the library has no CPU path)")
    torch.cuda.set_device(local)
    device = torch.device("cuda", local)
    if ws > 1:
        dist_init("nccl")

    from weight_only_int4_tma_gb300 import build as w4build
    w4build.build()
    import weight_only_int4_tma_gb300 as w4

    ex = dict(kernel=a.kernel, split_k=a.split_k, tile_m=a.tile_m, stages=a.stages,
              flags={"magic": 0, "lut": w4.W4A16_GEMM_DEQUANT_LUT,
                     "int": w4.W4A16_GEMM_DEQUANT_INT}[a.dequant])
    stream = torch.cuda.Stream(device=device)
    sampler = ClockSampler(local)
    sampler.start()
    time.sleep(0.3)

    if a.w4a8_only or a.mx_only:
        name = next(iter(si.MX_WORKLOADS if a.mx_only else si.W4A8_WORKLOADS))
        meas = measure_mx if a.mx_only else measure_w4a8
        x = meas(a, w4, device, stream, sampler, name, a.steps, a.warmup)
        sampler.stop()
        if rank == 0:
            print(json.dumps({
                "metric": x["metric"], "value": x["value"], "unit": x["unit"], "n_gpus": ws,
                "steps": a.steps, "warmup": a.warmup, "ms_per_step": x["ms_per_step"],
                "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
                "dtype": "fp4xfp8" if a.mx_only else "i8", "data": "synthetic",
                "config": {"workload": name, "shapes": x["shapes"], "step_bytes": x["step_bytes"],
                           "l2": x["l2"], "parallelism": f"replicas{ws}"},
                "roofline": x["roofline"], "per_shape": x["per_shape"], "cpu_baseline": None,
                "e2e": x["e2e"], "kernel": x["roofline"]["kernel"],
                "kernels_per_step": x["kernels_per_step"], "gpu_launches": x["gpu_launches"],
                "clocks": x["clocks"], "note": x["note"]}), flush=True)
        return

    shapes = workload_shapes(a)
    m = measure_workload(a, w4, device, stream, sampler, a.workload, shapes, ex, a.steps,
                         a.warmup, a.epilogue)
    extra = []
    if a.extra_workloads and not a.shape and a.epilogue == "none" and not any(ex.values()):
        for name in EXTRA_WORKLOADS:
            if name == a.workload:
                continue
            shp = si.WORKLOADS[name]
            x = measure_workload(a, w4, device, stream, sampler, name, shp, ex, a.steps,
                                 a.warmup)
            extra.append({
                "workload": name, "metric": metric_name(name, shp), "value": x.value,
                "unit": x.unit, "ms_per_step": x.elapsed_ms / x.steps, "steps": x.steps,
                "shapes": len(shp), "step_bytes": x.step_bytes, "step_flops": x.step_flops,
                "l2": f"inputs larger than L2: {x.copies} rotating copies of the packed "
                      f"weights ({x.copies * x.packed_per_step / 2**20:.0f} MiB per rotation)",
                "roofline": x.roofline, "per_shape": x.per_shape, "e2e": x.e2e,
                "kernels_per_step": x.counts, "gpu_launches": x.gpu_launches,
                "clocks": x.clocks})
        for name in si.W4A8_WORKLOADS:
            extra.append(measure_w4a8(a, w4, device, stream, sampler, name, a.steps, a.warmup))
        for name in si.MX_WORKLOADS:
            extra.append(measure_mx(a, w4, device, stream, sampler, name, a.steps, a.warmup))
    time.sleep(0.3)
    sampler.stop()

    cpu = None
    if rank == 0 and ws == 1 and not a.no_cpu_baseline:
        rate, desc, cores, used = cpu_oracle_rate(m.cases, m.shapes, budget_s=12.0)
        cpu = {"value": rate / 1e12, "unit": m.unit, "cores": cores, "kind": "oracle",
               "sample": f"{desc}; {used:.1f} s of CPU time"}

    if rank != 0:
        return
    line = {
        "metric": metric_name(a.workload, shapes),
        "value": m.value, "unit": m.unit, "n_gpus": ws, "steps": a.steps, "warmup": a.warmup,
        "ms_per_step": m.elapsed_ms / a.steps, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f16", "data": "synthetic",
        "config": {"workload": a.workload, "shapes": len(shapes),
                   **({"epilogue": a.epilogue} if a.epilogue != "none" else {}),
                   **({"shape_subset": a.shape} if a.shape else {}),
                   "step_bytes": m.step_bytes,
                   "step_flops": m.step_flops,
                   "l2": f"inputs larger than L2: {m.copies} rotating copies of the packed "
                         f"weights ({m.copies * m.packed_per_step / 2**20:.0f} MiB per rotation)",
                   "timing": f"CUDA graph of {m.G} steps replayed; CUDA events on the launch "
                             f"stream around the whole timed region", "parallelism": f"replicas{ws}",
                   "kernel": a.kernel, "split_k": a.split_k, "tile_m": a.tile_m,
                   "stages": a.stages, **({"dequant": a.dequant} if a.dequant != "magic" else {})},
        "roofline": m.roofline,
        "per_shape": m.per_shape,
        "cpu_baseline": cpu,
        "e2e": m.e2e,
        "kernel": m.dominant,
        "kernels_per_step": m.counts,
        "gpu_launches": m.gpu_launches,
        "clocks": m.clocks,
        "per_workload": extra,
    }
    print(json.dumps(line), flush=True)


def main():
    a = parse()
    if a.impl == "reference":
        run_reference(a)
    else:
        run_ours(a)
    import torch.distributed as dist
    if dist.is_available() and dist.is_initialized():
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
