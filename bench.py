#!/usr/bin/env python3
"""Throughput of the FP32 GEMM library on one GB300 (or N independent replicas).

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

One "step" is one C = alpha*op(A)*op(B) + beta*C call of the headline
workload: M = N = K = 4096, op = NN, A and B i.i.d. standard normal drawn from
seed 2, alpha = 1, beta = 0 (the largest case of the 512..4096 square sweep;
FLOPs per step = 2*M*N*K).  Inputs are resident in HBM when the timed region
starts; A + B + C = 192 MiB, more than the 129 MB L2, so no extra L2 flush is
done between steps.  Rank 0 prints ONE JSON line.

Keys beyond the throughput: ``e2e`` (the same metric through the C ABI with
every step's operands copied from pinned host memory and its result copied
back inside the timed region; the copies of neighbouring steps overlap a
step's product on separate streams, and the fully serial loop is reported in
``e2e.serial``), ``roofline`` (the dominant kernel's FLOP rate against the FP32
CUDA-core peak 2 * 128 * SMs * f_SM, at the 2070 MHz maximum SM clock),
``cpu_baseline`` (the CPU oracle timed on a bounded sample of the same product
on this host's cores), ``clocks`` (nvidia-smi samples taken during the timed
region), ``vs_size`` (TFLOP/s of the 512..4096 square sweep), ``configs``
(TFLOP/s of the other workload families; both from back-to-back eager calls),
``configs_graph`` (the same families' device time per call from CUDA-graph
replays, without the host's per-call cost), ``tensor_core_3xtf32`` (the
tensor-core kernel on the headline product), ``transpose`` (the transpose
kernel's HBM bandwidth at 4096 x 4096 and 16384 x 16384) and
``library_context`` (cuBLAS FP32 on the headline product, for context),
``strided_batched`` (a per-head attention Q K^T batch through
sgemm_strided_batched) and ``ladder`` (the pages' naive and 16 x 16
shared-memory-tiled kernels against the default path at 2048^3).

``--impl reference`` times the CPU oracle instead (the only other use of the
oracle here), on a bounded sample per step, and prints the same JSON line with
"impl": "reference".  Under torchrun with N > 1 only rank 0 runs it.
"""
import argparse
import hashlib
import glob
import json
import math
import os
import re
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

FP32_LANES_PER_SM = 128          # FP32 FMA units per Blackwell SM
RECIPE_SM_MAX_MHZ = 2070.0       # maximum SM clock of this GB300 pool
L2_BYTES = 129e6
NOMINAL_TF32_OVER_BF16 = 1.1 / 2.25   # dense tensor rates, GB300 nominal
FALLBACK_BF16_TFLOPS = 1900.0         # used only if no measured peak file
FALLBACK_HBM_GBS = 6800.0


# ----------------------------------------------------------------- helpers
# Sources each kernel family is built from; a stored ncu traffic figure is
# only used while the hash of its family's sources still matches.
KERNEL_SOURCES = {
    "simt": ["ptx.cuh", "internal.h", "simt_gemm.cuh", "simt_instances.cuh", "simt_tma_an.cu",
             "simt_tma_at.cu", "simt_cpasync_an.cu", "simt_cpasync_at.cu", "sk_fixup.cu"],
    "tc_3xtf32": ["ptx.cuh", "tc_3xtf32.cuh", "tc_3xtf32_pair.cuh", "tc_3xtf32.cu"],
    "transpose": ["transpose.cu"],
}


def kernel_source_hash(family: str) -> str:
    h = hashlib.sha256()
    for name in KERNEL_SOURCES[family]:
        path = os.path.join(ROOT, "dense_fp32_matrix_10_gb300", "csrc", name)
        h.update(name.encode())
        h.update(open(path, "rb").read())
    return h.hexdigest()[:16]


def stored_traffic(kernel_tag: str):
    """(bytes per launch, note) from the record of `kernel_tag` in
    profiles/traffic.json, if the hash of its family's sources still matches
    the one the capture was taken on."""
    family = next((f for f in ("tc_3xtf32", "transpose") if kernel_tag.startswith(f)), "simt")
    want = kernel_source_hash(family)
    try:
        records = json.load(open(os.path.join(ROOT, "profiles", "traffic.json")))["records"]
    except (OSError, ValueError, KeyError):
        return None, "no traffic records"
    rec = records.get(kernel_tag)
    if rec is None:
        return None, "no capture"
    if rec.get("source_hash") != want:
        return None, f"stale ({rec.get('summary')} taken on {rec.get('source_hash')}, now {want})"
    return int(rec["dram_bytes_per_launch"]), rec.get("summary")


def measured_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        return json.load(open(path))
    except (OSError, ValueError):
        return {}


class NvmlClockSampler:
    """SM clock, power and clock-event reasons read through NVML (the driver's
    libnvidia-ml, read-only queries) every 10 ms in a background thread, so
    that a timed region of a few tens of milliseconds still holds several
    samples; timestamps keep only the samples inside it.  Raises OSError where
    NVML cannot be loaded or the device not found (ClockSampler is then
    used)."""

    # clock-event reason bits of nvmlDeviceGetCurrentClocksEventReasons
    REASONS = {0x4: "sw_power_cap", 0x8: "hw_slowdown", 0x20: "sw_thermal_slowdown",
               0x40: "hw_thermal_slowdown", 0x80: "hw_power_brake_slowdown"}

    def __init__(self, gpu_uuid, period_s=0.01):
        import ctypes
        self.ct = ctypes
        try:
            self.nvml = ctypes.CDLL("libnvidia-ml.so.1")
        except OSError as e:
            raise OSError(f"NVML not loadable: {e}")
        if self.nvml.nvmlInit_v2() != 0:
            raise OSError("nvmlInit failed")
        self.handle = ctypes.c_void_p()
        if not gpu_uuid or self.nvml.nvmlDeviceGetHandleByUUID(
                gpu_uuid.encode(), ctypes.byref(self.handle)) != 0:
            raise OSError("device not found through NVML")
        fn = getattr(self.nvml, "nvmlDeviceGetCurrentClocksEventReasons", None)
        self.reasons_fn = fn or self.nvml.nvmlDeviceGetCurrentClocksThrottleReasons
        self.period = period_s
        self.samples = []
        self.stop_flag = threading.Event()
        self.thread = None

    def _sample(self):
        ct = self.ct
        sm, mx, pw, rs = ct.c_uint(), ct.c_uint(), ct.c_uint(), ct.c_ulonglong()
        ok = (self.nvml.nvmlDeviceGetClockInfo(self.handle, 1, ct.byref(sm)) == 0 and
              self.nvml.nvmlDeviceGetMaxClockInfo(self.handle, 1, ct.byref(mx)) == 0)
        if not ok:
            return None
        power = pw.value / 1000.0 if self.nvml.nvmlDeviceGetPowerUsage(self.handle, ct.byref(pw)) == 0 \
            else None
        bits = rs.value if self.reasons_fn(self.handle, ct.byref(rs)) == 0 else 0
        return (float(sm.value), float(mx.value), power, bits)

    def _run(self):
        while not self.stop_flag.is_set():
            smp = self._sample()
            if smp is not None:
                self.samples.append((time.time(), smp))
            self.stop_flag.wait(self.period)

    def start(self):
        self.thread = threading.Thread(target=self._run, daemon=True)
        self.thread.start()
        return self

    def stop(self):
        self.stop_flag.set()
        if self.thread is not None:
            self.thread.join(timeout=5)
        self.nvml.nvmlShutdown()

    def summary(self, t0: float, t1: float):
        inside = [p for (t, p) in self.samples if t0 <= t <= t1]
        window = "timed region"
        if not inside:
            near = sorted(self.samples, key=lambda s: min(abs(s[0] - t0), abs(s[0] - t1)))[:3]
            inside = [p for (_, p) in near]
            window = "nearest samples (timed region shorter than the sampling period)"
        if not inside:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["NVML gave no samples"],
                    "samples": 0, "source": "nvml"}
        pw = [p[2] for p in inside if p[2] is not None]
        reasons = sorted({name for p in inside for bit, name in self.REASONS.items() if p[3] & bit})
        return {"sm_mhz": statistics.median(p[0] for p in inside),
                "sm_max_mhz": max(p[1] for p in inside),
                "power_w_median": statistics.median(pw) if pw else None,
                "reasons": reasons, "samples": len(inside), "window": window,
                "source": "nvml, 10 ms"}


def clock_sampler(uuid):
    """NVML sampler where NVML is available, else nvidia-smi's."""
    try:
        return NvmlClockSampler(uuid)
    except (OSError, AttributeError):
        return ClockSampler(uuid)


class ClockSampler:
    """nvidia-smi samples every 100 ms in a background process; timestamps let
    us keep only the samples inside the timed region."""

    FIELDS = ("timestamp,index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_id):
        self.samples = []
        self.proc = None
        self.thread = None
        self.gpu = gpu_id

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "100", *(["-i", str(self.gpu)] if self.gpu is not None else [])],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except (OSError, ValueError):
            self.proc = None
            return self
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()
        return self

    def _read(self):
        for ln in self.proc.stdout:
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) >= 10:
                self.samples.append((time.time(), parts))

    def stop(self):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
        if self.thread is not None:
            self.thread.join(timeout=5)

    def summary(self, t0: float, t1: float):
        inside = [p for (t, p) in self.samples if t0 <= t <= t1]
        window = "timed region"
        if not inside:  # region shorter than one sample: take the nearest ones
            near = sorted(self.samples, key=lambda s: min(abs(s[0] - t0), abs(s[0] - t1)))[:3]
            inside = [p for (_, p) in near]
            window = "nearest samples (timed region shorter than the sampling period)"
        if not inside:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"],
                    "samples": 0}

        def num(x):
            try:
                return float(x)
            except ValueError:
                return None
        sm = [num(p[2]) for p in inside if num(p[2]) is not None]
        mx = [num(p[3]) for p in inside if num(p[3]) is not None]
        pw = [num(p[4]) for p in inside if num(p[4]) is not None]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for p in inside for i in range(4) if p[6 + i] == "Active"})
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(mx) if mx else None,
                "power_w_median": statistics.median(pw) if pw else None,
                "reasons": reasons, "samples": len(inside), "window": window,
                "source": "nvidia-smi, 100 ms"}


# ----------------------------------------------------------------- distributed
class Dist:
    def __init__(self):
        self.world = int(os.environ.get("WORLD_SIZE", "1"))
        self.rank = int(os.environ.get("RANK", "0"))
        self.local_rank = int(os.environ.get("LOCAL_RANK", "0"))
        self.pg = None

    def init(self, backend):
        if self.world > 1:
            import torch.distributed as dist
            dist.init_process_group(backend=backend)
            self.pg = dist

    def barrier(self):
        if self.pg is not None:
            self.pg.barrier()

    def max(self, value: float, device=None) -> float:
        """Maximum of `value` over ranks (the slowest rank sets the time)."""
        if self.pg is None:
            return value
        import torch
        t = torch.tensor([value], dtype=torch.float64, device=device)
        self.pg.all_reduce(t, op=self.pg.ReduceOp.MAX)
        return float(t.item())

    def close(self):
        if self.pg is not None:
            self.pg.destroy_process_group()


# ----------------------------------------------------------------- GPU timing
def time_gemm(sg, torch, case, A, B, C, steps, warmup, algo, stream, record_launches=False,
              per_call_events=True):
    """Warm up, then time `steps` back-to-back calls with CUDA events on
    `stream`.  Returns (ms per step from the region, mean per-launch ms from
    per-call events -- None without them --, launches counted).  Small
    products are host-bound: their region is timed without per-call events."""
    for _ in range(warmup):
        sg.gemm(A, B, C, case.alpha, case.beta, case.transA, case.transB, algo=algo, stream=stream)
    torch.cuda.synchronize()
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
          for _ in range(steps if per_call_events else 0)]
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    launches = 0
    start.record(stream)
    for i in range(steps):
        if per_call_events:
            ev[i][0].record(stream)
        sg.gemm(A, B, C, case.alpha, case.beta, case.transA, case.transB, algo=algo, stream=stream)
        if per_call_events:
            ev[i][1].record(stream)
        if record_launches:
            launches += sg.sgemm_last_launch_count()
    end.record(stream)
    torch.cuda.synchronize()
    region = start.elapsed_time(end) / steps
    calls = [a.elapsed_time(b) for a, b in ev]
    per_launch = sum(calls) / steps if per_call_events else None
    time_gemm.last_calls = calls   # per-call ms of the last timed region
    return region, per_launch, launches


def time_gemm_graph(sg, torch, case, A, B, C, algo, calls=20, replays=5):
    """Device time per call without host gaps: `calls` calls captured in one
    CUDA graph on a side stream (after an eager call there has sized the
    library's buffers), the graph replayed `replays` times between two CUDA
    events on that stream."""
    cs = torch.cuda.Stream()
    torch.cuda.synchronize()
    sg.gemm(A, B, C, case.alpha, case.beta, case.transA, case.transB, algo=algo, stream=cs)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=cs):
        for _ in range(calls):
            sg.gemm(A, B, C, case.alpha, case.beta, case.transA, case.transB, algo=algo,
                    stream=cs)
    with torch.cuda.stream(cs):
        g.replay()
    torch.cuda.synchronize()
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(cs):
        start.record(cs)
        for _ in range(replays):
            g.replay()
        end.record(cs)
    torch.cuda.synchronize()
    return start.elapsed_time(end) / (calls * replays)


def time_transpose(sg, torch, rows, cols, reps, stream, flush=None, read_back=False):
    """(mean, median) per-launch ms of sgemm_transpose on a rows x cols matrix:
    CUDA events around each launch on `stream`, the device synchronised after
    each timed launch.  `flush`, a buffer larger than L2, is rewritten before
    each launch, outside the events, and with `read_back` then read once more,
    so that the dirty lines the write left in L2 are written back before the
    timed launch instead of during it.  A short device-side spin is queued
    ahead of the first event, so that the host has enqueued the launch before
    the GPU reaches that event: the interval is the kernel's, not the host's
    launch latency."""
    X = torch.randn(rows, cols, device=stream.device)
    Y = torch.empty(cols, rows, device=stream.device)
    for _ in range(3):
        sg.transpose(X, Y, stream=stream)
    spin = getattr(torch.cuda, "_sleep", None)
    times = []
    with torch.cuda.stream(stream):
        for _ in range(reps):
            torch.cuda.synchronize()
            if flush is not None:
                flush.fill_(1.0)
                if read_back:
                    flush.sum()
            if spin is not None:
                spin(200_000)   # ~0.1 ms of GPU clock cycles
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record(stream)
            sg.transpose(X, Y, stream=stream)
            b.record(stream)
            torch.cuda.synchronize()
            times.append(a.elapsed_time(b))
    ok = bool(torch.equal(Y, X.t()))
    del X, Y
    times.sort()
    return sum(times) / reps, times[reps // 2], ok


def measure_tf32_peak(torch, dev, n=8192, reps=10):
    """TF32 tensor throughput of this GPU as cuBLAS delivers it: torch.matmul
    of two n x n FP32 matrices with TF32 allowed, best of `reps` (CUDA events).
    A library run (not inspected), used only as the roofline denominator of
    the 3xTF32 kernel.  None if it cannot run."""
    prev = torch.backends.cuda.matmul.allow_tf32
    try:
        torch.backends.cuda.matmul.allow_tf32 = True
        X = torch.randn(n, n, device=dev)
        Y = torch.randn(n, n, device=dev)
        Z = torch.empty(n, n, device=dev)
        for _ in range(3):
            torch.mm(X, Y, out=Z)
        best = float("inf")
        for _ in range(reps):
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record()
            torch.mm(X, Y, out=Z)
            e1.record()
            e1.synchronize()
            best = min(best, e0.elapsed_time(e1))
        del X, Y, Z
        return 2.0 * n ** 3 / (best * 1e-3) / 1e12
    except RuntimeError:
        return None
    finally:
        torch.backends.cuda.matmul.allow_tf32 = prev


def tflops(flops, ms):
    return flops / (ms * 1e-3) / 1e12


def job_rate(dist, flops_per_rank: float, ms_this_rank: float, device=None):
    """Whole-job rate over replicas: every rank did `flops_per_rank`, the job
    took as long as its slowest rank.  Returns (max ms over ranks, TFLOP/s of
    all ranks together)."""
    ms = dist.max(ms_this_rank, device)
    return ms, flops_per_rank * dist.world / (ms * 1e-3) / 1e12


def run_ours(args, dist):
    import torch
    import dense_fp32_matrix_10_gb300 as sg
    from dense_fp32_matrix_10_gb300 import workloads as W

    torch.cuda.set_device(dist.local_rank)
    dev = torch.device("cuda", dist.local_rank)
    dist.init("nccl")
    props = torch.cuda.get_device_properties(dev)
    sms = props.multi_processor_count
    stream = torch.cuda.current_stream(dev)

    case = {c.name: c for c in W.ALL_CASES}[args.workload] if args.workload else W.HEADLINE
    A, B, C = (t.to(dev) for t in W.make_inputs(case))
    flops = case.flops

    # ---- device-resident timed region
    uuid = str(getattr(props, "uuid", "") or "")
    sampler = clock_sampler(("GPU-" + uuid) if uuid and not uuid.startswith("GPU-") else (uuid or None))
    sampler.start()
    for _ in range(args.warmup):
        sg.gemm(A, B, C, case.alpha, case.beta, case.transA, case.transB, algo=args.algo, stream=stream)
    torch.cuda.synchronize()
    dist.barrier()
    torch.cuda.synchronize()
    t_wall0 = time.time()
    ms_region, ms_launch, launches = time_gemm(sg, torch, case, A, B, C, args.steps, 0, args.algo,
                                               stream, record_launches=True)
    calls = sorted(time_gemm.last_calls)
    t_wall1 = time.time()
    dist.barrier()
    sampler.stop()
    clocks = sampler.summary(t_wall0, t_wall1)
    # the timed steps' output (every step writes the same C), kept for the
    # parity check against the oracle's rows below
    C_timed = C.cpu().numpy() if dist.rank == 0 and not args.no_cpu_baseline else None
    ms_step, value = job_rate(dist, flops, ms_region, dev)

    # ---- end to end through the C ABI: pinned host operands in, result out.
    # Every step copies its A and B from pinned host memory, runs the product
    # and copies its C back.  Pipelined: two device buffer sets and three
    # streams (H2D, product, D2H) ordered by events, so the copies of
    # neighbouring steps overlap a step's product, as a serving loop would run;
    # the fully serial loop (one stream) is reported beside it.
    e2e = None
    e2e_steps = max(3, min(args.steps, 30)) if not args.no_e2e else 0
    if e2e_steps:
        hA = torch.empty(A.shape, dtype=torch.float32, pin_memory=True)
        hB = torch.empty(B.shape, dtype=torch.float32, pin_memory=True)
        hA.copy_(A)
        hB.copy_(B)
        hC = [torch.empty(C.shape, dtype=torch.float32, pin_memory=True) for _ in range(2)]
        dA = [A, torch.empty_like(A)]
        dB = [B, torch.empty_like(B)]
        dC = [C, torch.empty_like(C)]
        s_in, s_out = torch.cuda.Stream(dev), torch.cuda.Stream(dev)
        ev = lambda: torch.cuda.Event()
        ev_in, ev_comp, ev_out = [ev(), ev()], [ev(), ev()], [ev(), ev()]
        used = [False, False]

        def step(i):
            k = i % 2
            with torch.cuda.stream(s_in):
                if used[k]:
                    s_in.wait_event(ev_comp[k])          # the product of step i-2 read dA/dB[k]
                dA[k].copy_(hA, non_blocking=True)
                dB[k].copy_(hB, non_blocking=True)
                ev_in[k].record(s_in)
            stream.wait_event(ev_in[k])
            if used[k]:
                stream.wait_event(ev_out[k])             # C[k] of step i-2 has been copied out
            sg.gemm(dA[k], dB[k], dC[k], case.alpha, case.beta, case.transA, case.transB,
                    algo=args.algo, stream=stream)
            ev_comp[k].record(stream)
            with torch.cuda.stream(s_out):
                s_out.wait_event(ev_comp[k])
                hC[k].copy_(dC[k], non_blocking=True)
                ev_out[k].record(s_out)
            used[k] = True

        for i in range(2):
            step(i)
        torch.cuda.synchronize()
        dist.barrier()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        s_in.wait_event(e0)
        for i in range(2, 2 + e2e_steps):
            step(i)
        stream.wait_event(ev_out[(1 + e2e_steps) % 2])   # the last step's result is on the host
        stream.wait_event(ev_out[e2e_steps % 2])
        e1.record(stream)
        torch.cuda.synchronize()
        ms_e2e, e2e_rate = job_rate(dist, flops, e0.elapsed_time(e1) / e2e_steps, dev)

        # the fully serial loop: copy in, product, copy out on one stream
        s0, s1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        torch.cuda.synchronize()
        s0.record(stream)
        with torch.cuda.stream(stream):
            for _ in range(e2e_steps):
                A.copy_(hA, non_blocking=True)
                B.copy_(hB, non_blocking=True)
                sg.gemm(A, B, C, case.alpha, case.beta, case.transA, case.transB, algo=args.algo,
                        stream=stream)
                hC[0].copy_(C, non_blocking=True)
        s1.record(stream)
        torch.cuda.synchronize()
        ms_serial, serial_rate = job_rate(dist, flops, s0.elapsed_time(s1) / e2e_steps, dev)
        e2e = {"value": round(e2e_rate, 3), "unit": "TFLOP/s",
               "ms_per_step": round(ms_e2e, 4),
               "h2d_bytes_per_step": int(A.numel() * 4 + B.numel() * 4),
               "d2h_bytes_per_step": int(C.numel() * 4),
               "how": "pipelined: H2D / product / D2H on three streams, two buffer sets",
               "serial": {"value": round(serial_rate, 3), "ms_per_step": round(ms_serial, 4),
                          "how": "one stream: copy in, product, copy out"}}
        del dA[1], dB[1], dC[1]

    # ---- roofline of the dominant (only) kernel of a step
    peaks = measured_peaks()
    sm_max = float(peaks.get("sm_max_mhz") or RECIPE_SM_MAX_MHZ)
    peak = 2 * FP32_LANES_PER_SM * sms * sm_max * 1e6 / 1e12
    achieved = tflops(flops, ms_launch)
    algo_used = sg.sgemm_algo_name(sg.sgemm_select_algo(
        case.transA, case.transB, case.M, case.N, case.K, A.data_ptr(), A.stride(0), B.data_ptr(), B.stride(0),
        case.alpha, case.beta, C.data_ptr(), C.stride(0))) if args.algo == "auto" else args.algo
    tag = f"{algo_used}_{case.name}"
    traffic, traffic_src = stored_traffic(tag)
    roofline = {"bound": "alu", "achieved": round(achieved, 3), "peak": round(peak, 3),
                "unit": "TFLOP/s", "frac": round(achieved / peak, 4), "traffic": traffic,
                "peak_basis": f"FP32 FFMA: 2 x {FP32_LANES_PER_SM} lanes x {sms} SMs x {sm_max:.0f} MHz "
                              "(derived from unit counts and the maximum SM clock)",
                "kernel": tag, "traffic_source": traffic_src,
                "algorithmic_flops_per_launch": flops,
                "algorithmic_bytes_per_launch": int(4 * (case.M * case.K + case.K * case.N + case.M * case.N))}
    if clocks.get("sm_mhz"):
        roofline["frac_at_observed_clock"] = round(
            achieved / (2 * FP32_LANES_PER_SM * sms * clocks["sm_mhz"] * 1e6 / 1e12), 4)

    # ---- the tensor-core (3xTF32) kernel on the same workload
    tensor = None
    if not args.no_tensor:
        try:
            r, kms, _ = time_gemm(sg, torch, case, A, B, C, max(5, min(args.steps, 200)), 3,
                                  "tc_3xtf32", stream)
            tf32_meas = measure_tf32_peak(torch, dev)
            bf16 = float(peaks.get("bf16_tflops") or FALLBACK_BF16_TFLOPS)
            tf32_nominal = bf16 * NOMINAL_TF32_OVER_BF16
            tf32_peak = tf32_meas or tf32_nominal
            ach = tflops(flops, kms)
            tensor = {"value": round(tflops(flops, r), 3), "unit": "TFLOP/s",
                      "ms_per_step": round(r, 5), "algo": "tc_3xtf32",
                      "roofline": {"bound": "tensor", "achieved": round(ach, 3),
                                   "peak": round(tf32_peak, 1), "unit": "TFLOP/s",
                                   "frac": round(ach / tf32_peak, 4),
                                   "traffic": stored_traffic(f"tc_3xtf32_{case.name}")[0],
                                   "peak_basis": ("measured: cuBLAS TF32 (torch.matmul, allow_tf32) at "
                                                  "8192^3, best of 10, in this run"
                                                  if tf32_meas else
                                                  "TF32 dense = measured bf16 burst "
                                                  f"{bf16:.1f} x nominal 1.1/2.25"
                                                  + ("" if peaks.get("bf16_tflops") else " (fallback)")),
                                   "peak_nominal_from_bf16": round(tf32_nominal, 1),
                                   "peak_fp32_equivalent": round(tf32_peak / 3, 1),
                                   "frac_fp32_equivalent": round(3 * ach / tf32_peak, 4),
                                   "note": "3 TF32 MMAs per FP32 product; achieved counts 2MNK"}}
        except sg.SgemmError as e:
            tensor = {"unavailable": str(e)}

    # ---- the transpose kernel (the transpose page's 4096 x 4096 case, L2
    # flushed between launches, and a 1 GiB case larger than L2)
    transpose = None
    if not args.no_transpose:
        hbm = float(peaks.get("hbm_gbs") or FALLBACK_HBM_GBS)
        flush = torch.empty(64 * 1024 * 1024, device=dev)    # 256 MiB > L2
        transpose = {}
        for rows, cols, fl in ((4096, 4096, flush), (16384, 16384, None)):
            ms, ms_median, ok = time_transpose(sg, torch, rows, cols, 40, stream, fl,
                                               read_back=fl is not None)
            ms_dirty = (time_transpose(sg, torch, rows, cols, 40, stream, fl)[0]
                        if fl is not None else None)
            gbs = 8.0 * rows * cols / (ms * 1e-3) / 1e9
            transpose[f"{rows}x{cols}"] = {
                "ms": round(ms, 5), "ms_median": round(ms_median, 5), "same_as_torch_t": ok,
                "roofline": {"bound": "hbm", "achieved": round(gbs, 1), "peak": hbm,
                             "unit": "GB/s", "frac": round(gbs / hbm, 4),
                             "traffic": stored_traffic(f"transpose_{rows}x{cols}")[0],
                             "algorithmic_bytes_per_launch": 8 * rows * cols,
                             "peak_basis": "measured copy bandwidth" if peaks.get("hbm_gbs")
                                           else "fallback",
                             "l2": ("flushed between launches: 256 MiB written, then read "
                                    "(clean L2; the write's dirty lines are written back "
                                    "before the timed launch)") if fl is not None
                                   else "2 GiB per launch, larger than L2"}}
            if ms_dirty is not None:
                transpose[f"{rows}x{cols}"]["after_write_only_flush"] = {
                    "ms": round(ms_dirty, 5),
                    "gbs": round(8.0 * rows * cols / (ms_dirty * 1e-3) / 1e9, 1),
                    "note": "256 MiB written between launches, not read back: the launch also "
                            "writes back the flush's dirty L2 lines"}
        del flush

    # ---- strided batch (attention Q K^T shape) and the pages' kernel ladder
    batched = None
    if not args.no_batched:
        bt, bm_, bn_, bk_ = 96, 512, 512, 64
        Q = torch.randn(bt, bm_, bk_, device=dev)
        Kt = torch.randn(bt, bn_, bk_, device=dev)
        S = torch.empty(bt, bm_, bn_, device=dev)
        for _ in range(3):
            sg.gemm_strided_batched(Q, Kt, S, transB=True, stream=stream)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        torch.cuda.synchronize()
        e0.record(stream)
        for _ in range(50):
            sg.gemm_strided_batched(Q, Kt, S, transB=True, stream=stream)
        e1.record(stream)
        torch.cuda.synchronize()
        bms = e0.elapsed_time(e1) / 50
        bach = tflops(2.0 * bt * bm_ * bn_ * bk_, bms)
        batched = {"workload": f"{bt} x ({bm_}x{bk_}) . ({bk_}x{bn_})^T, NT (per-head Q K^T)",
                   "value": round(bach, 3), "unit": "TFLOP/s", "ms": round(bms, 5),
                   "roofline": {"bound": "alu", "achieved": round(bach, 3), "peak": round(peak, 3),
                                "unit": "TFLOP/s", "frac": round(bach / peak, 4),
                                "traffic": stored_traffic(f"simt_tma_nt_batch{bt}_{bm_}x{bn_}x{bk_}")[0],
                                "algorithmic_bytes_per_launch": 4 * bt * (bm_ * bk_ + bn_ * bk_ + bm_ * bn_)}}
        del Q, Kt, S
    ladder = None
    if not args.no_ladder:
        n = 2048
        La, Lb = torch.randn(n, n, device=dev), torch.randn(n, n, device=dev)
        Lc = torch.empty(n, n, device=dev)
        ladder = {"workload": f"{n}^3 NN", "unit": "TFLOP/s"}
        for algo_name in ("naive", "smem_tiled", "reg_2x2", "reg_4x4", "auto"):
            sg.gemm(La, Lb, Lc, algo=algo_name, stream=stream)
            reps = 3 if algo_name != "auto" else 20
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            torch.cuda.synchronize()
            e0.record(stream)
            for _ in range(reps):
                sg.gemm(La, Lb, Lc, algo=algo_name, stream=stream)
            e1.record(stream)
            torch.cuda.synchronize()
            ladder[algo_name] = round(tflops(2.0 * n ** 3, e0.elapsed_time(e1) / reps), 3)
        ladder["speedup_auto_over_naive"] = round(ladder["auto"] / ladder["naive"], 1)
        for rung in ("smem_tiled", "reg_2x2", "reg_4x4"):
            ladder[f"speedup_{rung}_over_naive"] = round(ladder[rung] / ladder["naive"], 2)
        del La, Lb, Lc

    # ---- the ownership contract: the same products with the library's scratch
    # limit at 0 (no workspace, nothing copied ahead), then the limit restored
    limit0 = None
    if not args.no_limit0:
        limit0 = {"what": "sgemm_set_scratch_limit(0): no library device memory; split tiles only "
                          "within clusters (else whole tiles), operands read in place"}
        sq = W.SQUARE_1024
        qA, qB, qC = (t.to(dev) for t in W.make_inputs(sq))
        # limit 0 first: no graph has used the library's buffers yet, so the
        # limit frees them all (a buffer a graph holds would stay and be reused)
        for lim_name, lim in (("limit_0", 0), ("unlimited", sg.SCRATCH_UNLIMITED)):
            sg.sgemm_set_scratch_limit(lim)
            r, _, _ = time_gemm(sg, torch, case, A, B, C, max(5, min(args.steps, 50)), 3, args.algo,
                                stream, per_call_events=False)
            us = 1000 * time_gemm_graph(sg, torch, sq, qA, qB, qC, args.algo)
            limit0[lim_name] = {case.name + "_tflops": round(tflops(flops, r), 3),
                                sq.name + "_graph_us": round(us, 2),
                                "library_bytes_held": int(sg.sgemm_get_scratch_limit()[1])}
        sg.sgemm_set_scratch_limit(sg.SCRATCH_UNLIMITED)
        del qA, qB, qC

    # ---- library context: cuBLAS FP32 (TF32 off) on the headline product
    library_context = None
    if not args.no_library_context:
        prev = torch.backends.cuda.matmul.allow_tf32
        torch.backends.cuda.matmul.allow_tf32 = False
        opA = A.t() if case.transA else A
        opB = B.t() if case.transB else B
        out = torch.empty(case.M, case.N, device=dev)
        for _ in range(3):
            torch.mm(opA, opB, out=out)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        torch.cuda.synchronize()
        e0.record()
        for _ in range(20):
            torch.mm(opA, opB, out=out)
        e1.record()
        torch.cuda.synchronize()
        torch.backends.cuda.matmul.allow_tf32 = prev
        library_context = {"cublas_fp32_tflops": round(tflops(flops, e0.elapsed_time(e1) / 20), 3),
                           "what": "torch.mm FP32, TF32 off (cuBLAS), same product; context only"}
        del out

    # ---- TFLOP/s vs size and the other workload families (rank 0 context)
    vs_size, families, families_graph = {}, {}, {}
    if not args.no_sweep:
        for sc in W.SWEEP:
            sA, sB, sC = (t.to(dev) for t in W.make_inputs(sc))
            n = max(5, min(200, int(2e11 / sc.flops)))
            r, _, _ = time_gemm(sg, torch, sc, sA, sB, sC, n, 3, args.algo, stream,
                                per_call_events=False)
            vs_size[str(sc.M)] = round(tflops(sc.flops, r), 3)
            del sA, sB, sC
        for sc in [W.SMALL_256, W.SQUARE_1024, W.NT_4096, *W.RAGGED]:
            sA, sB, sC0 = (t.to(dev) for t in W.make_inputs(sc))
            sC = sC0.clone()
            n = max(5, min(200, int(2e11 / sc.flops)))
            # beta != 0 updates C in place each call; the values drift but the
            # work per call is identical.
            r, _, _ = time_gemm(sg, torch, sc, sA, sB, sC, n, 3, args.algo, stream,
                                per_call_events=False)
            families[sc.name] = round(tflops(sc.flops, r), 3)
            us = 1000 * time_gemm_graph(sg, torch, sc, sA, sB, sC, args.algo)
            families_graph[sc.name] = {"us_per_call": round(us, 2),
                                       "tflops": round(tflops(sc.flops, us / 1000), 3)}
            del sA, sB, sC, sC0

    result = {
        "metric": "SGEMM FP32 TFLOP/s at 4096^3 (NN) and % of GB300 FP32 peak; TFLOP/s vs size",
        "value": round(value, 3), "unit": "TFLOP/s", "n_gpus": dist.world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(ms_step, 5), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f32",
        "data": "synthetic: seeded i.i.d. standard normal A, B (torch CPU generator, seed 2)",
        "config": {"workload": case.name, "M": case.M, "N": case.N, "K": case.K,
                   "op": "NT"[case.transA] + "NT"[case.transB],
                   "alpha": case.alpha, "beta": case.beta, "algo": algo_used,
                   "l2": "inputs (192 MiB) larger than L2 (129 MB); no flush between steps",
                   "parallelism": "replicas" if dist.world > 1 else "single GPU"},
        "pct_of_fp32_peak": round(100 * achieved / peak, 2),
        "per_call_ms": {"min": round(calls[0], 5), "median": round(calls[len(calls) // 2], 5),
                        "max": round(calls[-1], 5), "calls": len(calls)} if calls else None,
        "e2e": e2e, "roofline": roofline, "clocks": clocks, "gpu_launches": launches,
        "tensor_core_3xtf32": tensor, "transpose": transpose,
        "strided_batched": batched, "ladder": ladder,
        "library_context": library_context, "scratch_limit_0": limit0,
        "vs_size": vs_size, "configs": families,
        "configs_graph": families_graph or None,
        "device": {"name": props.name, "sms": sms, "cc": f"{props.major}.{props.minor}"},
    }
    if dist.rank == 0 and not args.no_cpu_baseline:
        result["cpu_baseline"] = cpu_baseline(case, A, B, seconds=args.cpu_seconds,
                                              keep_result=True)
        R = result["cpu_baseline"].pop("_result")
        if case.beta == 0.0:   # the sampled oracle rows are alpha * op(A) * op(B)
            result["parity"] = parity_stats(C_timed[:R.shape[0]], R, case.K)
    dist.close()
    return result


def parity_stats(G, R, K):
    """The timed output against the oracle's rows: relative Frobenius error
    and largest elementwise error, beside the tolerance the tests apply
    (1e-5 relative, 1e-4 * sqrt(K) absolute)."""
    import numpy as np
    G = G.astype(np.float64)
    diff = G - R
    rel = float(np.linalg.norm(diff) / max(np.linalg.norm(R), 1e-300))
    mx = float(np.max(np.abs(diff))) if diff.size else 0.0
    tol_abs = 1e-4 * float(np.sqrt(K))
    return {"rows": int(R.shape[0]), "rel_fro": rel, "max_abs": mx, "tol_rel_fro": 1e-5,
            "tol_max_abs": tol_abs, "within_tolerance": bool(rel <= 1e-5 and mx <= tol_abs),
            "what": "the timed steps' C against the FP64 oracle on the same rows"}


# ----------------------------------------------------------------- CPU oracle
def cpu_baseline(case, A=None, B=None, seconds=12.0, rows=None, keep_result=False):
    """The CPU oracle (as it stands) on the first `rows` output rows of the
    product, all columns, on every core this process may use (with
    keep_result, its output rides along under "_result")."""
    import numpy as np
    import oracle
    from dense_fp32_matrix_10_gb300 import workloads as W
    if A is None:
        A, B, _ = W.make_inputs(case)
    An = A.cpu().numpy() if hasattr(A, "cpu") else A
    Bn = B.cpu().numpy() if hasattr(B, "cpu") else B
    threads = oracle.default_threads()
    orc = oracle.default()
    if rows is None:  # calibrate on a small block, then size the sample to ~`seconds`
        probe = max(threads, 16)
        t0 = time.perf_counter()
        orc.sgemm_f64(case.transA, case.transB, case.alpha, np.ascontiguousarray(An[:probe]), Bn,
                      threads=threads)
        dt = max(time.perf_counter() - t0, 1e-3)
        rows = int(min(case.M, max(threads, probe * seconds / dt)))
    sub = np.ascontiguousarray(An[:rows])
    t0 = time.perf_counter()
    R = orc.sgemm_f64(case.transA, case.transB, case.alpha, sub, Bn, threads=threads)
    dt = time.perf_counter() - t0
    f = 2.0 * rows * case.N * case.K
    out = {"value": round(f / dt / 1e12, 6), "unit": "TFLOP/s", "cores": threads, "kind": "oracle",
           "sample": f"rows 0..{rows - 1} of the {case.M}x{case.N}x{case.K} NN product, all "
                     f"{case.N} columns ({f / 1e9:.1f} GFLOP in {dt:.1f} s, FP64 accumulation)",
           "seconds": round(dt, 2), "rows": rows}
    if keep_result:
        out["_result"] = R
    return out


def run_reference(args, dist):
    """The oracle on the host cores as the comparison arm (rank 0 only)."""
    from dense_fp32_matrix_10_gb300 import workloads as W
    case = W.HEADLINE
    A, B, _ = W.make_inputs(case)
    # each step: a bounded sample of rows, sized so that warmup + steps fit in a few minutes
    total_budget_s = 150.0
    per_step = max(0.5, total_budget_s / max(1, args.steps + args.warmup))
    probe = cpu_baseline(case, A, B, seconds=per_step)
    rows = probe["rows"]
    for _ in range(args.warmup):
        cpu_baseline(case, A, B, rows=rows)
    times = []
    for _ in range(args.steps):
        r = cpu_baseline(case, A, B, rows=rows)
        times.append(r["seconds"])
    ms = 1e3 * sum(times) / len(times)
    f = 2.0 * rows * case.N * case.K
    value = round(f / (ms * 1e-3) / 1e12, 6)
    return {
        "impl": "reference",
        "metric": "SGEMM FP32 TFLOP/s at 4096^3 (NN) and % of GB300 FP32 peak; TFLOP/s vs size",
        "value": value, "unit": "TFLOP/s", "n_gpus": dist.world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(ms, 3), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic: seeded i.i.d. standard normal A, B (torch CPU generator, seed 2)",
        "config": {"workload": case.name, "M": case.M, "N": case.N, "K": case.K,
                   "op": "NT"[case.transA] + "NT"[case.transB],
                   "alpha": case.alpha, "beta": case.beta,
                   "sample_rows_per_step": rows},
        "cpu_baseline": {"value": value, "unit": "TFLOP/s", "cores": probe["cores"],
                         "kind": "oracle",
                         "sample": f"rows 0..{rows - 1} of the {case.M}x{case.N}x{case.K} NN product, "
                                   f"all {case.N} columns, per step"},
        "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
        "gpu_launches": 0,
    }


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=500)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--algo", default="auto")
    ap.add_argument("--no-sweep", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-seconds", type=float, default=12.0)
    ap.add_argument("--workload", default=None,
                    help="time another workload family member instead of the headline "
                         "(e.g. nt_4096_uniform_s3); used to drive profiler captures")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-tensor", action="store_true",
                    help="skip the extra timing of the 3xTF32 tensor-core kernel")
    ap.add_argument("--no-transpose", action="store_true",
                    help="skip the extra timing of the transpose kernel")
    ap.add_argument("--no-library-context", action="store_true",
                    help="skip the cuBLAS FP32 context number")
    ap.add_argument("--no-batched", action="store_true",
                    help="skip the extra timing of a strided batch")
    ap.add_argument("--no-limit0", action="store_true",
                    help="skip the products timed under a scratch limit of 0")
    ap.add_argument("--no-ladder", action="store_true",
                    help="skip the naive / shared-memory-tiled comparison kernels")
    args = ap.parse_args(argv)
    if args.warmup < 3:
        ap.error("--warmup must be at least 3")
    dist = Dist()
    if args.impl == "reference":
        if dist.rank != 0:
            return 0
        print(json.dumps(run_reference(args, dist)), flush=True)
        return 0
    result = run_ours(args, dist)
    if dist.rank == 0:
        print(json.dumps(result), flush=True)
    return 0


if __name__ == "__main__":
    sys.exit(main())
