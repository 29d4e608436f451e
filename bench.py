"""Benchmark of the compensated-FP32 projection on GB300.

One step is one compensated projection y = x W^T of the 4096 x 4096 x 4096
square shape (x FP32 ~ N(0,1), W FP16 ~ N(0,0.02)) through the two-pass form
of the path, the two launches comp_gemm_f32x16_ws makes: comp_split_f32 writes
the FP16 hi/lo planes of x into a preallocated workspace, then comp_gemm_f16x2
runs both tensor-core products and the FP32 merge.  The metric is effective
FP32-GEMM throughput, 2*M*N*K per second.  The fused single-kernel
comp_gemm_f32x16 (one launch; x split in place in shared memory) is timed
beside it and reported under "kernels".

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

Timing: every step gets its own CUDA-event pair on the launching stream.
Before each step, outside the event pair, the L2 cache (129 MB, larger than
the 96 MB of inputs) is flushed: a 256 MiB buffer is written, then another
256 MiB buffer is read, so that the step starts with cold inputs and with L2
holding clean lines (the write-back of the flush's own dirty lines is not
charged to the step).  The K timed steps
are bracketed by a barrier and a device synchronisation on both sides, and
the slowest rank's time is reported.  N > 1 runs one independent replica per
GPU (the path has no exchange step), so scaling is weak.

--impl reference times the CPU oracle (test infrastructure) on the host cores
on a bounded sample of the same workload: the pages give no GPU code for this
path, so the oracle is the reference arm.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "comp-FP32 GEMM effective TFLOPS (2MNK/s) & % of FP16 TC roofline; split GB/s"
UNIT = "TFLOP/s"
WORKLOAD = "square"
PEAKS_FILE = os.path.join(ROOT, "MEASURED_PEAKS.json")
TRAFFIC_SUMMARY = os.path.join(ROOT, "profiles", "comp_gemm_f16x2_square.md")
KERNEL_SOURCE = os.path.join(ROOT, "compensated_fp32_projection_gb300", "csrc", "gemm_tc.cu")
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}


LEGS = ("step", "split", "product", "fused", "ws", "merge", "simt", "geglu")
BREAKDOWN_STEPS = 200  # steps of the second loop that times the split and the product of a step apart


def parse():
    p = argparse.ArgumentParser()
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=2000)
    p.add_argument("--warmup", type=int, default=10)
    p.add_argument("--impl", choices=["ours", "reference"], default="ours")
    p.add_argument("--no-cpu-baseline", action="store_true", help="skip the oracle CPU-baseline leg")
    p.add_argument("--leg", choices=LEGS, default=None,
                   help="time one leg alone on one shape (a small process for profiler captures); prints one "
                        "diagnostic line, not the bench line")
    p.add_argument("--config", default=WORKLOAD, help="shape of --leg: tiny, encoder, square, skinny, nonaligned")
    return p.parse_args()


def source_sha256():
    """SHA-256 over the library's sources, the header and this file (the GPU machine's
    copy of the repository has no git metadata)."""
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "compensated_fp32_projection_gb300", "csrc")
    files = sorted(os.path.join(csrc, f) for f in os.listdir(csrc)) + [
        os.path.join(ROOT, "include", "compfp32.h"), os.path.abspath(__file__)]
    for f in files:
        with open(f, "rb") as fh:
            h.update(os.path.basename(f).encode())
            h.update(fh.read())
    return h.hexdigest()


def run_metadata(dev):
    """GPU, driver, CUDA, SM count, source revision and host CPU of this run."""
    import platform

    import torch

    props = torch.cuda.get_device_properties(dev)
    meta = {"gpu": props.name, "sm_count": props.multi_processor_count,
            "compute_capability": f"{props.major}.{props.minor}",
            "torch": torch.__version__, "cuda_runtime_torch": torch.version.cuda,
            "source_sha256": source_sha256(), "host_arch": platform.machine()}
    try:
        out = subprocess.run(["nvidia-smi", "-i", str(dev.index), "--query-gpu=driver_version",
                              "--format=csv,noheader"], capture_output=True, text=True, timeout=20)
        meta["driver"] = out.stdout.strip() or None
    except (OSError, subprocess.SubprocessError):
        meta["driver"] = None
    try:
        out = subprocess.run(["nvcc", "--version"], capture_output=True, text=True, timeout=20)
        meta["nvcc"] = out.stdout.strip().splitlines()[-1] if out.stdout.strip() else None
    except (OSError, subprocess.SubprocessError):
        meta["nvcc"] = None
    try:
        out = subprocess.run(["git", "-C", ROOT, "rev-parse", "HEAD"], capture_output=True, text=True, timeout=20)
        meta["git_sha"] = out.stdout.strip() if out.returncode == 0 else None
    except (OSError, subprocess.SubprocessError):
        meta["git_sha"] = None
    model = None
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=20)
        for line in out.stdout.splitlines():
            if line.strip().startswith("Model name:"):
                model = line.split(":", 1)[1].strip()
                break
    except (OSError, subprocess.SubprocessError):
        pass
    if model is None:
        try:
            for line in open("/proc/cpuinfo"):
                if line.lower().startswith("model name"):
                    model = line.split(":", 1)[1].strip()
                    break
        except OSError:
            pass
    meta["host_cpu"] = model
    meta["host_cores"] = os.cpu_count()
    return meta


def dist_env():
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return rank, world, local


def max_over_ranks(value, dist, device):
    """The slowest rank's time (every rank receives it); value itself on one rank."""
    if dist is None:
        return value
    import torch

    t = torch.tensor([float(value)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_throughput(world, work_per_rank, seconds):
    """Whole-job rate: the work of all ranks (replicas, fixed work per rank) over
    the slowest rank's time."""
    return world * work_per_rank / seconds


def load_peaks():
    try:
        with open(PEAKS_FILE) as f:
            d = json.load(f)
        return {k: float(d[k]) for k in FALLBACK_PEAKS}, "measured"
    except (OSError, KeyError, ValueError):
        return dict(FALLBACK_PEAKS), "fallback"


def kernel_sha():
    with open(KERNEL_SOURCE, "rb") as f:
        return hashlib.sha256(f.read()).hexdigest()


def measured_traffic():
    """DRAM bytes per launch from the committed ncu summary, if it was taken on
    the current kernel source (else None)."""
    try:
        text = open(TRAFFIC_SUMMARY).read()
    except OSError:
        return None
    fields = {}
    for line in text.splitlines():
        if ":" in line and line.strip().startswith("- "):
            k, v = line.strip()[2:].split(":", 1)
            fields[k.strip()] = v.strip().strip("`")
    if fields.get("kernel source sha256") != kernel_sha():
        return None
    try:
        return int(fields["dram bytes per launch"])
    except (KeyError, ValueError):
        return None


class ClockSampler:
    """nvidia-smi samples of SM clock and throttle reasons while running."""

    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None
        self.lines: list[str] = []
        self.reader = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.QUERY}", "--format=csv,noheader,nounits",
                 "-lms", "50"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
            return
        self.reader = threading.Thread(target=self._read, daemon=True)
        self.reader.start()

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def stop(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.reader.join(timeout=2)
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
            for name, flag in zip(names, parts[5:9]):
                if flag.lower() == "active":
                    reasons.add(name)
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": smax, "reasons": sorted(reasons), "samples": len(sm)}


def oracle_cpu_baseline(x, W, target_s: float = 12.0):
    """The CPU oracle's compensated GEMM on the first rows of the workload, sized
    for about `target_s` seconds of host work.  Returns effective TFLOP/s and a
    description of the sample."""
    import numpy as np

    import oracle

    oracle.build()
    xn = x.numpy()
    wn = W.view(__import__("torch").int16).numpy().view(np.uint16)
    M, K = xn.shape
    N = wn.shape[0]
    t0 = time.perf_counter()
    oracle.gemm_comp(xn[:8], wn)  # calibration
    dt = time.perf_counter() - t0
    rows = int(min(M, max(8, 8 * target_s / max(dt, 1e-3))))
    t0 = time.perf_counter()
    oracle.gemm_comp(xn[:rows], wn)
    dt = time.perf_counter() - t0
    # one host thread on a smaller sample (about 3 s)
    rows1 = int(min(M, max(1, rows * 3.0 / max(dt * oracle.default_threads(), 1e-3))))
    t0 = time.perf_counter()
    oracle.gemm_comp(xn[:rows1], wn, threads=1)
    dt1 = time.perf_counter() - t0
    return {
        "value": 2.0 * rows * N * K / dt / 1e12,
        "unit": UNIT,
        "cores": oracle.default_threads(),
        "kind": "oracle",
        "sample": f"first {rows} of {M} rows of the square shape (all {N} columns, full K={K}), FP64 sums, "
                  f"{dt:.1f} s",
        "single_core": {"value": 2.0 * rows1 * N * K / dt1 / 1e12, "unit": UNIT, "cores": 1,
                        "sample": f"first {rows1} rows, {dt1:.1f} s"},
    }


def run_reference(args):
    """--impl reference: the CPU oracle, each step a bounded row sample."""
    rank, world, _ = dist_env()
    if rank != 0:
        return
    import numpy as np

    import oracle
    from compensated_fp32_projection_gb300 import workloads

    oracle.build()
    s = workloads.SHAPES[WORKLOAD]
    x, W = workloads.make_inputs(WORKLOAD)
    xn = x.numpy()
    wn = W.view(__import__("torch").int16).numpy().view(np.uint16)
    # one output row per step (all N columns, full K), through the oracle's
    # sampled mode: a bounded sample, so the whole run ends within minutes
    cols = np.arange(s.N, dtype=np.int64)

    def sample(i):
        r = np.full(s.N, i % s.M, dtype=np.int64)
        return oracle.gemm_comp(xn, wn, r, cols)

    for i in range(args.warmup):
        sample(i)
    times = []
    for i in range(args.steps):
        t0 = time.perf_counter()
        sample(i)
        times.append(time.perf_counter() - t0)
    per_step = statistics.mean(times)
    value = 2.0 * s.N * s.K / per_step / 1e12
    line = {
        "impl": "reference",
        "metric": METRIC,
        "value": value,
        "unit": UNIT,
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": per_step * 1e3,
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "f64",
        "data": "synthetic",
        "config": {"workload": f"{WORKLOAD} {s.M}x{s.N}x{s.K}, one output row per step (CPU oracle)",
                   "M": s.M, "N": s.N, "K": s.K},
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": oracle.default_threads(), "kind": "oracle",
                         "sample": f"1 row x {s.N} columns x K={s.K} per step (sampled mode), FP64 sums"},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


class L2Flush:
    """Cold, clean L2 before a timed launch: write a 256 MiB buffer (larger
    than the 129 MB L2), then read a second one so that the written lines are
    back in DRAM before the timed region starts."""

    def __init__(self, dev):
        import torch

        self.w = torch.empty(256 << 20, dtype=torch.uint8, device=dev)
        self.r = torch.zeros((256 << 20) // 8, dtype=torch.int64, device=dev)
        self.out = torch.empty((), dtype=torch.int64, device=dev)

    def __call__(self):
        import torch

        self.w.zero_()
        torch.sum(self.r, dim=0, out=self.out)


def time_kernel(fn, flush, stream, reps: int, warm: int = 3):
    """Median and mean of per-launch CUDA-event times (ms), L2 flushed before each."""
    import torch

    for _ in range(warm):
        flush()
        fn()
    ts = []
    for _ in range(reps):
        flush()
        a = torch.cuda.Event(enable_timing=True)
        b = torch.cuda.Event(enable_timing=True)
        a.record(stream)
        fn()
        b.record(stream)
        b.synchronize()
        ts.append(a.elapsed_time(b))
    return statistics.median(ts), statistics.mean(ts)


def time_back_to_back(fn, stream, reps: int = 200, warm: int = 10):
    """Mean per-call time (ms) of `reps` calls enqueued back to back (no flush:
    inputs warm in L2, launch latency overlapped with the previous call)."""
    import torch

    for _ in range(warm):
        fn()
    a = torch.cuda.Event(enable_timing=True)
    b = torch.cuda.Event(enable_timing=True)
    a.record(stream)
    for _ in range(reps):
        fn()
    b.record(stream)
    b.synchronize()
    return a.elapsed_time(b) / reps


def run_ours(args):
    import torch

    rank, world, local = dist_env()
    dist = None
    if world > 1:
        import torch.distributed as dist

        torch.cuda.set_device(local)
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    else:
        torch.cuda.set_device(0)
    dev = torch.device("cuda", torch.cuda.current_device())

    import __graft_entry__

    __graft_entry__.build()
    import compensated_fp32_projection_gb300 as pkg
    from compensated_fp32_projection_gb300 import workloads

    s = workloads.SHAPES[WORKLOAD]
    x_cpu, W_cpu = workloads.make_inputs(WORKLOAD)
    x = x_cpu.to(dev)
    W = W_cpu.to(dev)
    y = torch.empty((s.M, s.N), dtype=torch.float32, device=dev)
    ws = torch.empty(pkg.comp_gemm_workspace_bytes(s.M, s.K), dtype=torch.uint8, device=dev)
    hi = ws[: 2 * s.M * s.K].view(torch.float16).view(s.M, s.K)
    lo = ws[2 * s.M * s.K:].view(torch.float16).view(s.M, s.K)
    flush = L2Flush(dev)
    stream = torch.cuda.current_stream(dev)

    def split():
        pkg.comp_split_f32(x, hi, lo)

    def product():
        pkg.comp_gemm_f16x2(hi, lo, W, y)

    def step():
        split()
        product()

    def barrier():
        torch.cuda.synchronize(dev)
        if dist is not None:
            dist.barrier()
        torch.cuda.synchronize(dev)

    # the first call of the process (one-time set-up of the kernels' attributes
    # and the tensor-map encoder included), timed on the host around a
    # synchronised call, before any warm-up
    flush()
    torch.cuda.synchronize(dev)
    t0 = time.perf_counter()
    step()
    torch.cuda.synchronize(dev)
    first_call_ms = (time.perf_counter() - t0) * 1e3

    warm = max(3, args.warmup)
    for _ in range(warm):
        flush()
        step()
    barrier()
    sampler = ClockSampler(dev.index)
    sampler.start()
    time.sleep(0.3)  # let the sampler start
    barrier()
    events = []
    for _ in range(args.steps):
        flush()
        a = torch.cuda.Event(enable_timing=True)
        b = torch.cuda.Event(enable_timing=True)
        a.record(stream)
        step()
        b.record(stream)
        events.append((a, b))
    barrier()
    clocks = sampler.stop()
    times = [a.elapsed_time(b) for a, b in events]  # ms, whole step
    ms = max_over_ranks(statistics.mean(times), dist, dev)
    # the split and the product of a step, timed separately in a second loop:
    # an event between the two launches keeps the product from being launched
    # while the split still runs (its set-up then no longer overlaps the
    # split), so the steps of this loop are slower than the timed ones and the
    # product's time here includes its set-up
    breakdown = []
    for _ in range(min(args.steps, BREAKDOWN_STEPS)):
        flush()
        a = torch.cuda.Event(enable_timing=True)
        m = torch.cuda.Event(enable_timing=True)
        b = torch.cuda.Event(enable_timing=True)
        a.record(stream)
        split()
        m.record(stream)
        product()
        b.record(stream)
        breakdown.append((a, m, b))
    barrier()
    split_times = [a.elapsed_time(m) for a, m, _ in breakdown]
    product_times = [m.elapsed_time(b) for _, m, b in breakdown]
    breakdown_step_ms = statistics.mean(a.elapsed_time(b) for a, _, b in breakdown)
    st, where = pkg.device_status()
    if st != 0:
        raise RuntimeError(f"kernel fault word {where:#x}")

    flops = float(s.flops)
    value = job_throughput(world, flops, ms * 1e-3) / 1e12

    # end to end through the public API, pipelined like a serving loop: step i's
    # inputs go up on one copy stream while step i-1 computes and step i-2's
    # result comes down on another.  Every step still copies its own x and W
    # from pinned host memory and its own y back; three buffer sets, each reused
    # only after its previous result has left the device (with two, the upload
    # of step i+1 waits for the download of step i-1 and the link idles).
    nbuf = 3
    x_h = x_cpu.pin_memory()
    W_h = W_cpu.pin_memory()
    y_h = [torch.empty((s.M, s.N), dtype=torch.float32).pin_memory() for _ in range(nbuf)]
    bufs = [(torch.empty_like(x), torch.empty_like(W), torch.empty_like(y), torch.empty_like(ws))
            for _ in range(nbuf)]
    s_in, s_comp, s_out = (torch.cuda.Stream(dev) for _ in range(3))

    def run_e2e(nsteps):
        done_out = [None] * nbuf
        for i in range(nsteps):
            xb, Wb, yb, wsb = bufs[i % nbuf]
            if done_out[i % nbuf] is not None:
                s_in.wait_event(done_out[i % nbuf])
            with torch.cuda.stream(s_in):
                xb.copy_(x_h, non_blocking=True)
                Wb.copy_(W_h, non_blocking=True)
            ev_in = torch.cuda.Event()
            ev_in.record(s_in)
            s_comp.wait_event(ev_in)
            pkg.comp_gemm_f32x16_ws(xb, Wb, yb, workspace=wsb, stream=s_comp)
            ev_c = torch.cuda.Event()
            ev_c.record(s_comp)
            s_out.wait_event(ev_c)
            with torch.cuda.stream(s_out):
                y_h[i % nbuf].copy_(yb, non_blocking=True)
            ev_o = torch.cuda.Event()
            ev_o.record(s_out)
            done_out[i % nbuf] = ev_o
        return done_out

    e2e_steps = max(3, min(args.steps, 60))
    run_e2e(nbuf)
    barrier()
    a = torch.cuda.Event(enable_timing=True)
    b = torch.cuda.Event(enable_timing=True)
    a.record(s_in)
    run_e2e(e2e_steps)
    b.record(s_out)  # after the last result's copy, which depends on every earlier step
    barrier()
    e2e_ms = max_over_ranks(a.elapsed_time(b) / e2e_steps, dist, dev)

    peaks, peak_src = load_peaks()
    tensor_flops = 2.0 * flops  # two FP16 products per effective FP32 multiply-add
    achieved = tensor_flops / (statistics.mean(product_times) * 1e-3) / 1e12
    traffic = measured_traffic()
    split_in_step_gbs = 8.0 * s.M * s.K / (statistics.mean(split_times) * 1e-3) / 1e9

    # the standalone split and merge at the square shape's size (HBM bound), and the SIMT reference
    n = s.M * s.K
    xs = torch.randn(n, device=dev)
    hi = torch.empty(n, dtype=torch.float16, device=dev)
    lo = torch.empty(n, dtype=torch.float16, device=dev)
    med, mean = time_kernel(lambda: pkg.comp_split_f32(xs, hi, lo), flush, stream, 20)
    split_gbs = 8.0 * n / (mean * 1e-3) / 1e9
    a32 = torch.randn(n, device=dev)
    b32 = torch.randn(n, device=dev)
    o32 = torch.empty(n, device=dev)
    med, mean = time_kernel(lambda: pkg.comp_merge_f32(a32, b32, o32), flush, stream, 20)
    merge_gbs = 12.0 * n / (mean * 1e-3) / 1e9
    del xs, hi, lo, a32, b32, o32
    # the labelled sweep point far beyond L2: n = 2^28 (1 GiB of x; 3 GiB read
    # and written by the merge)
    nb = 1 << 28
    xs = torch.randn(nb, device=dev)
    hi = torch.empty(nb, dtype=torch.float16, device=dev)
    lo = torch.empty(nb, dtype=torch.float16, device=dev)
    med, mean = time_kernel(lambda: pkg.comp_split_f32(xs, hi, lo), flush, stream, 10)
    split_big_gbs = 8.0 * nb / (mean * 1e-3) / 1e9
    del hi, lo
    a32 = xs
    b32 = torch.randn(nb, device=dev)
    o32 = torch.empty(nb, device=dev)
    med, mean = time_kernel(lambda: pkg.comp_merge_f32(a32, b32, o32), flush, stream, 10)
    merge_big_gbs = 12.0 * nb / (mean * 1e-3) / 1e9
    med, fused_ms = time_kernel(lambda: pkg.comp_gemm_f32x16(x, W, y), flush, stream, 50)
    fused_tflops = flops / (fused_ms * 1e-3) / 1e12
    med, mean = time_kernel(lambda: pkg.comp_gemm_f32_simt(x, W, y), flush, stream, 3, warm=1)
    simt_tflops = flops / (mean * 1e-3) / 1e12
    # the GEGLU epilogue (bias and gate) in the product kernel, against the same
    # two-pass call without it; both through the public calls, same workspace
    g_ep = torch.Generator(device="cpu").manual_seed(7)
    b_ep = (torch.randn(s.N, generator=g_ep) * 0.5).to(dev)
    gate_ep = (torch.randn(s.M, s.N, generator=g_ep) * 2.0).to(dev)
    med, mean_plain = time_kernel(lambda: pkg.comp_gemm_f32x16_ws(x, W, y, workspace=ws), flush, stream, 20)
    med, mean_epi = time_kernel(lambda: pkg.comp_gemm_f32x16_epilogue(x, W, b_ep, gate_ep, y, workspace=ws), flush,
                                stream, 20)
    up_ep = torch.randn(s.M, s.N, generator=g_ep).to(dev)
    out_ep = torch.empty_like(up_ep)
    med, mean_geglu = time_kernel(lambda: pkg.comp_geglu_f32(gate_ep, up_ep, out_ep), flush, stream, 20)
    geglu_gbs = 12.0 * s.M * s.N / (mean_geglu * 1e-3) / 1e9
    del b_ep, gate_ep, up_ep, out_ep
    del xs, a32, b32, o32

    # the floor of this timing method: one trivial launch (a 16-element merge)
    # timed cold the same way as the configurations below
    f16a, f16b, f16o = (torch.zeros(16, device=dev) for _ in range(3))
    floor_med, _ = time_kernel(lambda: pkg.comp_merge_f32(f16a, f16b, f16o), flush, stream, 20)
    del f16a, f16b, f16o

    # the other configurations (parity cases), each through the workspace entry
    # point with the same flush; roofline time t* = max(tensor work / tensor peak,
    # algorithmic bytes / HBM peak)
    peaks_now, _ = load_peaks()
    others = {}
    for name in ("tiny", "encoder", "skinny", "nonaligned"):
        so = workloads.SHAPES[name]
        xo_c, Wo_c = workloads.make_inputs(name)
        xo, Wo = xo_c.to(dev), Wo_c.to(dev)
        yo = torch.empty((so.M, so.N), dtype=torch.float32, device=dev)
        wso = torch.empty(max(16, pkg.comp_gemm_workspace_bytes_mnk(so.M, so.N, so.K)), dtype=torch.uint8, device=dev)
        call = lambda: pkg.comp_gemm_f32x16_ws(xo, Wo, yo, workspace=wso)  # noqa: E731
        med, mean = time_kernel(call, flush, stream, 20)
        warm_ms = time_back_to_back(call, stream)
        byts = 4 * so.M * so.K + 2 * so.N * so.K + 4 * so.M * so.N
        t_star = max(4.0 * so.M * so.N * so.K / (peaks_now["bf16_tflops"] * 1e12), byts / (peaks_now["hbm_gbs"] * 1e9))
        padded = so.K % 8 != 0
        swapped = so.M <= 32 and not padded
        t128 = ((so.M + 127) // 128) * ((so.N + 127) // 128)
        t64 = ((so.M + 127) // 128) * ((so.N + 63) // 64)
        nk = ((so.K + 7) // 8 * 8 + 63) // 64
        few = so.M > 32 and (so.M <= 128 or so.M * so.N < 152 * 128 * 192)  # not the CTA-pair kernel
        narrow = few and t128 * 2 <= 152 and nk <= 32 and ((t64 * 2 <= 152 and nk >= 8) or t64 <= 152)
        narrow_split = narrow and t64 * 2 <= 152 and nk >= 8
        splitk = few and not narrow and ((t128 * 4 <= 152 and nk >= 16) or (t128 * 2 <= 152 and nk >= 8))
        if swapped:
            tiles_w = (so.N + 127) // 128
            nk_w = (so.K + 63) // 64
            ks_w = 4 if tiles_w * 4 <= 152 and nk_w >= 16 else 2 if tiles_w * 2 <= 152 and nk_w >= 8 else 1
            path = "one kernel: operands swapped (y^T = W x^T), split fused"
            if ks_w > 1:
                path += ", K split over clusters of %d CTAs" % ks_w
        elif padded:
            path = "one prep launch (x split into planes and W copied, both padded to K = %d), then the product " \
                   "kernel" % ((so.K + 7) // 8 * 8)
        else:
            path = "split + product kernel"
        if narrow_split:
            path += ", 128 x 64 tiles, K split over pairs of CTAs (ordered reduction through distributed shared memory)"
        elif narrow:
            path += ", 128 x 64 tiles, one CTA each"
        elif splitk:
            path += ", K split over clusters of CTAs (ordered reduction through distributed shared memory)"
        others[name] = {
            "M": so.M, "N": so.N, "K": so.K,
            "us": med * 1e3,
            "us_mean": mean * 1e3,
            "eff_TFLOP/s": 2.0 * so.M * so.N * so.K / (med * 1e-3) / 1e12,
            "GB/s": byts / (med * 1e-3) / 1e9,
            "frac_of_roofline": t_star / (med * 1e-3),
            "bound": "tensor" if t_star == 4.0 * so.M * so.N * so.K / (peaks_now["bf16_tflops"] * 1e12) else "hbm",
            "path": path,
            "us_back_to_back": warm_ms * 1e3,
        }
        del xo, Wo, yo, wso

    if rank != 0:
        if dist is not None:
            dist.barrier()
            dist.destroy_process_group()
        return

    meta = run_metadata(dev)
    cpu = None
    if world == 1 and not args.no_cpu_baseline:
        cpu = oracle_cpu_baseline(x_cpu, W_cpu)

    line = {
        "metric": METRIC,
        "value": value,
        "unit": UNIT,
        "n_gpus": world,
        "steps": args.steps,
        "warmup": warm,
        "ms_per_step": ms,
        "ms_per_step_median": statistics.median(times),
        "ms_per_step_min": min(times),
        "first_call_ms": first_call_ms,
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "f32",
        "data": "synthetic",
        "config": {
            "workload": f"{WORKLOAD} dense projection {s.M}x{s.N}x{s.K}: x FP32 N(0,1), W FP16 N(0,0.02) RNE, "
                        f"y FP32; two-pass: comp_split_f32 into a workspace, then comp_gemm_f16x2 (two FP16 "
                        f"tensor-core products, FP32 merge) - the launches of comp_gemm_f32x16_ws",
            "M": s.M,
            "N": s.N,
            "K": s.K,
            "seed": workloads.SEED_BASE + s.index,
            "x_sha256": hashlib.sha256(x_cpu.numpy().tobytes()).hexdigest(),
            "W_sha256": hashlib.sha256(W_cpu.view(torch.int16).numpy().tobytes()).hexdigest(),
            "l2": "flushed before every timed step, outside the event pair: 256 MiB written, then another "
                  "256 MiB read (cold inputs, clean L2)",
            "replicas": world,
        },
        "roofline": {
            "bound": "tensor",
            "kernel": "comp_f16x2_pair_kernel (comp_gemm_f16x2)",
            "achieved": achieved,
            "peak": peaks["bf16_tflops"],
            "unit": "TFLOP/s",
            "frac": achieved / peaks["bf16_tflops"],
            "traffic": traffic,
            "peak_source": f"{peak_src} dense bf16 burst (FP16 runs at the same tensor rate)",
            "work": "4*M*N*K tensor FLOP per launch (hi and lo products)",
            "kernel_time": f"mean of {len(product_times)} product launches, each timed between an event after the "
                           f"step's split and one after the product (a second loop of steps; with the event between "
                           f"them a step took {breakdown_step_ms:.4f} ms against {ms:.4f} without)",
            "step_frac_of_roofline": value / world / (peaks["bf16_tflops"] / 2.0),
        },
        "e2e": {
            "value": job_throughput(world, flops, e2e_ms * 1e-3) / 1e12,
            "unit": UNIT,
            "h2d_bytes_per_step": 4 * s.M * s.K + 2 * s.N * s.K,
            "d2h_bytes_per_step": 4 * s.M * s.N,
            "pipeline": "comp_gemm_f32x16_ws on a compute stream; inputs up and results down on two copy streams, "
                        "three buffer sets",
        },
        "gpu_launches": 2 * args.steps,
        "kernels": {
            "comp_split_f32 in step": {"n": s.M * s.K, "GB/s": split_in_step_gbs,
                                       "frac_of_hbm": split_in_step_gbs / peaks["hbm_gbs"]},
            "comp_gemm_f16x2 in step": {"ms": statistics.mean(product_times), "tensor TFLOP/s": achieved},
            "comp_gemm_f32x16 (fused: one launch, comp_f32x16_pair_kernel, x split in place in shared memory)": {
                "TFLOP/s": fused_tflops, "ms": fused_ms,
                "frac_of_roofline": fused_tflops / (peaks["bf16_tflops"] / 2.0)},
            "comp_split_f32": {"n": n, "GB/s": split_gbs, "frac_of_hbm": split_gbs / peaks["hbm_gbs"]},
            "comp_merge_f32": {"n": n, "GB/s": merge_gbs, "frac_of_hbm": merge_gbs / peaks["hbm_gbs"]},
            "comp_split_f32 (n = 2^28, beyond L2)": {"n": nb, "GB/s": split_big_gbs,
                                                     "frac_of_hbm": split_big_gbs / peaks["hbm_gbs"]},
            "comp_merge_f32 (n = 2^28, beyond L2)": {"n": nb, "GB/s": merge_big_gbs,
                                                     "frac_of_hbm": merge_big_gbs / peaks["hbm_gbs"]},
            "comp_gemm_f32_simt": {"TFLOP/s": simt_tflops},
            "comp_geglu_f32": {"n": s.M * s.N, "GB/s": geglu_gbs, "frac_of_hbm": geglu_gbs / peaks["hbm_gbs"]},
            "comp_gemm_f32x16_epilogue (bias in the product's epilogue, then the GEGLU dispatch)": {
                "ms": mean_epi, "eff TFLOP/s": flops / (mean_epi * 1e-3) / 1e12,
                "ms without the epilogue": mean_plain,
                "added gate bytes": 4 * s.M * s.N},
        },
        "other_configs": others,
        "other_configs_note": "us: median of 20 calls, each with L2 flushed first (cold); us_back_to_back: mean of "
                              "200 calls enqueued back to back (warm L2); one trivial launch timed cold the same "
                              "way takes %.2f us (the floor of this method)" % (floor_med * 1e3),
    }
    if clocks is not None:
        line["clocks"] = clocks
    if cpu is not None:
        line["cpu_baseline"] = cpu
        line["cpu_baseline"]["host_cpu"] = meta.get("host_cpu")
    line["run"] = meta
    print(json.dumps(line), flush=True)
    if dist is not None:
        dist.barrier()
        dist.destroy_process_group()


def run_leg(args):
    """One leg on one shape, W warm-up and K timed launches (each with its own
    CUDA-event pair, L2 flushed before each, outside the pair); prints one
    diagnostic line.  Sized for profiler captures: only this leg's buffers are
    allocated."""
    import torch

    torch.cuda.set_device(0)
    dev = torch.device("cuda", 0)
    import __graft_entry__

    __graft_entry__.build()
    import compensated_fp32_projection_gb300 as pkg
    from compensated_fp32_projection_gb300 import workloads

    s = workloads.SHAPES[args.config]
    x_cpu, W_cpu = workloads.make_inputs(args.config)
    x, W = x_cpu.to(dev), W_cpu.to(dev)
    y = torch.empty((s.M, s.N), dtype=torch.float32, device=dev)
    flush = L2Flush(dev)
    stream = torch.cuda.current_stream(dev)
    leg = args.leg
    if leg in ("step", "split", "product"):
        ws = torch.empty(pkg.comp_gemm_workspace_bytes(s.M, s.K), dtype=torch.uint8, device=dev)
        hi = ws[: 2 * s.M * s.K].view(torch.float16).view(s.M, s.K)
        lo = ws[2 * s.M * s.K:].view(torch.float16).view(s.M, s.K)
        pkg.comp_split_f32(x, hi, lo)
        fns = {"step": lambda: (pkg.comp_split_f32(x, hi, lo), pkg.comp_gemm_f16x2(hi, lo, W, y)),
               "split": lambda: pkg.comp_split_f32(x, hi, lo),
               "product": lambda: pkg.comp_gemm_f16x2(hi, lo, W, y)}
        fn = fns[leg]
        work = 2.0 * s.M * s.N * s.K if leg != "split" else 8.0 * s.M * s.K
    elif leg == "fused":
        fn, work = (lambda: pkg.comp_gemm_f32x16(x, W, y)), 2.0 * s.M * s.N * s.K
    elif leg == "ws":
        wso = torch.empty(max(16, pkg.comp_gemm_workspace_bytes_mnk(s.M, s.N, s.K)), dtype=torch.uint8, device=dev)
        fn, work = (lambda: pkg.comp_gemm_f32x16_ws(x, W, y, workspace=wso)), 2.0 * s.M * s.N * s.K
    elif leg == "simt":
        fn, work = (lambda: pkg.comp_gemm_f32_simt(x, W, y)), 2.0 * s.M * s.N * s.K
    elif leg in ("merge", "geglu"):
        a = torch.randn(s.M * s.N, device=dev)
        b = torch.randn(s.M * s.N, device=dev)
        o = torch.empty_like(a)
        fn = (lambda: pkg.comp_merge_f32(a, b, o)) if leg == "merge" else (lambda: pkg.comp_geglu_f32(a, b, o))
        work = 12.0 * s.M * s.N
    med, mean = time_kernel(fn, flush, stream, max(1, args.steps), warm=max(1, args.warmup))
    st, where = pkg.device_status()
    if st != 0:
        raise RuntimeError(f"kernel fault word {where:#x}")
    unit = "GB/s" if leg in ("split", "merge", "geglu") else "eff TFLOP/s"
    rate = work / (med * 1e-3) / (1e9 if unit == "GB/s" else 1e12)
    print(json.dumps({"leg": leg, "config": args.config, "M": s.M, "N": s.N, "K": s.K, "launches": args.steps,
                      "us_median": med * 1e3, "us_mean": mean * 1e3, unit: rate}), flush=True)


def main():
    args = parse()
    if args.impl == "reference":
        run_reference(args)
    elif args.leg is not None:
        run_leg(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
