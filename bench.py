#!/usr/bin/env python3
"""Benchmark of the PN decode GEMV on GB300; prints one JSON line.

Workload (default): pn3t GEMV, N = 17408 rows, K = 5120 (64 blocks of 34 bytes
per row, 37,879,808 bytes of packed weights), M = 1, fp16 x, fp32 y -- the
FFN gate/up shape of a 27B-class model at the tensorless pages' widths.  A
step is one GEMV over one batch (one token's x).  Other workloads:
``--config 0|2|3|4|5`` (3/4/5: one decoder layer's seven GEMVs in one fused
call at M = 1 / 8 / 16) and ``--config 6``, the prefill path (a 4096-token
prompt through the pn3t 5120->17408 tensor: fp16 rebuild + tcgen05 GEMM,
reported in TFLOP/s against the tensor-core roofline).

Timing: weights are resident in HBM; copies (together more than twice the
129 MB L2) are rotated so every step reads its weights from HBM.  Steps are
captured in CUDA graphs (launch overhead would otherwise exceed a 6 us kernel);
every graph is replayed once and the GPU kept busy with replays for half a
second before the timed region, which is exactly ``--steps`` steps timed with
CUDA events on the launching stream, after a barrier and a synchronize on both
sides; the max over ranks is taken.  ``value`` is the effective bandwidth:
algorithmic bytes per GEMV (packed weights + x + y) over the time per GEMV.
The default line also carries ``m8``, the metric's other half: the seven
GEMVs of the 27B-class layer at M = 8 in one fused call, timed the same way.
``e2e`` times the same GEMV through the public Python API with x copied from
pinned host memory and y copied back and synchronised every step.
``cpu_baseline`` times the CPU oracle on a bounded sample of rows.

Under torchrun (N > 1) every rank runs an independent replica of the workload
on its own GPU (weak scaling; no collective on the data path).

``--impl reference`` times the CPU oracle as the reference arm.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import re
import subprocess
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "PN GEMV µs and effective HBM GB/s (% of GB300 peak) at M=1 and M=8"
NOMINAL_HBM_GBS = 8000.0
FALLBACK_HBM_GBS = 6800.0
ROTATE_BYTES = 300e6           # > 2x the 129 MB L2
GRAPH_NODES = 1000


def parse_args():
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=100000)
    ap.add_argument("--warmup", type=int, default=2000)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--config", type=int, default=1, choices=[0, 1, 2, 3, 4, 5, 6])
    ap.add_argument("--algo", choices=["auto", "tc", "cuda_core", "cuda_core_staged"], default="auto")
    ap.add_argument("--e2e-steps", type=int, default=2000)
    ap.add_argument("--cpu-seconds", type=float, default=10.0,
                    help="target CPU time of the oracle baseline sample")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-m8", action="store_true",
                    help="leave out the M = 8 layer measurement that the default line carries as 'm8'")
    ap.add_argument("--m", type=int, default=0,
                    help="GEMV workloads: override the token count M (1 .. 16); 0 keeps the workload's")
    ap.add_argument("--hadamard", type=int, default=0,
                    help="rotate every tensor's activations with pn_hadamard (this block size) "
                         "before its GEMV, inside each step (0 = off)")
    ap.add_argument("--fused-hadamard", type=int, default=0,
                    help="GEMV on activations rotated inside the GEMV launch (pn_gemv_hadamard, this "
                         "block size; M <= 2; 0 = off)")
    ap.add_argument("--gptq", action="store_true",
                    help="time the device GPTQ-style quantiser (pn_gptq) on the workload's first tensor "
                         "with 256 calibration rows, and the oracle on a small sample")
    args = ap.parse_args()
    if args.fused_hadamard and args.hadamard:
        raise SystemExit("--hadamard and --fused-hadamard are exclusive")
    return args


# ----------------------------------------------------------------- helpers ---

def workload(cfg: int, m_override: int = 0):
    from bit_weight_only_pn_gb300 import synth
    c = synth.CONFIGS[cfg]
    if m_override and not c.get("prefill"):
        if not 1 <= m_override <= 16:
            raise SystemExit("--m must be in 1 .. 16")
        return f"{c['name']} (run at M={m_override})", list(c["tensors"]), m_override
    return c["name"], list(c["tensors"]), c["M"]


def cpu_model() -> str:
    """The host CPU's name from /proc/cpuinfo (model name, else the Arm part number)."""
    try:
        text = open("/proc/cpuinfo").read()
    except OSError:
        return "unknown"
    m = re.search(r"^model name\s*:\s*(.+)$", text, re.M)
    if m:
        return m.group(1).strip()
    impl = re.search(r"^CPU implementer\s*:\s*(\S+)", text, re.M)
    part = re.search(r"^CPU part\s*:\s*(\S+)", text, re.M)
    if impl and part:
        return f"Arm implementer {impl.group(1)} part {part.group(1)}"
    return "unknown"


def per_block(t: int) -> int:
    return 80 if t == 124 else 64


def algorithmic_bytes(tensors, M: int) -> int:
    """Packed weights + fp16 x + fp32 y of one step (what the method must move)."""
    total = 0
    for t, K, N in tensors:
        total += N * (K // per_block(t)) * 34 + 2 * M * K + 4 * M * N
    return total


def measured_peak():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as fh:
            d = json.load(fh)
        return float(d["hbm_gbs"]), "measured"
    except Exception:  # noqa: BLE001
        return FALLBACK_HBM_GBS, "fallback"


# The sources each workload's timed kernel is built from (its own file plus
# the shared device and host headers).
KERNEL_SOURCES = {
    "stream": ("pn_gemv_stream.cu", "pn_device.cuh", "pn_internal.h"),
    "tc": ("pn_gemv_tc.cu", "pn_device.cuh", "pn_internal.h"),
    "prefill": ("pn_prefill.cu", "pn_device.cuh", "pn_internal.h"),
}


def kernel_of(cfg: int) -> str:
    """Which kernel a workload times: the one-token kernel (M <= 2), the
    batch kernel (M = 3 .. 16) or the prefill GEMM."""
    from bit_weight_only_pn_gb300 import synth
    c = synth.CONFIGS[cfg]
    if c.get("prefill"):
        return "prefill"
    return "stream" if c["M"] <= 2 else "tc"


def code_only(text: str) -> str:
    """C/C++ source with comments removed and whitespace collapsed (string
    and character literals kept), so that editing a comment does not count
    as changing a kernel."""
    out, i, n = [], 0, len(text)
    while i < n:
        c = text[i]
        if c in "\"'":
            j = i + 1
            while j < n and text[j] != c:
                j += 2 if text[j] == "\\" else 1
            out.append(text[i:j + 1])
            i = j + 1
        elif text.startswith("//", i):
            j = text.find("\n", i)
            i = n if j < 0 else j
        elif text.startswith("/*", i):
            j = text.find("*/", i + 2)
            i = n if j < 0 else j + 2
            out.append(" ")
        else:
            out.append(c)
            i += 1
    return " ".join("".join(out).split())


def kernel_source_hash(kernel: str) -> str:
    """Hash of the code (comments and layout aside) of the sources a kernel
    is built from: a recorded ncu traffic figure is only used while that code
    is unchanged."""
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "bit_weight_only_pn_gb300", "csrc")
    for f in KERNEL_SOURCES[kernel]:
        with open(os.path.join(csrc, f), encoding="utf-8") as fh:
            h.update(f.encode() + b"\0" + code_only(fh.read()).encode())
    return h.hexdigest()[:16]


TRAFFIC_FILE = os.path.join("profiles", "traffic.json")


def recorded_traffic(cfg: int):
    """Per-launch DRAM bytes (read + write) of the workload's timed kernel from
    the committed ncu records (profiles/traffic.json), if they were taken on
    that kernel's current sources (else None)."""
    try:
        with open(os.path.join(ROOT, TRAFFIC_FILE)) as fh:
            records = json.load(fh)["records"]
    except (OSError, ValueError, KeyError):
        return None
    want = kernel_source_hash(kernel_of(cfg))
    for r in records:
        if int(r.get("config", -1)) == cfg and r.get("source") == want:
            return int(r["bytes_per_launch"])
    return None


class ClockSampler:
    """nvidia-smi clocks and throttle reasons, sampled every 100 ms."""
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.lines = []
        self.marks = []

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
            return
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append((time.time(), line.strip()))

    def mark(self):
        self.marks.append(time.time())

    def stop(self):
        if self.proc is None:
            return None
        time.sleep(0.25)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.thread.join(timeout=2)
        lo, hi = (self.marks[0], self.marks[-1]) if len(self.marks) >= 2 else (0, 1e30)
        sm, smax, reasons, n = [], None, set(), 0
        for ts, line in self.lines:
            if not (lo - 0.15 <= ts <= hi + 0.15):
                continue
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            n += 1
            try:
                sm.append(float(parts[1]))
                smax = float(parts[2])
            except ValueError:
                continue
            names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
            for name, v in zip(names, parts[5:9]):
                if v.lower() == "active":
                    reasons.add(name)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": smax, "reasons": sorted(reasons), "samples": 0}
        return {"sm_mhz": float(np.median(sm)), "sm_max_mhz": smax, "reasons": sorted(reasons),
                "samples": n}


# -------------------------------------------------------------- CPU oracle ---

def oracle_sample_rate(tensors, M, seconds, threads):
    """Time the CPU oracle on a bounded sample of the workload: a sample of
    every tensor's rows (all of them when one pass over the whole workload is
    short), passed over repeatedly for about `seconds` of wall time.  Returns
    (GB/s of algorithmic bytes, description, threads used, seconds)."""
    import oracle
    from bit_weight_only_pn_gb300 import synth
    o = oracle.Oracle()
    # calibrate on 64 rows of the first tensor (after one untimed call)
    t0, K0, N0 = tensors[0]
    W = o.pack(t0, synth.weight_rows(synth.weight_seed(9, 0), N0, K0, range(64)))
    x = synth.activations(synth.x_seed(9, 0), M, K0)
    o.gemv(t0, W, K0, x, want_abs=False)
    s = time.perf_counter()
    o.gemv(t0, W, K0, x, want_abs=False)
    per_row = (time.perf_counter() - s) / 64.0 / max(1, threads)
    total_rows = sum(N for _, _, N in tensors)
    frac = min(1.0, seconds / max(per_row * total_rows, 1e-9))
    work = []
    for e, (t, K, N) in enumerate(tensors):
        rows = min(N, max(16, int(N * frac)))
        w = synth.weight_rows(synth.weight_seed(9, e), N, K, range(rows))
        work.append((t, K, rows, o.pack(t, w), synth.activations(synth.x_seed(9, e), M, K)))

    def one_pass():
        for t, K, rows, W, x in work:
            o.gemv_threads(t, W, K, x, threads)

    s = time.perf_counter()
    one_pass()
    first = time.perf_counter() - s
    passes = max(1, int(round(seconds / max(first, 1e-6))))
    s = time.perf_counter()
    for _ in range(passes):
        one_pass()
    dt = time.perf_counter() - s
    nbytes = sum(rows * (K // per_block(t)) * 34 + 2 * M * K + 4 * M * rows for t, K, rows, _, _ in work)
    desc = ", ".join(f"{rows}/{N} rows of the {K}->{N} tensor" for (t, K, rows, _, _), (_, _, N) in zip(work, tensors))
    return (nbytes * passes / dt / 1e9, f"{desc}, M={M}, {passes} passes in {dt:.1f} s on {threads} threads",
            threads, dt)


# ------------------------------------------------------------- distributed ---

def dist_setup(args):
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        os.environ.setdefault("MASTER_ADDR", "127.0.0.1")
        dist.init_process_group("gloo", rank=rank, world_size=world)
    return world, rank, local


def dist_barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def dist_max(world, v: float) -> float:
    if world == 1:
        return v
    import torch
    import torch.distributed as dist
    t = torch.tensor([v], dtype=torch.float64)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


# ------------------------------------------------------------------- arms ----

def run_reference(args, world, rank):
    """The CPU oracle as the reference arm (rank 0 only): each step runs the
    oracle GEMV on a fixed sample of rows of every tensor, sized so that the
    warm-up and timed steps together take about two minutes."""
    if rank != 0:
        return
    import oracle
    from bit_weight_only_pn_gb300 import synth
    name, tensors, M = workload(args.config, args.m)
    o = oracle.Oracle()
    threads = os.cpu_count() or 1
    t0, K0, N0 = tensors[0]
    W = o.pack(t0, synth.weight_rows(synth.weight_seed(9, 0), N0, K0, range(64)))
    x = synth.activations(synth.x_seed(9, 0), M, K0)
    s0 = time.perf_counter()
    o.gemv(t0, W, K0, x, want_abs=False)
    per_row = (time.perf_counter() - s0) / 64.0
    budget = 120.0 / max(1, args.steps + args.warmup)
    total_rows = sum(N for _, _, N in tensors)
    frac = min(1.0, budget / max(per_row * total_rows, 1e-12))
    work = []
    for e, (t, K, N) in enumerate(tensors):
        rows = min(N, max(1, int(round(N * frac))))
        W = o.pack(t, synth.weight_rows(synth.weight_seed(9, e), N, K, range(rows)))
        work.append((t, K, rows, W, synth.activations(synth.x_seed(9, e), M, K)))
    sample_rows = sum(r for _, _, r, _, _ in work)
    use = threads if sample_rows >= 64 * threads else 1
    nbytes = sum(r * (K // per_block(t)) * 34 + 2 * M * K + 4 * M * r for t, K, r, _, _ in work)

    def one():
        for t, K, r, W, x in work:
            if use > 1:
                o.gemv_threads(t, W, K, x, use)
            else:
                o.gemv(t, W, K, x, want_abs=False)

    for _ in range(args.warmup):
        one()
    s0 = time.perf_counter()
    for _ in range(args.steps):
        one()
    dt = time.perf_counter() - s0
    value = nbytes * args.steps / dt / 1e9
    desc = ", ".join(f"{r}/{N} rows of {'pn3t' if t == 124 else 'pn4t'} {K}->{N}"
                     for (t, K, r, _, _), (_, _, N) in zip(work, tensors))
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "GB/s",
        "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": dt * 1e3 / max(1, args.steps),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic",
        "config": {"workload": name, "M": M,
                   "oracle": "plain C, fp64 accumulation, rows split over threads"},
        "cpu_baseline": {"value": value, "unit": "GB/s", "cores": use, "kind": "oracle",
                         "sample": f"each step: {desc}, M={M}"},
        "e2e": {"value": value, "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def run_prefill(args, world, rank, local):
    """The prefill path (config 6): one pn_prefill call per step -- the PN
    rows rebuilt as fp16 into a scratch buffer holding the whole tensor, then
    the tcgen05 GEMM with M tokens.  value = GEMM flops (2 M N K) per second."""
    import torch
    from bit_weight_only_pn_gb300 import build, pn, synth
    if rank == 0 or not os.path.exists(pn.LIBRARY):
        build.build()
    dist_barrier(world)
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    name, tensors, M = workload(args.config)
    (t, K, N), = tensors
    steps = min(args.steps, 200)              # a step is ~0.5 ms: 200 keep the timed region short
    warmup = min(max(args.warmup, 3), 20)
    flops = 2.0 * M * N * K
    w = torch.from_numpy(synth.weights(synth.weight_seed(args.config, 0), N, K)).to(dev)
    W = pn.pack(t, w)
    del w
    x = torch.from_numpy(synth.activations(synth.x_seed(args.config, 0), M, K)).to(dev)
    y = torch.empty((M, N), dtype=torch.float32, device=dev)
    scratch = torch.empty(N * K, dtype=torch.float16, device=dev)
    ws = pn.Workspace(N, dev)
    stream = torch.cuda.Stream(device=dev)

    def timed(fn, n):
        with torch.cuda.stream(stream):
            for _ in range(warmup):
                fn()
        torch.cuda.synchronize(dev)
        a = torch.cuda.Event(enable_timing=True)
        b = torch.cuda.Event(enable_timing=True)
        dist_barrier(world)
        torch.cuda.synchronize(dev)
        a.record(stream)
        with torch.cuda.stream(stream):
            for _ in range(n):
                fn()
        b.record(stream)
        torch.cuda.synchronize(dev)
        dist_barrier(world)
        return dist_max(world, a.elapsed_time(b)) / n

    step = lambda: pn.prefill(t, W, K, x, y=y, scratch=scratch, workspace=ws, stream=stream)
    props = torch.cuda.get_device_properties(local)
    uuid = getattr(props, "uuid", None)
    clocks = ClockSampler(f"GPU-{uuid}" if uuid is not None else local)
    clocks.start()
    time.sleep(0.3)
    clocks.mark()
    ms_per_step = timed(step, steps)
    clocks.mark()
    clock_info = clocks.stop()
    if ws.status(stream) != 0:
        raise RuntimeError("device-side error in the timed region")
    # the two kernels of a step, each timed alone on the same buffers
    w16 = scratch.view(N, K)
    ms_gemm = timed(lambda: pn.gemm_f16(w16, x, y=y, workspace=ws, stream=stream), steps)
    ms_unpack = timed(lambda: pn.unpack_f16(t, W, K, out=w16, stream=stream), steps)
    value = world * flops / (ms_per_step / 1e3) / 1e12

    e2e = None
    if args.e2e_steps > 0:
        xh = torch.from_numpy(synth.activations(synth.x_seed(args.config, 0) + 1000, M, K)).pin_memory()
        yh = torch.empty((M, N), dtype=torch.float32).pin_memory()

        def e2e_step():
            x.copy_(xh, non_blocking=True)
            step()
            yh.copy_(y, non_blocking=True)
            stream.synchronize()

        n_e2e = min(args.e2e_steps, 20)
        e_ms = timed(e2e_step, n_e2e)
        e2e = {"value": world * flops / (e_ms / 1e3) / 1e12, "unit": "TFLOP/s",
               "h2d_bytes_per_step": xh.numel() * 2, "d2h_bytes_per_step": yh.numel() * 4,
               "us_per_step": e_ms * 1e3, "steps": n_e2e,
               "path": "pinned x -> device, pn_prefill via the Python binding, y -> pinned host, "
                       "stream synchronised each step; PN weights resident"}

    peak = None
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as fh:
            peak = float(json.load(fh)["bf16_tflops"])
        peak_src = "measured cuBLAS bf16 burst (MEASURED_PEAKS.json bf16_tflops); fp16 runs at the bf16 rate"
    except (OSError, KeyError, ValueError):
        peak, peak_src = 1900.0, "fallback 1.9 PFLOP/s bf16 burst"
    achieved = flops / (ms_gemm / 1e3) / 1e12
    roofline = {"bound": "tensor", "achieved": achieved, "peak": peak, "unit": "TFLOP/s",
                "frac": achieved / peak, "traffic": recorded_traffic(args.config), "peak_source": peak_src,
                "kernel": "gemm_f16_kernel", "kernel_ms": ms_gemm}

    cpu = None
    if rank == 0 and not args.no_cpu_baseline:
        rate, desc, used = oracle_prefill_rate(t, K, N, M, args.cpu_seconds)
        cpu = {"value": rate, "unit": "TFLOP/s", "cores": used, "kind": "oracle", "sample": desc}
    if rank != 0:
        return
    line = {
        "metric": "PN prefill TFLOP/s (fp16 rebuild + tcgen05 GEMM)", "value": value, "unit": "TFLOP/s",
        "n_gpus": world, "steps": steps, "warmup": warmup, "ms_per_step": ms_per_step,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "f16 products, f32 accumulate", "data": "synthetic",
        "config": {"workload": name, "M": M, "tensors": [f"pn3t {K}->{N}"],
                   "scratch": f"fp16, all {N} rows ({N * K * 2 / 1e6:.0f} MB), one chunk",
                   "l2": "working set (PN rows, fp16 rows, x, y: 540 MB) larger than L2",
                   "launch": "direct launches, two per step (rebuild, GEMM)",
                   "parallelism": "replicas" if world > 1 else "1 GPU"},
        "ms_gemm": ms_gemm, "ms_unpack_f16": ms_unpack,
        "gpu_launches": 2 * steps,
        "roofline": roofline,
        "clocks": clock_info,
        "e2e": e2e,
        "cpu_baseline": cpu,
    }
    print(json.dumps(line), flush=True)


def oracle_prefill_rate(t, K, N, M, seconds):
    """The CPU oracle's prefill (fp16 rebuild + fp64 GEMM) on a sample of
    rows and tokens, repeated for about `seconds`; returns (TFLOP/s of the
    GEMM's 2 M N K, description, threads)."""
    import oracle
    from bit_weight_only_pn_gb300 import synth
    o = oracle.Oracle()
    rows, toks = 64, 64
    W = o.pack(t, synth.weight_rows(synth.weight_seed(9, 0), N, K, range(rows)))
    x = synth.activations(synth.x_seed(9, 0), toks, K)
    s = time.perf_counter()
    o.gemm_f16(o.unpack_f16(t, W, K), x, want_abs=False)
    first = time.perf_counter() - s
    passes = max(1, int(round(seconds / max(first, 1e-6))))
    s = time.perf_counter()
    for _ in range(passes):
        o.gemm_f16(o.unpack_f16(t, W, K), x, want_abs=False)
    dt = time.perf_counter() - s
    return (2.0 * rows * toks * K * passes / dt / 1e12,
            f"{rows}/{N} rows x {toks}/{M} tokens, {passes} passes in {dt:.1f} s on 1 thread", 1)


def run_reference_prefill(args, world, rank):
    """The CPU oracle as the reference arm of the prefill workload (rank 0):
    each step rebuilds and multiplies a fixed sample of rows and tokens."""
    if rank != 0:
        return
    from bit_weight_only_pn_gb300 import synth
    name, tensors, M = workload(args.config)
    (t, K, N), = tensors
    per_step = 120.0 / max(1, args.steps + args.warmup)
    rate, desc, used = oracle_prefill_rate(t, K, N, M, per_step)
    line = {
        "impl": "reference", "metric": "PN prefill TFLOP/s (fp16 rebuild + tcgen05 GEMM)", "value": rate,
        "unit": "TFLOP/s", "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": 2.0 * M * N * K / (rate * 1e12) * 1e3, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": name, "M": M, "oracle": "plain C, fp64 accumulation"},
        "cpu_baseline": {"value": rate, "unit": "TFLOP/s", "cores": used, "kind": "oracle", "sample": desc},
        "e2e": {"value": rate, "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


PREHEAT_S = 0.5              # untimed graph replays before every timed region
SLEEP_CYCLES = 400_000       # about 0.2 ms of GPU sleep ahead of each timed region


def measure_gemv(args, cfg, m_override, world, dev, e2e_steps):
    """Times one GEMV workload: `args.steps` steps (one fused launch each)
    after `args.warmup` warm-up steps, every captured graph replayed once and
    PREHEAT_S seconds of replays before the timed region, which covers exactly
    `args.steps` steps.  Returns a dict of the figures of the bench line."""
    import torch
    from bit_weight_only_pn_gb300 import pn, synth
    name, tensors, M = workload(cfg, m_override)
    default_m = workload(cfg)[2] == M
    algo = {"auto": pn.ALGO_AUTO, "tc": pn.ALGO_TENSOR_CORE, "cuda_core": pn.ALGO_CUDA_CORE,
            "cuda_core_staged": pn.ALGO_CUDA_CORE_STAGED}[args.algo]
    step_bytes = algorithmic_bytes(tensors, M)
    wbytes = sum(N * (K // per_block(t)) * 34 for t, K, N in tensors)
    copies = max(2, int(np.ceil(ROTATE_BYTES / wbytes)))

    # Inputs: seeded fp32 weights quantised on the device by pn_pack, x fp16.
    # Every tensor's x is a view into one contiguous buffer, and so is every
    # tensor's y of one weight copy (offsets M*K*2 bytes keep each x 16-byte
    # aligned), so an end-to-end step moves its inputs and its outputs with
    # one copy each way.
    x_offs = np.cumsum([0] + [M * K for _, K, _ in tensors])
    y_offs = np.cumsum([0] + [M * N for _, _, N in tensors])
    x_all = torch.empty(int(x_offs[-1]), dtype=torch.float16, device=dev)
    sets = []
    for e, (t, K, N) in enumerate(tensors):
        w = torch.from_numpy(synth.weights(synth.weight_seed(cfg, e), N, K)).to(dev)
        W0 = pn.pack(t, w)
        del w
        xs = x_all[int(x_offs[e]):int(x_offs[e + 1])].view(M, K)
        xs.copy_(torch.from_numpy(synth.activations(synth.x_seed(cfg, e), M, K)))
        sets.append((t, K, N, W0, xs))
    # with --hadamard every tensor's GEMV reads a rotated copy of its activations
    xr = [torch.empty_like(xs) for _, _, _, _, xs in sets] if args.hadamard else None
    rot, y_all = [], []
    for c in range(copies):
        entries = []
        y_all.append(torch.empty(int(y_offs[-1]), dtype=torch.float32, device=dev))
        for e, (t, K, N, W0, xs) in enumerate(sets):
            W = W0 if c == 0 else W0.clone()
            y = y_all[c][int(y_offs[e]):int(y_offs[e + 1])].view(M, N)
            entries.append((t, W, K, xr[e] if xr is not None else xs, y))
        rot.append(entries)
    total_rows = sum(N for _, _, N in tensors)
    ws = pn.Workspace(total_rows, dev)
    stream = torch.cuda.Stream(device=dev)

    def step(entries):
        if xr is not None:
            for (_, _, _, _, xs), xo in zip(sets, xr):
                pn.hadamard(xs, args.hadamard, out=xo, stream=stream)
        if args.fused_hadamard:
            if len(entries) == 1:
                t, W, K, x, y = entries[0]
                pn.gemv_hadamard(t, W, K, x, args.fused_hadamard, y=y, workspace=ws, stream=stream)
            else:
                pn.gemv_layer_hadamard(entries, M, args.fused_hadamard, workspace=ws, stream=stream)
        elif len(entries) == 1:
            t, W, K, x, y = entries[0]
            pn.gemv(t, W, K, x, y=y, workspace=ws, algo=algo, stream=stream)
        else:
            pn.gemv_layer(entries, M, workspace=ws, algo=algo, stream=stream)

    # warm up eagerly (also sets the kernel's shared-memory attribute)
    with torch.cuda.stream(stream):
        for i in range(max(3, min(args.warmup, 3 * copies))):
            step(rot[i % copies])
    torch.cuda.synchronize(dev)
    if ws.status(stream) != 0:
        raise RuntimeError("device-side error during warm-up")

    def capture(n, first=0):
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            for i in range(first, first + n):
                step(rot[i % copies])
        return g

    nodes = max(1, min(GRAPH_NODES, args.steps))
    g_full = capture(nodes)
    rem = args.steps % nodes
    g_rem = capture(rem, nodes) if rem else None
    reps = args.steps // nodes
    graphs = [g_full] + ([g_rem] if g_rem is not None else [])

    def preheat():
        """Replays every graph once (its first replay uploads it), the
        warm-up steps, then graph replays for PREHEAT_S seconds so that clocks
        and the overlap of back-to-back launches are at steady state."""
        with torch.cuda.stream(stream):
            for g in graphs:
                g.replay()
            for i in range(args.warmup):
                step(rot[i % copies])
        torch.cuda.synchronize(dev)
        t0 = time.perf_counter()
        n = 0
        while time.perf_counter() - t0 < PREHEAT_S:
            with torch.cuda.stream(stream):
                for _ in range(4):
                    g_full.replay()
            torch.cuda.synchronize(dev)
            n += 4
        return (time.perf_counter() - t0) * 1e3, n * nodes

    preheat_ms, preheat_steps = preheat()
    props = torch.cuda.get_device_properties(dev)
    uuid = getattr(props, "uuid", None)
    clocks = ClockSampler(f"GPU-{uuid}" if uuid is not None else dev.index)
    clocks.start()
    time.sleep(0.3)
    # keep the GPU busy while the sampler starts, then settle it again
    preheat()
    start = torch.cuda.Event(enable_timing=True)
    end = torch.cuda.Event(enable_timing=True)
    dist_barrier(world)
    torch.cuda.synchronize(dev)
    clocks.mark()
    # the GPU waits on a short sleep kernel while the host enqueues the start
    # event and the graphs, so no host launch latency falls inside the region
    with torch.cuda.stream(stream):
        torch.cuda._sleep(SLEEP_CYCLES)
    start.record(stream)
    with torch.cuda.stream(stream):
        for _ in range(reps):
            g_full.replay()
        if g_rem is not None:
            g_rem.replay()
    end.record(stream)
    torch.cuda.synchronize(dev)
    clocks.mark()
    dist_barrier(world)
    clock_info = clocks.stop()
    ms = start.elapsed_time(end)
    ms = dist_max(world, ms)
    status = ws.status(stream)
    if status != 0:
        raise RuntimeError(f"device-side error in the timed region: {status}")
    ms_per_step = ms / args.steps
    value = world * step_bytes * args.steps / (ms / 1e3) / 1e9

    # end to end through the public API: pinned x in, pinned y out, every step
    e2e = None
    if e2e_steps > 0:
        xh = torch.cat([torch.from_numpy(synth.activations(synth.x_seed(cfg, e) + 1000, M, K)).reshape(-1)
                        for e, (t, K, N) in enumerate(tensors)]).pin_memory()
        yh = torch.empty(int(y_offs[-1]), dtype=torch.float32).pin_memory()
        h2d = xh.numel() * 2
        d2h = yh.numel() * 4
        n_e2e = e2e_steps

        host_call = not args.hadamard and not args.fused_hadamard and algo == pn.ALGO_AUTO
        calls = [pn.LayerCall(entries, M, ws) for entries in rot] if host_call else None

        def e2e_step(i):
            if host_call:
                # one C-ABI call: x in from pinned host memory, the GEMVs, y out, wait
                calls[i % copies].host(xh, yh, stream=stream)
                return
            x_all.copy_(xh, non_blocking=True)          # every tensor's x (or the rotation's input)
            step(rot[i % copies])
            yh.copy_(y_all[i % copies], non_blocking=True)
            stream.synchronize()

        with torch.cuda.stream(stream):
            for i in range(min(20, n_e2e)):
                e2e_step(i)
            dist_barrier(world)
            torch.cuda.synchronize(dev)
            e0 = torch.cuda.Event(enable_timing=True)
            e1 = torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            for i in range(n_e2e):
                e2e_step(i)
            e1.record(stream)
            torch.cuda.synchronize(dev)
        e_ms = dist_max(world, e0.elapsed_time(e1))
        e2e = {"value": world * step_bytes * n_e2e / (e_ms / 1e3) / 1e9, "unit": "GB/s",
               "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
               "us_per_step": e_ms * 1e3 / n_e2e, "steps": n_e2e,
               "path": ("pn_gemv_layer_host through the Python binding (pn.LayerCall, arguments marshalled "
                        "once): pinned host x -> device (one copy "
                        "for all tensors), the GEMV launch, y -> pinned host (one copy), stream synchronised, "
                        "all inside one C-ABI call per step; weights resident") if host_call else
                       ("pinned x -> device (one copy for all tensors), the rotation and the GEMV via the "
                        "Python binding, y -> pinned host (one copy), stream synchronised each step; "
                        "weights resident")}

    # read-only ceiling on the same box and buffers: one pn_read_ranges
    # launch per step reads the step's weight copies once (16-byte loads, no
    # decode), in CUDA graphs like the GEMV steps, after the same pre-heat
    sink = torch.zeros(len(tensors), dtype=torch.int32, device=dev)

    def read_step(i):
        pn.read_ranges([W for (_, W, _, _, _) in rot[i % copies]], sink, stream=stream)

    with torch.cuda.stream(stream):
        for i in range(3 * copies):
            read_step(i)
        gr = torch.cuda.CUDAGraph()
        with torch.cuda.graph(gr, stream=stream):
            for i in range(nodes):
                read_step(i)
        gr.replay()
    torch.cuda.synchronize(dev)
    t0 = time.perf_counter()
    while time.perf_counter() - t0 < PREHEAT_S:
        with torch.cuda.stream(stream):
            for _ in range(4):
                gr.replay()
        torch.cuda.synchronize(dev)
    with torch.cuda.stream(stream):
        r0 = torch.cuda.Event(enable_timing=True)
        r1 = torch.cuda.Event(enable_timing=True)
        r_reps = max(1, reps)
        torch.cuda._sleep(SLEEP_CYCLES)
        r0.record(stream)
        for _ in range(r_reps):
            gr.replay()
        r1.record(stream)
    torch.cuda.synchronize(dev)
    r_us = r0.elapsed_time(r1) * 1e3 / (r_reps * nodes)
    read_ceiling = {"us_per_step": r_us, "gbs": wbytes / (r_us / 1e6) / 1e9,
                    "time_frac": r_us / (ms_per_step * 1e3),
                    "how": "pn_read_ranges over the same rotating PN weight copies (one launch per "
                           "step, 16-byte loads, no decode), CUDA graphs; time_frac = read time / GEMV time"}

    peak, peak_kind = measured_peak()
    per_gpu = step_bytes / (ms_per_step / 1e3) / 1e9
    roofline = {"bound": "hbm", "achieved": per_gpu, "peak": peak, "unit": "GB/s",
                "frac": per_gpu / peak,
                "traffic": recorded_traffic(cfg) if (default_m and not args.hadamard and not args.fused_hadamard
                                                     and args.algo == "auto")
                else None,
                "peak_source": f"{peak_kind} copy bandwidth (MEASURED_PEAKS.json hbm_gbs)"
                               if peak_kind == "measured" else "fallback 6.8 TB/s"}
    launches = args.steps * ((1 if len(tensors) == 1 or algo != pn.ALGO_CUDA_CORE else len(tensors))
                             + (len(tensors) if args.hadamard else 0))
    return {
        "name": name, "tensors": tensors, "M": M, "value": value, "ms_per_step": ms_per_step,
        "step_bytes": step_bytes, "wbytes": wbytes, "copies": copies, "nodes": nodes,
        "per_gpu": per_gpu, "roofline": roofline, "read_ceiling": read_ceiling, "clocks": clock_info,
        "e2e": e2e, "launches": launches, "preheat_ms": preheat_ms, "preheat_steps": preheat_steps,
    }


def run_ours(args, world, rank, local):
    import torch
    from bit_weight_only_pn_gb300 import build, pn
    if rank == 0 or not os.path.exists(pn.LIBRARY):
        build.build()             # no-op when the library is up to date
    dist_barrier(world)
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    r = measure_gemv(args, args.config, args.m, world, dev, args.e2e_steps)
    # the metric's other half: the skinny verification batch (M = 8) over the
    # 27B-class layer, timed the same way, in the same line
    m8 = None
    if not args.no_m8 and args.config != 4 and not args.m and not args.fused_hadamard:
        q = measure_gemv(args, 4, 0, world, dev, min(args.e2e_steps, 200))
        m8 = {"workload": q["name"], "M": q["M"], "us_per_gemv": q["ms_per_step"] * 1e3,
              "value": q["value"], "unit": "GB/s", "steps": args.steps, "warmup": args.warmup,
              "pct_of_nominal_8tbs": q["per_gpu"] / NOMINAL_HBM_GBS * 100.0,
              "algorithmic_bytes_per_step": q["step_bytes"],
              "roofline": q["roofline"], "read_ceiling": q["read_ceiling"], "clocks": q["clocks"],
              "e2e": q["e2e"], "gpu_launches": q["launches"], "preheat_ms": q["preheat_ms"]}
        del q
        torch.cuda.empty_cache()

    cpu = None
    if rank == 0 and not args.no_cpu_baseline:
        rate, desc, used, _ = oracle_sample_rate(r["tensors"], r["M"], args.cpu_seconds, os.cpu_count() or 1)
        rate1, desc1, _, _ = oracle_sample_rate(r["tensors"], r["M"], args.cpu_seconds / 2, 1)
        cpu = {"value": rate, "unit": "GB/s", "cores": used, "kind": "oracle", "sample": desc,
               "value_one_core": rate1, "sample_one_core": desc1, "cpu_model": cpu_model()}

    if rank != 0:
        return
    tensors = r["tensors"]
    line = {
        "metric": METRIC, "value": r["value"], "unit": "GB/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": r["ms_per_step"], "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f16 products, f32 accumulate",
        "data": "synthetic",
        "config": {"workload": r["name"], "M": r["M"],
                   "tensors": [f"{'pn3t' if t == 124 else 'pn4t'} {K}->{N}" for t, K, N in tensors],
                   "algorithmic_bytes_per_step": r["step_bytes"], "weight_bytes_per_step": r["wbytes"],
                   "l2": f"{r['copies']} rotating weight copies ({r['copies'] * r['wbytes'] / 1e6:.0f} MB > 2x L2)",
                   "launch": f"CUDA graph of {r['nodes']} steps, replayed; every graph replayed and "
                             f"{PREHEAT_S:.1f} s of replays untimed before the timed region",
                   "parallelism": "replicas" if world > 1 else "1 GPU",
                   "algo": args.algo,
                   "hadamard_block": args.hadamard or None,
                   "fused_hadamard_block": args.fused_hadamard or None},
        "us_per_gemv": r["ms_per_step"] * 1e3,
        "pct_of_nominal_8tbs": r["per_gpu"] / NOMINAL_HBM_GBS * 100.0,
        "gpu_launches": r["launches"],
        "preheat_ms": r["preheat_ms"],
        "roofline": r["roofline"],
        "read_ceiling": r["read_ceiling"],
        "clocks": r["clocks"],
        "e2e": r["e2e"],
        "m8": m8,
        "cpu_baseline": cpu,
    }
    print(json.dumps(line), flush=True)


def run_gptq(args, world, rank):
    """The offline quantiser (pn_gptq), not the GEMV: seconds per tensor on the
    device, and device against oracle on a small sample (K = 640, 64 rows)."""
    import numpy as np
    import torch
    from bit_weight_only_pn_gb300 import build, pn, synth
    if rank != 0:
        return
    build.build()
    dev = torch.device("cuda", 0)
    t, K, N = synth.CONFIGS[args.config]["tensors"][0]
    n = 256

    def inputs(N, K, seed):
        rng = np.random.default_rng(seed)
        w = synth.weights(synth.weight_seed(args.config, 0), N, K)
        A = rng.standard_normal((K, K)) * (0.3 / np.sqrt(K / 64)) + np.eye(K)
        X = (rng.standard_normal((n, K)) @ A).astype(np.float32)
        return w, X

    def time_device(w, X, reps):
        wd, Xd = torch.from_numpy(w).to(dev), torch.from_numpy(X).to(dev)
        pn.gptq(t, wd, Xd)                                    # warm-up (module load, allocations)
        torch.cuda.synchronize()
        t0 = time.perf_counter()
        for _ in range(reps):
            W = pn.gptq(t, wd, Xd)
        torch.cuda.synchronize()
        return (time.perf_counter() - t0) / reps, W

    w, X = inputs(N, K, 1)
    full_s, _ = time_device(w, X, max(1, min(args.steps, 3)))
    ws, Xs = inputs(64, 640, 2)
    small_s, Wsmall = time_device(ws, Xs, 3)
    o = None
    oracle_s = None
    try:
        import oracle as oracle_mod
        o = oracle_mod.Oracle()
        t0 = time.perf_counter()
        want = o.gptq(t, ws, Xs, 0.01)
        oracle_s = time.perf_counter() - t0
        same = bool(np.array_equal(Wsmall.cpu().numpy(), want))
    except Exception as e:                                    # the oracle is optional here
        same = f"oracle unavailable: {e}"
    flops = 2.0 * N * K * K / 2 + 4.0 * K ** 3 / 3 + 2.0 * n * K * K
    print(json.dumps({
        "metric": "PN GPTQ-style quantisation time (device, offline tool)", "value": full_s, "unit": "s",
        "higher_is_better": False, "n_gpus": 1, "steps": max(1, min(args.steps, 3)), "dtype": "f64",
        "data": "synthetic", "config": {"workload": f"{'pn3t' if t == 124 else 'pn4t'} {K}->{N}, "
                                                   f"{n} calibration rows", "parallelism": "1 GPU"},
        "fp64_gflop": flops / 1e9, "fp64_gflops_achieved": flops / full_s / 1e9,
        "small_sample": {"workload": f"K=640, 64 rows, {n} calibration rows", "device_s": small_s,
                         "oracle_s": oracle_s, "bytes_equal_oracle": same}}))


def main():
    args = parse_args()
    world, rank, local = dist_setup(args)
    from bit_weight_only_pn_gb300 import synth
    prefill = synth.CONFIGS[args.config].get("prefill", False)
    if args.gptq:
        run_gptq(args, world, rank)
    elif args.impl == "reference":
        run_reference_prefill(args, world, rank) if prefill else run_reference(args, world, rank)
    elif prefill:
        run_prefill(args, world, rank, local)
    else:
        run_ours(args, world, rank, local)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
