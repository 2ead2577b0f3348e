"""Benchmark of the complex chunkwise SSD forward (libssdc) on GB300.

One step = one forward pass of the whole scan (every row of the chunked
decomposition; one fused kernel launch on the TF32 path) over the single-layer
production workload (B=2, T=2048, H=16, D=N=64 complex, Q=64), inputs resident
in HBM. Metric: token-heads/s
(B*T*H per step). L2 is flushed (a 512 MiB write) before every timed step and
each step is timed on its stream with CUDA events.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
    python bench.py --backward [--workload ...] [--real-x]   (the backward pass)

Under torchrun each rank runs its own independent batch (weak scaling, no
collective on the data path); rank 0 prints one JSON line.
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

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from state_space_sequence_complex_gb300 import inputs  # noqa: E402

METRIC = "complex-SSD fwd token·heads/s at Q=64 and % of roofline (HBM or TF32)"  # the value is token·heads/s; the fraction is roofline.frac
UNIT = "token·heads/s"
FLUSH_BYTES = 512 << 20


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=1000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--precision", choices=["auto", "tf32", "fp32"], default="auto")
    ap.add_argument("--workload", choices=["layer", "train28", "qsweep", "long"], default="layer",
                    help="layer: the headline single-layer workload; the others are measurement modes "
                         "with device-generated inputs (no CPU baseline, no end-to-end figure)")
    ap.add_argument("--chunk", type=int, default=0, help="chunk size Q (default: the workload's)")
    ap.add_argument("--layers", type=int, default=0,
                    help="measurement mode: run this many of the workload's layers (default: all), e.g. one "
                         "training-batch layer for a profiler capture")
    ap.add_argument("--batch", type=int, default=0,
                    help="measurement mode: override the workload's batch size B (e.g. a smaller case of "
                         "the same shape for a profiler capture)")
    ap.add_argument("--segments", type=int, default=1,
                    help="measurement mode: process T in this many segments, each started from the "
                         "previous segment's final state (the initial-state entry point)")
    ap.add_argument("--bf16", action="store_true",
                    help="measurement mode: x, B_t and C_t in bfloat16 (ssd_complex_fwd_bf16), the rest fp32")
    ap.add_argument("--mimo", action="store_true",
                    help="measurement mode: the forward with the MIMO head mixer (ssd_complex_fwd_mimo: the scan "
                         "writes Re(y), a second kernel mixes it in place), timed against the mixer fused into "
                         "the scan's epilogue and against the plain forward plus a torch einsum")
    ap.add_argument("--state-only", action="store_true",
                    help="measurement mode: the final state alone (ssd_complex_final_state: reads x, B_t, dt; "
                         "no y), as the joining of time segments uses it")
    ap.add_argument("--real-x", action="store_true",
                    help="measurement mode: x real (x.im = NULL, only x.re is read), as in the model")
    ap.add_argument("--backward", action="store_true",
                    help="measurement mode: time the backward pass (ssd_complex_bwd, exact fp32) "
                         "on the workload, seeded with random output gradients")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    return ap.parse_args()


def dist_env():
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return rank, world, local


def rank_layer(rank: int) -> int:
    """Seed offset of rank `rank`'s batch: every rank runs its own independent
    batch of the workload (weak scaling, no data-path collective)."""
    return rank


def max_over_ranks(values, device=None):
    """Element-wise max of a list of floats over all ranks (identity when not
    distributed)."""
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return [float(v) for v in values]
    t = torch.tensor([float(v) for v in values], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return [float(v) for v in t.tolist()]


def peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    except Exception:
        return 6800.0, "fallback"


def fp32_flops_per_unit(w) -> dict:
    """Algorithmic real flops per token-head of each launch of the exact fp32 path (causal
    triangle only): chunk state S_loc = B^T (dec o x): 8 N D; state pass: 8 N D / Q; chunk
    scan: C B^T and P x over the causal triangle, 4 (Q+1) (N + D), and (C o e^Acs) S_in, 8 N D."""
    N, D, Q = w.N, w.D, w.Q
    return {"chunk_state": 8.0 * N * D, "state_pass": 8.0 * N * D / Q,
            "chunk_scan": 4.0 * (Q + 1) * (N + D) + 8.0 * N * D}


def bwd_flops_per_unit(w) -> dict:
    """Algorithmic real flops per token-head of each launch of the backward pass (causal
    triangle, every product counted once). Chunk states: the forward's S_loc = B^T (dec o x)
    (recomputed) and U = C'^H dY, 8 N D each; the two chunk recurrences: 8 N D / Q each;
    chunk gradients: per causal pair C B^T, P^H dY, dY x^H, V^T conj(C) and V conj(B)
    (24 N + 16 D), i.e. (Q+1)(12 N + 8 D) per token, plus the three state terms (24 N D);
    step-size gradients: about 12 per token; the per-head sum of dA: 2 per chunk."""
    N, D, Q = w.N, w.D, w.Q
    return {"chunk_states": 16.0 * N * D, "passes": 16.0 * N * D / Q,
            "bwd_chunk": (Q + 1) * (12.0 * N + 8.0 * D) + 24.0 * N * D + 16.0 * N + 8.0 * N * D / Q,
            "bwd_dt": 12.0, "bwd_dA": 2.0 / Q}


BWD_NAMES = ["chunk_states", "passes", "bwd_chunk", "bwd_dt", "bwd_dA"]


def bf16_peak_tflops() -> float:
    """The measured burst BF16 dense peak of MEASURED_PEAKS.json (0 if absent)."""
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            return float(json.load(f)["bf16_tflops"])
    except Exception:
        return 0.0


def fp32_alu_peak_tflops(dev_index: int):
    """FP32 FMA peak of the CUDA cores: SMs x 128 FP32 lanes x 2 flops x the maximum SM clock."""
    import torch
    sms = torch.cuda.get_device_properties(dev_index).multi_processor_count
    mhz = 2070.0
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            mhz = float(json.load(f).get("sm_max_mhz", mhz))
    except Exception:
        pass
    return sms * 128 * 2 * mhz * 1e6 / 1e12, f"derived: {sms} SMs x 128 FP32 lanes x 2 flops x {mhz:.0f} MHz"


def profiled_traffic(kernel: str):
    """DRAM bytes per launch (read + write) from the committed ncu summary of
    `kernel`, or None if the kernel source changed since that capture."""
    d = profiled_dram(kernel)
    return None if d is None else d["traffic"]


def profiled_dram(kernel: str):
    """DRAM bytes per launch from the committed ncu summary of `kernel`:
    {"traffic", "read", "write"} (read and write None where the summary gives
    only their sum), or None if the kernel source changed since that capture."""
    import hashlib
    files = {"fused_kernel": ("profiles/fused_kernel_single_layer.md",
                              "state_space_sequence_complex_gb300/csrc/ssdc_fused.cu"),
             "fused_tmem_kernel": ("profiles/fused_tmem_kernel_training_batch.md",
                                   "state_space_sequence_complex_gb300/csrc/ssdc_fused2.cu"),
             "bwd_chunk": ("profiles/bwd_chunk_single_layer.md",
                           "state_space_sequence_complex_gb300/csrc/ssdc_bwd.cu")}
    if kernel not in files:
        return None
    prof, src = (os.path.join(ROOT, f) for f in files[kernel])
    keys = ("traffic_bytes_per_launch", "dram_read_bytes_per_launch", "dram_write_bytes_per_launch",
            "source_sha256_16")
    try:
        fields = dict(line.split(": ", 1) for line in open(prof).read().splitlines() if ": " in line
                      and line.split(": ", 1)[0] in keys)
        digest = hashlib.sha256(open(src, "rb").read()).hexdigest()[:16]
        if fields.get("source_sha256_16", "").strip() != digest:
            return None
        get = lambda k: float(fields[k]) if k in fields else None
        return {"traffic": get("traffic_bytes_per_launch"), "read": get("dram_read_bytes_per_launch"),
                "write": get("dram_write_bytes_per_launch")}
    except Exception:
        return None


def algorithmic_bytes_per_unit(w) -> float:
    # x, B_t, C_t read and y written (complex64 = 8 B each element), dt read,
    # final state written once per sequence.
    return 16 * w.D + 16 * w.N + 4 + 8 * w.N * w.D / w.T


def input_bytes_per_unit(w, bf16=False, real_x=False, mimo=False, state_only=False) -> float:
    """algorithmic_bytes_per_unit with x, B_t, C_t in bfloat16 (2 bytes a plane element
    instead of 4: 4 D + 8 N fewer), a real x (no imaginary plane), the head mixer
    (only the mixed Re(y) leaves the call: 4 D fewer; the separate mixer's round trip
    of Re(y), 8 D more, is not counted as algorithmic) and / or the final state alone
    (ssd_complex_final_state: no C_t read and no y written, 8 N + 8 D fewer)."""
    b = algorithmic_bytes_per_unit(w)
    if state_only:
        b -= 8.0 * w.N + 8.0 * w.D
    if mimo:
        b -= 4.0 * w.D
    if bf16:
        b -= 4.0 * w.D + 8.0 * w.N
    if real_x:
        b -= (2.0 if bf16 else 4.0) * w.D
    return b


class ClockSampler:
    """nvidia-smi samples of SM clock and throttle reasons while running."""

    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None
        self.lines = []
        self.t = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "50"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.proc = None
            return
        self.t = threading.Thread(target=self._read, daemon=True)
        self.t.start()

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        if self.t:
            self.t.join(timeout=2)
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) < 8:
                continue
            try:
                sm.append(float(parts[0]))
                mx.append(float(parts[1]))
            except ValueError:
                continue
            for nm, v in zip(names, parts[4:8]):
                if v.lower().startswith("active"):
                    reasons.add(nm)
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(mx) if mx else None,
                "reasons": sorted(reasons), "samples": len(sm)}


def run_oracle_baseline(w, inp, max_seconds=12.0, max_reps=400):
    """Time the CPU oracle, as it stands, on the full workload, repeated."""
    from oracle import naive_scan_inputs
    from oracle.ssd_oracle import default_threads
    cores = default_threads()
    reps, t_total = 0, 0.0
    while reps < max_reps and t_total < max_seconds:
        t0 = time.perf_counter()
        naive_scan_inputs(inp, threads=cores)
        t_total += time.perf_counter() - t0
        reps += 1
    units = w.token_heads * reps
    return {"value": units / t_total, "unit": UNIT, "cores": cores, "kind": "oracle",
            "sample": f"full workload ({w.name}) x {reps} passes, {t_total:.1f} s"}


def reference_arm(args, w):
    rank, world, _ = dist_env()
    if rank != 0:
        return
    from oracle import naive_scan_inputs
    from oracle.ssd_oracle import default_threads
    inp = inputs.generate(w)
    cores = default_threads()
    # each step is one full pass of the workload on the host cores
    for _ in range(args.warmup):
        naive_scan_inputs(inp, threads=cores)
    times = []
    for _ in range(args.steps):
        t0 = time.perf_counter()
        naive_scan_inputs(inp, threads=cores)
        times.append(time.perf_counter() - t0)
    ms = 1000.0 * sum(times) / len(times)
    value = w.token_heads / (ms / 1000.0)
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": w.name, "B": w.B, "T": w.T, "H": w.H, "D": w.D, "N": w.N,
                   "chunk_size": w.Q, "seed": w.seed},
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": cores, "kind": "oracle",
                         "sample": f"full workload per step ({w.name})"},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def reduce_param_grads(dA_re, dA_im):
    """Data-parallel backward: every rank holds the gradients of its own batch rows;
    dA, the gradient of the per-head parameter A, sums over all rows, so its two
    planes are summed over the ranks (one all-reduce). Identity on one rank."""
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return
    buf = torch.cat([dA_re.reshape(-1), dA_im.reshape(-1)])
    dist.all_reduce(buf, op=dist.ReduceOp.SUM)
    dA_re.copy_(buf[:dA_re.numel()].view_as(dA_re))
    dA_im.copy_(buf[dA_re.numel():].view_as(dA_im))


def device_layer_inputs(w, layer, dev, g):
    """The inputs of one layer of `w` drawn on the device (torch generator seeded with
    seed + layer) from the distributions of `inputs`: x, A, B_t, C_t planes and dt."""
    import torch
    g.manual_seed(w.seed + layer)
    Bn, T, H, D, N = w.B, w.T, w.H, w.D, w.N
    s = math.sqrt(0.5)
    A_re = torch.empty(H, device=dev).uniform_(w.re_lo, w.re_hi, generator=g)
    sign = torch.where(torch.rand(H, device=dev, generator=g) < 0.5, -1.0, 1.0)
    A_im = torch.empty(H, device=dev).uniform_(0.35, 2.20, generator=g) * sign
    dt = torch.randn(Bn, T, H, device=dev, generator=g) * w.dt_std + w.dt_mean
    cp = lambda F: [torch.randn(Bn, T, H, F, device=dev, generator=g) * s for _ in range(2)]
    (x_re, x_im), (B_re, B_im), (C_re, C_im) = cp(D), cp(N), cp(N)
    return [x_re, x_im, A_re, A_im, B_re, B_im, C_re, C_im, dt]


def backward_workload(args, w):
    """Measurement mode for the backward pass: one step = ssd_complex_bwd over every layer
    of the workload (inputs and output gradients drawn on the device), L2 flushed before
    each step. With --real-x the model's case: x real, a loss of Re(y) alone (dy.im null)
    and no final-state gradient. Under torchrun each rank runs its own batch (data
    parallel, weak scaling) and every step all-reduces dA over the ranks."""
    import torch
    from state_space_sequence_complex_gb300 import build, ssdc
    rank, world, local = dist_env()
    if world > 1:
        import torch.distributed as dist
        torch.cuda.set_device(local)
        dist.init_process_group("nccl" if dist.is_nccl_available() else "gloo")
    else:
        torch.cuda.set_device(0)
    dev = torch.device("cuda", torch.cuda.current_device())
    build.build()
    ssdc.load()
    Q = args.chunk or w.Q
    g = torch.Generator(device=dev)
    s = math.sqrt(0.5)
    layers = []
    for i in range(w.layers):
        L = device_layer_inputs(w, i + 1000 * rank_layer(rank), dev, g)
        dy = [torch.randn(w.B, w.T, w.H, w.D, device=dev, generator=g) * s for _ in range(2)]
        dfs = [torch.randn(w.B, w.H, w.N, w.D, device=dev, generator=g) * s for _ in range(2)]
        if args.real_x:
            L[1], dy[1], dfs = None, None, [None, None]
        layers.append(L + dy + dfs)
    # --precision tf32: the chunk gradients on the TF32 tensor cores (Q <= 64)
    precision = "tf32" if args.precision == "tf32" else "fp32"
    b = ssdc.Backward(w.B, w.T, w.H, w.N, w.D, Q, precision, device=dev)

    def run():
        for L in layers:
            b(*L)
            reduce_param_grads(b.grads["dA_re"], b.grads["dA_im"])
    flush = torch.empty(FLUSH_BYTES // 4, dtype=torch.float32, device=dev)
    stream = torch.cuda.current_stream()
    for i in range(max(args.warmup, 3)):
        flush.fill_(float(i))
        run()
    torch.cuda.synchronize()
    sampler = ClockSampler(dev.index)
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    sampler.start()
    time.sleep(0.1)
    ev = []
    for k in range(args.steps):
        flush.fill_(float(k))
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        run()
        e1.record(stream)
        ev.append((e0, e1))
    torch.cuda.synchronize()
    clocks = sampler.stop()
    if world > 1:
        torch.distributed.barrier()
    st = ssdc.ssd_complex_status(b.workspace)
    if st != ssdc.SSDC_OK:
        raise SystemExit(f"device status after timed steps: {ssdc.strerror(st)}")
    ms = sum(a.elapsed_time(e) for a, e in ev) / len(ev)
    ms = max_over_ranks([ms], device=dev)[0]
    ssdc.timing_enable(True)
    per_kernel = []
    for k in range(min(args.steps, 50)):
        flush.fill_(float(k))
        for L in layers:
            b(*L)
            per_kernel.append(ssdc.timing_read())
    ssdc.timing_enable(False)
    nk = min(len(p) for p in per_kernel)
    kmeans = [sum(p[i] for p in per_kernel) / len(per_kernel) for i in range(nk)]
    names = BWD_NAMES if nk == len(BWD_NAMES) else [f"launch{i}" for i in range(nk)]
    top = int(np.argmax(kmeans))
    wq = w.with_(Q=Q)
    fl_unit = bwd_flops_per_unit(wq)
    fl = fl_unit.get(names[top], 0.0) * w.token_heads
    alu_peak, alu_kind = fp32_alu_peak_tflops(dev.index)
    bound, kind_top = "alu", alu_kind
    top_peak = alu_peak
    if precision == "tf32" and names[top] == "bwd_chunk":  # a tensor-core kernel
        bound, top_peak = "tensor", bf16_peak_tflops() * 1.1 / 2.25
        kind_top = "measured cuBLAS bf16 TFLOP/s x the nominal TF32 / BF16 ratio 1.1 / 2.25"
    tf = fl / (kmeans[top] / 1000.0) / 1e12
    # minimum HBM bytes per token-head: x, dy, dx (8 D each, 4 D when real), B_t, C_t, dB_t,
    # dC_t (8 N each), dt and ddt (4 each)
    xb = 4.0 if args.real_x else 8.0
    bytes_unit = 3 * xb * w.D + 32.0 * w.N + 8.0
    units = w.token_heads * w.layers * world
    if rank != 0:
        return
    cpu = None
    if (world == 1 and w.name == inputs.LAYER.name and Q == w.Q and not args.no_cpu_baseline
            and not args.real_x):
        cpu = run_oracle_grad_baseline(w)
    # the FP32 ALU fraction of the whole step (SIMT kernels) is reported either way
    line = {
        "metric": "complex-SSD bwd token·heads/s (" + ("TF32 chunk gradients" if precision == "tf32"
                                                       else "exact fp32 gradients") + " of every input)",
        "value": units / (ms / 1000.0), "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "tf32" if precision == "tf32" else "f32",
        "data": "synthetic, drawn on the device per layer",
        "config": {"workload": f"{w.name} Q{Q} backward" + (", real x, Re(y) loss" if args.real_x else ""),
                   "B": w.B, "T": w.T, "H": w.H, "D": w.D, "N": w.N, "chunk_size": Q,
                   "layers": w.layers, "real_x": bool(args.real_x), "precision": precision,
                   "l2": f"flushed before every timed step ({FLUSH_BYTES >> 20} MiB write)",
                   "parallelism": f"data parallel: {world} batch(es), dA all-reduced each step"},
        "roofline": {"bound": bound, "kernel": names[top], "achieved": tf, "peak": top_peak,
                     "peak_kind": kind_top, "unit": "TFLOP/s", "frac": tf / top_peak,
                     "traffic": profiled_traffic(names[top]) if w.name == inputs.LAYER.name and Q == w.Q
                     and not args.real_x and precision == "fp32" else None,
                     "algorithmic_flops_per_launch": fl,
                     "step_alu_frac": sum(fl_unit.values()) * units / world / (ms / 1000.0) / 1e12 / alu_peak,
                     "hbm_step_frac": bytes_unit * units / world / (ms / 1000.0) / 1e9 / peaks()[0],
                     "kernel_ms": {n: m for n, m in zip(names, kmeans)}},
        "cpu_baseline": cpu,
        "e2e": None,
        "gpu_launches": nk * w.layers * args.steps,
        "clocks": clocks,
    }
    print(json.dumps(line), flush=True)


def run_oracle_grad_baseline(w, max_seconds=12.0, max_reps=100):
    """Time the gradient oracle, as it stands, on the full workload, repeated."""
    from oracle import naive_grad_inputs
    from oracle.ssd_oracle import default_threads
    inp = inputs.generate(w)
    og = inputs.output_grads(w.B, w.T, w.H, w.D, w.N, seed=w.seed + 1000)
    dy = og.dy_re + 1j * og.dy_im
    dfs = og.dfs_re + 1j * og.dfs_im
    cores = default_threads()
    reps, t_total = 0, 0.0
    while reps < max_reps and t_total < max_seconds:
        t0 = time.perf_counter()
        naive_grad_inputs(inp, dy, dfs, threads=cores)
        t_total += time.perf_counter() - t0
        reps += 1
    return {"value": w.token_heads * reps / t_total, "unit": UNIT, "cores": cores, "kind": "oracle",
            "sample": f"full workload ({w.name}) backward x {reps} passes, {t_total:.1f} s"}


def other_workload(args, w):
    """Measurement mode for the training-batch, chunk-sweep and long-memory workloads: inputs
    drawn on the device from the same distributions (torch generator seeded per layer), one
    step = every layer of the workload back to back, L2 flushed before each step. With
    --segments K each layer's sequence is processed as K consecutive segments, every segment
    started from the previous one's final state (updated in place)."""
    import torch
    from state_space_sequence_complex_gb300 import build, ssdc
    torch.cuda.set_device(0)
    dev = torch.device("cuda", 0)
    build.build()
    ssdc.load()
    Q = args.chunk or w.Q
    g = torch.Generator(device=dev)

    def layer_inputs(layer):
        return device_layer_inputs(w, layer, dev, g)

    K = max(1, args.segments)
    if w.T % K != 0:
        raise SystemExit(f"--segments {K} does not divide T={w.T}")
    Ts = w.T // K

    def split(L):  # contiguous per-segment copies of the (B, T, ...) inputs; A is per head
        return [[t if t.dim() == 1 else t[:, k * Ts:(k + 1) * Ts].contiguous() for t in L] for k in range(K)]

    layers = [split(layer_inputs(i)) for i in range(w.layers)]
    if args.bf16:  # bfloat16 activations: x, B_t, C_t (the draws rounded to nearest even)
        for L in layers:
            for seg in L:
                for i in (0, 1, 4, 5, 6, 7):
                    seg[i] = seg[i].to(torch.bfloat16)
    if args.real_x:  # no imaginary plane for x
        for L in layers:
            for seg in L:
                seg[1] = None
    precision = args.precision
    if precision == "auto":
        precision = "tf32" if ssdc.ssd_complex_fwd_supported(ssdc.dims(w.B, Ts, w.H, w.N, w.D, "tf32"), Q) == 0 else "fp32"
    if args.bf16 and precision != "tf32":
        raise SystemExit("--bf16 runs on the TF32 path only")
    if args.mimo and (precision != "tf32" or args.bf16 or K > 1):
        raise SystemExit("--mimo runs on the TF32 path, fp32 inputs, unsegmented")
    if args.state_only and (args.bf16 or args.mimo):
        raise SystemExit("--state-only takes fp32 inputs and no mixer")
    if args.state_only:
        f = ssdc.FinalState(w.B, Ts, w.H, w.N, w.D, Q, precision, device=dev)
    elif args.mimo:
        # identity plus a cross-head part, as a trained mixer would have
        W = (torch.eye(w.H, device=dev) + 0.3 * torch.randn(w.H, w.H, device=dev, generator=g)).contiguous()
        f = ssdc.MimoForward(w.B, Ts, w.H, w.N, w.D, Q, device=dev)
    else:
        f = ssdc.Forward(w.B, Ts, w.H, w.N, w.D, Q, precision, device=dev, bf16_inputs=args.bf16)

    def run_layer(L, timed=False):
        for k, seg in enumerate(L):
            if args.state_only:  # x, A, B_t, dt
                sel = [seg[i] for i in (0, 1, 2, 3, 4, 5, 8)]
                if k == 0:
                    f(*sel)
                else:
                    f(*sel, s0_re=f.fs_re, s0_im=f.fs_im)
            elif args.mimo:
                f(*seg, W)
            elif k == 0:
                f(*seg)
            else:
                f(*seg, s0_re=f.fs_re, s0_im=f.fs_im)
            if timed:
                per_kernel.append(ssdc.timing_read())
    flush = torch.empty(FLUSH_BYTES // 4, dtype=torch.float32, device=dev)
    stream = torch.cuda.current_stream()
    per_kernel, ev = [], []
    for i in range(max(args.warmup, 3)):
        flush.fill_(float(i))
        for L in layers:
            run_layer(L)
    torch.cuda.synchronize()
    sampler = ClockSampler(dev.index)
    torch.cuda.synchronize()
    sampler.start()
    time.sleep(0.1)
    for k in range(args.steps):
        flush.fill_(float(k))
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for L in layers:
            run_layer(L)
        e1.record(stream)
        ev.append((e0, e1))
    torch.cuda.synchronize()
    clocks = sampler.stop()
    st = f.status()
    if st != ssdc.SSDC_OK:
        raise SystemExit(f"device status after timed steps: {ssdc.strerror(st)}")
    ms = sum(a.elapsed_time(b) for a, b in ev) / len(ev)
    # per-launch device times from the library's own events, in a separate pass (reading
    # them waits for each call, which would stall the timed steps)
    ssdc.timing_enable(True)
    for k in range(min(args.steps, 50)):
        flush.fill_(float(k))
        for L in layers:
            run_layer(L, timed=True)
    ssdc.timing_enable(False)
    nk = min(len(p) for p in per_kernel)
    kmeans = [sum(p[i] for p in per_kernel) / len(per_kernel) for i in range(nk)]
    path = ssdc.last_path()
    names = {1: [{"fused_tmem": "fused_tmem_kernel", "state_tmem": "state_tmem_kernel"}.get(path, "fused_kernel")],
             2: ["chunk_state", "state_pass"],
             3: ["chunk_state", "state_pass", "chunk_scan"]}.get(
        nk, [f"launch{i}" for i in range(nk)])
    if args.mimo and nk == 2:  # the scan (either fused kernel), then the in-place head mixer
        names = [{"fused_tmem": "fused_tmem_kernel"}.get(path, "fused_kernel"), "head_mix"]
    top = int(np.argmax(kmeans))
    peak, peak_kind = peaks()
    wq = w.with_(Q=Q, T=Ts)
    # per launch; a segment after the first also reads its initial state (8 N D bytes per sequence)
    bytes_per_launch = (input_bytes_per_unit(wq, bf16=args.bf16, real_x=args.real_x, mimo=args.mimo,
                                             state_only=args.state_only) * wq.token_heads
                        + 8.0 * w.N * w.D * w.B * w.H * (K - 1) / K)
    launch_ms = sum(kmeans)
    units = w.token_heads * w.layers
    line = {
        "metric": METRIC, "value": units / (ms / 1000.0), "unit": UNIT, "n_gpus": 1, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None,
        "dtype": ("bf16 inputs, tf32" if args.bf16 else "tf32") if precision == "tf32" else "f32",
        "data": "synthetic, drawn on the device per layer",
        "config": {"workload": f"{w.name} Q{Q}" + (f" in {K} segments of T={Ts}, state carried" if K > 1 else "")
                   + (f", {w.layers} layer(s) run" if args.layers > 0 else "")
                   + (f", batch {w.B}" if args.batch > 0 else "")
                   + (", real x" if args.real_x else "") + (", bf16 x/B/C" if args.bf16 else "")
                   + (", head mixer on Re(y) (scan, then the in-place mixer kernel)" if args.mimo else "")
                   + (", final state alone (no y)" if args.state_only else ""),
                   "real_x": bool(args.real_x), "bf16_inputs": bool(args.bf16),
                   "B": w.B, "T": w.T, "H": w.H, "D": w.D, "N": w.N,
                   "chunk_size": Q, "layers": w.layers, "segments": K, "precision": precision,
                   "path": path,
                   "l2": f"flushed before every timed step ({FLUSH_BYTES >> 20} MiB write)"},
        "roofline": {"bound": "hbm", "kernel": names[top], "achieved": bytes_per_launch / (launch_ms / 1000.0) / 1e9,
                     "peak": peak, "peak_kind": f"{peak_kind} HBM copy GB/s (burst)", "unit": "GB/s",
                     "frac": bytes_per_launch / (launch_ms / 1000.0) / 1e9 / peak, "traffic": None,
                     "algorithmic_bytes_per_launch": bytes_per_launch,
                     "kernel_ms": {n: m for n, m in zip(names, kmeans)}},
        "cpu_baseline": None,
        "e2e": None,
        "gpu_launches": nk * w.layers * K * args.steps,
        "clocks": clocks,
    }
    if args.mimo:
        # the alternatives: the mixer fused into the scan's epilogue (one launch), and the plain
        # forward (y written) followed by the same mixer as a torch einsum on Re(y); each timed with
        # CUDA events, L2 flushed before each step
        fp = ssdc.Forward(w.B, Ts, w.H, w.N, w.D, Q, precision, device=dev)
        mixed = [None]

        def plain(L):
            for seg in L:
                fp(*seg)

        def mixer(L):
            mixed[0] = torch.einsum("gh,bthd->btgd", W, fp.y_re)

        def timed(fn, n):
            for i in range(3):
                flush.fill_(float(i))
                for L in layers:
                    fn(L)
            tot = 0.0
            for k in range(n):
                flush.fill_(float(k))
                e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                e0.record(stream)
                for L in layers:
                    fn(L)
                e1.record(stream)
                torch.cuda.synchronize()
                tot += e0.elapsed_time(e1)
            return tot / n
        def fused(L):
            for seg in L:
                f(*seg, W)

        n = max(3, min(args.steps, 50))
        with ssdc.option(ssdc.OPT_MIMO_FUSED, 1):
            fused_ms = timed(fused, n)
        scan_ms = timed(plain, n)
        mixer_ms = timed(mixer, n)
        line["alternatives"] = {"fused_epilogue_ms": fused_ms,
                                "torch_einsum": {"scan_ms": scan_ms, "mixer_ms": mixer_ms,
                                                 "total_ms": scan_ms + mixer_ms},
                                "what": "ms_per_step is the default call (the scan writes Re(y), then the "
                                        "mixer kernel); fused_epilogue_ms the same call with the mixer in "
                                        "the scan's epilogue (SSDC_OPT_MIMO_FUSED = 1); torch_einsum the plain "
                                        "forward (path chosen as usual, y written) plus a torch einsum over Re(y)"}
    print(json.dumps(line), flush=True)


def main():
    args = parse()
    if args.backward:
        if args.impl == "reference" or args.segments > 1:
            raise SystemExit("the backward measurement runs with --impl ours, unsegmented")
        w = inputs.ALL[args.workload]
        if args.layers > 0:
            w = w.with_(layers=args.layers)
        if args.batch > 0:
            w = w.with_(B=args.batch)
        backward_workload(args, w)
        return
    if (args.workload != "layer" or args.segments > 1 or args.real_x or args.batch > 0 or args.bf16 or args.mimo
            or args.state_only):
        if args.impl == "reference" or args.gpus != 1:
            raise SystemExit("the measurement workloads run on one GPU with --impl ours")
        w = inputs.ALL[args.workload]
        if args.layers > 0:
            w = w.with_(layers=args.layers)
        if args.batch > 0:
            w = w.with_(B=args.batch)
        other_workload(args, w)
        return
    w = inputs.LAYER
    if args.impl == "reference":
        reference_arm(args, w)
        return
    import torch
    from state_space_sequence_complex_gb300 import build, ssdc

    rank, world, local = dist_env()
    if world > 1:
        import torch.distributed as dist
        torch.cuda.set_device(local)
        dist.init_process_group("nccl" if dist.is_nccl_available() else "gloo")
    else:
        torch.cuda.set_device(0)
    dev = torch.device("cuda", torch.cuda.current_device())
    build.build()
    ssdc.load()

    # each rank processes its own independently seeded batch (weak scaling)
    inp = inputs.generate(w, layer=rank_layer(rank))
    host = {k: torch.from_numpy(np.ascontiguousarray(v)) for k, v in inp.arrays().items()}
    d_in = {k: v.to(dev) for k, v in host.items()}
    Bn, T, H, N, D = inp.dims

    precision = args.precision
    if precision == "auto":
        precision = "tf32" if ssdc.ssd_complex_fwd_supported(ssdc.dims(Bn, T, H, N, D, "tf32"), w.Q) == 0 else "fp32"
    f = ssdc.Forward(Bn, T, H, N, D, w.Q, precision, device=dev)
    stream = torch.cuda.current_stream()
    order = ["x_re", "x_im", "A_re", "A_im", "B_re", "B_im", "C_re", "C_im", "dt"]
    call = lambda: f(*[d_in[k] for k in order])
    flush = torch.empty(FLUSH_BYTES // 4, dtype=torch.float32, device=dev)

    for i in range(max(args.warmup, 3)):
        flush.fill_(float(i))
        call()
    torch.cuda.synchronize()
    st = f.status()
    if st != ssdc.SSDC_OK:
        raise SystemExit(f"device status after warm-up: {ssdc.strerror(st)}")

    # ---- timed region: device-resident inputs, one library call per step ----
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
          for _ in range(args.steps)]
    sampler = ClockSampler(dev.index)
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    sampler.start()
    time.sleep(0.1)
    launches_per_step = 0
    for k in range(args.steps):
        flush.fill_(float(k))
        ev[k][0].record(stream)
        call()
        ev[k][1].record(stream)
        launches_per_step = ssdc.last_launch_count()
    torch.cuda.synchronize()
    clocks = sampler.stop()
    if world > 1:
        torch.distributed.barrier()
    step_ms = [a.elapsed_time(b) for a, b in ev]
    ms = sum(step_ms) / len(step_ms)
    st = f.status()
    if st != ssdc.SSDC_OK:
        raise SystemExit(f"device status after timed steps: {ssdc.strerror(st)}")
    # per-launch device times from the library's own events (the roofline's kernel time), in
    # a separate pass: reading them waits for each call, which would stall the timed steps
    ssdc.timing_enable(True)
    per_kernel = []
    for k in range(min(args.steps, 200)):
        flush.fill_(float(k))
        call()
        per_kernel.append(ssdc.timing_read())
    ssdc.timing_enable(False)

    # ---- back to back without the L2 flush (consecutive layers of a model): host time
    # per call (argument checks, cached launch set-up, the launch) against device time
    # per call; the GPU never waits for the host while the host time is the smaller ----
    b2b_calls = 200
    torch.cuda.synchronize()
    b0, b1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    b0.record(stream)
    t0 = time.perf_counter()
    for _ in range(b2b_calls):
        call()
    host_s = time.perf_counter() - t0
    b1.record(stream)
    torch.cuda.synchronize()
    back_to_back = {"calls": b2b_calls, "host_us_per_call": 1e6 * host_s / b2b_calls,
                    "device_us_per_call": 1000.0 * b0.elapsed_time(b1) / b2b_calls,
                    "l2": "not flushed between calls"}

    # ---- end to end through the C ABI with host buffers (ssd_complex_fwd_host): every
    # step copies its inputs from pinned host memory, runs the scan and copies y and the
    # final state back; the call returns when they are in host memory ----
    pinned = {k: v.pin_memory() for k, v in host.items()}
    hf = ssdc.HostForward(Bn, T, H, N, D, w.Q, precision, device=dev)
    h2d = sum(v.numel() * 4 for v in pinned.values())
    d2h = 2 * (hf.y_re.numel() + hf.fs_re.numel()) * 4
    e2e_step = lambda: hf(*[pinned[k] for k in order], stream=stream)

    for i in range(3):
        e2e_step()
    torch.cuda.synchronize()
    e2e_steps = max(3, min(args.steps, 200))
    e2e_ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
              for _ in range(e2e_steps)]
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    for k in range(e2e_steps):
        flush.fill_(float(k))
        e2e_ev[k][0].record(stream)
        e2e_step()
        e2e_ev[k][1].record(stream)
    torch.cuda.synchronize()
    e2e_ms = sum(a.elapsed_time(b) for a, b in e2e_ev) / e2e_steps

    # max over ranks
    ms, e2e_ms = max_over_ranks([ms, e2e_ms], device=dev)

    units = w.token_heads * world
    value = units / (ms / 1000.0)
    e2e_value = units / (e2e_ms / 1000.0)

    # dominant kernel: the launch with the largest mean device time
    nk = min(len(p) for p in per_kernel)
    kmeans = [sum(p[i] for p in per_kernel) / len(per_kernel) for i in range(nk)]
    path = ssdc.last_path()
    names = {1: ["fused_tmem_kernel" if path == "fused_tmem" else "fused_kernel"],
             3: ["chunk_state", "state_pass", "chunk_scan"]}.get(
        nk, [f"launch{i}" for i in range(nk)])
    top = int(np.argmax(kmeans))
    peak, peak_kind = peaks()
    bytes_per_launch = algorithmic_bytes_per_unit(w) * w.token_heads
    achieved = bytes_per_launch / (kmeans[top] / 1000.0) / 1e9
    step_achieved = bytes_per_launch / (ms / 1000.0) / 1e9 / 1.0

    dram = profiled_dram(names[top])
    roofline = {"bound": "hbm", "kernel": names[top], "achieved": achieved, "peak": peak,
                "peak_kind": f"{peak_kind} HBM copy GB/s (burst)", "unit": "GB/s",
                "frac": achieved / peak, "traffic": None if dram is None else dram["traffic"],
                "algorithmic_bytes_per_launch": bytes_per_launch,
                "kernel_ms": {n: m for n, m in zip(names, kmeans)},
                "step_frac": step_achieved / peak}
    if dram is not None and dram["read"] is not None:
        # the write count of one captured launch misses the part of y still in L2 when the
        # kernel ends (written back later): reads are the comparable figure
        roofline["traffic_read"] = dram["read"]
        roofline["traffic_write"] = dram["write"]
        roofline["traffic_note"] = ("ncu DRAM bytes of one launch; y lines still dirty in L2 at kernel "
                                    "end are written back after it, so write < y bytes")
    if precision == "tf32" and len(kmeans) == 1:
        # context: the same launch against the TF32 tensor peak (the file's BF16 peak times the
        # nominal TF32 / BF16 ratio), with the algorithmic (causal) flops
        fl = sum(fp32_flops_per_unit(w).values()) * w.token_heads
        tf32_peak = bf16_peak_tflops() * 1.1 / 2.25
        roofline["tf32_flops_per_launch"] = fl
        roofline["tf32_frac"] = fl / (kmeans[top] / 1000.0) / 1e12 / tf32_peak if tf32_peak else None
    if precision == "fp32" and names[top] in ("chunk_state", "state_pass", "chunk_scan"):
        # the exact path computes on the CUDA cores: its dominant launch against the FP32 FMA peak
        fl = fp32_flops_per_unit(w)[names[top]] * w.token_heads
        alu_peak, alu_kind = fp32_alu_peak_tflops(dev.index)
        tf = fl / (kmeans[top] / 1000.0) / 1e12
        roofline = {"bound": "alu", "kernel": names[top], "achieved": tf, "peak": alu_peak,
                    "peak_kind": alu_kind, "unit": "TFLOP/s", "frac": tf / alu_peak, "traffic": None,
                    "algorithmic_flops_per_launch": fl,
                    "kernel_ms": {n: m for n, m in zip(names, kmeans)},
                    "hbm_step_frac": step_achieved / peak}

    if rank != 0:
        return
    cpu = None
    if world == 1 and not args.no_cpu_baseline:
        cpu = run_oracle_baseline(w, inp)
    line = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "tf32" if precision == "tf32" else "f32", "data": "synthetic",
        "config": {"workload": w.name, "B": w.B, "T": w.T, "H": w.H, "D": w.D, "N": w.N,
                   "chunk_size": w.Q, "seed": w.seed, "precision": precision, "path": path,
                   "l2": f"flushed before every timed step ({FLUSH_BYTES >> 20} MiB write)",
                   "parallelism": f"weak: {world} independent batch(es), no collective"},
        "roofline": roofline,
        "cpu_baseline": cpu,
        "e2e": {"value": e2e_value, "unit": UNIT, "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                "ms_per_step": e2e_ms},
        "gpu_launches": launches_per_step * args.steps,
        "clocks": clocks,
        "back_to_back": back_to_back,
    }
    print(json.dumps(line), flush=True)


if __name__ == "__main__":
    main()
