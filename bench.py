"""Benchmark of the fused attention forward on GB300.

One step = one fused attention forward over the whole workload (one kernel
launch), inputs resident in HBM.  Prints ONE JSON line on rank 0.  Without
``--steps`` the timed region is sized from the warm-up to about 5 s of device
time.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME]
                    [--impl ours|reference]

Metric: attention forward TFLOP/s = 4 * B * H_q * S_q * S_kv * D (halved when
causal) / time, and its fraction of the measured dense BF16 peak.

Extra keys: ``roofline`` (the kernel against the measured tensor peak),
``e2e`` (the same metric through the host-buffer C entry point, copies timed),
``cpu_baseline`` (the fp64 oracle on a bounded sample of the same workload,
on the host cores), ``clocks`` (nvidia-smi samples during the timed region),
``gpu_launches``.

Multi-GPU: one process per GPU under torchrun; each rank runs an independent
replica of the workload (the path has no exchange step), the timed region is
bracketed by barriers, and the time is the maximum over ranks.
``--impl reference`` times the fp64 CPU oracle as the reference arm.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "attention fwd TFLOP/s (bf16, fp32 acc) and % of GB300 dense BF16 peak"
FALLBACK_BF16_TFLOPS = 1900.0
L2_BYTES = 129 * 1024 * 1024
TRAFFIC_FILE = os.path.join(ROOT, "profiles", "attn_fwd_traffic.json")
KERNEL_SOURCES = ["attention_pipelining_gb300/csrc/attn_fwd_sm103.cu",
                  "attention_pipelining_gb300/csrc/attn_tiles.cuh",
                  "attention_pipelining_gb300/csrc/ptx.cuh"]
CS_TRAFFIC_FILE = os.path.join(ROOT, "profiles", "chunk_scan_traffic.json")
CS_KERNEL_SOURCES = ["attention_pipelining_gb300/csrc/chunk_scan_sm103.cu",
                     "attention_pipelining_gb300/csrc/ptx.cuh"]


# ----------------------------------------------------------------- helpers

def kernel_source_hash(sources=None) -> str:
    h = hashlib.sha256()
    for rel in (sources or KERNEL_SOURCES):
        with open(os.path.join(ROOT, rel), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return float(d["bf16_tflops"]), float(d.get("bf16_tflops_sustained", d["bf16_tflops"])), "measured"
    except Exception:
        return FALLBACK_BF16_TFLOPS, FALLBACK_BF16_TFLOPS * 0.9, "fallback"


def load_hbm_peak():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            return float(json.load(f)["hbm_gbs"]), "measured"
    except Exception:
        return 6800.0, "fallback"


def flush_bytes_for(in_bytes: int) -> int:
    """Bytes to write between timed steps: none when the inputs alone are
    larger than L2 (each step then reads them from DRAM), else a buffer of
    four times L2."""
    return 0 if in_bytes > L2_BYTES else 4 * L2_BYTES


def l2_note(in_bytes: int, flush_bytes: int) -> str:
    if flush_bytes == 0:
        return f"inputs larger than L2 ({in_bytes / 1e6:.0f} MB > {L2_BYTES / 1e6:.0f} MB), no flush"
    return f"L2 flushed before each timed step ({flush_bytes / 1e6:.0f} MB written, outside the timed events)"


def time_steps(step, steps, stream, dev, flush_bytes):
    """Device seconds of `steps` calls of step() on `stream`.  Without a
    flush one pair of CUDA events brackets all steps; with one, a buffer of
    `flush_bytes` is written before each step, outside a pair of events per
    step, and the per-step times are summed."""
    import torch
    if flush_bytes <= 0:
        start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        start.record(stream)
        for _ in range(steps):
            step()
        end.record(stream)
        torch.cuda.synchronize(dev)
        return start.elapsed_time(end) / 1e3
    buf = torch.empty(flush_bytes, dtype=torch.uint8, device=dev)
    events = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
              for _ in range(steps)]
    with torch.cuda.stream(stream):
        for i in range(steps):
            buf.fill_(i & 0xFF)
            events[i][0].record(stream)
            step()
            events[i][1].record(stream)
    torch.cuda.synchronize(dev)
    return sum(a.elapsed_time(b) for a, b in events) / 1e3


MIN_TIMED_SECONDS = 5.0     # default length of the timed region (device time)
MIN_DEFAULT_STEPS = 20
MAX_DEFAULT_STEPS = 20000


def warm_up(step, warmup, stream, dev, world):
    """Runs the untimed warm-up steps and returns their mean device seconds
    per step (max over ranks), which sizes the timed region when no step
    count is given."""
    import torch
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    start.record(stream)
    for _ in range(warmup):
        step()
    end.record(stream)
    torch.cuda.synchronize(dev)
    return max_over_ranks(start.elapsed_time(end) / 1e3 / warmup, world)


def timed_steps(requested, per_step_s):
    """The step count to time: the one asked for, else enough steps for
    MIN_TIMED_SECONDS of device time (within MIN/MAX_DEFAULT_STEPS)."""
    if requested is not None:
        return requested
    want = math.ceil(MIN_TIMED_SECONDS / max(per_step_s, 1e-9))
    return int(min(MAX_DEFAULT_STEPS, max(MIN_DEFAULT_STEPS, want)))


def load_traffic(path=TRAFFIC_FILE, sources=None):
    """DRAM bytes per launch from the committed ncu summary, if it was taken on
    the current kernel source (else None)."""
    try:
        with open(path) as f:
            d = json.load(f)
    except Exception:
        return None
    if d.get("kernel_source_hash") != kernel_source_hash(sources):
        return None
    return d


def chunk_scan_traffic(w):
    """(DRAM bytes per launch, note) of the chunk scan on workload w from the
    committed capture, scaled by the batch size when w differs from the
    captured workload only in a larger B (the same CTAs, 32 heads each, in
    more waves: inputs, output and traffic grow with B); (None, None) if the
    capture is stale or of other shapes."""
    d = load_traffic(CS_TRAFFIC_FILE, CS_KERNEL_SOURCES)
    if d is None:
        return None, None
    shape = d.get("shape", {})
    if any(shape.get(k) != getattr(w, k) for k in ("L", "H", "P", "G", "Q")):
        return None, None
    if w.B < shape.get("B", 0):
        return None, None            # smaller grids choose smaller head blocks
    if shape.get("B") == w.B:
        return d["dram_bytes_per_launch"], f"ncu capture of {d['workload']}"
    return (d["dram_bytes_per_launch"] * w.B / shape["B"],
            f"ncu capture of {d['workload']}, scaled by B {w.B} / {shape['B']}")


class ClockSampler:
    """nvidia-smi clocks and throttle reasons, sampled while the timed region runs."""

    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int, interval_ms: int = 50):
        self.gpu = gpu_index
        self.interval = interval_ms
        self.proc = None
        self.out = None

    def start(self):
        try:
            self.out = tempfile.NamedTemporaryFile("w+", suffix=".csv", delete=False)
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.QUERY}",
                 "--format=csv,noheader,nounits", "-lms", str(self.interval)],
                stdout=self.out, stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None

    def stop(self) -> dict:
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        self.out.flush()
        self.out.seek(0)
        lines = self.out.read().splitlines()
        self.out.close()
        os.unlink(self.out.name)
        return parse_clock_rows(lines)


def parse_clock_rows(lines) -> dict:
    """Summary of nvidia-smi CSV rows (noheader, nounits) of ClockSampler.QUERY."""
    sm, smax, reasons, power = [], [], set(), []
    names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
    for line in lines:
        r = [x.strip() for x in line.split(",")]
        if len(r) < 9:
            continue
        try:
            sm.append(float(r[1]))
            smax.append(float(r[2]))
            power.append(float(r[3]))
        except ValueError:
            continue
        for name, val in zip(names, r[5:9]):
            if val.lower() == "active":
                reasons.add(name)
    return {
        "sm_mhz": statistics.median(sm) if sm else None,
        "sm_max_mhz": max(smax) if smax else None,
        "power_w_max": max(power) if power else None,
        "samples": len(sm),
        "reasons": sorted(reasons),
    }


def dist_env():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def init_dist(world: int, backend: str):
    import torch.distributed as dist
    if world > 1 and not dist.is_initialized():
        os.environ.setdefault("MASTER_ADDR", "127.0.0.1")
        dist.init_process_group(backend=backend)
    return dist


def max_over_ranks(x: float, world: int) -> float:
    """Maximum of a per-rank scalar (time) over all ranks."""
    if world == 1:
        return x
    import torch
    import torch.distributed as dist
    dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([x], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def barrier(world: int):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


# ----------------------------------------------------------------- CPU oracle timing

def time_oracle_rows(q, k, v, w, rows) -> float:
    import oracle
    t0 = time.perf_counter()
    oracle.attn_rows(q, k, v, rows, w.causal, w.scale)
    return time.perf_counter() - t0


def row_flops(w, rows) -> float:
    """FLOPs of the sampled rows under the metric's convention (4*S_kv*D per
    row, causal rows counting only their visible keys)."""
    import numpy as np
    i = rows % w.S_q
    vis = np.minimum(i + 1, w.S_kv) if w.causal else np.full(rows.shape, w.S_kv)
    return float(4.0 * w.D * vis.sum())


def sample_rows(w, n: int, seed: int = 0):
    import numpy as np
    rng = np.random.default_rng(seed)
    total = w.B * w.H_q * w.S_q
    return np.sort(rng.choice(total, size=min(n, total), replace=False)).astype(np.int64)


def calibrate_oracle(q, k, v, w, target_s: float):
    """Row count whose oracle time is about target_s seconds."""
    n = 64
    while True:
        rows = sample_rows(w, n)
        dt = time_oracle_rows(q, k, v, w, rows)
        if dt >= 0.5 or n >= w.B * w.H_q * w.S_q:
            break
        n *= 4
    per_row = dt / len(rows)
    return max(1, int(target_s / per_row))


def host_cpu_model() -> str:
    """The host CPU's model name (lscpu, else /proc/cpuinfo), for the CPU
    baseline's record."""
    import subprocess
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        for line in out.splitlines():
            if line.strip().lower().startswith("model name"):
                return line.split(":", 1)[1].strip()
    except Exception:
        pass
    try:
        with open("/proc/cpuinfo") as f:
            for line in f:
                if line.lower().startswith("model name"):
                    return line.split(":", 1)[1].strip()
    except Exception:
        pass
    import platform
    return platform.machine() or "unknown"


def cpu_baseline(q, k, v, w, target_s: float = 12.0) -> dict:
    import oracle
    n = calibrate_oracle(q, k, v, w, target_s)
    rows = sample_rows(w, n, seed=1)
    dt = time_oracle_rows(q, k, v, w, rows)
    return {
        "value": row_flops(w, rows) / dt / 1e12,
        "unit": "TFLOP/s",
        "cores": oracle.num_threads(),
        "cpu_model": host_cpu_model(),
        "kind": "oracle",
        "sample": f"{len(rows)} of {w.B * w.H_q * w.S_q} output rows of {w.name} "
                  f"(random rows, each over its full visible key range), fp64, {dt:.1f} s",
    }


# ----------------------------------------------------------------- arms

def run_reference(args, w):
    """The fp64 CPU oracle as the reference arm (rank 0 only)."""
    import oracle
    from attention_pipelining_gb300.synthetic import make_workload
    world, rank, _ = dist_env()
    if rank != 0:
        return
    oracle.build()
    q, k, v = make_workload(w)
    budget = 150.0
    if args.steps is None:
        args.steps = 5
    n = calibrate_oracle(q, k, v, w, budget / max(1, args.steps + args.warmup))
    for s in range(args.warmup):
        time_oracle_rows(q, k, v, w, sample_rows(w, n, seed=100 + s))
    total_t, total_f = 0.0, 0.0
    for s in range(args.steps):
        rows = sample_rows(w, n, seed=s)
        total_t += time_oracle_rows(q, k, v, w, rows)
        total_f += row_flops(w, rows)
    value = total_f / total_t / 1e12
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "TFLOP/s",
        "n_gpus": 0, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": total_t / args.steps * 1e3, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": w.name, **{kk: vv for kk, vv in w.as_dict().items() if kk != "name"},
                   "sample_rows_per_step": n},
        "cpu_baseline": {"value": value, "unit": "TFLOP/s", "cores": oracle.num_threads(),
                         "cpu_model": host_cpu_model(), "kind": "oracle",
                         "sample": f"{n} random output rows of {w.name} per step, fp64"},
        "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def run_ours(args, w):
    import torch
    import attention_pipelining_gb300 as ap
    from attention_pipelining_gb300.synthetic import make_workload

    world, rank, local = dist_env()
    torch.cuda.set_device(local)
    init_dist(world, "nccl")
    ap.build()
    dev = torch.device("cuda", local)

    q_cpu, k_cpu, v_cpu = make_workload(w)
    q, k, v = q_cpu.to(dev), k_cpu.to(dev), v_cpu.to(dev)
    o = torch.empty_like(q)
    lse = torch.empty((w.B, w.H_q, w.S_q), dtype=torch.float32, device=dev)
    in_bytes = (q.numel() + k.numel() + v.numel()) * 2
    out_bytes = o.numel() * 2 + lse.numel() * 4
    stream = torch.cuda.current_stream(dev)

    splitkv = (w.path == "splitkv")
    if splitkv:
        splits = ap.splitkv_default_splits(w.B, w.H_q, w.H_kv, w.S_q, w.S_kv, w.causal)
        ws = torch.empty(int(ap._load().attn_splitkv_workspace_bytes(w.B, w.H_q, w.S_q, w.D, splits)),
                         dtype=torch.uint8, device=dev)

        def run_path(qq, kk, vv):
            return ap.attn_fwd_splitkv(qq, kk, vv, w.causal, w.scale, num_splits=splits,
                                       workspace=ws, stream=stream)

        def step():
            ap._check(ap._load().attn_fwd_splitkv(
                q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), lse.data_ptr(),
                ws.data_ptr(), ws.numel(), w.B, w.H_q, w.H_kv, w.S_q, w.S_kv, w.D, int(w.causal),
                float(w.scale), splits, stream.cuda_stream), "attn_fwd_splitkv")
    else:
        def step():
            ap.attn_fwd_out(q, k, v, o, lse, w.causal, w.scale, stream)

    args.steps = timed_steps(args.steps, warm_up(step, args.warmup, stream, dev, world))
    if ap.device_status(reset=True) != 0:
        raise RuntimeError("a kernel wait timed out during warm-up")

    flush = flush_bytes_for(in_bytes)
    visible = os.environ.get("CUDA_VISIBLE_DEVICES")
    smi_index = int(visible.split(",")[local]) if visible and visible.split(",")[local].isdigit() else local
    sampler = ClockSampler(smi_index)
    sampler.start()
    time.sleep(0.2)
    barrier(world)
    torch.cuda.synchronize(dev)
    t_local = time_steps(step, args.steps, stream, dev, flush)
    barrier(world)
    clocks = sampler.stop()
    t = max_over_ranks(t_local, world)
    if ap.device_status(reset=True) != 0:
        raise RuntimeError("a kernel wait timed out in the timed region")

    # end to end through the host-buffer entry point: pinned host inputs in,
    # host outputs back, copies inside the timed region
    e2e_steps = max(1, min(args.steps, args.e2e_steps))
    qh, kh, vh = q_cpu.pin_memory(), k_cpu.pin_memory(), v_cpu.pin_memory()
    oh = torch.empty_like(q_cpu).pin_memory()
    lh = torch.empty((w.B, w.H_q, w.S_q), dtype=torch.float32).pin_memory()

    def e2e_step():
        if splitkv:
            # the split-KV entry takes device buffers: pinned host copies in and out
            q.copy_(qh, non_blocking=True)
            k.copy_(kh, non_blocking=True)
            v.copy_(vh, non_blocking=True)
            step()
            oh.copy_(o, non_blocking=True)
            lh.copy_(lse, non_blocking=True)
        else:
            ap.attn_fwd_host(qh, kh, vh, oh, lh, q, k, v, o, lse, w.causal, w.scale, stream)

    for _ in range(2):
        e2e_step()
    torch.cuda.synchronize(dev)
    barrier(world)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(e2e_steps):
        e2e_step()
    e1.record(stream)
    torch.cuda.synchronize(dev)
    barrier(world)
    t_e2e = max_over_ranks(e0.elapsed_time(e1) / 1e3, world)

    if rank != 0:
        return
    peak, peak_sustained, peak_kind = load_peaks()
    hbm_peak = load_hbm_peak()
    flops = w.flops
    value = world * flops * args.steps / t / 1e12
    per_launch = t_local / args.steps
    achieved = flops / per_launch / 1e12
    traffic = load_traffic()
    line = {
        "metric": METRIC,
        "value": value,
        "unit": "TFLOP/s",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": t / args.steps * 1e3,
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "bf16",
        "data": "synthetic",
        "config": {
            "workload": w.name, "B": w.B, "H_q": w.H_q, "H_kv": w.H_kv, "S_q": w.S_q,
            "S_kv": w.S_kv, "D": w.D, "causal": w.causal, "k_scale": w.k_scale,
            "scale": w.scale, "seed": w.seed, "parallelism": f"replicas x{world}",
            "l2": l2_note(in_bytes, flush),
        },
        "pct_of_peak": 100.0 * achieved / peak,
        "roofline": ({
            "bound": "tensor",
            "achieved": achieved,
            "peak": peak,
            "unit": "TFLOP/s",
            "frac": achieved / peak,
            "peak_kind": f"{peak_kind} bf16 dense (burst)",
            "frac_of_sustained": achieved / peak_sustained,
            "traffic": (traffic["dram_bytes_per_launch"] if traffic else None),
            "algorithmic_flops_per_launch": flops,
            "kernel": "attn_fwd_kernel",
        } if not splitkv else {
            "bound": "hbm",
            "achieved": w.io_bytes / per_launch / 1e9,
            "peak": hbm_peak[0],
            "unit": "GB/s",
            "frac": w.io_bytes / per_launch / 1e9 / hbm_peak[0],
            "peak_kind": f"{hbm_peak[1]} HBM copy",
            "traffic": None,
            "algorithmic_bytes_per_launch": w.io_bytes,
            "kernel": "attn_fwd_kernel (split KV) + splitkv_combine_kernel, timed together",
            "num_splits": splits,
        }),
        "e2e": {
            "value": world * flops * e2e_steps / t_e2e / 1e12,
            "unit": "TFLOP/s",
            "h2d_bytes_per_step": in_bytes,
            "d2h_bytes_per_step": out_bytes,
            "steps": e2e_steps,
        },
        "gpu_launches": args.steps * (2 if splitkv else 1),
        "clocks": clocks,
    }
    if not args.no_cpu_baseline:
        import oracle
        oracle.build()
        line["cpu_baseline"] = cpu_baseline(q_cpu, k_cpu, v_cpu, w, args.cpu_seconds)
    print(json.dumps(line), flush=True)


def run_bwd(args, w):
    """The backward on the same workload: one step = dQ, dK, dV for one
    upstream gradient, inputs (q, k, v, O, LSE, dO) resident in HBM.
    attn_bwd (prep, dK/dV with dQ, dQ conversion), or with
    --bwd-deterministic attn_bwd_deterministic (prep, dK/dV, dQ).  FLOPs: the
    five GEMMs of a FlashAttention backward, 2.5 x the forward's count
    (halved when causal)."""
    import torch
    import attention_pipelining_gb300 as ap
    from attention_pipelining_gb300.synthetic import make_workload

    world, rank, local = dist_env()
    torch.cuda.set_device(local)
    init_dist(world, "nccl")
    ap.build()
    dev = torch.device("cuda", local)
    q_cpu, k_cpu, v_cpu = make_workload(w)
    g = torch.Generator().manual_seed(w.seed + 1)
    do_cpu = torch.randn(q_cpu.shape, generator=g).to(torch.bfloat16)
    q, k, v, dout = (t.to(dev) for t in (q_cpu, k_cpu, v_cpu, do_cpu))
    o, lse = ap.attn_fwd(q, k, v, w.causal, w.scale)
    dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
    ws = torch.empty(ap.bwd_workspace_bytes(w.B, w.H_q, w.H_kv, w.S_q, w.D), dtype=torch.uint8,
                     device=dev)
    stream = torch.cuda.current_stream(dev)

    det = bool(args.bwd_deterministic)
    fused = not det

    def step():
        ap.attn_bwd(q, k, v, o, lse, dout, w.causal, w.scale, workspace=ws, out=(dq, dk, dv),
                    stream=stream, deterministic=det)

    in_bytes = sum(t.numel() * t.element_size() for t in (q, k, v, dout, o, lse))

    args.steps = timed_steps(args.steps, warm_up(step, args.warmup, stream, dev, world))
    if ap.device_status(reset=True) != 0:
        raise RuntimeError("a kernel wait timed out during warm-up")
    flush = flush_bytes_for(in_bytes)
    visible = os.environ.get("CUDA_VISIBLE_DEVICES")
    smi_index = int(visible.split(",")[local]) if visible and visible.split(",")[local].isdigit() else local
    sampler = ClockSampler(smi_index)
    sampler.start()
    time.sleep(0.2)
    barrier(world)
    torch.cuda.synchronize(dev)
    t_local = time_steps(step, args.steps, stream, dev, flush)
    barrier(world)
    clocks = sampler.stop()
    t = max_over_ranks(t_local, world)
    if ap.device_status(reset=True) != 0:
        raise RuntimeError("a kernel wait timed out in the timed region")

    # end to end through the host-buffer backward (attn_bwd_host): pinned
    # host inputs in, gradients back, copies inside the timed region
    e2e_steps = max(1, min(args.steps, args.e2e_steps))
    host_in = [t.pin_memory() for t in (q_cpu, k_cpu, v_cpu)] + \
        [o.cpu().pin_memory(), lse.cpu().pin_memory(), do_cpu.pin_memory()]
    host_out = [torch.empty(t.shape, dtype=t.dtype).pin_memory() for t in (dq, dk, dv)]

    def e2e_step():
        ap.attn_bwd_host(*host_in, *host_out, q, k, v, o, lse, dout, dq, dk, dv, w.causal,
                         w.scale, ws, stream=stream)

    for _ in range(2):
        e2e_step()
    torch.cuda.synchronize(dev)
    barrier(world)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(e2e_steps):
        e2e_step()
    e1.record(stream)
    torch.cuda.synchronize(dev)
    barrier(world)
    t_e2e = max_over_ranks(e0.elapsed_time(e1) / 1e3, world)
    if rank != 0:
        return
    peak, peak_sustained, peak_kind = load_peaks()
    flops = 2.5 * w.flops
    per_launch = t_local / args.steps
    achieved = flops / per_launch / 1e12
    out_bytes = sum(t.numel() * t.element_size() for t in (dq, dk, dv))
    line = {
        "metric": "attention bwd TFLOP/s (bf16, fp32 acc; 2.5x the forward's FLOPs)",
        "value": world * flops * args.steps / t / 1e12,
        "unit": "TFLOP/s",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": t / args.steps * 1e3,
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "bf16",
        "data": "synthetic",
        "pass": "bwd",
        "config": {
            "workload": w.name, "B": w.B, "H_q": w.H_q, "H_kv": w.H_kv, "S_q": w.S_q,
            "S_kv": w.S_kv, "D": w.D, "causal": w.causal, "k_scale": w.k_scale,
            "scale": w.scale, "seed": w.seed, "parallelism": f"replicas x{world}",
            "l2": l2_note(in_bytes, flush),
            "path": "deterministic (dQ kernel)" if det else "fused dQ",
        },
        "pct_of_peak": 100.0 * achieved / peak,
        "roofline": {
            "bound": "tensor",
            "achieved": achieved,
            "peak": peak,
            "unit": "TFLOP/s",
            "frac": achieved / peak,
            "peak_kind": f"{peak_kind} bf16 dense (burst)",
            "frac_of_sustained": achieved / peak_sustained,
            "traffic": None,
            "algorithmic_flops_per_launch": flops,
            "kernel": ("attn_bwd_prep + attn_bwd_dkdv (with dQ) + attn_bwd_dq_convert"
                       if fused else "attn_bwd_prep + attn_bwd_dkdv + attn_bwd_dq") +
                      ", timed together",
        },
        "e2e": {
            "value": world * flops * e2e_steps / t_e2e / 1e12,
            "unit": "TFLOP/s",
            "h2d_bytes_per_step": in_bytes,
            "d2h_bytes_per_step": out_bytes,
            "steps": e2e_steps,
        },
        "gpu_launches": args.steps * 3,
        "clocks": clocks,
    }
    if not args.no_cpu_baseline:
        import oracle
        oracle.build()
        line["cpu_baseline"] = cpu_baseline_bwd(q_cpu, k_cpu, v_cpu, do_cpu, w, args.cpu_seconds)
    print(json.dumps(line), flush=True)


def cpu_baseline_bwd(q, k, v, dout, w, target_s: float = 12.0) -> dict:
    """The fp64 backward oracle on a bounded sample: dQ of random query rows
    (each formed from its full softmax row), counted at 2.5x the rows' forward
    FLOPs."""
    import oracle
    bo = oracle.bwd_default()
    n = 8
    while True:
        rows = sample_rows(w, n, seed=1)
        t0 = time.perf_counter()
        bo.dq_rows(q, k, v, dout, rows, w.causal, w.scale)
        dt = time.perf_counter() - t0
        if dt >= target_s / 4 or n >= w.B * w.H_q * w.S_q:
            break
        n = min(w.B * w.H_q * w.S_q, max(n * 2, int(n * target_s / max(dt, 1e-3) / 2)))
    flops = 2.5 * row_flops(w, rows)
    return {"value": flops / dt / 1e12, "unit": "TFLOP/s", "cores": oracle.default().num_threads(),
            "cpu_model": host_cpu_model(),
            "kind": "oracle",
            "sample": f"dQ of {len(rows)} random query rows of {w.name} (each over its full "
                      f"visible key range), fp64, {dt:.1f} s"}


def run_chunk_scan(args, name):
    """The Mamba2 chunk scan (chunk_scan_fwd) on one of the chunk-scan
    workloads: one step = one launch over the whole batch, inputs resident in
    HBM (drawn on the device with the recipe's distributions)."""
    import torch
    import attention_pipelining_gb300 as ap
    from attention_pipelining_gb300.synthetic import CHUNK_SCAN_WORKLOADS, make_chunk_scan_workload

    w = CHUNK_SCAN_WORKLOADS[name]
    world, rank, local = dist_env()
    torch.cuda.set_device(local)
    init_dist(world, "nccl")
    ap.build()
    dev = torch.device("cuda", local)
    cb, dA_cs, dt, x = make_chunk_scan_workload(w, device=f"cuda:{local}")
    out = torch.empty_like(x)
    stream = torch.cuda.current_stream(dev)

    def step():
        ap.chunk_scan(cb, dA_cs, dt, x, out=out, stream=stream)

    in_bytes = sum(tt.numel() * tt.element_size() for tt in (cb, dA_cs, dt, x))

    args.steps = timed_steps(args.steps, warm_up(step, args.warmup, stream, dev, world))
    if ap.device_status(reset=True) != 0:
        raise RuntimeError("a kernel wait timed out during warm-up")
    flush = flush_bytes_for(in_bytes)
    visible = os.environ.get("CUDA_VISIBLE_DEVICES")
    smi_index = int(visible.split(",")[local]) if visible and visible.split(",")[local].isdigit() else local
    sampler = ClockSampler(smi_index)
    sampler.start()
    time.sleep(0.2)
    barrier(world)
    torch.cuda.synchronize(dev)
    t_local = time_steps(step, args.steps, stream, dev, flush)
    barrier(world)
    clocks = sampler.stop()
    t = max_over_ranks(t_local, world)
    if ap.device_status(reset=True) != 0:
        raise RuntimeError("a kernel wait timed out in the timed region")

    # end to end through the host-buffer entry (chunk_scan_fwd_host): pinned
    # host inputs in, the output back, copies inside the timed region
    e2e_steps = max(1, min(args.steps, args.e2e_steps))
    dev_in = [cb, dA_cs, dt, x]
    host_in = [tt.cpu().pin_memory() for tt in dev_in]
    host_out = torch.empty(out.shape, dtype=out.dtype).pin_memory()

    def e2e_step():
        ap.chunk_scan_host(*host_in, host_out, *dev_in, out, stream=stream)

    for _ in range(2):
        e2e_step()
    torch.cuda.synchronize(dev)
    barrier(world)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(e2e_steps):
        e2e_step()
    e1.record(stream)
    torch.cuda.synchronize(dev)
    barrier(world)
    t_e2e = max_over_ranks(e0.elapsed_time(e1) / 1e3, world)
    if rank != 0:
        return
    hbm_peak = load_hbm_peak()
    per_launch = t_local / args.steps
    traffic, traffic_note = chunk_scan_traffic(w)
    line = {
        "metric": "Mamba2 chunk scan TFLOP/s (bf16 products, fp32 acc; 2 P per visible key)",
        "value": world * w.flops * args.steps / t / 1e12,
        "unit": "TFLOP/s",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": t / args.steps * 1e3,
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "bf16",
        "data": "synthetic",
        "pass": "chunkscan",
        "config": {
            "workload": w.name, "B": w.B, "L": w.L, "H": w.H, "P": w.P, "G": w.G, "Q": w.Q,
            "seed": w.seed, "parallelism": f"replicas x{world}",
            "l2": l2_note(in_bytes, flush),
        },
        "roofline": {
            "bound": "hbm",
            "achieved": w.io_bytes / per_launch / 1e9,
            "peak": hbm_peak[0],
            "unit": "GB/s",
            "frac": w.io_bytes / per_launch / 1e9 / hbm_peak[0],
            "peak_kind": f"{hbm_peak[1]} HBM copy",
            "traffic": traffic,
            "traffic_source": traffic_note,
            "algorithmic_bytes_per_launch": w.io_bytes,
            "kernel": "chunk_scan_kernel",
        },
        "e2e": {
            "value": world * w.flops * e2e_steps / t_e2e / 1e12,
            "unit": "TFLOP/s",
            "h2d_bytes_per_step": in_bytes,
            "d2h_bytes_per_step": out.numel() * out.element_size(),
            "steps": e2e_steps,
        },
        "gpu_launches": args.steps,
        "clocks": clocks,
    }
    if not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline_chunk_scan(w, args.cpu_seconds)
    print(json.dumps(line), flush=True)


def cpu_baseline_chunk_scan(w, target_s: float = 12.0) -> dict:
    """The fp64 chunk-scan oracle on a bounded sample: random output rows of
    one batch item of the workload's shapes (inputs drawn on the CPU with the
    same recipe), counted at 2 P FLOPs per visible key."""
    import numpy as np
    import oracle
    from attention_pipelining_gb300.synthetic import make_chunk_scan
    cs = oracle.chunk_scan_default()
    cb, dA_cs, dt, x = make_chunk_scan(1, w.L, w.H, w.P, w.G, w.Q, w.seed)
    total = w.L * w.H
    rng = np.random.default_rng(0)
    n = 256
    while True:
        rows = np.sort(rng.choice(total, size=min(n, total), replace=False)).astype(np.int64)
        t0 = time.perf_counter()
        cs.rows(cb, dA_cs, dt, x, rows)
        dt_s = time.perf_counter() - t0
        if dt_s >= target_s / 4 or n >= total:
            break
        n = min(total, max(n * 2, int(n * target_s / max(dt_s, 1e-3) / 2)))
    m = (rows // w.H) % w.Q                      # row within its chunk
    flops = float(2.0 * w.P * (m + 1).sum())
    return {"value": flops / dt_s / 1e12, "unit": "TFLOP/s",
            "cores": oracle.default().num_threads(), "cpu_model": host_cpu_model(),
            "kind": "oracle",
            "sample": f"{len(rows)} random output rows of one batch item of {w.name}, fp64, "
                      f"{dt_s:.1f} s"}


def run_trace(args, w):
    """Timeline of the first CTAs from the trace instantiation (not a bench line)."""
    import torch
    import attention_pipelining_gb300 as ap
    from attention_pipelining_gb300 import trace as tr
    from attention_pipelining_gb300.synthetic import make_workload
    ap.build()
    q, k, v = (t.cuda() for t in make_workload(w))
    for _ in range(args.warmup):
        ap.attn_fwd(q, k, v, w.causal, w.scale)
    torch.cuda.synchronize()
    n_blocks = min((w.S_kv + 127) // 128, ap.MAX_TRACE_BLOCKS)
    _, _, t = ap.attn_fwd_trace(q, k, v, w.causal, w.scale, ctas=args.trace, blocks=n_blocks)
    out = {"workload": w.name, "traced_ctas": args.trace, **tr.summarize(t.numpy(), n_blocks)}
    if args.trace_out:
        import numpy as np
        np.save(args.trace_out, t.numpy())
    print(json.dumps(out), flush=True)


def main(argv=None):
    from attention_pipelining_gb300.synthetic import HEADLINE, WORKLOADS
    ap_ = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap_.add_argument("--gpus", type=int, default=1)
    ap_.add_argument("--steps", type=int, default=None,
                     help="timed steps (default: enough for %g s of device time)" % MIN_TIMED_SECONDS)
    ap_.add_argument("--warmup", type=int, default=10)
    ap_.add_argument("--workload", default=HEADLINE, choices=sorted(WORKLOADS))
    ap_.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap_.add_argument("--e2e-steps", type=int, default=50)
    ap_.add_argument("--cpu-seconds", type=float, default=12.0)
    ap_.add_argument("--no-cpu-baseline", action="store_true")
    ap_.add_argument("--trace", type=int, default=0,
                     help="print a timeline summary of the first N CTAs instead of a bench line")
    ap_.add_argument("--trace-out", default="", help="also save the raw trace (.npy)")
    ap_.add_argument("--bwd-deterministic", action="store_true",
                     help="--pass bwd: time attn_bwd_deterministic (dQ by its own kernel)")
    ap_.add_argument("--pass", dest="which", default="fwd", choices=["fwd", "bwd", "chunkscan"],
                     help="bwd: time the backward (attn_bwd) instead of the forward; "
                          "chunkscan: time the Mamba2 chunk scan (see --cs-workload)")
    ap_.add_argument("--cs-workload", default=None,
                     help="chunk-scan workload for --pass chunkscan (default: the 64 x 8192 one)")
    args = ap_.parse_args(argv)
    if args.warmup < 3:
        ap_.error("--warmup must be >= 3")
    if args.steps is not None and args.steps < 1:
        ap_.error("--steps must be >= 1")
    w = WORKLOADS[args.workload]
    if args.trace > 0:
        run_trace(args, w)
        return
    if args.impl == "reference":
        run_reference(args, w)
    elif args.which == "bwd":
        run_bwd(args, w)
    elif args.which == "chunkscan":
        from attention_pipelining_gb300.synthetic import CHUNK_SCAN_HEADLINE, CHUNK_SCAN_WORKLOADS
        name = args.cs_workload or CHUNK_SCAN_HEADLINE
        if name not in CHUNK_SCAN_WORKLOADS:
            ap_.error(f"--cs-workload must be one of {sorted(CHUNK_SCAN_WORKLOADS)}")
        run_chunk_scan(args, name)
    else:
        run_ours(args, w)
    world, _, _ = dist_env()
    if world > 1:
        import torch.distributed as dist
        if dist.is_initialized():
            dist.barrier()
            dist.destroy_process_group()


if __name__ == "__main__":
    main()
