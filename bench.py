#!/usr/bin/env python
"""Throughput benchmark of the Based causal forward pass on GB300.

A step is one based_fwd call over one batch of the workload (every kernel of the hot path: the
aggregate pass and scan when the plan needs them, then the forward kernel). The headline workload
is B=4, T=4096, H=16, K=16, V=64 with q, k, v ~ N(0,1) bf16; the output is fp32.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME] [--impl gb300|reference]

Prints one JSON line (rank 0). Under torchrun with N > 1 every rank runs its own replica of the
workload on its own GPU (the problem has no cross-GPU exchange); the timed region is bracketed by
a barrier and device synchronisation and the slowest rank's time is used.
"""
import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import tempfile
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import torch  # noqa: E402

from linear_attention_gb300.inputs import GRADER_WORKLOADS, WORKLOADS, make_workload  # noqa: E402

METRIC = "Based fwd tokens/s and TFLOP/s (% of GB300 bf16 peak) at B4 T4096 H16 K16 V64"
L2_BYTES = 129 * 1024 * 1024
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}


def canonical_flops(B, T, H, K, V, C=64):
    """FLOPs credited to one forward pass from the shape alone (the spec's canonical_work)."""
    P = 1 + K + K * K
    return B * H * T * (4 * P * V + 2 * C * (K + V))


def algorithmic_bytes(B, T, H, K, V, out_bytes=4):
    """q, k, v read once (bf16) and o written once (fp32, or bf16 with out_bytes=2)."""
    return B * T * H * (2 * K * 2 + V * 2 + V * out_bytes)


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return d, "measured"
    return dict(FALLBACK_PEAKS), "fallback"


def kernel_source_sha():
    h = hashlib.sha256()
    for rel in ("linear_attention_gb300/csrc/based_kernels.cuh",
                "linear_attention_gb300/csrc/sm103_ptx.cuh"):
        with open(os.path.join(ROOT, rel), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def ncu_traffic(workload):
    """DRAM bytes per launch of the forward kernel from the committed ncu summary, if it was taken
    on the current kernel source; else None."""
    p = os.path.join(ROOT, "profiles", f"based_fwd_kernel_{workload}_traffic.json")
    if not os.path.exists(p):
        return None
    with open(p) as f:
        d = json.load(f)
    if d.get("kernel_source_sha") != kernel_source_sha():
        return None
    return d.get("dram_bytes_per_launch")


class ClockSampler:
    """nvidia-smi clocks/throttle sampling while the timed region runs."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.gpu = gpu_index
        self.proc = None
        self.path = None

    def start(self):
        fd, self.path = tempfile.mkstemp(prefix="clocks_", suffix=".csv")
        os.close(fd)
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
        except OSError:
            self.proc = None
        return self

    def nsamples(self):
        try:
            with open(self.path) as f:
                return sum(1 for line in f if line.strip())
        except OSError:
            return 0

    def stop(self):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
        rows = []
        try:
            with open(self.path) as f:
                for line in f:
                    parts = [x.strip() for x in line.split(",")]
                    if len(parts) >= 9:
                        rows.append(parts)
            os.unlink(self.path)
        except OSError:
            pass
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"], "samples": 0}

        def num(x):
            try:
                return float(x)
            except ValueError:
                return None

        sm = [num(r[1]) for r in rows if num(r[1]) is not None]
        smax = [num(r[2]) for r in rows if num(r[2]) is not None]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i in range(4) if r[5 + i] == "Active"})
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(smax) if smax else None, "reasons": reasons,
                "samples": len(rows)}


def dist_setup():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        backend = "nccl" if torch.cuda.is_available() else "gloo"
        if backend == "nccl":
            torch.cuda.set_device(local)
        dist.init_process_group(backend)
    return world, rank, local


def dist_max(x, world, device):
    if world == 1:
        return x
    import torch.distributed as dist
    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def dist_barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def job_value(tokens_per_step, steps, elapsed_ms, world):
    """Whole-job throughput: every rank processes its own replica of the workload, the time is the
    slowest rank's."""
    return world * tokens_per_step * steps / (elapsed_ms * 1e-3)


def workload_config(w, extra=None):
    cfg = {"workload": f"Based fwd {w.name}: B={w.B} T={w.T} H={w.H} K={w.K} V={w.V}",
           "B": w.B, "T": w.T, "H": w.H, "K": w.K, "V": w.V,
           "scale": w.scale if w.scale is not None else "K^-0.5",
           "inputs": f"q,k,v ~ N(0,1) bf16, seed {w.seed}; fp32 output"}
    if extra:
        cfg.update(extra)
    return cfg


# ------------------------------------------------------------------------------------------------
# CPU oracle arm (also the cpu_baseline of the GPU arm)
# ------------------------------------------------------------------------------------------------
def oracle_inputs(w):
    q, k, v = make_workload(w)
    return q.double().numpy(), k.double().numpy(), v.double().numpy()


def time_oracle(w, qkv, heads, nthreads):
    import oracle
    q, k, v = qkv
    sc = oracle.default_scale(w.K) if w.scale is None else float(w.scale)
    t0 = time.perf_counter()
    oracle.chunked(q, k, v, sc, chunk=256, heads=heads, nthreads=nthreads)
    return time.perf_counter() - t0


def cpu_baseline(w, budget_s=12.0):
    """The oracle as it stands on the host cores: repeated passes over sampled heads until about
    budget_s of wall time; tokens/s scaled to the whole workload."""
    import oracle
    qkv = oracle_inputs(w)
    nthreads = oracle.default_threads()
    nh = w.B * w.H
    heads = list(range(nh))
    t_all = time_oracle(w, qkv, heads, nthreads)  # one full pass
    passes, total = 1, t_all
    while total + t_all <= budget_s:
        total += time_oracle(w, qkv, heads, nthreads)
        passes += 1
    tok_s = w.B * w.T * passes / total
    return {"value": tok_s, "unit": "tokens/s", "cores": nthreads, "kind": "oracle",
            "sample": f"{passes} full pass(es) over all {nh} heads of the workload, fp64 chunked "
                      f"feature-map form (chunk 256), {total:.2f} s wall"}


def run_reference(args, w, world, rank):
    if rank != 0:
        return 0
    import oracle
    oracle.build()
    qkv = oracle_inputs(w)
    nthreads = oracle.default_threads()
    nh = w.B * w.H
    # size each step so that warmup + steps end within about two minutes
    t_head = time_oracle(w, qkv, [0], 1)
    budget = 120.0 / max(1, args.steps + args.warmup)
    per_head_wall = t_head / max(1, min(nthreads, nh))
    n = int(max(1, min(nh, budget / max(per_head_wall, 1e-6))))
    heads = list(range(n))
    for _ in range(args.warmup):
        time_oracle(w, qkv, heads, nthreads)
    times = [time_oracle(w, qkv, heads, nthreads) for _ in range(args.steps)]
    t = sum(times)
    tokens = w.B * w.T * (n / nh) * args.steps
    value = tokens / t
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "tokens/s",
        "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": 1e3 * t / args.steps, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": workload_config(w),
        "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": nthreads, "kind": "oracle",
                         "sample": f"{n} of {nh} heads per step, whole rows, fp64 chunked "
                                   f"feature-map form; tokens scaled by {n}/{nh}"},
        "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


# ------------------------------------------------------------------------------------------------
# GPU arm
# ------------------------------------------------------------------------------------------------
def run_gpu(args, w, world, rank, local):
    from linear_attention_gb300 import build as lbuild
    lbuild.build()
    from linear_attention_gb300.based import (based_fwd, based_fwd_bf16_out, based_fwd_host,
                                              based_fwd_timed, device_status, kernel_count)

    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    B, T, H, K, V = w.B, w.T, w.H, w.K, w.V
    q0, k0, v0 = make_workload(w)
    obf = args.out == "bf16"
    out_dtype = torch.bfloat16 if obf else torch.float32
    wbytes = algorithmic_bytes(B, T, H, K, V, 2 if obf else 4)

    def fwd(s, stream=None):
        if obf:
            based_fwd_bf16_out(*s[:3], scale=w.scale, out=s[3], stream=stream)
        else:
            based_fwd(*s[:3], scale=w.scale, out=s[3], stream=stream)

    def fwd_timed(s, eb, ee, stream):
        if obf:
            based_fwd_bf16_out(*s[:3], scale=w.scale, out=s[3], stream=stream, events=(eb, ee))
        else:
            based_fwd_timed(s[0], s[1], s[2], s[3], eb, ee, scale=w.scale, stream=stream)
    # rotate enough input/output sets that consecutive steps never find their data in L2
    nsets = max(2, -(-3 * L2_BYTES // wbytes) + 1)
    sets = []
    for i in range(nsets):
        sets.append((q0.to(dev), k0.to(dev), v0.to(dev),
                     torch.empty(B, T, H, V, dtype=out_dtype, device=dev)))
    stream = torch.cuda.current_stream(dev)
    ev_b = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    ev_e = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    for e in ev_b + ev_e:
        e.record(stream)  # creates the handles the library records into
    t_start, t_stop = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize(dev)

    # warm-up: W steps, then keep stepping for at least 1 s so clocks settle under load
    clocks = ClockSampler(local).start() if (rank == 0 and not args.profile) else None
    for i in range(max(3, args.warmup)):
        fwd(sets[i % nsets])
    torch.cuda.synchronize(dev)
    t_end = time.time() + (0.0 if args.profile else 1.0)
    i = 0
    while time.time() < t_end or (clocks is not None and clocks.nsamples() < 3 and
                                  time.time() < t_end + 5):
        for _ in range(20):
            fwd(sets[i % nsets])
            i += 1
        torch.cuda.synchronize(dev)

    # timed region: exactly K steps, back to back as a caller issues them
    dist_barrier(world)
    torch.cuda.synchronize(dev)
    t_start.record(stream)
    for j in range(args.steps):
        fwd(sets[j % nsets], stream)
    t_stop.record(stream)
    torch.cuda.synchronize(dev)
    dist_barrier(world)
    clk = clocks.stop() if clocks is not None else None
    elapsed_ms = t_start.elapsed_time(t_stop)
    # the forward kernel alone: K more steps with CUDA events recorded on the launch stream right
    # around it (this launches it without overlap with the kernel before it, so its duration is
    # not shortened by early start)
    torch.cuda.synchronize(dev)
    for j in range(args.steps):
        fwd_timed(sets[j % nsets], ev_b[j], ev_e[j], stream)
    torch.cuda.synchronize(dev)
    fwd_ms = [ev_b[j].elapsed_time(ev_e[j]) for j in range(args.steps)]
    elapsed_ms = dist_max(elapsed_ms, world, dev)
    status = device_status(local, clear=True)
    if status != 0:
        raise RuntimeError(f"a kernel gave up a bounded wait (status {status:#x})")

    ms_per_step = elapsed_ms / args.steps
    tokens_per_step = B * T
    value = job_value(tokens_per_step, args.steps, elapsed_ms, world)
    flops = canonical_flops(B, T, H, K, V)
    peaks, peak_kind = load_peaks()
    hbm = float(peaks["hbm_gbs"])
    tc = float(peaks["bf16_tflops"])
    fwd_avg_ms = sum(fwd_ms) / len(fwd_ms)
    achieved_gbs = wbytes / (fwd_avg_ms * 1e-3) / 1e9
    t_roof_ms = max(wbytes / (hbm * 1e9), flops / (tc * 1e12)) * 1e3
    launches = kernel_count(B, T, H, K, V)

    # end-to-end through the host entry point: pinned host inputs -> GPU -> pinned host output
    e2e = None
    if obf:
        e2e = {"value": None, "unit": "tokens/s",
               "note": "the host entry point (based_fwd_host) returns fp32 only"}
    elif not args.profile:
        qh, kh, vh = q0.pin_memory(), k0.pin_memory(), v0.pin_memory()
        oh = torch.empty(B, T, H, V, dtype=torch.float32).pin_memory()
        for _ in range(3):
            based_fwd_host(qh, kh, vh, scale=w.scale, out=oh, device=dev)
        n_e2e = max(3, min(args.steps, 20))
        dist_barrier(world)
        t0 = time.perf_counter()
        for _ in range(n_e2e):
            based_fwd_host(qh, kh, vh, scale=w.scale, out=oh, device=dev)
        t_e2e = dist_max(time.perf_counter() - t0, world, dev)
        e2e = {"value": world * tokens_per_step * n_e2e / t_e2e, "unit": "tokens/s",
               "h2d_bytes_per_step": B * T * H * (2 * K + V) * 2,
               "d2h_bytes_per_step": B * T * H * V * 4, "steps": n_e2e,
               "ms_per_step": 1e3 * t_e2e / n_e2e}

    if rank != 0:
        return 0
    cpu = None if (args.no_cpu_baseline or args.profile or world > 1) else cpu_baseline(w)
    line = {
        "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms_per_step,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic",
        "config": workload_config(w, {
            "l2": f"{nsets} rotating input/output sets ({nsets * wbytes / 2**20:.0f} MiB > 3x L2)",
            "output": "bf16" if obf else "fp32",
            "launch": f"stream launches, one {'based_fwd_bf16_out' if obf else 'based_fwd'} call per step "
                      f"({launches} kernel(s): the forward kernel alone when the ranges that start "
                      "inside a head run lead-ins; else aggregate, scan when a prefix chains more "
                      "than four partial states, forward, the later ones as programmatic "
                      "dependents)"}),
        "tflops": flops / (ms_per_step * 1e-3) / 1e12,
        "pct_bf16_peak": 100.0 * flops / (ms_per_step * 1e-3) / (tc * 1e12),
        "pct_roofline_step": 100.0 * t_roof_ms / ms_per_step,
        "roofline": {"bound": "hbm", "achieved": achieved_gbs, "peak": hbm, "unit": "GB/s",
                     "frac": achieved_gbs / hbm, "traffic": ncu_traffic(w.name),
                     "kernel": "based_fwd_kernel", "kernel_ms": fwd_avg_ms,
                     "kernel_timing": "CUDA events around the forward kernel on its launch stream, "
                                      "K steps after the timed region, launched without overlap",
                     "algorithmic_bytes": wbytes, "peak_source": f"{peak_kind} (hbm_gbs)",
                     # the whole call (every kernel of the step) against the same bound
                     "call_achieved": wbytes / (ms_per_step * 1e-3) / 1e9,
                     "call_frac": wbytes / (ms_per_step * 1e-3) / 1e9 / hbm,
                     "call_roofline_ms": t_roof_ms,
                     "kernel_source_sha": kernel_source_sha()},
        "gpu_launches": launches * args.steps,
        "clocks": clk,
        "e2e": e2e,
        "cpu_baseline": cpu,
    }
    print(json.dumps(line), flush=True)
    return 0


def main():
    ap = argparse.ArgumentParser(description=__doc__.split("\n\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--workload", default="headline", choices=sorted(WORKLOADS) + sorted(GRADER_WORKLOADS))
    ap.add_argument("--impl", default="gb300", choices=["gb300", "reference"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--out", default="fp32", choices=["fp32", "bf16"],
                    help="output dtype (fp32 is the contract's default; bf16 uses based_fwd_bf16_out)")
    ap.add_argument("--profile", action="store_true",
                    help="only the W warm-up and K timed steps (for running under ncu)")
    args = ap.parse_args()
    if args.steps < 1:
        ap.error("--steps must be >= 1")
    w = WORKLOADS[args.workload] if args.workload in WORKLOADS else GRADER_WORKLOADS[args.workload]
    if args.impl == "reference":
        # the CPU oracle arm: rank 0 alone runs it, other ranks exit without work
        world = int(os.environ.get("WORLD_SIZE", "1"))
        rank = int(os.environ.get("RANK", "0"))
        return run_reference(args, w, world, rank)
    world, rank, local = dist_setup()
    try:
        return run_gpu(args, w, world, rank, local)
    finally:
        if world > 1:
            import torch.distributed as dist
            dist.destroy_process_group()


if __name__ == "__main__":
    sys.exit(main())
