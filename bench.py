"""Benchmark of the batched constrained logits sampler.

One step = one sampler call (penalties, bias, grammar mask, temperature, top-k ->
top-p -> min-p, exponential race, logprob) over one batch of the penalties+bias
workload: B=192 rows, V=151936, fp32 logits, Zipf histories of 0-4096 ids, 16
logit_bias entries per row, bitmasks on 25% of rows, mixed parameters.  --workload
selects another batch (1-5: the tiny, decode-mix, grammar, penalties and
verify-scale configurations; 6-7: all-greedy and all-untruncated batches on the
single-sweep fast path).

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference] [--workload n]

--gpus N > 1 runs N replicas, one process per GPU: under a launcher that sets
WORLD_SIZE (torchrun) it must equal N; without one, bench.py starts
torch.distributed.run itself.

Prints one JSON line (rank 0).  Inputs are rotated over three resident copies of the
batch (3 x 122 MB, more than twice the 129 MB L2), so no step reads a batch that the
previous step left in L2.  Per-launch times come from CUDA events on the launching
stream; SM clocks are sampled with nvidia-smi during the timed region.
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

METRIC = "rows/s & HBM GB/s (% of peak), fused mask+top-k/p sample, B=192 V=151936"
WORKLOAD = 4
MODE_FAST_SWEEP = 4  # clsample.h CLSAMPLE_MODE_FAST_SWEEP
N_SETS = 3
FALLBACK_HBM_GBS = 6800.0
NOMINAL_HBM_GBS = 8000.0  # GB300 HBM3e, nominal


def parse(argv=None):
    p = argparse.ArgumentParser()
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=1000)
    p.add_argument("--warmup", type=int, default=20)
    p.add_argument("--impl", default="ours", choices=["ours", "reference"])
    p.add_argument("--workload", type=int, default=WORKLOAD)
    p.add_argument("--no-e2e", action="store_true")
    p.add_argument("--no-cpu", action="store_true")
    return p.parse_args(argv)


def dist_env():
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return rank, world, local


def launch_plan(args, env, argv):
    """How `--gpus N` runs: ("run", None) in this process; ("spawn", cmd) to start N
    ranks with torch.distributed.run; ("error", message) when a launcher's world size
    disagrees with --gpus."""
    if args.gpus < 1:
        return "error", f"--gpus {args.gpus}: at least one GPU"
    world = env.get("WORLD_SIZE")
    if world is not None:
        if int(world) != args.gpus:
            return "error", f"--gpus {args.gpus} but the launcher started WORLD_SIZE={world} ranks"
        return "run", None
    if args.gpus == 1:
        return "run", None
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", f"--nproc-per-node={args.gpus}",
           "--master-addr", "127.0.0.1", "--master-port", str(env.get("MASTER_PORT", "29531")),
           os.path.abspath(__file__), *argv]
    return "spawn", cmd


def peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    except Exception:
        return FALLBACK_HBM_GBS, "fallback"


def kernel_source_hash():
    """Hash of the CUDA sources and the C header (ties a committed ncu traffic figure
    to the kernel it was measured on)."""
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "constrained_logits_sampling_gb300", "csrc")
    paths = sorted(os.path.join(csrc, n) for n in os.listdir(csrc) if n.endswith((".cu", ".cuh")))
    for p in paths + [os.path.join(ROOT, "include", "clsample.h")]:
        with open(p, "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def traffic_from_profile(workload_name):
    """DRAM bytes per launch from the committed ncu summary, if it was taken on the
    current kernel source; else None."""
    path = os.path.join(ROOT, "profiles", "traffic.json")
    try:
        with open(path) as f:
            d = json.load(f)
    except Exception:
        return None
    for c in d.get("captures", [d]):
        if c.get("kernel_source_sha") == kernel_source_hash() and c.get("workload") == workload_name:
            return c.get("dram_bytes_per_launch")
    return None


class ClockSampler:
    """nvidia-smi clocks and throttle reasons, sampled every 20 ms."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.gpu = gpu_index
        self.proc = None
        self.lines = []

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "20"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.t = threading.Thread(target=self._read, daemon=True)
            self.t.start()
        except Exception:
            self.proc = None

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
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for l in self.lines:
            parts = [x.strip() for x in l.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                smax.append(float(parts[2]))
            except ValueError:
                continue
            for n, v in zip(names, parts[5:9]):
                if v.lower() in ("active", "1"):
                    reasons.add(n)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(smax) if smax else None,
                "reasons": sorted(reasons), "samples": len(sm)}


def cpu_baseline(batch, sample_rows, min_repeats=3, min_seconds=1.0, max_repeats=40, single_rows=8):
    """The oracle as it stands, on the host cores, on a bounded sample of the batch:
    whole passes over the sample until about `min_seconds` of wall time (10-30 s of
    CPU work on a many-core host), at least `min_repeats` of them; then the same on one
    thread over a smaller sample."""
    from oracle import oracle as O

    def timed(sub, nthreads):
        O.sample(sub, nthreads=nthreads, want_transformed=False)  # warm-up (page-in, thread start)
        t0 = time.perf_counter()
        threads, repeats = 1, 0
        while repeats < min_repeats or (time.perf_counter() - t0 < min_seconds and repeats < max_repeats):
            threads = O.sample(sub, nthreads=nthreads, want_transformed=False)["threads"]
            repeats += 1
        return time.perf_counter() - t0, int(threads), repeats

    sub = batch.rows(range(min(sample_rows, batch.B)))
    dt, threads, repeats = timed(sub, 0)
    sub1 = batch.rows(range(min(single_rows, batch.B)))
    dt1, _, repeats1 = timed(sub1, 1)
    return {"value": sub.B * repeats / dt, "unit": "rows/s", "cores": threads, "kind": "oracle",
            "sample": f"{sub.B} rows of workload {batch.name} (B={batch.B}, V={batch.V}) x {repeats} repeats, "
                      f"{dt:.2f} s wall on {threads} threads (about {dt * threads:.0f} s of CPU work)",
            "single_thread": {"value": sub1.B * repeats1 / dt1, "unit": "rows/s", "cores": 1,
                              "sample": f"{sub1.B} rows x {repeats1} repeats, {dt1:.2f} s on one thread"}}


def run_reference(args, rank, world):
    if rank != 0:
        return 0
    from constrained_logits_sampling_gb300.workloads import make_workload
    from oracle import oracle as O
    O.build()
    b = make_workload(args.workload)
    sample_rows = min(32, b.B)
    sub = b.rows(range(sample_rows))
    for _ in range(max(args.warmup, 0)):
        O.sample(sub, nthreads=0)
    t0 = time.perf_counter()
    threads = 1
    for _ in range(args.steps):
        threads = O.sample(sub, nthreads=0)["threads"]
    dt = time.perf_counter() - t0
    value = sample_rows * args.steps / dt
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "rows/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": dt / args.steps * 1e3,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f32+f64",
        "data": "synthetic",
        "config": {"workload": workload_text(b, args.workload), "sample_rows_per_step": sample_rows},
        "cpu_baseline": {"value": value, "unit": "rows/s", "cores": int(threads), "kind": "oracle",
                         "sample": f"{sample_rows} rows of {b.name} per step, {args.steps} steps"},
        "e2e": {"value": value, "unit": "rows/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


def max_over_ranks(values, dist=None, device=None):
    """Element-wise max of a list of floats over the ranks (the timing rule: the slowest
    rank's time counts); the list unchanged on one process."""
    if dist is None:
        return [float(v) for v in values]
    import torch
    t = torch.tensor([float(v) for v in values], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return [float(v) for v in t.tolist()]


def rows_per_second(rows_per_rank, world, steps, total_ms):
    """Whole-job throughput: every rank processes rows_per_rank rows per step (weak
    scaling), over the slowest rank's time for `steps` steps."""
    return rows_per_rank * world * steps / (total_ms / 1e3)


def workload_text(b, n):
    from constrained_logits_sampling_gb300.workloads import WORKLOADS
    return f"{b.name} (workload {n}): " + WORKLOADS.get(n, "").split(": ", 1)[-1]


def main():
    args = parse()
    how, what = launch_plan(args, os.environ, sys.argv[1:])
    if how == "error":
        print(json.dumps({"error": what}), flush=True)
        return 2
    if how == "spawn":
        return subprocess.call(what)
    rank, world, local = dist_env()
    if args.impl == "reference":
        return run_reference(args, rank, world)

    import numpy as np
    import torch

    from constrained_logits_sampling_gb300 import build as cuda_build
    from constrained_logits_sampling_gb300.sampler import Sampler, batch_to_device
    from constrained_logits_sampling_gb300.workloads import make_workload

    torch.cuda.set_device(local)
    dist = None
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    cuda_build.build()
    dev = torch.device("cuda", local)
    b = make_workload(args.workload)
    s = Sampler(b.B, b.V)
    sets = []
    for i in range(N_SETS):
        kw = batch_to_device(b, dev)
        logits = kw.pop("logits")
        out = {"tokens": torch.empty(b.B, dtype=torch.int32, device=dev),
               "logprobs": torch.empty(b.B, dtype=torch.float32, device=dev)}
        sets.append((s.make_args(logits, tokens=out["tokens"], logprobs=out["logprobs"], **kw), kw, logits, out))
    stream = torch.cuda.current_stream()
    torch.cuda.synchronize()

    def barrier():
        if dist is not None:
            dist.barrier()
        torch.cuda.synchronize()

    for i in range(args.warmup):
        s.apply(sets[i % N_SETS][0], stream)
    barrier()
    # The K timed steps are captured into one CUDA graph, so the host's launch cost does
    # not leave the GPU idle between steps; every step is the ordering kernel and the
    # sampler kernel.
    graph = torch.cuda.CUDAGraph()
    cap_stream = torch.cuda.Stream(device=dev)
    cap_stream.wait_stream(stream)
    with torch.cuda.graph(graph, stream=cap_stream):
        for i in range(args.steps):
            s.apply(sets[i % N_SETS][0], cap_stream)
    graph.replay()  # one untimed replay: the graph's first launch uploads it
    barrier()
    clocks = ClockSampler(local)
    clocks.start()
    time.sleep(0.2)  # nvidia-smi's first sample lands before the timed region starts
    barrier()
    t_all0 = torch.cuda.Event(enable_timing=True)
    t_all1 = torch.cuda.Event(enable_timing=True)
    t_all0.record(stream)
    graph.replay()
    t_all1.record(stream)
    barrier()
    clk = clocks.stop()
    total_ms = t_all0.elapsed_time(t_all1)
    # each kernel alone: the two halves of a step with events between them (the launch
    # queue stays ahead of the GPU, so the events bracket the kernels themselves)
    n_split = min(args.steps, 100)
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(n_split)]
    for i in range(n_split):
        a_i = sets[i % N_SETS][0]
        ev[i][0].record(stream)
        s.prepare(a_i, stream)
        ev[i][1].record(stream)
        s.sample(a_i, stream)
        ev[i][2].record(stream)
    barrier()
    order_ms = sum(e[0].elapsed_time(e[1]) for e in ev) / n_split
    mean_launch_ms = sum(e[1].elapsed_time(e[2]) for e in ev) / n_split  # the sampler kernel
    total_ms, mean_launch_ms, order_ms = max_over_ranks([total_ms, mean_launch_ms, order_ms], dist, dev)
    ms_per_step = total_ms / args.steps
    value = rows_per_second(b.B, world, args.steps, total_ms)

    # ---- end to end through the public API: host inputs -> device -> sampler -> host
    e2e = None
    if not args.no_e2e:
        host = {}
        kw0 = batch_to_device(b, "cpu")
        for k, v in kw0.items():
            if isinstance(v, torch.Tensor):
                host[k] = v.pin_memory()
            else:
                host[k] = v
        h2d = sum(v.numel() * v.element_size() for v in host.values() if isinstance(v, torch.Tensor))
        out_host = {"tokens": torch.empty(b.B, dtype=torch.int32).pin_memory(),
                    "logprobs": torch.empty(b.B, dtype=torch.float32).pin_memory()}
        d2h = sum(v.numel() * v.element_size() for v in out_host.values())
        e2e_steps = max(10, min(args.steps, 50))

        # two buffer sets: the upload of step i + 1 (copy stream) overlaps the sampling of
        # step i (compute stream); every step still uploads its inputs from pinned host
        # memory and reads its tokens and logprobs back inside the timed region
        copy_stream = torch.cuda.Stream(device=dev)
        bufs = []
        for _ in range(2):
            dkw = {k: (torch.empty_like(v, device=dev) if isinstance(v, torch.Tensor) else v) for k, v in host.items()}
            bufs.append({"kw": dkw, "uploaded": torch.cuda.Event(), "consumed": torch.cuda.Event()})
        for bset in bufs:
            bset["consumed"].record(stream)

        def upload(i):
            bset = bufs[i % 2]
            with torch.cuda.stream(copy_stream):
                copy_stream.wait_event(bset["consumed"])
                for k, v in host.items():
                    if isinstance(v, torch.Tensor):
                        bset["kw"][k].copy_(v, non_blocking=True)
                bset["uploaded"].record(copy_stream)

        def sample_step(i):
            bset = bufs[i % 2]
            stream.wait_event(bset["uploaded"])
            kw_i = dict(bset["kw"])
            lg = kw_i.pop("logits")
            out = s(lg, **kw_i)
            bset["consumed"].record(stream)
            out_host["tokens"].copy_(out["tokens"], non_blocking=True)
            out_host["logprobs"].copy_(out["logprobs"], non_blocking=True)

        def e2e_run(nsteps):
            upload(0)
            for i in range(nsteps):
                if i + 1 < nsteps:
                    upload(i + 1)
                sample_step(i)

        e2e_run(3)
        barrier()
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        copy_stream.wait_event(e0)
        e2e_run(e2e_steps)
        e1.record(stream)
        barrier()
        e_ms = max_over_ranks([e0.elapsed_time(e1)], dist, dev)[0]
        e2e = {"value": rows_per_second(b.B, world, e2e_steps, e_ms), "unit": "rows/s",
               "h2d_bytes_per_step": int(h2d), "d2h_bytes_per_step": int(d2h), "steps": e2e_steps}

    if rank != 0:
        if dist is not None:
            dist.destroy_process_group()
        return 0

    peak, peak_kind = peaks()
    alg = b.algorithmic_bytes()
    sweep = bool(getattr(b, "mode", 0) & MODE_FAST_SWEEP)
    hb = b.host_bytes()
    if sweep:
        # the single-sweep kernel reads everything itself: logits, bitmask, parameters and
        # the history and logit_bias CSRs (each CTA scans its rows' lists), writes outputs
        alg_kernel = alg
        kernel = ("sweep_kernel (single pass, one CTA per (row, 8192-token slice); no preparation launch; "
                  "the row's last CTA draws)")
    else:
        # the sampler kernel reads the logits, the bitmask and the per-row parameters and
        # writes the outputs; the history and logit_bias CSRs are read by the preparation
        # launch ahead of it (which hands the sampler a short list per slice instead)
        alg_kernel = alg - sum(hb.get(k, 0) for k in ("hist_offs", "hist_ids", "bias_offs", "bias_ids", "bias_vals"))
        kernel = ("sampler_kernel (one CTA per (row, slice), launched with programmatic serialisation after "
                  "order_kernel, the preparation launch: row order and per-row penalty/bias lists)")
    achieved = alg_kernel / (mean_launch_ms / 1e3) / 1e9
    line = {
        "metric": METRIC,
        "value": value,
        "unit": "rows/s",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": ms_per_step,
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "bf16" if b.logits_bf16 else "f32",
        "data": "synthetic",
        "config": {
            "workload": workload_text(b, args.workload),
            "rows_per_gpu": b.B,
            "l2": f"inputs rotated over {N_SETS} resident copies ({N_SETS * alg / 1e6:.0f} MB > 2 x L2)",
            "parallelism": f"replicas x{world} (rows are independent)",
        },
        "hbm_gbs": alg / (ms_per_step / 1e3) / 1e9,
        "roofline": {
            "bound": "hbm",
            "achieved": achieved,
            "peak": peak,
            "unit": "GB/s",
            "frac": achieved / peak,
            "frac_of_nominal_8tbs": achieved / NOMINAL_HBM_GBS,
            "peak_kind": f"{peak_kind} (MEASURED_PEAKS.json hbm_gbs)" if peak_kind == "measured" else "fallback",
            "traffic": traffic_from_profile(b.name),
            "algorithmic_bytes_per_launch": alg_kernel,
            "mean_launch_us": mean_launch_ms * 1e3,
            "kernel": kernel,
            "order_kernel_us": None if sweep else order_ms * 1e3,
            "step_algorithmic_gbs": alg / (ms_per_step / 1e3) / 1e9,
        },
        "gpu_launches": (1 if sweep else 2) * args.steps,
        "clocks": clk,
        "e2e": e2e,
    }
    if not args.no_cpu:
        line["cpu_baseline"] = cpu_baseline(b, sample_rows=b.B)
    print(json.dumps(line), flush=True)
    if dist is not None:
        dist.destroy_process_group()
    return 0


if __name__ == "__main__":
    sys.exit(main())
