"""Benchmark of the verify-and-accept step on GB300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                    [--workload vocab248k|batch64|tree60|small]

One step is one spec_verify_sample call (the whole chain path: row
statistics, accept scan, residual or bonus draw) on one batch.  The default
workload is the one the headline metric is quoted on: B=1 request, k=4
drafted tokens, V=248,320 bf16 logits (9 verified rows per step).  Inputs
rotate over 64 resident input sets (286 MB, more than twice the 126 MB L2) so
no step reads logits from L2; the calls are replayed from a CUDA graph.

Printed JSON line (rank 0): value = verified rows/s over all ranks, roofline
of the dominant kernel against the measured HBM copy bandwidth, the oracle's
CPU rate on the machine's host cores, the end-to-end rate through the C ABI with
host buffers, SM clocks sampled during the run.

Multi-GPU: under torchrun every rank runs the same workload on its own GPU
(independent replicas, no collective on the data path); the timing is the
max over ranks.  --impl reference times the fp64 oracle on the host cores.
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
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "verified logit rows/sec at V=248,320; achieved HBM GB/s vs GB300 peak"
FALLBACK_HBM_GBS = 6800.0
L2_BYTES = 126 * 1024 * 1024
PROFILE_DIR = os.path.join(ROOT, "profiles")
KERNEL_SOURCES = ["speculative_decoding_verification_02_gb300/csrc/chain.cu",
                  "speculative_decoding_verification_02_gb300/csrc/common.cuh"]


# --------------------------------------------------------------- workloads

def make_workload(name: str):
    from speculative_decoding_verification_02_gb300 import workloads as W
    if name == "vocab248k":
        return W.chain_vocab248k(W.SEED_BASE + 3, B=1), "chain sampling verify, B=1, k=4, V=248,320 bf16 " \
            "(t~N(0,3) with 5 ids +8, d=0.8t+N(0,1), T=1)"
    if name == "batch64":
        return W.chain_batch64(), "chain sampling verify, B=64, k=8, V=128,256 bf16 " \
            "(t~N(0,2.5), d=t+N(0,s) s in {0.3,1,2}, T=0.7)"
    if name == "small":
        return W.chain_small(), "chain sampling verify, B=4, k=4, V=2048 fp32 (t~N(0,2), d=t+N(0,0.5), T=1)"
    raise ValueError(name)


def row_bytes(prob) -> int:
    """Algorithmic bytes of one call's streaming pass: every target and draft
    row read once."""
    B, R, V = prob["target"].shape
    es = 2 if prob["target"].dtype == np.uint16 else 4
    return B * (2 * R - 1) * V * es


# ------------------------------------------------------------------ clocks

class ClockSampler:
    """nvidia-smi clocks and throttle reasons every 200 ms while running."""
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.path = os.path.join(ROOT, "gpurun_out", f"clocks_gpu{gpu_index}.csv")

    def __enter__(self):
        try:
            os.makedirs(os.path.dirname(self.path), exist_ok=True)
            self.f = open(self.path, "w")
            self.proc = subprocess.Popen(["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                                          "-lms", "200", "-i", str(self.gpu)], stdout=self.f,
                                         stderr=subprocess.DEVNULL)
        except (OSError, FileNotFoundError):
            self.proc = None
        return self

    def __exit__(self, *a):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
            self.f.close()

    def summary(self) -> dict:
        if self.proc is None or not os.path.exists(self.path):
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        sms, maxs, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in open(self.path):
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                sms.append(float(parts[1]))
                maxs.append(float(parts[2]))
            except ValueError:
                continue
            for n, v in zip(names, parts[5:9]):
                if v.lower() == "active":
                    reasons.add(n)
        if not sms:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"]}
        return {"sm_mhz": statistics.median(sms), "sm_max_mhz": max(maxs), "reasons": sorted(reasons),
                "samples": len(sms)}


# ----------------------------------------------------------------- helpers

def peak_hbm():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            return float(json.load(f)["hbm_gbs"]), "measured"
    except (OSError, KeyError, ValueError):
        return FALLBACK_HBM_GBS, "fallback"


def source_sha() -> str:
    h = hashlib.sha256()
    for rel in KERNEL_SOURCES:
        with open(os.path.join(ROOT, rel), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def profiled_traffic(kernel: str, workload: str):
    """DRAM bytes per launch from the committed ncu summary of this kernel and
    workload, if the kernel sources are unchanged since the capture."""
    path = os.path.join(PROFILE_DIR, f"{kernel}_{workload}.md")
    if not os.path.exists(path):
        return None
    vals = {}
    for line in open(path):
        if ":" in line and line.strip().startswith("- "):
            k, v = line.strip()[2:].split(":", 1)
            vals[k.strip()] = v.strip().strip("`")
    if vals.get("source_sha") != source_sha():
        return None
    try:
        return float(vals["dram_bytes_per_launch"])
    except (KeyError, ValueError):
        return None


def dist_env():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


def reduce_max(value: float, device) -> float:
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()):
        return value
    t = torch.tensor([value], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def reduce_sum(value: float, device) -> float:
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()):
        return value
    t = torch.tensor([value], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.SUM)
    return float(t.item())


def barrier():
    import torch.distributed as dist
    if dist.is_available() and dist.is_initialized():
        dist.barrier()


# --------------------------------------------------------------- CPU oracle

def oracle_rate(prob, target_seconds: float, max_requests: int | None = None):
    """Rows/s of the fp64 oracle on this host's cores over a bounded sample of
    the workload (requests replicated from the problem, one call)."""
    import oracle
    B, R, V = prob["target"].shape
    threads = oracle.max_threads()
    # calibrate with one request, then size the sample to ~target_seconds
    t0 = time.perf_counter()
    oracle.verify_sample(prob["target"][:1], prob["draft_logits"][:1], prob["draft"][:1], prob["uniforms"][:1],
                         prob["T"], threads=1)
    one = max(time.perf_counter() - t0, 1e-6)
    n = max(1, int(target_seconds * threads / one))
    if max_requests:
        n = min(n, max_requests)
    idx = np.arange(n) % B
    tgt = np.broadcast_to(prob["target"][:1], (n,) + prob["target"].shape[1:]) if B == 1 else prob["target"][idx]
    dl = np.broadcast_to(prob["draft_logits"][:1], (n,) + prob["draft_logits"].shape[1:]) if B == 1 \
        else prob["draft_logits"][idx]
    t0 = time.perf_counter()
    oracle.verify_sample(tgt, dl, prob["draft"][idx], prob["uniforms"][idx], prob["T"], threads=threads)
    dt = time.perf_counter() - t0
    rows = n * (2 * R - 1)
    return rows / dt, threads, n, dt


# ------------------------------------------------------------ reference arm

def run_reference(args, workload_name):
    ws, rank, _ = dist_env()
    if rank != 0:
        return 0
    prob, desc = make_workload(workload_name)
    import oracle
    B, R, V = prob["target"].shape
    rows_per_step = B * (2 * R - 1)
    threads = min(oracle.max_threads(), B)   # the oracle parallelises over requests
    budget = float(os.environ.get("SPEC_REF_SECONDS", "60"))
    t_start = time.perf_counter()
    steps_done = 0
    for _ in range(args.warmup):
        oracle.verify_sample(prob["target"], prob["draft_logits"], prob["draft"], prob["uniforms"], prob["T"],
                             threads=threads)
        if time.perf_counter() - t_start > budget / 4:
            break
    t0 = time.perf_counter()
    for _ in range(args.steps):
        oracle.verify_sample(prob["target"], prob["draft_logits"], prob["draft"], prob["uniforms"], prob["T"],
                             threads=threads)
        steps_done += 1
        if time.perf_counter() - t0 > budget:
            break
    dt = time.perf_counter() - t0
    value = steps_done * rows_per_step / dt
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": "rows/s", "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * dt / steps_done,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic", "config": {"workload": desc, "rows_per_step": rows_per_step},
            "cpu_baseline": {"kind": "oracle", "value": value, "unit": "rows/s", "cores": threads,
                             "sample": f"{steps_done} of {args.steps} steps timed (cap {budget:.0f} s), "
                                       f"one call of the workload each"},
            "e2e": {"value": value, "unit": "rows/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)
    return 0


# -------------------------------------------------------------- our arm

def run_ours(args, workload_name):
    import torch
    import torch.distributed as dist

    ws, rank, local = dist_env()
    if ws > 1 and not dist.is_initialized():
        dist.init_process_group("nccl")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)

    import __graft_entry__
    __graft_entry__.build()
    from speculative_decoding_verification_02_gb300 import api

    prob, desc = make_workload(workload_name)
    B, R, V = prob["target"].shape
    k = R - 1
    rows_per_step = B * (2 * k + 1)
    step_bytes = row_bytes(prob)

    def to_dev(x):
        x = np.ascontiguousarray(x)
        if x.dtype == np.uint16:
            return torch.from_numpy(x.view(np.int16)).view(torch.bfloat16).to(dev)
        return torch.from_numpy(x).to(dev)

    # rotating input sets: enough copies that one cycle is > 2x L2
    nsets = max(4, min(256, int(np.ceil(2 * L2_BYTES / step_bytes))))
    nsets = int(2 ** np.ceil(np.log2(nsets)))
    T0, D0 = to_dev(prob["target"]), to_dev(prob["draft_logits"])
    X0, U0 = to_dev(prob["draft"]), to_dev(prob["uniforms"])
    sets = []
    rng = torch.Generator(device="cpu").manual_seed(1234)
    for s in range(nsets):
        # each set: the same logits at a different address, its own uniforms
        u = torch.rand((B, k + 1), generator=rng).clamp_(max=1 - 2 ** -24).to(dev)
        sets.append(dict(T=T0.clone(), D=D0.clone(), X=X0.clone(), U=u if s else U0.clone()))
    outs = [None] * nsets
    stream = torch.cuda.Stream(device=dev)

    def call(i, out=None):
        st = sets[i % nsets]
        return api.spec_verify_sample(st["T"], st["D"], st["X"], st["U"], prob["T"], out=out, stream=stream)

    with torch.cuda.stream(stream):
        for i in range(nsets):
            outs[i] = call(i)
    launches_per_call = None
    n0 = api.launch_count()
    with torch.cuda.stream(stream):
        call(0, outs[0])
    launches_per_call = api.launch_count() - n0
    torch.cuda.synchronize(dev)

    # one graph cycles once through every input set
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.stream(stream):
        with torch.cuda.graph(graph, stream=stream):
            for i in range(nsets):
                call(i, outs[i])
    rem = args.steps % nsets
    graph_rem = None
    if rem:
        graph_rem = torch.cuda.CUDAGraph()
        with torch.cuda.stream(stream):
            with torch.cuda.graph(graph_rem, stream=stream):
                for i in range(rem):
                    call(i, outs[i])
    torch.cuda.synchronize(dev)

    sampler = ClockSampler(local)
    with sampler:
        # warm-up: W steps
        with torch.cuda.stream(stream):
            for _ in range(args.warmup // nsets):
                graph.replay()
            for i in range(args.warmup % nsets):
                call(i, outs[i])
        torch.cuda.synchronize(dev)
        barrier()
        torch.cuda.synchronize(dev)
        ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        ev0.record(stream)
        with torch.cuda.stream(stream):
            for _ in range(args.steps // nsets):
                graph.replay()
            if graph_rem is not None:
                graph_rem.replay()
        ev1.record(stream)
        torch.cuda.synchronize(dev)
        barrier()
        ms = ev0.elapsed_time(ev1)
    clocks = sampler.summary()
    ms_max = reduce_max(ms, dev)
    total_rows = reduce_sum(args.steps * rows_per_step, dev)
    value = total_rows / (ms_max / 1e3)

    # kernel timing pass: the same calls, each kernel bracketed by events
    api.trace_enable(True)
    api.trace_collect()
    with torch.cuda.stream(stream):
        for i in range(4 * nsets):
            call(i, outs[i % nsets])
    torch.cuda.synchronize(dev)
    trace = api.trace_collect()
    api.trace_enable(False)
    dom = max(trace.items(), key=lambda kv: kv[1][0])
    dom_name, (dom_ms, dom_n) = dom
    dom_avg_s = dom_ms / dom_n / 1e3
    achieved = step_bytes / dom_avg_s / 1e9 if dom_name.startswith("chain_stats") else None
    peak, peak_kind = peak_hbm()

    # end to end through the C ABI with host buffers: H2D inputs, call, D2H results
    steps_e2e = max(3, min(args.steps, 2000))
    h_sets = []
    for s in range(nsets):
        h_sets.append({k2: v.cpu().pin_memory() for k2, v in sets[s].items()})
    d_in = {k2: torch.empty_like(v) for k2, v in sets[0].items()}
    d_out = call(0)
    h_out = {k2: torch.empty(v.shape, dtype=v.dtype, pin_memory=True) for k2, v in d_out.items()
             if k2 in ("accepted", "out_tokens", "n_emit", "status")}
    h2d = sum(v.numel() * v.element_size() for v in h_sets[0].values())
    d2h = sum(v.numel() * v.element_size() for v in h_out.values())
    torch.cuda.synchronize(dev)

    def e2e_step(i):
        hs = h_sets[i % nsets]
        for k2 in d_in:
            d_in[k2].copy_(hs[k2], non_blocking=True)
        o = api.spec_verify_sample(d_in["T"], d_in["D"], d_in["X"], d_in["U"], prob["T"], out=d_out, stream=stream)
        for k2 in h_out:
            h_out[k2].copy_(o[k2], non_blocking=True)

    with torch.cuda.stream(stream):
        for i in range(min(args.warmup, 50)):
            e2e_step(i)
    torch.cuda.synchronize(dev)
    barrier()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    t_wall = time.perf_counter()
    e0.record(stream)
    with torch.cuda.stream(stream):
        for i in range(steps_e2e):
            e2e_step(i)
    e1.record(stream)
    torch.cuda.synchronize(dev)
    wall = time.perf_counter() - t_wall
    e2e_ms = max(e0.elapsed_time(e1), 1e3 * wall)
    e2e_ms = reduce_max(e2e_ms, dev)
    e2e_value = reduce_sum(steps_e2e * rows_per_step, dev) / (e2e_ms / 1e3)

    cpu = None
    if rank == 0 and not args.no_cpu_baseline:
        rate, threads, n, dt = oracle_rate(prob, target_seconds=float(os.environ.get("SPEC_CPU_SECONDS", "10")))
        cpu = {"value": rate, "unit": "rows/s", "cores": threads, "kind": "oracle",
               "sample": f"{n} requests of the workload in one oracle call ({dt:.1f} s, fp64, OpenMP)"}

    if rank == 0:
        traffic = profiled_traffic(dom_name, workload_name)
        line = {
            "metric": METRIC, "value": value, "unit": "rows/s", "n_gpus": ws, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": ms_max / args.steps, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f32", "data": "synthetic",
            "config": {"workload": desc, "rows_per_step": rows_per_step, "logits": "bf16" if
                       prob["target"].dtype == np.uint16 else "fp32",
                       "bytes_per_step": step_bytes, "parallelism": f"replicas x{ws}",
                       "l2": f"inputs rotate over {nsets} resident sets ({nsets * step_bytes / 2**20:.0f} MiB > L2)",
                       "launch": f"CUDA graph of {nsets} calls", "hbm_gbs_whole_step":
                           step_bytes * args.steps / (ms_max / 1e3) / 1e9},
            "roofline": {"bound": "hbm", "kernel": dom_name, "achieved": achieved, "peak": peak,
                         "peak_kind": peak_kind, "unit": "GB/s",
                         "frac": (achieved / peak) if achieved else None,
                         "traffic": traffic, "avg_launch_us": dom_avg_s * 1e6,
                         "algorithmic_bytes_per_launch": step_bytes,
                         "kernels": {n: {"avg_us": 1e3 * t / c, "launches": c} for n, (t, c) in trace.items()}},
            "cpu_baseline": cpu,
            "e2e": {"value": e2e_value, "unit": "rows/s", "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                    "steps": steps_e2e},
            "gpu_launches": int(launches_per_call * args.steps),
            "clocks": clocks,
        }
        print(json.dumps(line), flush=True)
    if dist.is_initialized():
        dist.destroy_process_group()
    return 0


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200_000)
    ap.add_argument("--warmup", type=int, default=2_000)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default="vocab248k", choices=["vocab248k", "batch64", "small"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    args = ap.parse_args(argv)
    if args.warmup < 3:
        args.warmup = 3
    if args.impl == "reference":
        return run_reference(args, args.workload)
    return run_ours(args, args.workload)


if __name__ == "__main__":
    sys.exit(main())
