"""Benchmark of the verify-and-accept step on GB300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                    [--workload vocab248k|batch64|topkp64|small|tree60|tree60wor|draw64|ngram|eagle2]
                    [--chain-path auto|two_pass|fused|chunked] [--no-configs]

One step is one pass of the path over one batch:
  vocab248k  spec_verify_sample, B=1, k=4, V=248,320 bf16 (the default: the
             workload the headline metric is quoted on; 9 rows per step)
  batch64    spec_verify_sample, B=64, k=8, V=128,256 bf16 (1,088 rows)
  topkp64    the batch64 rows verified with top_k=50, top_p=0.9 (drafts from
             the drafter's own top-50; spec_verify_sample_topkp)
  small      spec_verify_sample, B=4, k=4, V=2,048 fp32 (36 rows)
  tree60     spec_verify_tree, 16 trees of 60 nodes, V=128,256 bf16
             (960 node rows per step)
  tree60wor  the same trees with siblings drafted without replacement,
             spec_verify_tree_ex with SPEC_TREE_SIBLINGS_WITHOUT_REPLACEMENT
  draw64     spec_sample (drafter-side draw), B=64 rows of V=128,256 bf16
  ngram      spec_ngram_draft on 64 histories of 4,096 tokens, then
             spec_verify_greedy of the drafts, V=32,000 fp32 (320 rows)
  eagle2     spec_tree_rerank on 16 EAGLE-2-shaped candidate trees of 511
             nodes, keeping 60 (value = candidate nodes per second)
Inputs rotate over enough resident copies that one cycle reads more than
twice the 126 MB L2, so no step finds its logits in L2; the calls are
replayed from a CUDA graph.

Printed JSON line (rank 0): value = verified rows/s over all ranks; a
roofline entry for the kernel with the largest share of device time (its
algorithmic bytes per launch over its CUDA-event time, against the measured
HBM copy bandwidth); the oracle's rate on the host cores; the end-to-end
rate through the C ABI with host buffers (H2D of the inputs and D2H of the
results inside the timed region); SM clocks sampled during the run.

Multi-GPU: under torchrun every rank runs the same workload on its own GPU
(independent replicas, no collective on the data path); the timing is the
max over ranks.  --impl reference times the fp64 oracle on the host cores.
"""
from __future__ import annotations

import argparse
import contextlib
import hashlib
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "verified logit rows/sec at V=248,320; achieved HBM GB/s vs GB300 peak"
FALLBACK_HBM_GBS = 6800.0
L2_BYTES = 126 * 1024 * 1024
PROFILE_DIR = os.path.join(ROOT, "profiles")
CSRC = "speculative_decoding_verification_02_gb300/csrc"
_CHAIN = [f"{CSRC}/chain.cu", f"{CSRC}/chain_fused.cu", f"{CSRC}/chain_common.cuh", f"{CSRC}/common.cuh",
          f"{CSRC}/segments.cuh"]
KERNEL_SOURCES = {"chain": _CHAIN,
                  "filter": _CHAIN + [f"{CSRC}/filter.cu"],
                  "tree": [f"{CSRC}/tree.cu", f"{CSRC}/common.cuh", f"{CSRC}/segments.cuh"],
                  "ngram": [f"{CSRC}/ngram.cu"] + _CHAIN,
                  "draw": _CHAIN,
                  "rerank": [f"{CSRC}/rerank.cu", f"{CSRC}/common.cuh"]}


# ----------------------------------------------------------------- helpers

def to_dev(x, dev):
    import torch
    x = np.ascontiguousarray(x)
    if x.dtype == np.uint16:
        return torch.from_numpy(x.view(np.int16)).view(torch.bfloat16).to(dev)
    return torch.from_numpy(x).to(dev)


def elem_bytes(a) -> int:
    return 2 if a.dtype == np.uint16 else 4


def peak_hbm():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            return float(json.load(f)["hbm_gbs"]), "measured"
    except (OSError, KeyError, ValueError):
        return FALLBACK_HBM_GBS, "fallback"


def source_sha(kind: str) -> str:
    h = hashlib.sha256()
    for rel in KERNEL_SOURCES[kind]:
        with open(os.path.join(ROOT, rel), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def profiled_traffic(kernel: str, workload: str, kind: str):
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
    if vals.get("source_sha") != source_sha(kind):
        return None
    try:
        return float(vals["dram_bytes_per_launch"])
    except (KeyError, ValueError):
        return None


def dist_env():
    return (int(os.environ.get("WORLD_SIZE", "1")), int(os.environ.get("RANK", "0")),
            int(os.environ.get("LOCAL_RANK", "0")))


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


class ClockSampler:
    """nvidia-smi clocks and throttle reasons every 200 ms while running.

    A timed region of a few milliseconds falls between two samples, so the
    caller keeps the GPU under the same (untimed) load before and after it
    until samples have landed (keep_busy); the summary gives the samples
    inside the timed region when there are any, else those of the load
    around it, and says which."""
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap,timestamp")

    def __init__(self, gpu_index: int, path=None):
        self.gpu = gpu_index
        self.proc = None
        self.keep = path is not None
        self.path = path or os.path.join(tempfile.gettempdir(), f"spec_bench_clocks_{os.getpid()}_{gpu_index}.csv")
        self.window = None  # (start, end) of the timed region, wall clock

    def count(self) -> int:
        try:
            with open(self.path) as f:
                return sum(1 for _ in f)
        except OSError:
            return 0

    def keep_busy(self, work, new_samples: int, max_seconds: float):
        """Runs work() repeatedly until new_samples more samples are written
        (or max_seconds pass)."""
        if self.proc is None:
            return
        c0, t0 = self.count(), time.time()
        while self.count() < c0 + new_samples and time.time() - t0 < max_seconds:
            work()

    def __enter__(self):
        try:
            os.makedirs(os.path.dirname(self.path), exist_ok=True)
            self.f = open(self.path, "w")
            self.proc = subprocess.Popen(["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                                          "-lms", "200", "-i", str(self.gpu)], stdout=self.f,
                                         stderr=subprocess.DEVNULL)
        except OSError:
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

    def _samples(self):
        """(timestamp, SM MHz, max MHz, active throttle reasons) per sample,
        read once; a temporary sample file is removed after reading."""
        if getattr(self, "_rows", None) is not None:
            return self._rows
        import datetime
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        rows = []
        for line in open(self.path):
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 10:
                continue
            try:
                sm, mx = float(parts[1]), float(parts[2])
            except ValueError:
                continue
            try:
                ts = datetime.datetime.strptime(parts[9], "%Y/%m/%d %H:%M:%S.%f").timestamp()
            except ValueError:
                ts = None
            rows.append((ts, sm, mx, {n for n, v in zip(names, parts[5:9]) if v.lower() == "active"}))
        if not self.keep:
            try:
                os.remove(self.path)
            except OSError:
                pass
        self._rows = rows
        return rows

    def summary(self) -> dict:
        if self.proc is None or (not os.path.exists(self.path) and getattr(self, "_rows", None) is None):
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        rows = self._samples()
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"]}
        inside = [r for r in rows if self.window and r[0] is not None and
                  self.window[0] <= r[0] <= self.window[1]]
        use = inside or rows
        return {"sm_mhz": statistics.median(r[1] for r in use), "sm_max_mhz": max(r[2] for r in use),
                "reasons": sorted(set().union(*(r[3] for r in use))), "samples": len(use),
                "window": "timed region" if inside else "the same load just before and after the timed region"}


# --------------------------------------------------------------- workloads

class ChainWorkload:
    """spec_verify_sample on one chain problem (filtered when top_k / top_p
    are set)."""
    kind = "chain"
    top_k, top_p = 0, 1.0

    def __init__(self, name):
        from speculative_decoding_verification_02_gb300 import workloads as W
        if name == "vocab248k":
            self.prob = W.chain_vocab248k(W.SEED_BASE + 3, B=1)
            self.desc = ("chain sampling verify, B=1, k=4, V=248,320 bf16 "
                         "(t~N(0,3) with 5 ids +8, d=0.8t+N(0,1), T=1)")
        elif name == "batch64":
            self.prob = W.chain_batch64()
            self.desc = ("chain sampling verify, B=64, k=8, V=128,256 bf16 "
                         "(t~N(0,2.5), d=t+N(0,s), s in {0.3,1,2}, T=0.7)")
        elif name == "topkp64":
            self.top_k, self.top_p = 50, 0.9
            self.kind = "filter"
            self.prob = W.chain_batch64_topk(top_k=self.top_k)
            self.desc = ("top-k / top-p filtered chain sampling verify, top_k=50, top_p=0.9, B=64, k=8, "
                         "V=128,256 bf16 (the batch64 rows, T=0.7; drafts from the drafter's own top-50)")
        else:
            self.prob = W.chain_small()
            self.desc = "chain sampling verify, B=4, k=4, V=2048 fp32 (t~N(0,2), d=t+N(0,0.5), T=1)"
        p = self.prob
        self.B, R, self.V = p["target"].shape
        self.k = R - 1
        self.es = elem_bytes(p["target"])
        self.rows_per_step = self.B * (2 * self.k + 1)
        self.set_bytes = self.rows_per_step * self.V * self.es
        self.logits = "bf16" if self.es == 2 else "fp32"
        if name != "vocab248k":
            self.metric = f"verified logit rows/sec at V={self.V:,}; achieved HBM GB/s vs GB300 peak"

    def device_set(self, dev, i):
        import torch
        p = self.prob
        g = torch.Generator().manual_seed(1000 + i)
        u = torch.rand((self.B, self.k + 1), generator=g).clamp_(max=1 - 2 ** -24) if i else \
            torch.from_numpy(p["uniforms"])
        return dict(T=to_dev(p["target"], dev), D=to_dev(p["draft_logits"], dev), X=to_dev(p["draft"], dev),
                    U=u.to(dev))

    def call(self, s, out, stream):
        from speculative_decoding_verification_02_gb300 import api
        return api.spec_verify_sample(s["T"], s["D"], s["X"], s["U"], self.prob["T"], top_k=self.top_k,
                                      top_p=self.top_p, out=out, stream=stream)

    result_keys = ("accepted", "out_tokens", "n_emit", "status")

    def kernel_bytes(self, name, outs):
        """Algorithmic bytes of one launch of kernel `name`, averaged over the
        rotating sets (the draw's bytes depend on where each call stopped)."""
        row = self.V * self.es
        if name.startswith(("chain_stats", "chain_fused", "chain_filter")):
            return self.set_bytes  # every row once (the fused kernel's draw re-reads two from L2)
        if name.startswith("chain_sample_accept"):
            tot = 0.0
            for o in outs:
                acc = o["accepted"].cpu().numpy()
                # a rejection reads the target and draft rows of the rejected
                # position, a full accept the bonus row
                tot += sum(2 * row if a < self.k else row for a in acc)
            return tot / len(outs)
        return None

    def step_bytes(self, outs):
        """Algorithmic bytes of one step: every verified row read once."""
        return self.set_bytes

    def oracle_call(self, n, threads):
        """At least n requests through the oracle: a single-request workload is
        broadcast to n requests (no copy), a batch is verified whole, repeatedly."""
        import oracle
        p = self.prob
        if self.B == 1:
            tgt = np.broadcast_to(p["target"][:1], (n,) + p["target"].shape[1:])
            dl = np.broadcast_to(p["draft_logits"][:1], (n,) + p["draft_logits"].shape[1:])
            idx = np.zeros(n, dtype=np.int64)
            oracle.verify_sample(tgt, dl, p["draft"][idx], p["uniforms"][idx], p["T"], top_k=self.top_k,
                                 top_p=self.top_p, threads=threads)
            return n * (2 * self.k + 1)
        reps = max(1, -(-n // self.B))
        for _ in range(reps):
            oracle.verify_sample(p["target"], p["draft_logits"], p["draft"], p["uniforms"], p["T"], top_k=self.top_k,
                                 top_p=self.top_p, threads=threads)
        return reps * self.B * (2 * self.k + 1)


class DrawWorkload:
    """spec_sample: the drafter-side draw x ~ softmax(d/T) with its
    probability, on the first draft row of each batch64 request."""
    kind = "draw"
    unit = "rows/s"

    def __init__(self, name):
        from speculative_decoding_verification_02_gb300 import workloads as W
        p = W.chain_batch64()
        self.rows = np.ascontiguousarray(p["draft_logits"][:, 0])
        self.T = p["T"]
        self.B, self.V = self.rows.shape
        self.u = np.random.default_rng(W.SEED_BASE + 7).random(self.B, dtype=np.float32)
        self.desc = ("drafter-side draw x ~ softmax(d/T) with q(x), B=64 rows of V=128,256 bf16 "
                     "(batch64's first draft rows: d=t+N(0,s), t~N(0,2.5)), T=0.7")
        self.metric = f"drawn logit rows/sec at V={self.V:,}; achieved HBM GB/s vs GB300 peak"
        self.es = 2
        self.rows_per_step = self.B
        self.set_bytes = self.B * self.V * self.es
        self.logits = "bf16"

    def device_set(self, dev, i):
        import torch
        g = torch.Generator().manual_seed(2000 + i)
        u = torch.rand(self.B, generator=g).clamp_(max=1 - 2 ** -24) if i else torch.from_numpy(self.u)
        return dict(L=to_dev(self.rows, dev), U=u.to(dev))

    def call(self, s, out, stream):
        from speculative_decoding_verification_02_gb300 import api
        return api.spec_sample(s["L"], s["U"], self.T, out=out, stream=stream)

    result_keys = ("tokens", "probs", "status")

    def kernel_bytes(self, name, outs):
        """The statistics pass reads every row once; the draw re-reads (at
        most) the row it draws from."""
        if name.startswith(("chain_stats", "chain_fused")):
            return self.set_bytes
        if name.startswith("chain_sample_accept"):
            return self.B * self.V * self.es
        return None

    def step_bytes(self, outs):
        return self.set_bytes

    def oracle_call(self, n, threads):
        """At least n draws through the oracle (verification with no draft)."""
        import oracle
        reps = max(1, -(-n // self.B))
        empty = np.zeros((self.B, 0, self.V), self.rows.dtype)
        for _ in range(reps):
            oracle.verify_sample(self.rows[:, None], empty, np.zeros((self.B, 0), np.int32), self.u[:, None], self.T,
                                 threads=threads)
        return reps * self.B


class TreeWorkload:
    """spec_verify_tree on 16 draft trees of 60 nodes."""
    kind = "tree"

    def __init__(self, name):
        from speculative_decoding_verification_02_gb300 import api
        from speculative_decoding_verification_02_gb300 import workloads as W
        self.wor = name == "tree60wor"
        self.flags = api.TREE_SIBLINGS_WITHOUT_REPLACEMENT if self.wor else 0
        self.prob = (W.tree_problem(W.SEED_BASE + 5, 16, 60, 6, 10, 128256, "bf16", 1.0, siblings="without_replacement")
                     if self.wor else W.tree60())
        self.desc = ("EAGLE-style tree verify, B=16, 60-node trees of depth 6 with <=10 children, "
                     "V=128,256 bf16 (t~N(0,3) with 5 ids +8, d=0.8t+N(0,1)), T=1" +
                     (", siblings drawn from q without replacement and verified with the matching rule"
                      if self.wor else ""))
        p = self.prob
        self.B, self.N, self.V = p["target"].shape
        self.es = 2
        self.metric = f"verified tree-node logit rows/sec at V={self.V:,}; achieved HBM GB/s vs GB300 peak"
        self.rows_per_step = self.B * self.N
        self.set_bytes = 2 * self.B * self.N * self.V * self.es
        self.logits = "bf16"
        self.kids = [set(int(x) for x in p["parents"][b] if x >= 0) for b in range(self.B)]

    def device_set(self, dev, i):
        p = self.prob
        return dict(T=to_dev(p["target"], dev), D=to_dev(p["draft_logits"], dev), P=to_dev(p["parents"], dev),
                    X=to_dev(p["node_tok"], dev), U=to_dev(p["uniforms"], dev))

    def call(self, s, out, stream):
        from speculative_decoding_verification_02_gb300 import api
        return api.spec_verify_tree(s["T"], s["D"], s["P"], s["X"], s["U"], self.prob["T"], self.prob["depth"],
                                    flags=self.flags, out=out, stream=stream)

    result_keys = ("accepted_len", "path_nodes", "out_tokens", "n_emit", "status")

    def kernel_bytes(self, name, outs):
        """Rows the walk must read: each visited node's target row, and its
        draft row when it has children (sibling passes re-read cached data)."""
        row = self.V * self.es
        tot = 0.0
        for o in outs:
            path = o["path_nodes"].cpu().numpy()
            for b in range(self.B):
                for u in path[b]:
                    if u >= 0:
                        tot += row * (2 if int(u) in self.kids[b] else 1)
        return tot / len(outs)

    def step_bytes(self, outs):
        """The rows on the walked paths (read-everything would be set_bytes)."""
        return self.kernel_bytes("tree_walk", outs)

    def oracle_call(self, n, threads):
        """At least n requests: the batch of trees is verified whole, repeatedly."""
        import oracle
        p = self.prob
        reps = max(1, -(-n // self.B))
        for _ in range(reps):
            oracle.verify_tree(p["target"], p["draft_logits"], p["parents"], p["node_tok"], p["uniforms"], p["T"],
                               p["depth"], threads=threads,
                               variant=oracle.TREE_VARIANT_WITHOUT_REPLACEMENT if self.wor else 0)
        return reps * self.B * self.N


class EagleWorkload:
    """spec_tree_rerank on 16 EAGLE-2-shaped candidate trees of 511 nodes."""
    kind = "rerank"
    oracle_threads = 1  # the oracle's rerank runs on one thread
    metric = "EAGLE-2 candidate-tree nodes post-processed per second (value, top-60 rerank, flatten, mask)"
    unit = "nodes/s"

    def __init__(self, name):
        from speculative_decoding_verification_02_gb300 import workloads as W
        self.prob = W.eagle2_candidates()
        self.m = 60
        p = self.prob
        self.B, self.N = p["parents"].shape
        self.desc = (f"EAGLE-2 tree post-processing, B={self.B} candidate trees of {self.N} nodes (depth 6, "
                     f"10 nodes expanded per layer, 10 children each), keep m={self.m}, uint8 mask")
        self.rows_per_step = self.B * self.N
        self.set_bytes = self.B * self.N * 12
        self.logits = "none"

    def device_set(self, dev, i):
        p = self.prob
        return dict(P=to_dev(p["parents"], dev), C=to_dev(p["conf"], dev), X=to_dev(p["node_tok"], dev))

    def call(self, s, out, stream):
        from speculative_decoding_verification_02_gb300 import api
        return api.spec_tree_rerank(s["P"], s["C"], self.m, node_tok=s["X"], out=out, stream=stream)

    result_keys = ("sel_nodes", "sel_parents", "sel_depth", "sel_tok", "n_sel", "status")

    def kernel_bytes(self, name, outs):
        """Inputs (parents, confidences, tokens) and outputs (five int32/fp32
        values per kept node, the m x m mask)."""
        return self.B * (self.N * 12 + self.m * 20 + self.m * self.m)

    def step_bytes(self, outs):
        return self.kernel_bytes("tree_rerank", outs)

    def oracle_call(self, n, threads):
        import oracle
        p = self.prob
        reps = max(1, -(-n // self.B))
        for _ in range(reps):
            oracle.tree_rerank(p["parents"], p["conf"], self.m, node_tok=p["node_tok"])
        return reps * self.rows_per_step


class NgramWorkload:
    """spec_ngram_draft, then spec_verify_greedy of its drafts."""
    kind = "ngram"

    def __init__(self, name):
        from speculative_decoding_verification_02_gb300 import workloads as W
        self.prob = W.ngram_problem(W.SEED_BASE + 2, boost=10.0)
        self.desc = ("n-gram history-lookup draft + greedy verify, B=64, int32 history 4096 over V=32,000 "
                     "with planted repeated spans 8-32, window 3, k=4; target N(0,1) fp32")
        p = self.prob
        self.B, self.H = p["history"].shape
        self.k, self.V, self.w = p["k"], p["V"], p["window"]
        self.es = 4
        self.rows_per_step = self.B * (self.k + 1)
        self.metric = f"drafted and greedily verified logit rows/sec at V={self.V:,}; achieved HBM GB/s vs GB300 peak"
        self.set_bytes = self.rows_per_step * self.V * 4 + self.B * self.H * 4
        self.logits = "fp32"

    def device_set(self, dev, i):
        p = self.prob
        return dict(H=to_dev(p["history"], dev), L=to_dev(p["hist_len"], dev), T=to_dev(p["target"], dev))

    def call(self, s, out, stream):
        from speculative_decoding_verification_02_gb300 import api
        o1 = out[0] if out else None
        o2 = out[1] if out else None
        d = api.spec_ngram_draft(s["H"], s["L"], self.w, self.k, out=o1, stream=stream)
        g = api.spec_verify_greedy(s["T"], d["draft"], d["draft_len"], out=o2, stream=stream)
        return (d, g)

    result_keys = None

    def kernel_bytes(self, name, outs):
        if name == "ngram_draft":
            return self.B * self.H * 4
        if name.startswith(("chain_stats", "chain_fused")):
            tot = 0.0
            for d, _ in outs:
                lens = d["draft_len"].cpu().numpy()
                tot += float(np.sum(lens + 1)) * self.V * self.es
            return tot / len(outs)
        return None

    def step_bytes(self, outs):
        """The histories and the verified rows (draft_len + 1 per request)."""
        return self.B * self.H * 4 + self.kernel_bytes("chain_stats_greedy", outs)

    def oracle_call(self, n, threads):
        import oracle
        p = self.prob
        reps = max(1, n // self.B)
        for _ in range(reps):
            d, dl, _ = oracle.ngram_draft(p["history"], p["hist_len"], self.w, self.k)
            oracle.verify_greedy(p["target"], d, dl)
        return reps * self.rows_per_step


# the pages' other configs whose workloads every run also measures (the
# headline --workload is vocab248k: config 3)
CONFIG_WORKLOADS = ("batch64", "ngram", "tree60", "topkp64")

WORKLOADS = {"vocab248k": ChainWorkload, "batch64": ChainWorkload, "small": ChainWorkload, "topkp64": ChainWorkload,
             "tree60": TreeWorkload, "tree60wor": TreeWorkload, "draw64": DrawWorkload, "ngram": NgramWorkload, "eagle2": EagleWorkload}


def oracle_rate(wl, target_seconds: float):
    """Rows/s of the fp64 oracle on this host's cores over a bounded sample of
    the workload: whole requests, in rounds whose size grows until the timed
    rounds together last about target_seconds."""
    import oracle
    threads = getattr(wl, "oracle_threads", None) or oracle.max_threads()
    wl.oracle_call(1, threads)            # untimed: thread pool and caches warm
    n, rows, dt = max(1, threads), 0, 0.0
    while dt < target_seconds:
        t0 = time.perf_counter()
        rows += wl.oracle_call(n, threads)
        last = time.perf_counter() - t0
        dt += last
        # next round: the rest of the time budget at the rate seen so far, at most 4x
        n = max(1, min(4 * n, int(n * max(target_seconds - dt, 0.0) / max(last, 1e-6)) + 1))
    return rows / dt, threads, rows, dt


# ------------------------------------------------------------ reference arm

def run_reference(args):
    ws, rank, _ = dist_env()
    if rank != 0:
        return 0
    import oracle
    wl = WORKLOADS[args.workload](args.workload)
    threads = getattr(wl, "oracle_threads", None) or min(oracle.max_threads(), wl.B)  # over requests
    budget = float(os.environ.get("SPEC_REF_SECONDS", "60"))
    t_start = time.perf_counter()
    for _ in range(args.warmup):
        wl.oracle_call(wl.B, threads)
        if time.perf_counter() - t_start > budget / 4:
            break
    steps_done = rows = 0
    t0 = time.perf_counter()
    for _ in range(args.steps):
        rows += wl.oracle_call(wl.B, threads)
        steps_done += 1
        if time.perf_counter() - t0 > budget:
            break
    dt = time.perf_counter() - t0
    value = rows / dt
    unit = getattr(wl, "unit", "rows/s")
    line = {"impl": "reference", "metric": getattr(wl, "metric", METRIC), "value": value, "unit": unit,
            "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * dt / steps_done,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic", "config": {"workload": wl.desc, "rows_per_step": wl.rows_per_step},
            "cpu_baseline": {"kind": "oracle", "value": value, "unit": unit, "cores": threads,
                             "sample": f"{steps_done} of {args.steps} steps timed (cap {budget:.0f} s), "
                                       f"one batch of the workload each"},
            "e2e": {"value": value, "unit": unit, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)
    return 0


# -------------------------------------------------------------- our arm

def _external_event():
    """A timing event that, recorded during stream capture, becomes an
    event-record node of the graph (None when this torch lacks the option)."""
    import torch
    try:
        return torch.cuda.Event(enable_timing=True, external=True)
    except TypeError:
        return None


def timed_graphs(wl, sets, outs, stream, steps):
    """Exactly `steps` calls cycling over the input sets, as CUDA graphs to
    replay in order: [(graph, replays), ...], and the two timing events.  The
    first graph's first node and the last graph's last node record the events,
    so the measured span starts with the first kernel, not with a graph
    launch; each graph is replayed once here, untimed, so that no replay in
    the timed region is a graph's first."""
    import torch
    nsets = len(sets)
    ev0, ev1 = _external_event(), _external_event()
    in_graph = ev0 is not None and ev1 is not None

    def capture(n, head=False, tail=False):
        g = torch.cuda.CUDAGraph()
        with torch.cuda.stream(stream):
            with torch.cuda.graph(g, stream=stream):
                if head and in_graph:
                    ev0.record(stream)
                for i in range(n):
                    wl.call(sets[i], outs[i], stream)
                if tail and in_graph:
                    ev1.record(stream)
        return g

    full, rem = divmod(steps, nsets)
    if full == 0:
        plan = [(capture(rem, True, True), 1)]
    elif rem:
        plan = [(capture(nsets, head=True), 1)]
        if full > 1:
            plan.append((capture(nsets), full - 1))
        plan.append((capture(rem, tail=True), 1))
    elif full == 1:
        plan = [(capture(nsets, True, True), 1)]
    else:
        plan = [(capture(nsets, head=True), 1)]
        if full > 2:
            plan.append((capture(nsets), full - 2))
        plan.append((capture(nsets, tail=True), 1))
    if not in_graph:
        ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(stream):
        for g, _ in plan:
            g.replay()
    return plan, ev0, ev1, in_graph


def kernel_times(wl, sets, outs, stream, reps=8):
    """{kernel: (microseconds per launch, launches per step)}: the calls of one
    input cycle captured into a graph with every kernel launched `reps` times
    back to back between a pair of CUDA events on its launching stream
    (spec_trace_repeat), timed on the graph's last replay; the bracket over
    reps is the kernel's duration without one launch's set-up."""
    import torch
    from speculative_decoding_verification_02_gb300 import api
    dev = stream.device
    api.trace_enable(True)
    api.trace_repeat(reps)
    api.trace_collect()
    g = torch.cuda.CUDAGraph()
    try:
        with torch.cuda.stream(stream):
            with torch.cuda.graph(g, stream=stream):
                for i in range(len(sets)):
                    wl.call(sets[i], outs[i], stream)
    finally:
        api.trace_enable(False)
        api.trace_repeat(1)
    torch.cuda.synchronize(dev)
    with torch.cuda.stream(stream):
        for _ in range(3):
            g.replay()
    torch.cuda.synchronize(dev)
    trace = api.trace_collect()
    del g
    return {k: (1e3 * t_ms / cnt / reps, cnt / len(sets)) for k, (t_ms, cnt) in trace.items()}


def measure(name, args, dev, stream, want_clocks=True):
    """Times one workload: exactly args.steps calls after args.warmup, inputs
    rotating over resident sets that put more than twice the L2 between
    reuses.  Returns (workload, result dict, sets, outs)."""
    import torch
    from speculative_decoding_verification_02_gb300 import api
    wl = WORKLOADS[name](name)
    nsets = max(2, int(np.ceil(2 * L2_BYTES / wl.set_bytes)))
    nsets = min(256, int(2 ** np.ceil(np.log2(nsets))))
    if wl.kind == "tree":
        nsets = 6   # a walk reads ~1/8 of a set; six sets put ~2.4x L2 between reuses
    sets = [wl.device_set(dev, i) for i in range(nsets)]
    with torch.cuda.stream(stream):
        outs = [wl.call(sets[i], None, stream) for i in range(nsets)]
    n0 = api.launch_count()
    with torch.cuda.stream(stream):
        wl.call(sets[0], outs[0], stream)
    launches_per_call = api.launch_count() - n0
    torch.cuda.synchronize(dev)
    plan, ev0, ev1, in_graph = timed_graphs(wl, sets, outs, stream, args.steps)
    load_graph = torch.cuda.CUDAGraph()  # untimed load around the timed region (no timing nodes)
    with torch.cuda.stream(stream):
        with torch.cuda.graph(load_graph, stream=stream):
            for i in range(nsets):
                wl.call(sets[i], outs[i], stream)
    torch.cuda.synchronize(dev)

    sampler = ClockSampler(dev.index, args.clock_log) if want_clocks else None
    with (sampler or contextlib.nullcontext()):
        with torch.cuda.stream(stream):
            for _ in range(args.warmup // nsets):
                load_graph.replay()
            for i in range(args.warmup % nsets):
                wl.call(sets[i], outs[i], stream)
        torch.cuda.synchronize(dev)

        def load():
            with torch.cuda.stream(stream):
                for _ in range(8):
                    load_graph.replay()
            torch.cuda.synchronize(dev)

        if sampler:
            sampler.keep_busy(load, 2, 3.0)
        barrier()
        torch.cuda.synchronize(dev)
        t_start = time.time()
        if not in_graph:
            ev0.record(stream)
        with torch.cuda.stream(stream):
            for g, n in plan:
                for _ in range(n):
                    g.replay()
        if not in_graph:
            ev1.record(stream)
        torch.cuda.synchronize(dev)
        t_end = time.time()
        barrier()
        ms = ev0.elapsed_time(ev1)
        if sampler:
            sampler.window = (t_start, t_end)
            sampler.keep_busy(load, 1, 1.5)
    del plan, load_graph
    ms_max = reduce_max(ms, dev)
    ws, _, _ = dist_env()
    value = reduce_sum(args.steps * wl.rows_per_step, dev) / (ms_max / 1e3)
    ms_step = ms_max / args.steps

    peak, peak_kind = peak_hbm()
    kt = kernel_times(wl, sets, outs, stream)
    kernels = {}
    busy = sum(us * per for us, per in kt.values())
    for kname, (us, per) in kt.items():
        nbytes = wl.kernel_bytes(kname, outs)
        kernels[kname] = {"avg_us": us, "launches_per_step": per, "share": us * per / busy,
                          "algorithmic_bytes_per_launch": nbytes,
                          "achieved_gbs": (nbytes / (us * 1e-6) / 1e9) if nbytes else None}
    dom = max(kernels, key=lambda n: kernels[n]["avg_us"] * kernels[n]["launches_per_step"])
    achieved = kernels[dom]["achieved_gbs"]
    step_bytes = wl.step_bytes(outs)
    res = {
        "metric": getattr(wl, "metric", METRIC), "value": value, "unit": getattr(wl, "unit", "rows/s"),
        "steps": args.steps, "ms_per_step": ms_step,
        "config": {"workload": wl.desc, "rows_per_step": wl.rows_per_step, "logits": wl.logits,
                   "parallelism": f"replicas x{ws}",
                   "l2": (f"inputs rotate over {min(nsets, args.steps)} of {nsets} resident sets "
                          f"({nsets * wl.set_bytes / 2**20:.0f} MiB), more than twice the L2 between reuses"
                          if nsets * wl.set_bytes > 2 * L2_BYTES else
                          f"inputs L2-resident ({nsets} sets, {nsets * wl.set_bytes / 2**20:.1f} MiB): a "
                          f"latency-bound workload with little data"),
                   "launch": f"CUDA graphs of {nsets} calls; timing events are graph nodes" if in_graph else
                             f"CUDA graphs of {nsets} calls", "chain_path": args.chain_path},
        "roofline": {"bound": "hbm", "kernel": dom, "achieved": achieved, "peak": peak, "peak_kind": peak_kind,
                     "unit": "GB/s", "frac": (achieved / peak) if achieved else None,
                     "traffic": profiled_traffic(dom, name, wl.kind),
                     "avg_launch_us": kernels[dom]["avg_us"],
                     "algorithmic_bytes_per_launch": kernels[dom]["algorithmic_bytes_per_launch"],
                     "step_bytes": step_bytes,
                     "step_frac": step_bytes / (ms_step * 1e-3) / 1e9 / peak if step_bytes else None,
                     "kernel_timing": "each kernel launched 8 times back to back between CUDA events "
                                      "in a graph replay; avg_us = bracket / 8",
                     "kernels": kernels},
        "gpu_launches": int(launches_per_call * args.steps),
    }
    if sampler:
        res["clocks"] = sampler.summary()
    return wl, res, sets, outs


def run_ours(args):
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
    api.set_chain_path({"auto": api.CHAIN_AUTO, "two_pass": api.CHAIN_TWO_PASS, "fused": api.CHAIN_FUSED,
                        "chunked": api.CHAIN_CHUNKED}[args.chain_path])
    stream = torch.cuda.Stream(device=dev)
    wl, res, sets, outs = measure(args.workload, args, dev, stream)

    # end to end through the C ABI with host buffers: H2D inputs, call, D2H
    # results.  Double-buffered like a serving loop: while step i's call and
    # its D2H copies run on the compute stream, step i+1's inputs are copied
    # from pinned host memory into the other device buffer on a copy stream.
    # One CUDA graph holds a cycle of W steps (W a multiple of the host sets
    # and of the two buffers) with exactly these dependencies: a buffer's
    # copy waits for the call that last read it, a call waits for its copy.
    # Every step's copies are inside the timed region.
    n_host = max(1, min(4, len(sets), int(1e9 // max(wl.set_bytes, 1))))
    W = n_host if n_host % 2 == 0 else 2 * n_host
    steps_e2e = max(W, min(args.steps, int(2e9 // max(wl.set_bytes, 1)), 2000) // W * W)
    h_sets = [{k2: v.cpu().pin_memory() for k2, v in sets[i].items()} for i in range(n_host)]
    d_ins = [{k2: torch.empty_like(v) for k2, v in sets[0].items()} for _ in range(2)]
    del sets, outs
    d_outs = []
    with torch.cuda.stream(stream):
        for bf in range(2):
            o = wl.call(d_ins[bf], None, stream)
            d_outs.append(o)
    keys = wl.result_keys
    h_outs = []
    for bf in range(2):
        h_outs.append([{k2: torch.empty(v.shape, dtype=v.dtype, pin_memory=True) for k2, v in oo.items()
                        if keys is None or k2 in keys}
                       for oo in (d_outs[bf] if isinstance(d_outs[bf], tuple) else (d_outs[bf],))])
    h2d = sum(v.numel() * v.element_size() for v in h_sets[0].values())
    d2h = sum(v.numel() * v.element_size() for ho in h_outs[0] for v in ho.values())
    copy_stream = torch.cuda.Stream(device=dev)
    torch.cuda.synchronize(dev)

    def copy_in(j, bf):
        for k2 in d_ins[bf]:
            d_ins[bf][k2].copy_(h_sets[j][k2], non_blocking=True)

    def call_out(bf):
        o = wl.call(d_ins[bf], d_outs[bf], stream)
        for ho, oo in zip(h_outs[bf], o if isinstance(o, tuple) else (o,)):
            for k2 in ho:
                ho[k2].copy_(oo[k2], non_blocking=True)

    def cycle():  # W pipelined steps; called inside a capture on `stream`
        copied = [torch.cuda.Event() for _ in range(W)]
        done = [torch.cuda.Event() for _ in range(W)]
        copy_stream.wait_stream(stream)  # fork from the capture
        for i in range(W):
            bf = i % 2
            with torch.cuda.stream(copy_stream):
                if i >= 2:
                    copy_stream.wait_event(done[i - 2])  # the call that last read this buffer
                copy_in(i % n_host, bf)
                copied[i].record(copy_stream)
            stream.wait_event(copied[i])
            with torch.cuda.stream(stream):
                call_out(bf)
                done[i].record(stream)
        stream.wait_stream(copy_stream)  # join

    with torch.cuda.stream(stream):  # warm-up outside any graph
        for i in range(2):
            copy_in(i % n_host, i % 2)
            call_out(i % 2)
    torch.cuda.synchronize(dev)
    g_e2e = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g_e2e, stream=stream):
        cycle()
    with torch.cuda.stream(stream):
        g_e2e.replay()  # once untimed
    torch.cuda.synchronize(dev)
    barrier()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    t_wall = time.perf_counter()
    e0.record(stream)
    with torch.cuda.stream(stream):
        for _ in range(steps_e2e // W):
            g_e2e.replay()
    e1.record(stream)
    torch.cuda.synchronize(dev)
    wall = time.perf_counter() - t_wall
    e2e_ms = reduce_max(max(e0.elapsed_time(e1), 1e3 * wall), dev)
    e2e_value = reduce_sum(steps_e2e * wl.rows_per_step, dev) / (e2e_ms / 1e3)
    len_h = n_host
    del g_e2e, h_sets, d_ins, d_outs, h_outs

    # the other workloads of the pages' configs, measured in the same run
    configs = {}
    if not args.no_configs:
        cargs = argparse.Namespace(**vars(args))
        cargs.steps = max(1, min(args.steps, args.config_steps))
        cargs.warmup = max(3, min(args.warmup, 200))
        for name in CONFIG_WORKLOADS:
            if name == args.workload:
                continue
            _, r, s_, o_ = measure(name, cargs, dev, stream, want_clocks=False)
            del s_, o_
            torch.cuda.empty_cache()
            configs[name] = r

    cpu = None
    if rank == 0 and not args.no_cpu_baseline:
        rate, threads, nrows, dt = oracle_rate(wl, float(os.environ.get("SPEC_CPU_SECONDS", "10")))
        cpu = {"value": rate, "unit": getattr(wl, "unit", "rows/s"), "cores": threads, "kind": "oracle",
               "sample": f"{nrows} {getattr(wl, 'unit', 'rows/s').split('/')[0]} of the workload's requests "
                         f"through the oracle ({dt:.1f} s, fp64"
                         f"{', OpenMP over requests' if threads > 1 else ', one thread'})"}

    if rank == 0:
        line = {"metric": res["metric"], "value": res["value"], "unit": res["unit"], "n_gpus": ws,
                "steps": args.steps, "warmup": args.warmup, "ms_per_step": res["ms_per_step"],
                "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f32",
                "data": "synthetic", "config": res["config"], "roofline": res["roofline"],
                "cpu_baseline": cpu,
                "e2e": {"value": e2e_value, "unit": res["unit"], "h2d_bytes_per_step": h2d,
                        "d2h_bytes_per_step": d2h, "steps": steps_e2e,
                        "launch": f"double-buffered: step i+1's H2D copies (copy stream, {len_h} pinned host "
                                  "sets in turn) overlap step i's C-ABI call and D2H copies; one CUDA graph "
                                  f"per cycle of {W} steps"},
                "gpu_launches": res["gpu_launches"], "clocks": res["clocks"]}
        if configs:
            line["configs"] = configs
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
    ap.add_argument("--workload", default="vocab248k", choices=sorted(WORKLOADS))
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-configs", action="store_true",
                    help="time only --workload (not the other configs' workloads as well)")
    ap.add_argument("--config-steps", type=int, default=20_000,
                    help="steps of each other config's workload (at most --steps)")
    ap.add_argument("--clock-log", default=None,
                    help="keep the nvidia-smi clock samples in this CSV file (default: a temporary file)")
    ap.add_argument("--chain-path", choices=["auto", "two_pass", "fused", "chunked"], default="auto",
                    help="chain verification path (same results; for profiling one path)")
    args = ap.parse_args(argv)
    args.warmup = max(args.warmup, 3)
    if args.impl == "reference":
        return run_reference(args)
    return run_ours(args)


if __name__ == "__main__":
    sys.exit(main())
