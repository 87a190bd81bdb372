"""bench.py host logic without a GPU: the reference arm's JSON line, and the
max-over-ranks / sum-over-ranks reductions of the multi-GPU path on two
gloo ranks."""
import json
import os
import socket

import numpy as np
import pytest
import torch.distributed as dist
import torch.multiprocessing as mp

import bench


def test_reference_arm_json_line(capsys, monkeypatch):
    monkeypatch.setenv("SPEC_REF_SECONDS", "5")
    assert bench.main(["--impl", "reference", "--workload", "small", "--steps", "3", "--warmup", "1"]) == 0
    line = json.loads(capsys.readouterr().out.strip().splitlines()[-1])
    for key in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step", "higher_is_better",
                "scaling", "vs_baseline", "dtype", "data", "config", "cpu_baseline", "e2e"):
        assert key in line, key
    assert line["impl"] == "reference" and line["value"] > 0 and line["unit"] == "rows/s"
    assert line["e2e"]["value"] == line["value"] and line["e2e"]["h2d_bytes_per_step"] == 0
    assert line["cpu_baseline"]["kind"] == "oracle" and line["cpu_baseline"]["cores"] >= 1


def test_reference_arm_other_ranks_exit_quietly(capsys, monkeypatch):
    monkeypatch.setenv("RANK", "1")
    monkeypatch.setenv("WORLD_SIZE", "2")
    assert bench.main(["--impl", "reference", "--workload", "small", "--steps", "2"]) == 0
    assert capsys.readouterr().out.strip() == ""


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE="2",
                      LOCAL_RANK=str(rank))
    dist.init_process_group("gloo", rank=rank, world_size=2)
    ws, r, local = bench.dist_env()
    mx = bench.reduce_max(10.0 * (rank + 1), "cpu")
    sm = bench.reduce_sum(9.0, "cpu")
    bench.barrier()
    q.put((r, ws, mx, sm))
    dist.destroy_process_group()


def test_two_rank_reductions_gloo():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = sorted(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    # timing is the max over ranks, rows add up: value = sum(rows) / max(time)
    assert res == [(0, 2, 20.0, 18.0), (1, 2, 20.0, 18.0)]


def test_clock_summary_prefers_samples_inside_the_timed_region(tmp_path):
    import datetime
    s = bench.ClockSampler(0)
    s.path = str(tmp_path / "clocks.csv")
    s.proc = object()                       # as if nvidia-smi had been started
    t0 = datetime.datetime(2026, 1, 2, 3, 4, 5)
    rows = [(0.0, 1500, "Not Active"), (0.2, 2070, "Not Active"), (0.4, 2055, "Active"), (0.6, 1200, "Not Active")]
    with open(s.path, "w") as f:
        for dt, mhz, cap in rows:
            ts = (t0 + datetime.timedelta(seconds=dt)).strftime("%Y/%m/%d %H:%M:%S.%f")[:-3]
            f.write(f"0, {mhz}, 2070, 900.1, 0x4, Not Active, Not Active, Not Active, {cap}, {ts}\n")
    base = t0.timestamp()
    s.window = (base + 0.1, base + 0.5)
    c = s.summary()
    assert c["window"] == "timed region" and c["samples"] == 2
    assert c["sm_mhz"] == 2062.5 and c["sm_max_mhz"] == 2070 and c["reasons"] == ["sw_power_cap"]
    s.window = (base + 5.0, base + 5.1)     # a region between samples: the load around it
    c = s.summary()
    assert c["samples"] == 4 and c["window"].startswith("the same load")


def test_topkp64_workload_recipe():
    """The filtered-verification bench workload: the batch64 rows with
    top_k = 50, top_p = 0.9, every draft among its draft row's 50 largest
    logits, and the filter kernel's algorithmic bytes = every row once."""
    wl = bench.WORKLOADS["topkp64"]("topkp64")
    p = wl.prob
    assert (wl.top_k, wl.top_p, wl.kind) == (50, 0.9, "filter")
    assert (wl.B, wl.k, wl.V) == (64, 8, 128_256) and wl.rows_per_step == 64 * 17
    from speculative_decoding_verification_02_gb300 import workloads as W
    for b in range(0, 64, 7):
        for i in range(wl.k):
            row = W.logits_as_f64(p["draft_logits"][b, i])
            assert row[p["draft"][b, i]] >= np.sort(row)[-50]
    assert wl.kernel_bytes("chain_filter_rows", None) == wl.set_bytes == 64 * 17 * 128_256 * 2
    assert "filter.cu" in " ".join(bench.KERNEL_SOURCES["filter"])
