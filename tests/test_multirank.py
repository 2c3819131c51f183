"""The benchmark's replica scaling logic with two gloo ranks on CPU: the
path has no exchange step, so ranks only agree on the slowest rank's time
and the job's value counts every rank's decoded bytes."""
import os
import socket

import pytest

torch = pytest.importorskip("torch")
import torch.distributed as dist  # noqa: E402
import torch.multiprocessing as mp  # noqa: E402


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _worker(rank, world, port, times, result):
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    ms = bench.max_over_ranks(times[rank], torch.device("cpu"), world)
    result[rank] = ms
    dist.destroy_process_group()


def test_max_over_ranks_and_whole_job_value():
    world = 2
    times = [12.5, 20.0]
    mgr = mp.get_context("spawn").Manager()
    result = mgr.dict()
    mp.start_processes(_worker, args=(world, _free_port(), times, result), nprocs=world, join=True,
                       start_method="spawn")
    assert result[0] == result[1] == 20.0
    import bench
    # two ranks, 256 MiB each, 10 steps in 20 ms
    assert bench.whole_job_gbs(1 << 28, 2, 10, 20.0) == pytest.approx(2 * 10 * (1 << 28) / 0.020 / 1e9)
    assert bench.max_over_ranks(3.0, torch.device("cpu"), 1) == 3.0


def test_cpu_baseline_parallel_fields():
    """The all-core oracle baseline reports the threads it ran and the
    values it decoded (a 4-stripe layer cut to a few chunks per stripe)."""
    import bench
    import oracle
    import workloads
    blob = oracle.encode_layer([workloads.normal_tensor((3, 4096 * 64 + 5), 0.02, seed=5)])
    r = bench.cpu_baseline_parallel(blob, budget_s=5.0, threads=3)
    assert r["cores"] == 3 and r["kind"] == "oracle" and r["value"] > 0
    assert r["sample"].startswith("193 chunks of 4096 values")


def test_cpu_article_style_fields():
    """The article-style decoder's timing: one core over whole stripes,
    then the whole layer with one thread per stripe, decoded and input
    rates both positive, and the sample naming what ran."""
    import numpy as np
    import bench
    import oracle
    import workloads
    blob = oracle.encode_layer([np.tile(workloads.tiny(), 17)[: (1 << 25) + 5003]])    # two stripes
    r = bench.cpu_article_style(blob, budget_s=0.0)
    assert r["one_core"] > 0 and r["all_cores"] > 0
    assert r["input_gbs"]["one_core"] > 0 and r["input_gbs"]["all_cores"] > 0
    assert r["cores"] == min(2, os.cpu_count() or 1)
    assert "not the oracle" in r["kind"]
    assert "(2 stripes" in r["sample"] and r["sample"].startswith("one core: 64 MiB decoded")


def test_reference_arm_json_line():
    """`bench.py --impl reference` (the oracle on the host cores) prints one
    JSON line with the contract's keys: impl, metric, value, unit, timing,
    the cpu_baseline describing the run and an e2e with no host traffic."""
    import json
    import subprocess
    import sys
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    r = subprocess.run([sys.executable, os.path.join(root, "bench.py"), "--impl", "reference", "--workload", "tiny",
                        "--steps", "1", "--warmup", "1"], capture_output=True, text=True, timeout=600, cwd=root)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [ln for ln in r.stdout.splitlines() if ln.startswith("{")]
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["unit"] == "GB/s" and d["value"] > 0
    assert d["higher_is_better"] is True and d["steps"] == 1 and d["n_gpus"] == 1
    assert d["config"]["workload"] == "tiny"
    cb = d["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["cores"] >= 1 and cb["value"] == d["value"] and cb["sample"]
    assert d["e2e"]["value"] == d["value"] and d["e2e"]["h2d_bytes_per_step"] == 0 and d["e2e"]["d2h_bytes_per_step"] == 0
