#!/usr/bin/env python3
"""Benchmark: decoded bf16 GB/s of the k3huf GPU decoder on GB300, its HBM
roofline fraction, and the compression ratio of the workload.

Default workload: the streaming ring, 14 trunk layers (seeds 10..23, 23 GiB
of bf16, 126 tensors with one code table each).  A step is one pass of the
whole decode path over the 14 layers' containers, already resident in HBM:
per layer, host-side header validation and launch, the per-CTA table
builds, chunk seek, Huffman decode of the high bytes, merge with the raw
low bytes, integrity check.  The K timed steps run back to back with early
start (each launch's table build overlaps the previous launch's end)
between one pair of CUDA events, right after a sustained run of the same
loop that lasts at least a second and a half; the clock sampler covers
both.  The outputs of the timed steps are compared with the generated
tensors, every byte of every layer.  ``single_launch`` times launches one
at a time beside it.  ``e2e`` is the streaming ring itself: every step
copies the 14 containers from pinned host memory into two device slots
(cudaMemcpyAsync on a copy stream, double buffered against the decode on a
compute stream) and reads the status word back.

The single-layer workloads time one layer per step the same way, and their
``e2e`` copies the container in and the decoded weights out every step.

Usage: python bench.py [--gpus N] [--steps K] [--warmup W]
                       [--workload ring|projection|tiny|heavy_tail|trunk_layer|ring_file|gemv|encode]
                       [--impl reference]
For N > 1 run under torchrun: every rank decodes its own replica (the path
has no exchange step), timing is the max over ranks and ``value`` counts
the bytes all ranks decoded.
"""
from __future__ import annotations

import argparse
import ctypes
import hashlib
import itertools
import json
import math
import os
import platform
import statistics
import subprocess
import sys
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import workloads  # noqa: E402

METRIC = "decoded bf16 GB/s on 1 GB300 and % of HBM roofline; compression ratio"
UNIT = "GB/s"
FALLBACK_HBM_GBS = 6800.0
L2_BYTES = 129 * 1024 * 1024


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--workload", default="ring",
                    choices=["tiny", "projection", "heavy_tail", "trunk_layer", "ring", "ring_file", "encode", "gemv"])
    ap.add_argument("--impl", default="gpu", choices=["gpu", "reference"])
    ap.add_argument("--variant", type=int, default=0, help="codes per lookup: 0 default (2), 1, 2")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--ring-layers", type=int, default=None, help="layers streamed (ring: 14, ring_file: 4)")
    ap.add_argument("--sustain-ms", type=float, default=1500.0,
                    help="ring: length of the sustained run before the timed steps")
    ap.add_argument("--feed-dir", default=None, help="directory of the ring_file container file (default: temp dir)")
    ap.add_argument("--feed-threads", type=int, default=8, help="pread threads of the storage feed")
    ap.add_argument("--sub-syms", type=int, default=None, help="values per sub-stream in the container")
    return ap.parse_args()


def dist_env():
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return rank, world, local


def describe(name):
    d = {"workload": name, "recipe": workloads.WORKLOADS[name]}
    return d


def l2_note(blob_bytes, out_bytes):
    return "inputs larger than L2" if blob_bytes + out_bytes > 2 * L2_BYTES else "L2 flushed between steps"


def shared_config(name, layers, world):
    """The config keys both arms print: the workload, its sizes and its
    container sizes.  layers: (n_tensors, raw_bytes, blob_bytes, chunk_syms,
    sub_syms) per layer."""
    raw = sum(x[1] for x in layers)
    blob = sum(x[2] for x in layers)
    return {**describe(name), "layers": len(layers), "tensors": sum(x[0] for x in layers), "values": raw // 2,
            "raw_bytes": raw, "blob_bytes": blob, "compression_ratio": round(raw / blob, 4),
            "compression_rate": round(blob / raw, 4), "chunk_syms": layers[0][3], "sub_syms": layers[0][4],
            "l2": l2_note(max(x[2] for x in layers), max(x[1] for x in layers)),
            "parallelism": f"replicas x{world}"}


def cpu_model():
    """The host CPU's model name (lscpu, else /proc/cpuinfo)."""
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        for line in out.splitlines():
            if line.lower().startswith("model name:"):
                return line.split(":", 1)[1].strip()
    except Exception:
        pass
    try:
        with open("/proc/cpuinfo") as f:
            for line in f:
                if line.split(":")[0].strip().lower() in ("model name", "cpu part"):
                    return line.split(":", 1)[1].strip()
    except OSError:
        pass
    return platform.processor() or platform.machine()


def make_layer(name, sub_syms=None):
    """(tensors, container) of a named single-layer workload."""
    import lossless_bf16_weight_k3huf_gb300 as k3
    tensors = workloads.workload(name)
    kw = {} if sub_syms is None else {"sub_syms": sub_syms}
    blob = k3.encode_layer(tensors, **kw)
    return tensors, blob


def measured_peak():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(p) as f:
            v = float(json.load(f)["hbm_gbs"])
        return v, "measured"
    except Exception:
        return FALLBACK_HBM_GBS, "fallback"


def kernel_src_sha(src="k3huf_decode.cu"):
    p = os.path.join(ROOT, "lossless_bf16_weight_k3huf_gb300", "csrc", src)
    return hashlib.sha256(open(p, "rb").read()).hexdigest()[:16]


def ncu_traffic(workload, alg_bytes_per_launch=None):
    """DRAM bytes per launch from the committed ncu summary, if it was taken
    on the current kernel source; else None.  An entry taken on another
    workload of the same shape (``scale_by_alg``) is scaled to this one's
    algorithmic bytes per launch."""
    p = os.path.join(ROOT, "profiles", "traffic.json")
    try:
        with open(p) as f:
            t = json.load(f).get(workload)
        if t and t.get("kernel_src_sha") == kernel_src_sha(t.get("kernel_src", "k3huf_decode.cu")):
            v = float(t["dram_bytes_per_launch"])
            if t.get("scale_by_alg") and alg_bytes_per_launch:
                v *= alg_bytes_per_launch / float(t["alg_bytes_per_launch"])
            return round(v)
    except Exception:
        pass
    return None


class ClockSampler:
    """nvidia-smi clock / throttle samples while the timed region runs."""
    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.gpu = gpu_index
        self.proc = None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.Q}", "--format=csv,noheader,nounits",
                 "-lms", "50"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.proc = None
        time.sleep(0.25)
        return self

    def __exit__(self, *a):
        time.sleep(0.25)
        self.lines = []
        if self.proc is not None:
            self.proc.terminate()
            try:
                out, _ = self.proc.communicate(timeout=5)
            except Exception:
                self.proc.kill()
                out, _ = self.proc.communicate()
            self.lines = [l for l in out.splitlines() if l.strip()]

    def summary(self):
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for l in getattr(self, "lines", []):
            f = [x.strip() for x in l.split(",")]
            try:
                sm.append(float(f[1]))
                mx.append(float(f[2]))
            except (ValueError, IndexError):
                continue
            for n, v in zip(names, f[5:9]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx), "reasons": sorted(reasons),
                "samples": len(sm)}


def cpu_baseline(blob, budget_s=12.0):
    """The oracle's bit-serial decoder (single thread), timed on a bounded
    sample: whole chunks of the workload's stripes, in order, until the
    time budget is used."""
    import oracle
    info = oracle.layer_info(blob)
    out = np.zeros(info["out_bytes"], dtype=np.uint8)
    cs = info["chunk_syms"]
    sdir = 64 + 256 * info["n_tables"] + 32 * info["n_tensors"]
    values = 0
    chunks = 0
    t0 = time.perf_counter()
    step = 64
    done = False
    for s in range(info["n_stripes"]):
        e = sdir + 32 * s
        nv = int.from_bytes(blob[e + 24:e + 28].tobytes(), "little")
        nch = -(-nv // cs)
        for c in range(0, nch, step):
            n = min(step, nch - c)
            rc = oracle.decode_chunks(blob, s, c, n, out)
            if rc != 0:
                raise RuntimeError(f"oracle decode failed: {rc}")
            values += min(nv, (c + n) * cs) - c * cs
            chunks += n
            if time.perf_counter() - t0 > budget_s:
                done = True
                break
        if done:
            break
    dt = time.perf_counter() - t0
    return {"value": round(2 * values / dt / 1e9, 4), "unit": UNIT, "cores": 1, "kind": "oracle",
            "cpu_model": cpu_model(), "host_cores": os.cpu_count(),
            "sample": f"{chunks} chunks of {cs} values ({2 * values / 2**20:.1f} MiB decoded) in {dt:.1f} s, "
                      f"bit-serial oracle decoder, one thread"}


def cpu_article_style(blob, budget_s=4.0):
    """The article-style scalar decoder (12-bit table, 64-bit accumulator,
    even plane merged in a loop of its own; oracle/k3huf_pagestyle.c): whole
    stripes on one core until the budget is used, then the whole layer with
    one thread per stripe (the article's unit of parallelism) on up to every
    host core.  Decoded bf16 GB/s, and compressed input GB/s beside it."""
    import threading
    import oracle
    info = oracle.layer_info(blob)
    out = np.zeros(info["out_bytes"], dtype=np.uint8)
    sdir = 64 + 256 * info["n_tables"] + 32 * info["n_tensors"]
    nv = [int.from_bytes(blob[sdir + 32 * s + 24:sdir + 32 * s + 28].tobytes(), "little")
          for s in range(info["n_stripes"])]
    sb = [int.from_bytes(blob[sdir + 32 * s + 8:sdir + 32 * s + 16].tobytes(), "little")
          for s in range(info["n_stripes"])]
    hi = np.empty(1 << 25, np.uint8)
    out.fill(1)                              # pages touched before the timed loops
    hi.fill(1)
    one_v = one_b = 0
    t0 = time.perf_counter()
    for s in range(info["n_stripes"]):
        if oracle.pagestyle_decode_stripe(blob, s, out, hi):
            raise RuntimeError("article-style decode failed")
        one_v += nv[s]
        one_b += sb[s]
        if time.perf_counter() - t0 > budget_s:
            break
    dt1 = time.perf_counter() - t0
    threads = min(os.cpu_count() or 1, info["n_stripes"])
    lock = threading.Lock()
    state = {"next": 0, "rc": 0}

    scratch = [np.ones(1 << 25, np.uint8) for _ in range(threads)]

    def work(h):
        while True:
            with lock:
                s = state["next"]
                state["next"] += 1
            if s >= info["n_stripes"]:
                return
            rc = oracle.pagestyle_decode_stripe(blob, s, out, h)
            with lock:
                state["rc"] |= rc

    pool = [threading.Thread(target=work, args=(h,)) for h in scratch]
    t0 = time.perf_counter()
    for t in pool:
        t.start()
    for t in pool:
        t.join()
    dtn = time.perf_counter() - t0
    if state["rc"]:
        raise RuntimeError("article-style decode failed")
    return {"one_core": round(2 * one_v / dt1 / 1e9, 4), "all_cores": round(2 * sum(nv) / dtn / 1e9, 4),
            "unit": UNIT, "cores": threads, "cpu_model": cpu_model(),
            "input_gbs": {"one_core": round(one_b / dt1 / 1e9, 4), "all_cores": round(sum(sb) / dtn / 1e9, 4)},
            "kind": "article-style scalar table decoder (not the oracle)",
            "sample": f"one core: {2 * one_v / 2**20:.0f} MiB decoded in {dt1:.3f} s; all cores: the whole layer "
                      f"({info['n_stripes']} stripes, one thread each on {threads} cores) in {dtn:.3f} s"}


def cpu_baseline_parallel(blob, budget_s=10.0, threads=None):
    """The same oracle decoder run stripe-parallel on every host core:
    threads take blocks of 64 chunks, stripes interleaved, from a shared
    list until the time budget is used (ctypes releases the GIL during each
    call)."""
    import threading
    import oracle
    threads = threads or os.cpu_count() or 1
    info = oracle.layer_info(blob)
    out = np.zeros(info["out_bytes"], dtype=np.uint8)
    cs = info["chunk_syms"]
    sdir = 64 + 256 * info["n_tables"] + 32 * info["n_tensors"]
    step = 64
    per_stripe = []
    for s in range(info["n_stripes"]):
        e = sdir + 32 * s
        nv = int.from_bytes(blob[e + 24:e + 28].tobytes(), "little")
        per_stripe.append([(s, c, min(step, -(-nv // cs) - c), min(nv, (c + step) * cs) - c * cs)
                           for c in range(0, -(-nv // cs), step)])
    units = [u for blk in itertools.zip_longest(*per_stripe) for u in blk if u is not None]
    lock = threading.Lock()
    state = {"next": 0, "values": 0, "chunks": 0, "rc": 0}
    t0 = time.perf_counter()

    def work():
        while time.perf_counter() - t0 < budget_s:
            with lock:
                if state["next"] >= len(units):
                    return
                s, c, n, v = units[state["next"]]
                state["next"] += 1
            rc = oracle.decode_chunks(blob, s, c, n, out)
            with lock:
                state["rc"] |= rc
                state["values"] += v
                state["chunks"] += n

    pool = [threading.Thread(target=work) for _ in range(threads)]
    for t in pool:
        t.start()
    for t in pool:
        t.join()
    dt = time.perf_counter() - t0
    if state["rc"]:
        raise RuntimeError(f"oracle decode failed: {state['rc']}")
    return {"value": round(2 * state["values"] / dt / 1e9, 4), "unit": UNIT, "cores": threads, "kind": "oracle",
            "cpu_model": cpu_model(), "host_cores": os.cpu_count(),
            "sample": f"{state['chunks']} chunks of {cs} values ({2 * state['values'] / 2**20:.1f} MiB decoded) "
                      f"in {dt:.3f} s, bit-serial oracle decoder, {threads} threads over stripe-interleaved "
                      f"64-chunk blocks"}


def _reference_layers(name):
    """The reference arm's view of a workload: the tensors of each layer, one
    layer at a time (a generator), so that the 14-layer ring never sits in
    host memory whole."""
    if name == "ring":
        for s in workloads.ring_layers():
            yield workloads.trunk_layer(seed=s)
    else:
        yield workloads.workload(name)


def run_reference(args):
    """The oracle as it stands, on the host cores.  The config's container
    sizes come from the oracle's own sizing pass over every layer of the
    workload; each step decodes a bounded sample with the oracle's
    bit-serial decoder, on one thread: for the trunk layers (and the ring of
    them) the whole 576x8192 tensor of the first layer, as its own
    container (every tensor of a trunk layer has a code table of its own);
    for a single-tensor workload the first 256 chunks of its first stripe."""
    rank, world, local = dist_env()
    if rank != 0:
        return
    from concurrent.futures import ThreadPoolExecutor
    import oracle
    name = {"ring_file": "trunk_layer", "encode": "heavy_tail", "gemv": "projection"}.get(args.workload,
                                                                                         args.workload)
    sizes, sample_tensors, first = [], None, True
    # sizing runs in C (ctypes releases the GIL) while the next layer is drawn
    with ThreadPoolExecutor(4) as ex:
        futs = []
        for tensors in _reference_layers(name):
            raw = sum(2 * t.size for t in tensors)
            futs.append((len(tensors), raw, ex.submit(oracle.container_bytes, tensors)))
            if first:
                sample_tensors = [tensors[4]] if name in ("ring", "trunk_layer") else tensors
                first = False
            while len([f for f in futs if not f[2].done()]) > 3:
                time.sleep(0.05)
        for n_t, raw, f in futs:
            sizes.append((n_t, raw, f.result(), 4096, 256))
    blob = oracle.encode_layer(sample_tensors)
    info = oracle.layer_info(blob)
    out = np.zeros(info["out_bytes"], dtype=np.uint8)
    cs = info["chunk_syms"]
    sdir = 64 + 256 * info["n_tables"] + 32 * info["n_tensors"]
    nv0 = int.from_bytes(blob[sdir + 24:sdir + 28].tobytes(), "little")
    whole = name in ("ring", "trunk_layer")
    n_chunks = -(-nv0 // cs) if whole else min(-(-nv0 // cs), 256)
    sample_values = min(nv0, n_chunks * cs)

    def step():
        rc = oracle.decode_chunks(blob, 0, 0, n_chunks, out)
        if rc:
            raise RuntimeError(rc)

    for _ in range(args.warmup):
        step()
    t0 = time.perf_counter()
    for _ in range(args.steps):
        step()
    dt = time.perf_counter() - t0
    value = 2 * sample_values * args.steps / dt / 1e9
    if whole:
        sample = (f"per step the whole 576x8192 tensor ({sample_values} values, {n_chunks} chunks) of the first "
                  f"layer, as its own container, bit-serial oracle decoder, one thread")
    else:
        sample = (f"per step the first {n_chunks} chunks ({sample_values} values) of stripe 0, bit-serial oracle "
                  f"decoder, one thread")
    line = {
        "impl": "reference", "metric": METRIC, "value": round(value, 4), "unit": UNIT, "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(dt / args.steps * 1e3, 3),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "u8", "data": "synthetic",
        "config": shared_config(name, sizes, world),
        "cpu_baseline": {"value": round(value, 4), "unit": UNIT, "cores": 1, "kind": "oracle", "sample": sample,
                         "cpu_model": cpu_model(), "host_cores": os.cpu_count()},
        "e2e": {"value": round(value, 4), "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def max_over_ranks(ms: float, device, world: int) -> float:
    """The slowest rank's time: every rank decodes its own replica, so the
    job finishes when the last one does."""
    if world <= 1:
        return ms
    import torch
    import torch.distributed as dist
    t = torch.tensor([ms], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    dist.barrier()
    return float(t.item())


def whole_job_gbs(raw_bytes_per_rank: int, world: int, steps: int, ms: float) -> float:
    """Decoded GB/s of the whole job: the bytes all ranks decoded over the
    max-over-ranks time."""
    return raw_bytes_per_rank * world * steps / (ms / 1e3) / 1e9


def main():
    args = parse()
    if args.impl == "reference":
        run_reference(args)
        return
    import torch
    import lossless_bf16_weight_k3huf_gb300 as k3
    rank, world, local = dist_env()
    if world > 1:
        import torch.distributed as dist
        torch.cuda.set_device(local)
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    else:
        torch.cuda.set_device(0)
    dev = torch.device("cuda", torch.cuda.current_device())
    k3._build.build()
    k3.set_decoder_variant(args.variant)
    if args.workload == "ring":
        return bench_ring(args, rank, world, local, dev)
    if args.workload == "ring_file":
        return bench_ring_file(args, rank, world, local, dev)
    if args.workload == "encode":
        return bench_encode(args, rank, world, local, dev)
    if args.workload == "gemv":
        return bench_gemv(args, rank, world, local, dev)

    tensors, blob = make_layer(args.workload, args.sub_syms)
    info = k3.layer_info(blob)
    hdr = blob[: info["hdr_bytes"]].copy()
    raw = info["raw_bytes"]
    d_blob = torch.from_numpy(blob).to(dev)
    d_out = torch.empty(info["out_bytes"], dtype=torch.uint8, device=dev)
    d_st = torch.zeros(1, dtype=torch.int32, device=dev)
    d_work = torch.zeros(k3.WORK_BYTES // 4, dtype=torch.int32, device=dev)   # pool of the last items
    stream = torch.cuda.Stream(device=dev)
    launches_per_step = -(-info["n_stripes"] // 64)
    l2_note = ("inputs larger than L2" if info["blob_bytes"] + info["out_bytes"] > 2 * L2_BYTES
               else "L2 flushed between steps")
    flush = None if info["blob_bytes"] + info["out_bytes"] > 2 * L2_BYTES else \
        torch.empty(2 * L2_BYTES, dtype=torch.uint8, device=dev)

    # early start: each launch's CTAs take the SMs the previous launch frees
    # and build their tables there (the previous kernel never writes d_blob)
    def step():
        if flush is not None:
            flush.fill_(1)
        k3.decode_layer(hdr, d_blob, d_out, d_st, stream=stream, work=d_work, early_start=True)

    with torch.cuda.stream(stream):
        for _ in range(max(3, args.warmup)):
            step()
    stream.synchronize()
    # correctness of the benchmarked output (bytes equal the original tensors)
    ok = d_st.item() == 0
    for t, x in zip(range(info["n_tensors"]), tensors):
        ti = k3.tensor_info(hdr, t)
        a = ti["out_offset"]
        ref = torch.from_numpy(np.asarray(x, np.uint16).reshape(-1).view(np.int16)).to(dev)
        ok = ok and torch.equal(d_out[a:a + 2 * ti["n_values"]].view(torch.int16), ref)
        del ref
    if not ok:
        raise SystemExit("decode output differs from the input tensors")

    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(args.steps)]
    with ClockSampler(dev.index) as clk:
        t_start = torch.cuda.Event(enable_timing=True)
        t_end = torch.cuda.Event(enable_timing=True)
        with torch.cuda.stream(stream):
            t_start.record(stream)
            for i in range(args.steps):
                if flush is not None:
                    # an L2 flush between steps: events bracket each decode
                    flush.fill_(1)
                    ev[i][0].record(stream)
                k3.decode_layer(hdr, d_blob, d_out, d_st, stream=stream, work=d_work, early_start=True)
                if flush is not None:
                    ev[i][1].record(stream)
            t_end.record(stream)
        stream.synchronize()
    torch.cuda.synchronize()
    total_ms = t_start.elapsed_time(t_end)
    # without a flush the timed region holds the K decode steps back to back
    # (an event recorded between two launches would end the early start)
    kernel_ms = [a.elapsed_time(b) for a, b in ev] if flush is not None else [total_ms / args.steps] * args.steps
    dev_ms = sum(kernel_ms)                      # decode time only (excludes any L2 flush)
    dev_ms = max_over_ranks(dev_ms, dev, world)
    ms_per_step = dev_ms / args.steps
    value = whole_job_gbs(raw, world, args.steps, dev_ms)

    # single launches, each between its own pair of events (so none starts
    # early), after 5 more warm-ups: median and min of 20, in us per launch
    single = []
    with torch.cuda.stream(stream):
        for i in range(25):
            if flush is not None:
                flush.fill_(1)
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record(stream)
            k3.decode_layer(hdr, d_blob, d_out, d_st, stream=stream, work=d_work)
            b.record(stream)
            if i >= 5:
                single.append((a, b))
    stream.synchronize()
    single_us = sorted(a.elapsed_time(b) * 1e3 / launches_per_step for a, b in single)

    # end to end through the C ABI with host buffers
    e2e = bench_e2e(k3, blob, hdr, info, dev, stream, max(4, min(args.steps, 20)))

    if rank != 0:
        if world > 1:
            torch.distributed.destroy_process_group()
        return
    peak, peak_kind = measured_peak()
    alg = info["blob_bytes"] + info["raw_bytes"]
    avg_launch_ms = statistics.mean(kernel_ms) / launches_per_step
    achieved = alg / launches_per_step / (avg_launch_ms / 1e3) / 1e9
    single_achieved = alg / launches_per_step / (statistics.median(single_us) / 1e6) / 1e9
    traffic = ncu_traffic(args.workload, alg // launches_per_step)
    line = {
        "metric": METRIC, "value": round(value, 2), "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": max(3, args.warmup), "ms_per_step": round(ms_per_step, 5), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "u8", "data": "synthetic",
        "config": shared_config(args.workload, [(info["n_tensors"], raw, info["blob_bytes"], info["chunk_syms"],
                                                 info["sub_syms"])], world),
        "method": {"decoder": ["2 codes/lookup", "1 code/lookup", "2 codes/lookup"][args.variant],
                   "call": "k3huf_decode_layer_ex (work area: the last sixteenth of each CTA's items pooled "
                           "across the CTAs; early start: a launch's CTAs start on the SMs the previous launch "
                           "frees)",
                   "timing": ("CUDA events around each decode, L2 flushed between steps" if flush is not None
                              else "CUDA events around the K back-to-back decode steps")},
        "roofline": {"bound": "hbm", "achieved": round(achieved, 1), "peak": peak, "unit": "GB/s",
                     "frac": round(achieved / peak, 4), "peak_kind": f"{peak_kind} copy bandwidth",
                     "traffic": traffic, "algorithmic_bytes_per_launch": alg // launches_per_step,
                     "frac_of_8TBs": round(achieved / 8000.0, 4),
                     "single_launch": {"achieved": round(single_achieved, 1),
                                       "frac": round(single_achieved / peak, 4),
                                       "median_us": round(statistics.median(single_us), 2),
                                       "note": "launches one at a time, an event pair around each, no early "
                                               "start"}},
        "e2e": e2e,
        "gpu_launches": launches_per_step * args.steps,
        "single_launch_us": {"median": round(statistics.median(single_us), 2), "min": round(single_us[0], 2),
                             "of": len(single_us), "note": "outside the timed region: launches one at a time, "
                                                           "event pair around each, no early start"},
        "clocks": clk.summary(),
        "timed_region_ms": round(total_ms, 3),
    }
    if world == 1 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline_parallel(blob)
        line["cpu_baseline"]["one_core"] = cpu_baseline(blob, budget_s=6.0)["value"]
        line["cpu_baseline"]["article_style"] = cpu_article_style(blob)
    print(json.dumps(line), flush=True)
    if world > 1:
        torch.distributed.destroy_process_group()


def bench_e2e(k3, blob, hdr, info, dev, stream, steps):
    """End to end through the C ABI with host buffers: every step copies the
    container from pinned host memory to HBM, decodes it, and copies the
    decoded weights back to pinned host memory.  Steps are pipelined on
    three streams (copy in, decode, copy out) with two buffer sets, so the
    two copy directions and the decode of consecutive steps overlap; the
    timed region spans all steps, first copy to last copy back."""
    import torch
    h_blob = torch.from_numpy(blob).pin_memory()
    h_out = [torch.empty(info["out_bytes"], dtype=torch.uint8).pin_memory() for _ in range(2)]
    d_blob = [torch.empty(blob.size, dtype=torch.uint8, device=dev) for _ in range(2)]
    d_out = [torch.empty(info["out_bytes"], dtype=torch.uint8, device=dev) for _ in range(2)]
    d_st = torch.zeros(1, dtype=torch.int32, device=dev)
    d_work = torch.zeros(k3.WORK_BYTES // 4, dtype=torch.int32, device=dev)   # pool of the last items
    s_in, s_out = torch.cuda.Stream(device=dev), torch.cuda.Stream(device=dev)
    ev_in = [torch.cuda.Event() for _ in range(2)]
    ev_dec = [torch.cuda.Event() for _ in range(2)]
    ev_out = [torch.cuda.Event() for _ in range(2)]

    def run(n):
        for i in range(n):
            b = i % 2
            if i >= 2:
                s_in.wait_event(ev_dec[b])            # decode i-2 finished reading d_blob[b]
            with torch.cuda.stream(s_in):
                d_blob[b].copy_(h_blob, non_blocking=True)
                ev_in[b].record(s_in)
            stream.wait_event(ev_in[b])
            if i >= 2:
                stream.wait_event(ev_out[b])          # copy-out i-2 finished reading d_out[b]
            k3.decode_layer(hdr, d_blob[b], d_out[b], d_st, stream=stream, work=d_work)
            ev_dec[b].record(stream)
            s_out.wait_event(ev_dec[b])
            with torch.cuda.stream(s_out):
                h_out[b].copy_(d_out[b], non_blocking=True)
                ev_out[b].record(s_out)

    run(2)
    torch.cuda.synchronize()
    a = torch.cuda.Event(enable_timing=True)
    z = torch.cuda.Event(enable_timing=True)
    a.record(s_in)
    run(steps)
    s_out.wait_stream(stream)
    z.record(s_out)
    torch.cuda.synchronize()
    ms = a.elapsed_time(z) / steps
    if d_st.item() != 0:
        raise SystemExit("end-to-end decode reported a fault")
    return {"value": round(info["raw_bytes"] / (ms / 1e3) / 1e9, 2), "unit": UNIT,
            "h2d_bytes_per_step": int(blob.size), "d2h_bytes_per_step": int(info["out_bytes"]),
            "ms_per_step": round(ms, 4), "steps": steps, "pipelined": "copy-in / decode / copy-out streams"}


def _fill(bufs, value, stream):
    import torch
    with torch.cuda.stream(stream):
        for b in bufs:
            b.fill_(value)


def bench_ring(args, rank, world, local, dev):
    """The 14 trunk layers of the streaming ring.  value: decode only, every
    layer's container resident in HBM, K steps of the 14 layers back to back
    with early start between one pair of CUDA events, right after a
    sustained run of the same loop; the outputs of the timed steps are then
    compared with the generated tensors, every byte.  e2e: the ring from
    pinned host memory (two device slots, copy stream against compute
    stream), each step ending with a read of the status word."""
    import torch
    import lossless_bf16_weight_k3huf_gb300 as k3
    seeds = workloads.ring_layers(n_layers=args.ring_layers or 14)
    t_prep = time.perf_counter()
    L = []                   # per layer: hdr, info, pinned container, device container, output, expected output
    blob0 = None
    for s in seeds:
        tensors = workloads.trunk_layer(seed=s)
        blob = k3.encode_layer(tensors)
        info = k3.layer_info(blob)
        hdr = blob[: info["hdr_bytes"]].copy()
        h_blob = torch.from_numpy(blob).pin_memory()
        d_blob = h_blob.to(dev)
        d_ref = torch.zeros(info["out_bytes"], dtype=torch.uint8, device=dev)
        regions = []
        for t, x in enumerate(tensors):
            ti = k3.tensor_info(hdr, t)
            a, b = ti["out_offset"], ti["out_offset"] + 2 * ti["n_values"]
            d_ref[a:b].copy_(torch.from_numpy(x.reshape(-1).view(np.uint8)))
            regions.append((a, b))
        L.append({"hdr": hdr, "info": info, "h": h_blob, "d": d_blob, "ref": d_ref, "regions": regions,
                  "out": torch.empty(info["out_bytes"], dtype=torch.uint8, device=dev)})
        if blob0 is None:
            blob0 = blob
        del tensors, blob
    prep_s = time.perf_counter() - t_prep
    raw = sum(x["info"]["raw_bytes"] for x in L)
    blob_total = sum(x["info"]["blob_bytes"] for x in L)
    alg = blob_total + raw                                  # container read + bf16 written, all layers
    n_layers = len(L)
    outs = [x["out"] for x in L]
    work = torch.zeros(k3.WORK_BYTES // 4, dtype=torch.int32, device=dev)
    st = torch.zeros(1, dtype=torch.int32, device=dev)
    stream = torch.cuda.Stream(device=dev)

    def step():
        for x in L:
            k3.decode_layer(x["hdr"], x["d"], x["out"], st, stream=stream, work=work, early_start=True)

    def verify(what):
        torch.cuda.synchronize()
        if st.item() != 0:
            raise SystemExit(f"{what}: decode reported status {st.item()}")
        for i, x in enumerate(L):
            for a, b in x["regions"]:
                if not torch.equal(x["out"][a:b], x["ref"][a:b]):
                    raise SystemExit(f"{what}: layer {i} differs from its input tensors in bytes [{a}, {b})")

    def timed_steps(n):
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        with torch.cuda.stream(stream):
            e0.record(stream)
            for _ in range(n):
                step()
            e1.record(stream)
        return e0, e1

    warm = max(3, args.warmup)
    with torch.cuda.stream(stream):
        for _ in range(warm):
            step()
    stream.synchronize()
    w0, w1 = timed_steps(2)
    stream.synchronize()
    est_ms = w0.elapsed_time(w1) / 2
    n_sustain = max(1, int(math.ceil(args.sustain_ms / est_ms)))
    # the outputs are overwritten with a pattern, so the check after the timed
    # steps sees only what they wrote
    _fill(outs, 0xA5, stream)
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    with ClockSampler(dev.index) as clk:
        s0, s1 = timed_steps(n_sustain)
        _fill(outs, 0xA5, stream)
        t0, t1 = timed_steps(args.steps)
        stream.synchronize()
    torch.cuda.synchronize()
    timed_ms = t0.elapsed_time(t1)
    sustain_ms = s0.elapsed_time(s1)
    verify("timed steps")
    dev_ms = max_over_ranks(timed_ms, dev, world)
    value = whole_job_gbs(raw, world, args.steps, dev_ms)

    # launches one at a time (event pair around each, no early start)
    single = []
    with torch.cuda.stream(stream):
        for rep in range(3):
            for x in L:
                a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                a.record(stream)
                k3.decode_layer(x["hdr"], x["d"], x["out"], st, stream=stream, work=work)
                b.record(stream)
                if rep:
                    single.append((a, b, x["info"]["blob_bytes"] + x["info"]["raw_bytes"]))
    stream.synchronize()
    single_us = sorted(a.elapsed_time(b) * 1e3 for a, b, _ in single)
    single_gbs = sorted(n / (a.elapsed_time(b) / 1e3) / 1e9 for a, b, n in single)

    # end to end: the ring from pinned host memory, status word read back
    ring = k3.Ring(max(x["h"].numel() for x in L), 2)
    h_layers = [x["h"] for x in L]
    ring.run(h_layers, outs, st)
    torch.cuda.synchronize()
    _fill(outs, 0xA5, stream)
    torch.cuda.synchronize()
    e2e_steps = max(2, min(args.steps, 20))
    walls, stats = [], []
    with ClockSampler(dev.index) as clk_e2e:
        for _ in range(e2e_steps):
            w = time.perf_counter()
            stats.append(ring.run(h_layers, outs, st))
            status = int(st.item())
            walls.append(time.perf_counter() - w)
            if status:
                raise SystemExit(f"ring decode reported status {status}")
    ring.close()
    verify("ring (e2e)")
    e2e_s = sum(walls)
    dec = sum(x["decode_ms"] for x in stats)
    cp = sum(x["copy_ms"] for x in stats)
    tot = sum(x["total_ms"] for x in stats)

    if rank != 0:
        if world > 1:
            torch.distributed.destroy_process_group()
        return
    peak, peak_kind = measured_peak()
    launches = n_layers * args.steps
    achieved = alg * args.steps / (timed_ms / 1e3) / 1e9
    traffic = ncu_traffic("ring", alg // n_layers)
    clocks = clk.summary()
    clocks["window"] = "the sustained run and the timed steps"
    line = {
        "metric": METRIC, "value": round(value, 2), "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": warm, "ms_per_step": round(dev_ms / args.steps, 4), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "u8", "data": "synthetic",
        "config": shared_config("ring", [(x["info"]["n_tensors"], x["info"]["raw_bytes"], x["info"]["blob_bytes"],
                                          x["info"]["chunk_syms"], x["info"]["sub_syms"]) for x in L], world),
        "method": {"call": "k3huf_decode_layer_ex per layer (work area; early start: a launch's CTAs start on "
                           "the SMs the previous launch frees)",
                   "timing": "CUDA events around the K steps of 14 back-to-back decodes; the containers "
                             "resident in HBM (inputs larger than L2)",
                   "verified": "after the timed steps every byte of the 14 layers' outputs equals the generated "
                               "tensors (outputs overwritten with a pattern before the timed steps)",
                   "prep_s": round(prep_s, 1)},
        "roofline": {"bound": "hbm", "achieved": round(achieved, 1), "peak": peak, "unit": "GB/s",
                     "frac": round(achieved / peak, 4), "peak_kind": f"{peak_kind} copy bandwidth",
                     "traffic": traffic, "algorithmic_bytes_per_launch": alg // n_layers,
                     "frac_of_8TBs": round(achieved / 8000.0, 4),
                     "single_launch": {"achieved": round(statistics.median(single_gbs), 1),
                                       "frac": round(statistics.median(single_gbs) / peak, 4),
                                       "median_us": round(statistics.median(single_us), 2),
                                       "min_us": round(single_us[0], 2), "of": len(single_us),
                                       "note": "launches one at a time, an event pair around each, no early "
                                               "start"}},
        "sustained": {"steps": n_sustain, "ms": round(sustain_ms, 1),
                      "gbs": round(raw * n_sustain / (sustain_ms / 1e3) / 1e9, 2),
                      "note": "the same loop run just before the timed steps, under the same clock sampler"},
        "e2e": {"value": round(raw * e2e_steps / e2e_s / 1e9, 2), "unit": UNIT, "h2d_bytes_per_step": blob_total,
                "d2h_bytes_per_step": 4, "steps": e2e_steps, "ms_per_step": round(e2e_s / e2e_steps * 1e3, 2),
                "decode_only_gbs": round(raw * e2e_steps / (dec / 1e3) / 1e9, 2),
                "copy_only_gbs_h2d": round(blob_total * e2e_steps / (cp / 1e3) / 1e9, 2),
                "exposed_copy_ms_per_step": round((tot - dec) / e2e_steps, 2),
                "call": "k3huf_ring_run: two device slots, cudaMemcpyAsync of each container on a copy stream "
                        "against the decode on a compute stream; host wall time per step including the "
                        "read of the 4-byte status word", "clocks": clk_e2e.summary()},
        "gpu_launches": launches,
        "clocks": clocks,
        "timed_region_ms": round(timed_ms, 3),
    }
    if world == 1 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline_parallel(blob0)
        line["cpu_baseline"]["sample"] += " (layer 1 of the 14)"
        line["cpu_baseline"]["one_core"] = cpu_baseline(blob0, budget_s=6.0)["value"]
        line["cpu_baseline"]["article_style"] = cpu_article_style(blob0)
    print(json.dumps(line), flush=True)
    if world > 1:
        torch.distributed.destroy_process_group()


def bench_encode(args, rank, world, local, dev):
    """GPU encoder on the heavy-tail tensor: the container built on the
    device from a device-resident tensor.  The call plans the codes and the
    layout on the device and synchronises once, at the end, so K calls in a
    row are timed with CUDA events around them (the host's share of each
    call included); they are made through the C ABI with their arguments
    marshalled once, and the Python binding's time per call is reported
    beside it.  The container is
    checked byte for byte against the CPU encoder's (which the host tests
    check against the oracle's)."""
    import torch
    import lossless_bf16_weight_k3huf_gb300 as k3
    x = workloads.heavy_tail()
    n = x.size
    raw = 2 * n
    t0 = time.perf_counter()
    ref = k3.encode_layer([x])
    cpu_enc_s = time.perf_counter() - t0
    h_x = torch.from_numpy(x.view(np.int16)).pin_memory()
    d_x = h_x.to(dev)
    scratch = torch.empty(k3.encode_scratch_bytes([n]), dtype=torch.uint8, device=dev)
    # one call per encode: the output buffer holds any container of n values
    out_buf = torch.empty(k3.encode_bound([n]), dtype=torch.uint8, device=dev)
    blob = k3.encode_layer_gpu([d_x], scratch=scratch, out=out_buf)
    if not np.array_equal(blob.cpu().numpy(), ref):
        raise SystemExit("GPU container differs from the CPU encoder's")
    for _ in range(max(0, args.warmup - 1)):
        k3.encode_layer_gpu([d_x], scratch=scratch, out=out_buf)
    torch.cuda.synchronize()
    # the C ABI call, its arguments marshalled once
    enc = k3._lib().k3huf_encode_layer_gpu
    c_ptrs = (ctypes.c_void_p * 1)(d_x.data_ptr())
    c_nv = (ctypes.c_uint64 * 1)(n)
    c_size = ctypes.c_size_t(0)
    c_args = (1, c_ptrs, c_nv, 4096, 256, 0, scratch.data_ptr(), scratch.numel(), out_buf.data_ptr(),
              out_buf.numel(), ctypes.byref(c_size), torch.cuda.current_stream(dev).cuda_stream)
    for _ in range(3):
        if enc(*c_args) != 0:
            raise SystemExit("k3huf_encode_layer_gpu failed")
    torch.cuda.synchronize()
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with ClockSampler(dev.index) as clk:
        ev0.record()
        for _ in range(args.steps):
            if enc(*c_args) != 0:
                raise SystemExit("k3huf_encode_layer_gpu failed")
        ev1.record()
        torch.cuda.synchronize()
    t = ev0.elapsed_time(ev1) / 1e3 / args.steps
    if c_size.value != blob.numel():
        raise SystemExit("container size changed between calls")
    # the same calls through the Python binding (host wall time)
    tb = []
    for _ in range(max(3, args.steps // 2)):
        t0 = time.perf_counter()
        k3.encode_layer_gpu([d_x], scratch=scratch, out=out_buf)
        torch.cuda.synchronize()
        tb.append(time.perf_counter() - t0)
    tb = sorted(tb)[len(tb) // 2]
    # end to end: input from pinned host memory, container back to pinned host memory
    h_blob = torch.empty(blob.numel(), dtype=torch.uint8).pin_memory()
    d_in = torch.empty_like(d_x)                   # the input's device buffer, reused every step
    e2e = []
    for _ in range(max(3, args.steps // 4)):
        t0 = time.perf_counter()
        d_in.copy_(h_x, non_blocking=True)
        b = k3.encode_layer_gpu([d_in], scratch=scratch, out=out_buf)
        h_blob.copy_(b, non_blocking=True)
        torch.cuda.synchronize()
        e2e.append(time.perf_counter() - t0)
    te = sum(e2e) / len(e2e)
    peak, peak_kind = measured_peak()
    alg = raw + blob.numel()                      # one read of the input, one write of the container
    line = {
        "metric": "encoded bf16 GB/s on 1 GB300 (GPU encoder, container identical to the CPU encoder's)",
        "value": round(raw / t / 1e9, 2), "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(t * 1e3, 3), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "u8", "data": "synthetic",
        "config": {**describe("encode"), "values": n, "raw_bytes": raw, "blob_bytes": int(blob.numel()),
                   "compression_ratio": round(raw / blob.numel(), 4),
                   "passes": ("histogram; code lengths, codes and layout planned on the device; one pass per "
                              "4096-value chunk: bit counts, chunk and sub-stream index (decoupled look-back), "
                              "packing, low bytes (2 reads of the input); the words neighbouring chunks share "
                              "joined and the padding zeroed"),
                   "call": ("one k3huf_encode_layer_gpu per step (C ABI, CUDA events around the steps) into a "
                            "buffer of k3huf_encode_bound bytes"),
                   "python_binding_ms_per_call": round(tb * 1e3, 3),
                   "cpu_encoder_gbs": round(raw / cpu_enc_s / 1e9, 3),
                   "cpu_encoder_threads": os.cpu_count(), "l2": "inputs larger than L2"},
        "roofline": {"bound": "hbm", "achieved": round(alg / t / 1e9, 1), "peak": peak, "unit": "GB/s",
                     "frac": round(alg / t / 1e9 / peak, 4), "peak_kind": f"{peak_kind} copy bandwidth",
                     "traffic": ncu_traffic("encode"), "algorithmic_bytes_per_call": alg},
        "e2e": {"value": round(raw / te / 1e9, 2), "unit": UNIT, "h2d_bytes_per_step": raw,
                "d2h_bytes_per_step": int(blob.numel())},
        "gpu_launches": 4 * args.steps,                 # histogram, planner, one-pass packing, seams
        "clocks": clk.summary(),
    }
    if rank == 0 and not args.no_cpu_baseline:
        import oracle
        t0 = time.perf_counter()
        m = 1 << 25
        oracle.encode_layer([x[:m]])
        dt = time.perf_counter() - t0
        line["cpu_baseline"] = {"value": round(2 * m / dt / 1e9, 4), "unit": UNIT, "cores": 1, "kind": "oracle",
                                "sample": f"first {m} values (one stripe, {2 * m >> 20} MiB) encoded by the oracle in {dt:.1f} s, one thread"}
    if rank == 0:
        print(json.dumps(line), flush=True)


def bench_gemv(args, rank, world, local, dev):
    """Decode fused into a matrix-vector product: y = W x with W held as a
    k3huf container and decoded on chip, against the unfused path (decode W
    into HBM, then cuBLAS GEMV through torch.mv on the bf16 weights).  The
    value is weight bytes (bf16) per second of the fused call."""
    import torch
    import lossless_bf16_weight_k3huf_gb300 as k3
    rows, cols = 8192, 16384
    w = workloads.projection(rows=rows, cols=cols).reshape(rows, cols)
    blob = k3.encode_layer([w])
    info = k3.layer_info(blob)
    hdr = blob[: info["hdr_bytes"]].copy()
    d_blob = torch.from_numpy(blob).to(dev)
    x_bits = workloads.normal_tensor((cols,), 1.0, 4).reshape(-1)
    x = torch.from_numpy(x_bits.view(np.int16)).to(dev)
    x_bf = x.view(torch.bfloat16)
    y = torch.zeros(rows, dtype=torch.float32, device=dev)
    st = torch.zeros(1, dtype=torch.int32, device=dev)
    d_out = torch.empty(info["out_bytes"], dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream()
    # correctness against the unfused path
    k3.gemv_layer(hdr, d_blob, 0, cols, x, y, st)
    k3.decode_layer(hdr, d_blob, d_out, st)
    W = d_out[: 2 * rows * cols].view(torch.bfloat16).view(rows, cols)
    ref = (W.float() @ x_bf.float())
    torch.cuda.synchronize()
    if st.item() != 0:
        raise SystemExit("fused GEMV reported a fault")
    mag = W.float().abs() @ x_bf.float().abs()
    if not bool(((y - ref).abs() <= 1e-4 * mag + 1e-30).all()):
        raise SystemExit("fused GEMV disagrees with decode + matmul")

    def fused():
        # y = W x in one call: its zeroing kernel and the GEMV start early,
        # so a call's table build overlaps the previous call's end
        k3.gemv_layer(hdr, d_blob, 0, cols, x, y, st, zero_y=True, early_start=True)

    def unfused():
        k3.decode_layer(hdr, d_blob, d_out, st)
        torch.mv(W, x_bf)

    def timed(fn, steps):
        for _ in range(max(3, args.warmup)):
            fn()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        torch.cuda.synchronize()
        e0.record(stream)
        for _ in range(steps):
            fn()
        e1.record(stream)
        torch.cuda.synchronize()
        return e0.elapsed_time(e1) / steps / 1e3

    with ClockSampler(dev.index) as clk:
        t_f = timed(fused, args.steps)
    t_u = timed(unfused, args.steps)
    t_mv = timed(lambda: torch.mv(W, x_bf), args.steps)

    # several vectors at once: one decode of W for all of them (k3huf_gemv_layer_batch)
    # against decode into HBM + cuBLAS GEMM, and cuBLAS on the uncompressed weights
    curve = []
    for n_vec in (2, 4, 8):
        xs = np.concatenate([workloads.normal_tensor((cols,), 1.0, 4 + b).reshape(-1) for b in range(n_vec)])
        X = torch.from_numpy(xs.view(np.int16)).to(dev).view(n_vec, cols)
        Xb = X.view(torch.bfloat16)
        Y = torch.zeros((n_vec, rows), dtype=torch.float32, device=dev)
        k3.gemv_layer_batch(hdr, d_blob, 0, cols, X, Y, st, zero_y=True)
        refB = (W.float() @ Xb.float().t()).t()
        magB = (W.float().abs() @ Xb.float().abs().t()).t()
        torch.cuda.synchronize()
        if st.item() != 0 or not bool(((Y - refB).abs() <= 1e-4 * magB + 1e-30).all()):
            raise SystemExit(f"batched fused GEMV ({n_vec} vectors) disagrees with decode + matmul")
        del refB, magB
        tb_f = timed(lambda: k3.gemv_layer_batch(hdr, d_blob, 0, cols, X, Y, st, zero_y=True, early_start=True),
                     args.steps)

        def unfused_b():
            k3.decode_layer(hdr, d_blob, d_out, st)
            torch.mm(W, Xb.t())

        tb_u = timed(unfused_b, args.steps)
        tb_c = timed(lambda: torch.mm(W, Xb.t()), args.steps)
        curve.append({"n_vec": n_vec, "fused_ms": round(tb_f * 1e3, 4), "decode_then_cublas_ms": round(tb_u * 1e3, 4),
                      "cublas_uncompressed_ms": round(tb_c * 1e3, 4)})
    raw = 2 * rows * cols
    peak, peak_kind = measured_peak()
    alg = info["blob_bytes"] + 2 * cols + 4 * rows * 2          # container, x, y read and written
    line = {
        "metric": "bf16 weight GB/s of y = W x with W decoded on chip (fused decode + GEMV) on 1 GB300",
        "value": round(raw / t_f / 1e9, 2), "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(t_f * 1e3, 4), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f32", "data": "synthetic",
        "config": {**describe("gemv"), "rows": rows, "cols": cols, "raw_bytes": raw,
                   "blob_bytes": info["blob_bytes"], "compression_ratio": round(raw / info["blob_bytes"], 4),
                   "unfused_ms": round(t_u * 1e3, 4), "speedup_vs_unfused": round(t_u / t_f, 3),
                   "cublas_gemv_bf16_ms": round(t_mv * 1e3, 4),
                   "call": "k3huf_gemv_layer_ex (y zeroed by the call, early start)",
                   "note": "unfused = k3huf_decode_layer into HBM, then torch.mv (cuBLAS) on the bf16 weights",
                   "batch_curve": [{"n_vec": 1, "fused_ms": round(t_f * 1e3, 4),
                                    "decode_then_cublas_ms": round(t_u * 1e3, 4),
                                    "cublas_uncompressed_ms": round(t_mv * 1e3, 4)}] + curve,
                   "l2": "inputs larger than L2"},
        "roofline": {"bound": "hbm", "achieved": round(alg / t_f / 1e9, 1), "peak": peak, "unit": "GB/s",
                     "frac": round(alg / t_f / 1e9 / peak, 4), "peak_kind": f"{peak_kind} copy bandwidth",
                     "traffic": ncu_traffic("gemv"), "algorithmic_bytes_per_call": alg},
        "e2e": {"value": round(raw / t_f / 1e9, 2), "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0,
                "note": "weights resident compressed in HBM; no host traffic per call"},
        "gpu_launches": 2 * args.steps,                 # zeroing kernel + fused GEMV
        "clocks": clk.summary(),
    }
    if rank == 0:
        print(json.dumps(line), flush=True)


def _fs_of(path):
    """Filesystem type and device of the mount holding path (best effort)."""
    best = ("?", "?", "")
    try:
        with open("/proc/mounts") as f:
            for line in f:
                dev, mnt, fstype = line.split()[:3]
                if os.path.realpath(path).startswith(mnt) and len(mnt) >= len(best[2]):
                    best = (fstype, dev, mnt)
    except OSError:
        pass
    return {"fstype": best[0], "device": best[1], "mount": best[2]}


def _drop_cache(path):
    """Ask the kernel to drop the file's pages (a buffered feed then reads
    the device, not the page cache)."""
    fd = os.open(path, os.O_RDONLY)
    try:
        os.posix_fadvise(fd, 0, 0, os.POSIX_FADV_DONTNEED)
    finally:
        os.close(fd)


def bench_ring_file(args, rank, world, local, dev):
    """Storage feed: trunk layers written once to a container file, then read
    back every step (O_DIRECT where the filesystem allows it, the file's
    pages dropped from the page cache before each step) into the pinned
    ring, copied to HBM and decoded.  The value is end to end: decoded bytes
    over the host wall time from the first read to the last decode."""
    import shutil
    import tempfile
    import torch
    import lossless_bf16_weight_k3huf_gb300 as k3
    n_layers = args.ring_layers or 4
    seeds = workloads.ring_layers(n_layers=n_layers)
    blobs, infos = [], []
    for s in seeds:
        tensors = workloads.trunk_layer(seed=s)
        blobs.append(k3.encode_layer(tensors))
        infos.append(k3.layer_info(blobs[-1]))
        del tensors
    total = sum(b.size for b in blobs)
    d = tempfile.mkdtemp(prefix="k3huf_feed_", dir=args.feed_dir)
    path = os.path.join(d, "layers.k3huf")
    try:
        if shutil.disk_usage(d).free < total + (1 << 30):
            raise SystemExit(f"not enough free space in {d} for {total} bytes")
        offs = k3.write_layers(path, blobs)
        sizes = [b.size for b in blobs]
        del blobs
        feed = k3.Feed(path, threads=args.feed_threads)
        out_bytes = max(i["out_bytes"] for i in infos)
        outs = [torch.empty(out_bytes, dtype=torch.uint8, device=dev) for _ in range(2)]
        d_outs = [outs[i % 2] for i in range(n_layers)]
        st = torch.zeros(1, dtype=torch.int32, device=dev)
        ring = k3.Ring(max(sizes), 2, staged=True)
        for _ in range(max(1, args.warmup)):
            _drop_cache(path)
            ring.run_file(feed, offs, sizes, d_outs, st)
        if st.item() != 0:
            raise SystemExit("file-fed decode reported a fault")
        stats = []
        with ClockSampler(dev.index) as clk:
            for _ in range(args.steps):
                _drop_cache(path)
                stats.append(ring.run_file(feed, offs, sizes, d_outs, st))
        direct = feed.direct
        ring.close()
        feed.close()
        fs = _fs_of(d)
    finally:
        shutil.rmtree(d, ignore_errors=True)
    raw = sum(i["raw_bytes"] for i in infos)
    tot = sum(s["total_ms"] for s in stats)
    rd = sum(s["read_ms"] for s in stats)
    dec = sum(s["decode_ms"] for s in stats)
    cp = sum(s["copy_ms"] for s in stats)
    value = raw * args.steps / (tot / 1e3) / 1e9
    peak, peak_kind = measured_peak()
    achieved = (total + raw) / (dec / args.steps / 1e3) / 1e9
    launches = sum(-(-i["n_stripes"] // 64) for i in infos)
    line = {
        "metric": METRIC, "value": round(value, 2), "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(tot / args.steps, 3), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "u8", "data": "synthetic",
        "config": {**describe("ring_file"), "layers": n_layers, "raw_bytes": raw, "blob_bytes": total,
                   "compression_ratio": round(raw / total, 4), "o_direct": bool(direct),
                   "feed_threads": args.feed_threads, "filesystem": fs,
                   "read_gbs": round(total * args.steps / (rd / 1e3) / 1e9, 2),
                   "decode_only_gbs": round(raw * args.steps / (dec / 1e3) / 1e9, 2),
                   "copy_only_gbs_h2d": round(total * args.steps / (cp / 1e3) / 1e9, 2),
                   "read_share_of_wall": round(rd / tot, 3),
                   "l2": "inputs larger than L2"},
        "roofline": {"bound": "hbm", "achieved": round(achieved, 1), "peak": peak, "unit": "GB/s",
                     "frac": round(achieved / peak, 4), "peak_kind": f"{peak_kind} copy bandwidth",
                     "traffic": None},
        "e2e": {"value": round(value, 2), "unit": UNIT, "h2d_bytes_per_step": total, "d2h_bytes_per_step": 0},
        "gpu_launches": launches * args.steps,
        "clocks": clk.summary(),
    }
    if rank == 0:
        print(json.dumps(line), flush=True)


if __name__ == "__main__":
    main()
