#!/usr/bin/env python
"""Benchmark: condensate-set attention decode on B300.

One step = one decode query per sequence through topo_attn_forward: score
every key of the KV cache, select C_i (anchor + window + top-k), softmax and
PV over C_i.  The excluded-mass diagnostic is off the timed path.  The default
workload is the million-token decode (B=1, 32/8 heads, d=128, n=1,048,576,
bf16, W=64, k=32); the K cache (2.1 GB) is far larger than L2, so no flush is
needed between steps.

Prints one JSON line (rank 0).  --impl reference times the CPU oracle on the
same workload instead (bounded sample per step).
"""
from __future__ import annotations

import argparse
import json
import math
import os
import statistics
import subprocess
import tempfile
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402

import synth  # noqa: E402

METRIC = "condensate-attn decode queries/s at n=128K–1M; achieved HBM GB/s vs peak"
PREFILL_METRIC = "condensate-attn chunked-prefill scoring TFLOP/s at n=65536 (bf16 tensor peak)"
WORKLOADS = {"decode-1m": 4, "decode-128k-b16": 2, "decode-32k": 1, "prefill-64k": 3}


def workload_desc(w: synth.Workload) -> str:
    return (f"{w.name}: B={w.B} Hq={w.Hq} Hkv={w.Hkv} d={w.d} n={w.n} nq={w.nq} W={w.W} "
            f"k={w.k} {w.dtype} planted={w.planted}")


def load_peaks() -> dict:
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return {"hbm_gbs": float(d["hbm_gbs"]), "bf16_tflops": float(d["bf16_tflops"]),
                "bf16_tflops_sustained": float(d.get("bf16_tflops_sustained", 0.0)),
                "source": "measured"}
    return {"hbm_gbs": 6400.0, "bf16_tflops": 1800.0, "bf16_tflops_sustained": 1400.0,
            "source": "fallback"}


def rank_workload(w: synth.Workload, rank: int) -> synth.Workload:
    """Each rank serves its own sequences: same shapes, its own seeds (weak
    scaling; no data-path collective)."""
    return w.with_(seed=w.seed + 7919 * rank) if rank else w


def job_rate(ms_local: float, queries_per_rank: int, world: int):
    """Whole-job time (max over ranks, gloo all-reduce on the host) and rate:
    queries of all ranks / that time."""
    ms = ms_local
    if world > 1:
        import torch
        import torch.distributed as dist
        tt = torch.tensor([ms], dtype=torch.float64)
        dist.all_reduce(tt, op=dist.ReduceOp.MAX)
        ms = float(tt.item())
    return ms, queries_per_rank * world / (ms / 1000.0)


def dist_env():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


class ClockSampler:
    """nvidia-smi sampling of SM clocks and throttle reasons during a region."""
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu: int):
        self.gpu = gpu
        self.proc = None
        # the raw samples go to TOPO_CLOCKS_DIR (default: the system temp dir);
        # the JSON line carries their summary
        out_dir = os.environ.get("TOPO_CLOCKS_DIR") or tempfile.gettempdir()
        self.path = os.path.join(out_dir, f"clocks_gpu{gpu}.csv")

    def __enter__(self):
        os.makedirs(os.path.dirname(self.path), exist_ok=True)
        try:
            self.f = open(self.path, "w")
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "100"], stdout=self.f,
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

    def summary(self) -> dict:
        if self.proc is None or not os.path.exists(self.path):
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"]}
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in open(self.path):
            parts = [x.strip() for x in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                smax.append(float(parts[2]))
            except ValueError:
                continue
            for nm, val in zip(names, parts[5:9]):
                if val.lower() == "active":
                    reasons.add(nm)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"]}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(smax),
                "samples": len(sm), "reasons": sorted(reasons)}


def oracle_rate(w: synth.Workload, x: dict, budget_s: float, rows_cap: int | None = None):
    """Time the CPU oracle (as it stands) on a bounded sample of rows."""
    import oracle
    P = oracle.make_params(w.B, w.Hq, w.Hkv, w.d, w.n, w.nq, w.W, w.k, w.scale, w.dtype)
    nthreads = oracle.threads()
    total_rows = w.B * w.Hq * w.nq
    probe = min(total_rows, max(1, nthreads))
    t0 = time.perf_counter()
    oracle.topo_attn(P, x["q"], x["k"], x["v"], rows=np.arange(probe), want=("out",),
                     nthreads=nthreads)
    t_probe = time.perf_counter() - t0
    rows = probe
    if t_probe < budget_s:
        more = int(probe * (budget_s - t_probe) / max(t_probe, 1e-9))
        more = min(more, total_rows - probe) if rows_cap is None else min(more, rows_cap - probe)
        if more > 0:
            t1 = time.perf_counter()
            oracle.topo_attn(P, x["q"], x["k"], x["v"], rows=np.arange(probe, probe + more),
                             want=("out",), nthreads=nthreads)
            t_probe += time.perf_counter() - t1
            rows += more
    queries = rows / (w.Hq * w.nq)
    return {"value": queries / t_probe, "unit": "queries/s", "cores": nthreads,
            "kind": "oracle",
            "sample": f"{rows} of the {w.Hq * w.nq} query-head rows of one query "
                      f"({workload_desc(w)}), {t_probe:.2f} s"}


def prefill_oracle_rate(w: synth.Workload, x: dict, budget_s: float):
    """The CPU oracle on a seeded uniform sample of prefill rows; rate in
    scoring TFLOP/s (2 d flops per causal (query, key) pair)."""
    import oracle
    P = oracle.make_params(w.B, w.Hq, w.Hkv, w.d, w.n, w.n, w.W, w.k, w.scale, w.dtype)
    nthreads = oracle.threads()
    rng = np.random.default_rng(20260211)
    total = w.B * w.Hq * w.n
    rows, t, flops = 0, 0.0, 0.0
    batch = max(1, nthreads)
    while t < budget_s and rows < total:
        sel = np.sort(rng.choice(total, size=batch, replace=False))
        t0 = time.perf_counter()
        oracle.topo_attn(P, x["q"], x["k"], x["v"], rows=sel, want=("out",), nthreads=nthreads)
        t += time.perf_counter() - t0
        flops += float((2.0 * w.d * ((sel % w.n) + 1)).sum())
        rows += batch
    return {"value": flops / t / 1e12, "unit": "TFLOP/s", "cores": nthreads, "kind": "oracle",
            "sample": f"{rows} uniformly drawn query-head rows of {workload_desc(w)}, {t:.2f} s"}


def bench_reference(args, w: synth.Workload):
    world, rank, _ = dist_env()
    if rank != 0:
        return
    x = synth.make(w)
    import oracle
    P = oracle.make_params(w.B, w.Hq, w.Hkv, w.d, w.n, w.nq, w.W, w.k, w.scale, w.dtype)
    nthreads = oracle.threads()
    total_rows = w.B * w.Hq * w.nq
    # rows per step so that warmup + steps stay within ~150 s
    t0 = time.perf_counter()
    oracle.topo_attn(P, x["q"], x["k"], x["v"], rows=np.arange(1), want=("out",),
                     nthreads=nthreads)
    t_row = time.perf_counter() - t0
    per_step = max(1, min(total_rows, int(150.0 / max(1, args.steps + args.warmup) /
                                          max(t_row, 1e-9) * min(nthreads, total_rows))))
    per_step = min(per_step, total_rows)
    times = []
    for s in range(args.warmup + args.steps):
        rows = (np.arange(per_step) + s * per_step) % total_rows
        t1 = time.perf_counter()
        oracle.topo_attn(P, x["q"], x["k"], x["v"], rows=rows, want=("out",),
                         nthreads=nthreads)
        if s >= args.warmup:
            times.append(time.perf_counter() - t1)
    t = sum(times)
    value = (per_step * len(times) / (w.Hq * w.nq)) / t
    cpu = {"value": value, "unit": "queries/s", "cores": nthreads, "kind": "oracle",
           "sample": f"{per_step} query-head rows per step of {workload_desc(w)}"}
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": "queries/s",
            "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": 1000.0 * t / len(times), "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64 (float32 ranking score)",
            "data": "synthetic", "config": {"workload": workload_desc(w)},
            "cpu_baseline": cpu,
            "e2e": {"value": value, "unit": "queries/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


# the sources that determine the tensor-core decode kernel and its launch
DECODE_KERNEL_SOURCES = ("topo_tc_kernels.cuh", "topo_kernels.cuh", "topo_device.cuh",
                         "tc_device.cuh", "topo_api.cu")


def kernel_source_hash(files=DECODE_KERNEL_SOURCES) -> str:
    import hashlib
    h = hashlib.sha256()
    for name in files:
        with open(os.path.join(ROOT, "dynamic_sparse_transformer_qk_b300", "csrc", name),
                  "rb") as f:
            h.update(name.encode())
            h.update(f.read())
    return h.hexdigest()


def traffic_from_profile(kernel: str, workload: str):
    """DRAM bytes per launch from the committed ncu summary, only while the
    kernel's sources are the ones the counters were taken on."""
    p = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(p):
        return None
    try:
        with open(p) as f:
            d = json.load(f)
        ent = d.get(kernel, {}).get(workload)
        if ent and ent.get("kernel_source_hash") == kernel_source_hash():
            return float(ent["dram_bytes_per_launch"])
    except Exception:
        return None
    return None


def decode_alg_bytes(w: synth.Workload) -> int:
    """Algorithmic bytes of one decode step: K read once, the 1+W+k V rows of
    C_i per query head, the anchor and window K rows per KV head (logits), q
    in and out."""
    es = 2 if w.dtype == "bf16" else 4
    cset = min(w.n, 1 + w.W + w.k)
    k_bytes = w.B * w.Hkv * w.n * w.d * es
    gather = w.B * w.Hq * cset * w.d * es + w.B * w.Hkv * (1 + w.W) * w.d * es
    io = w.B * w.Hq * w.d * (es + 4)
    return k_bytes + gather + io


def measure_decode(args, w: synth.Workload, dev, rank: int, world: int, local: int, *,
                   steps: int, e2e: bool = True, dense: bool = True,
                   cpu_budget: float = 0.0, x: dict | None = None) -> dict:
    """One decode step per sequence through topo_attn_forward, timed as CUDA
    graph replays with CUDA events; returns the figures of one JSON record."""
    import torch
    import torch.distributed as dist
    import dynamic_sparse_transformer_qk_b300 as topo

    if x is None:
        # every rank serves its own sequences (weak scaling, no data-path collective)
        x = synth.make(rank_workload(w, rank))

    def to_dev(a):
        t = torch.from_numpy(a)
        return (t.view(torch.bfloat16) if w.dtype == "bf16" else t).to(dev)

    q, k, v = to_dev(x["q"]), to_dev(x["k"]), to_dev(x["v"])
    out = torch.empty((w.B, w.Hq, w.nq, w.d), dtype=torch.float32, device=dev)
    ws = topo.Workspace(dev)
    stream = torch.cuda.current_stream(dev)

    def step():
        topo.forward(q, k, v, W=w.W, topk=w.k, n=w.n, scale=w.scale, out=out, workspace=ws)

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    # the timed steps replay one captured step (counter clear + kernel), so the
    # Python binding's per-call host time stays out of the device timing
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        step()
    torch.cuda.synchronize()
    es = 2 if w.dtype == "bf16" else 4
    k_bytes = w.B * w.Hkv * w.n * w.d * es
    l2_flush = k_bytes < 2 * 126 * 2 ** 20
    flush = torch.empty(256 * 2 ** 20, dtype=torch.uint8, device=dev) if l2_flush else None
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
          for _ in range(steps)]
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize()
    with ClockSampler(local) as clk:
        time.sleep(0.3)
        t_wall = time.perf_counter()
        for i in range(steps):
            if flush is not None:
                flush.zero_()  # evict the K cache from L2 between timed steps
            ev[i][0].record(stream)
            graph.replay()
            ev[i][1].record(stream)
        torch.cuda.synchronize()
        t_wall = time.perf_counter() - t_wall
        # keep sampling a moment so short regions still get clock samples
        if t_wall < 0.5 and not args.profile:
            extra = max(1, int(0.5 / max(t_wall / steps, 1e-6)))
            for _ in range(min(extra, 20000)):
                graph.replay()
            torch.cuda.synchronize()
    per = [a.elapsed_time(b) for a, b in ev]
    ms, value = job_rate(sum(per) / len(per), w.B, world)
    queries = w.B * world

    alg_bytes = decode_alg_bytes(w)
    peaks = load_peaks()
    achieved = alg_bytes / (ms / 1000.0) / 1e9
    roofline = {"bound": "hbm", "achieved": achieved, "peak": peaks["hbm_gbs"], "unit": "GB/s",
                "frac": achieved / peaks["hbm_gbs"],
                "peak_source": f"{peaks['source']} (MEASURED_PEAKS.json hbm_gbs)",
                "kernel": "topo_select_tc_kernel",
                "algorithmic_bytes_per_launch": alg_bytes,
                "timing": "CUDA events around each replay of the captured step "
                          "(counter memset, select kernel, dependent tail kernel)",
                "traffic": traffic_from_profile("topo_select_tc_kernel",
                                                "decode-1m" if w.n == 1048576 and w.B == 1
                                                else "none")}
    rec = {"ms_per_step": ms, "value": value, "unit": "queries/s", "roofline": roofline,
           "clocks": clk.summary(), "queries_per_step": queries,
           # per step: the select kernel and its dependent tail kernel
           "gpu_launches": 2 * steps,
           "config": {"workload": workload_desc(w),
                      "l2": (f"K cache {k_bytes / 1e9:.3f} GB < 2x L2: 256 MB write between "
                             "timed steps" if l2_flush else
                             f"K cache {k_bytes / 1e9:.2f} GB per GPU >> 126 MB L2; no flush")}}
    if args.profile:
        return rec
    if e2e:
        # end to end through the public API: pinned host q and the appended K/V
        # row go up, out comes back, every step
        hq = torch.from_numpy(x["q"]).pin_memory()
        hk_row = torch.from_numpy(np.ascontiguousarray(x["k"][:, :, w.n - 1])).pin_memory()
        hv_row = torch.from_numpy(np.ascontiguousarray(x["v"][:, :, w.n - 1])).pin_memory()
        hout = torch.empty_like(out, device="cpu").pin_memory()
        kview = k.view(torch.uint16) if w.dtype == "bf16" else k
        vview = v.view(torch.uint16) if w.dtype == "bf16" else v
        qview = q.view(torch.uint16) if w.dtype == "bf16" else q

        def e2e_step():
            qview.copy_(hq, non_blocking=True)
            kview[:, :, w.n - 1].copy_(hk_row, non_blocking=True)
            vview[:, :, w.n - 1].copy_(hv_row, non_blocking=True)
            step()
            hout.copy_(out, non_blocking=True)

        for _ in range(args.warmup):
            e2e_step()
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        if world > 1:
            dist.barrier()
        e0.record(stream)
        for _ in range(steps):
            e2e_step()
        e1.record(stream)
        torch.cuda.synchronize()
        ems, _ = job_rate(e0.elapsed_time(e1) / steps, w.B, world)
        h2d = hq.numel() * hq.element_size() + 2 * hk_row.numel() * hk_row.element_size()
        d2h = hout.numel() * hout.element_size()
        rec["e2e"] = {"value": queries / (ems / 1000.0), "unit": "queries/s",
                      "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h}
    if dense:
        # the dense (full attention) path on the same cache, for comparison
        dout = torch.empty_like(out)
        dws = topo.Workspace(dev)
        for _ in range(3):
            topo.dense_forward(q, k, v, n=w.n, scale=w.scale, out=dout, workspace=dws)
        torch.cuda.synchronize()
        dgraph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(dgraph):
            topo.dense_forward(q, k, v, n=w.n, scale=w.scale, out=dout, workspace=dws)
        torch.cuda.synchronize()
        nd = max(3, steps // 4)
        dsum = 0.0
        for _ in range(nd):
            if flush is not None:
                flush.zero_()
            d0, d1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            d0.record(stream)
            dgraph.replay()
            d1.record(stream)
            torch.cuda.synchronize()
            dsum += d0.elapsed_time(d1)
        dense_ms = dsum / nd
        dense_bytes = 2 * k_bytes + w.B * w.Hq * w.d * (es + 4)
        rec["dense_attn"] = {"ms_per_step": dense_ms,
                             "gbs": dense_bytes / (dense_ms / 1000.0) / 1e9,
                             "hbm_frac": dense_bytes / (dense_ms / 1000.0) / 1e9
                             / peaks["hbm_gbs"],
                             "sparse_speedup": dense_ms / ms}
    if rank == 0 and world == 1 and cpu_budget > 0:
        rec["cpu_baseline"] = oracle_rate(w, x, budget_s=cpu_budget)
    del q, k, v
    return rec


def measure_layers(args, dev, local: int, *, steps: int, L: int = 32, n: int = 131072,
                   cpu_budget: float = 0.0) -> dict:
    """One decode step through L layers (topo_attn_layers_forward): layer l
    has its own q and its own K/V cache of n tokens (32/8 heads, d=128,
    bf16); pillar layers (every 16th, from layer 0) attend densely, the
    others use windows 256 / 128 / 64 by depth third and k = 32.  Timed as
    CUDA graph replays; beside it, the same step with every layer dense."""
    import torch
    import dynamic_sparse_transformer_qk_b300 as topo

    base = synth.CONFIGS[1].with_(n=n, name=f"decode n={n} bf16 32/8 heads, {L} layers")
    sch = topo.layer_schedule(L, pillar_every=16, windows=(256, 128, 64), topk=32)
    qs, ks, vs = [], [], []
    x0 = None
    for l in range(L):
        x = synth.make(base.with_(seed=base.seed + 101 * (l + 1)))
        if l == 1:
            x0 = x  # a sparse layer's inputs, for the CPU baseline
        qs.append(torch.from_numpy(x["q"]).view(torch.bfloat16).to(dev))
        ks.append(torch.from_numpy(x["k"]).view(torch.bfloat16).to(dev))
        vs.append(torch.from_numpy(x["v"]).view(torch.bfloat16).to(dev))
    outs = [torch.empty((1, base.Hq, 1, base.d), dtype=torch.float32, device=dev)
            for _ in range(L)]
    stream = torch.cuda.current_stream(dev)

    def timed(schedule):
        ws = topo.Workspace(dev)

        def step():
            topo.layers_forward(qs, ks, vs, schedule, n=n, scale=base.scale, outs=outs,
                                workspace=ws)

        for _ in range(args.warmup):
            step()
        torch.cuda.synchronize()
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph):
            step()
        torch.cuda.synchronize()
        ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
              for _ in range(steps)]
        for a, b in ev:
            a.record(stream)
            graph.replay()
            b.record(stream)
        torch.cuda.synchronize()
        return sum(a.elapsed_time(b) for a, b in ev) / steps

    with ClockSampler(local) as clk:
        time.sleep(0.2)
        ms = timed(sch)
        dense_sch = [dict(s, dense=True) for s in sch]
        dense_ms = timed(dense_sch)
    es = 2
    k_bytes = base.Hkv * n * base.d * es
    io = base.Hq * base.d * (es + 4)
    alg = sum(2 * k_bytes + io if s["dense"] else decode_alg_bytes(base.with_(W=s["W"], k=s["topk"]))
              for s in sch)
    peaks = load_peaks()
    achieved = alg / (ms / 1000.0) / 1e9
    rec = {"ms_per_step": ms, "value": 1000.0 / ms, "unit": "queries/s",
           "roofline": {"bound": "hbm", "achieved": achieved, "peak": peaks["hbm_gbs"],
                        "unit": "GB/s", "frac": achieved / peaks["hbm_gbs"],
                        "peak_source": f"{peaks['source']} (MEASURED_PEAKS.json hbm_gbs)",
                        "algorithmic_bytes_per_step": alg,
                        "kernel": "topo_select_tc_kernel (sparse layers) + dense_tc_kernel (pillars)",
                        "timing": f"CUDA events around each replay of the captured {L}-layer step",
                        "traffic": None},
           "all_dense_ms_per_step": dense_ms, "pillar_speedup_vs_all_dense": dense_ms / ms,
           "clocks": clk.summary(),
           # per step: select + tail kernels per sparse layer, one dense kernel per pillar
           "gpu_launches": sum(1 if s["dense"] else 2 for s in sch) * steps,
           "config": {"workload": f"{L} layers x (decode n={n}, 32/8 heads, d=128, bf16); "
                                  "pillars (dense) at layers 0 and 16; W 256/128/64 by depth "
                                  "third; k=32; every layer its own seeded q, K, V",
                      "schedule": [("dense" if s["dense"] else f"W{s['W']}") for s in sch],
                      "l2": f"{2 * k_bytes * L / 1e9:.1f} GB of K/V >> 126 MB L2; no flush"}}
    if cpu_budget > 0:
        # the oracle on one sparse layer's rows, scaled to the whole step (the
        # dense layers cost about as much per row as the sparse ones there)
        r = oracle_rate(base.with_(W=sch[1]["W"]), x0, budget_s=cpu_budget)
        rec["cpu_baseline"] = dict(r, value=r["value"] / L,
                                   sample=r["sample"] + f"; scaled to {L} layers per query")
    del qs, ks, vs
    return rec


def bench_ours(args, w: synth.Workload):
    import torch
    import torch.distributed as dist

    world, rank, local = dist_env()
    if world > 1:
        dist.init_process_group("gloo", init_method="env://")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    rec = measure_decode(args, w, dev, rank, world, local, steps=args.steps,
                         dense=args.dense and not args.profile,
                         cpu_budget=0.0 if args.no_cpu_baseline else args.cpu_budget)
    if args.profile:
        if rank == 0:
            print(json.dumps({"profile": True, "ms_per_step": rec["ms_per_step"],
                              "value": rec["value"], "workload": workload_desc(w)}), flush=True)
        return
    subs = []
    if world == 1 and args.workloads:
        # the other workloads of the benchmark, one sub-record each (same
        # rules: inputs resident in HBM, CUDA events, clocks sampled)
        sub_steps = max(3, min(args.steps, 10))
        bcfg = synth.CONFIGS[2]
        r = measure_decode(args, bcfg, dev, rank, world, local, steps=args.steps, e2e=True,
                           dense=True, cpu_budget=0.0 if args.no_cpu_baseline else 5.0)
        subs.append(dict(name="decode-128k-b16", metric=METRIC, **r))
        torch.cuda.empty_cache()
        r = measure_decode(args, synth.CONFIGS[1], dev, rank, world, local, steps=args.steps,
                           e2e=True, dense=True,
                           cpu_budget=0.0 if args.no_cpu_baseline else 5.0)
        subs.append(dict(name="decode-32k", metric=METRIC, **r))
        torch.cuda.empty_cache()
        r = measure_layers(args, dev, local, steps=sub_steps,
                           cpu_budget=0.0 if args.no_cpu_baseline else 5.0)
        subs.append(dict(name="decode-32-layers-128k", metric=METRIC, **r))
        torch.cuda.empty_cache()
        px = synth.make(synth.CONFIGS[3])
        for W in synth.PREFILL_WINDOWS:
            wp = synth.CONFIGS[3].with_(W=W)
            r = measure_prefill(args, wp, dev, local, steps=sub_steps, x=px, e2e=False,
                                cpu_budget=0.0 if args.no_cpu_baseline else 5.0)
            subs.append(dict(name=f"prefill-64k-W{W}", metric=PREFILL_METRIC, **r))
            torch.cuda.empty_cache()
        del px
    if rank != 0:
        if world > 1:
            dist.barrier()
        return
    line = {
        "metric": METRIC, "value": rec["value"], "unit": "queries/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": rec["ms_per_step"],
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16"
        if w.dtype == "bf16" else "f32",
        "data": "synthetic: seeded N(0,1) Q/K/V, Q+=3u, sink K[0]+=6u, "
                f"{w.planted} planted keys per KV head",
        "config": dict(rec["config"], queries_per_step=rec["queries_per_step"],
                       timed_outputs="out only (idx and excluded mass off the timed path)"),
        "hbm_gbs": rec["roofline"]["achieved"], "hbm_frac_of_peak": rec["roofline"]["frac"],
        "roofline": rec["roofline"], "e2e": rec.get("e2e"), "clocks": rec["clocks"],
        "gpu_launches": rec["gpu_launches"], "cpu_baseline": rec.get("cpu_baseline"),
    }
    if "dense_attn" in rec:
        line["dense_attn"] = rec["dense_attn"]
    if subs:
        line["workloads"] = subs
    elif world > 1:
        line["workloads_note"] = "sub-workloads are measured at N=1 only"
    print(json.dumps(line), flush=True)
    if world > 1:
        dist.barrier()


def measure_prefill(args, w: synth.Workload, dev, local: int, *, steps: int,
                    x: dict | None = None, e2e: bool = True, cpu_budget: float = 0.0) -> dict:
    """Chunked causal prefill (n=65536, chunks of 4096 rows): one step = the
    whole sequence through topo_attn_score_select (the scored value) and
    through topo_attn_forward (reported beside it), chunk by chunk."""
    import torch
    import dynamic_sparse_transformer_qk_b300 as topo

    if x is None:
        x = synth.make(w)

    def to_dev(a):
        return torch.from_numpy(a).view(torch.bfloat16).to(dev)

    q, k, v = to_dev(x["q"]), to_dev(x["k"]), to_dev(x["v"])
    chunk = w.chunk
    nch = w.n // chunk
    qs = [q[:, :, c * chunk:(c + 1) * chunk].contiguous() for c in range(nch)]
    out = torch.empty((w.B, w.Hq, w.n, w.d), dtype=torch.float32, device=dev)
    outs = [out[:, :, c * chunk:(c + 1) * chunk] for c in range(nch)]
    obufs = [torch.empty((w.B, w.Hq, chunk, w.d), dtype=torch.float32, device=dev)
             for _ in range(nch)]
    idxs = [torch.empty((w.B, w.Hq, chunk, 1 + w.W + w.k), dtype=torch.int32, device=dev)
            for _ in range(nch)]
    ws = topo.Workspace(dev)
    stream = torch.cuda.current_stream(dev)

    def step():
        for c in range(nch):
            topo.forward(qs[c], k, v, W=w.W, topk=w.k, n=(c + 1) * chunk, scale=w.scale,
                         out=obufs[c], workspace=ws)

    def select_step():
        for c in range(nch):
            topo.score_select(qs[c], k, W=w.W, topk=w.k, n=(c + 1) * chunk, scale=w.scale,
                              idx=idxs[c], workspace=ws)

    if args.profile:
        # profiling: the last chunk call alone (warm-up calls, then `steps` calls)
        c = nch - 1
        for _ in range(args.warmup + steps):
            topo.forward(qs[c], k, v, W=w.W, topk=w.k, n=(c + 1) * chunk, scale=w.scale,
                         out=obufs[c], workspace=ws)
        torch.cuda.synchronize()
        return {"profile": True, "workload": workload_desc(w), "chunk_call": c}

    def timed(fn, nsteps):
        for _ in range(args.warmup):
            fn()
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for _ in range(nsteps):
            fn()
        e1.record(stream)
        torch.cuda.synchronize()
        return e0.elapsed_time(e1) / nsteps

    with ClockSampler(local) as clk:
        ms = timed(step, steps)
        sel_ms = timed(select_step, steps)
    flops = 2.0 * w.Hq * w.d * (w.n * (w.n + 1) / 2.0) * w.B
    peaks = load_peaks()
    value = flops / (sel_ms / 1000.0) / 1e12
    roofline = {"bound": "tensor", "achieved": value, "peak": peaks["bf16_tflops"],
                "unit": "TFLOP/s", "frac": value / peaks["bf16_tflops"],
                "peak_source": f"{peaks['source']} (MEASURED_PEAKS.json bf16_tflops, burst)",
                "kernel": "prefill_scan_kernel (+ K-scale and exact-rescoring finalize)",
                "algorithmic_flops_per_step": flops,
                "timing": f"CUDA events around {nch} topo_attn_score_select chunk calls",
                "traffic": None}
    rec = {"ms_per_step": sel_ms, "value": value, "unit": "TFLOP/s", "roofline": roofline,
           "forward_ms_per_sequence": ms, "clocks": clk.summary(),
           "gpu_launches": 3 * nch * steps,
           "config": {"workload": workload_desc(w), "chunk": chunk,
                      "l2": "K cache 134 MB per chunk call > 126 MB L2; no flush"}}
    if e2e:
        # end to end: the sequence's q, k, v go up from pinned host memory, out comes back
        hq = torch.from_numpy(x["q"]).pin_memory()
        hk = torch.from_numpy(x["k"]).pin_memory()
        hv = torch.from_numpy(x["v"]).pin_memory()
        hout = torch.empty(out.shape, dtype=torch.float32).pin_memory()
        qv, kv_, vv = q.view(torch.uint16), k.view(torch.uint16), v.view(torch.uint16)

        def e2e_step():
            qv.copy_(hq, non_blocking=True)
            kv_.copy_(hk, non_blocking=True)
            vv.copy_(hv, non_blocking=True)
            for c in range(nch):
                qs[c].copy_(q[:, :, c * chunk:(c + 1) * chunk])
                topo.forward(qs[c], k, v, W=w.W, topk=w.k, n=(c + 1) * chunk, scale=w.scale,
                             out=outs[c], workspace=ws)
            hout.copy_(out, non_blocking=True)

        e2e_ms = timed(e2e_step, max(1, steps // 2))
        h2d = sum(t.numel() * t.element_size() for t in (hq, hk, hv))
        d2h = hout.numel() * hout.element_size()
        rec["e2e"] = {"value": flops / (e2e_ms / 1000.0) / 1e12, "unit": "TFLOP/s",
                      "ms_per_step": e2e_ms, "h2d_bytes_per_step": h2d,
                      "d2h_bytes_per_step": d2h}
    if cpu_budget > 0:
        rec["cpu_baseline"] = prefill_oracle_rate(w, x, budget_s=cpu_budget)
    return rec


def bench_prefill(args, w: synth.Workload):
    """The chunked prefill as the headline line (--workload prefill-64k)."""
    import torch

    world, rank, local = dist_env()
    if rank != 0:
        return
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    rec = measure_prefill(args, w, dev, local, steps=args.steps,
                          cpu_budget=0.0 if args.no_cpu_baseline else args.cpu_budget)
    if rec.get("profile"):
        print(json.dumps(rec), flush=True)
        return
    line = {
        "metric": PREFILL_METRIC, "value": rec["value"], "unit": "TFLOP/s", "n_gpus": 1,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": rec["ms_per_step"],
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic: seeded N(0,1) Q/K/V, Q+=3u, sink K[0]+=6u, "
                f"{w.planted} planted keys per KV head",
        "config": rec["config"], "forward_ms_per_sequence": rec["forward_ms_per_sequence"],
        "roofline": rec["roofline"], "clocks": rec["clocks"], "e2e": rec.get("e2e"),
        "gpu_launches": rec["gpu_launches"], "cpu_baseline": rec.get("cpu_baseline"),
    }
    print(json.dumps(line), flush=True)


def eps_report(args):
    """The pages' exactness argument rests on the dense-softmax mass left out of
    C_i being below the float32 ULP.  Per workload: that excluded mass eps
    (GPU, every row; sampled rows for the 64K prefill), and on oracle-sampled
    rows the largest excluded weight against 2^-23 and the anchor's weight."""
    import torch
    import oracle
    import dynamic_sparse_transformer_qk_b300 as topo
    rng = np.random.default_rng(20260211)
    cases = [(i, synth.CONFIGS[i]) for i in (0, 1, 2, 4)]
    cases += [(3, synth.CONFIGS[3].with_(W=W)) for W in synth.PREFILL_WINDOWS]
    for cid, w in cases:
        x = synth.make(w)

        def dev(a):
            t = torch.from_numpy(a)
            return (t.view(torch.bfloat16) if w.dtype == "bf16" else t).cuda()

        q, k, v = dev(x["q"]), dev(x["k"]), dev(x["v"])
        nrows = w.B * w.Hq * w.nq
        if cid == 3:
            # last chunk of the chunked prefill (rows 61,440..65,535)
            c = w.n // w.chunk - 1
            qc = q[:, :, c * w.chunk:].contiguous()
            _, _, excl = topo.forward(qc, k, v, W=w.W, topk=w.k, n=w.n, scale=w.scale,
                                      want_excl=True)
            flat = np.arange(nrows).reshape(w.B, w.Hq, w.nq)[:, :, c * w.chunk:].reshape(-1)
            gexcl = excl.cpu().numpy().reshape(-1).astype(np.float64)
            sample = np.sort(rng.choice(flat, size=64, replace=False))
        else:
            _, _, excl = topo.forward(q, k, v, W=w.W, topk=w.k, n=w.n, scale=w.scale,
                                      want_excl=True)
            gexcl = excl.cpu().numpy().reshape(-1).astype(np.float64)
            sample = np.sort(rng.choice(nrows, size=min(nrows, 256), replace=False))
        torch.cuda.synchronize()
        P = oracle.make_params(w.B, w.Hq, w.Hkv, w.d, w.n, w.nq, w.W, w.k, w.scale, w.dtype)
        o = oracle.topo_attn(P, x["q"], x["k"], x["v"], rows=sample, want=("excl", "wmax", "p0"))
        ulp, half = 2.0 ** -23, 2.0 ** -24
        line = {
            "workload": workload_desc(w), "rows": int(gexcl.size),
            "eps_median": float(np.median(gexcl)), "eps_max": float(gexcl.max()),
            "eps_below_half_ulp_frac": float((gexcl < half).mean()),
            "oracle_rows": int(sample.size),
            "wmax_over_ulp_median": float(np.median(o["wmax"] / ulp)),
            "wmax_over_ulp_max": float(o["wmax"].max() / ulp),
            "wmax_below_ulp_frac": float((o["wmax"] < ulp).mean()),
            "anchor_weight_median": float(np.median(o["p0"])),
        }
        print(json.dumps(line), flush=True)


def main():
    ap = argparse.ArgumentParser(description=__doc__)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=100)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", choices=sorted(WORKLOADS), default="decode-1m")
    ap.add_argument("--no-dense", dest="dense", action="store_false")
    ap.add_argument("--no-workloads", dest="workloads", action="store_false",
                    help="headline decode line only (no batched-decode and prefill sub-records)")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-budget", type=float, default=15.0)
    ap.add_argument("--n", type=int, default=0,
                    help="override the causal length (profiling runs on smaller caches)")
    ap.add_argument("--profile", action="store_true",
                    help="time the steps only: no e2e, dense, clock padding or CPU baseline")
    ap.add_argument("--eps-report", action="store_true",
                    help="report the excluded softmax mass against the float32 ULP per workload")
    ap.add_argument("--window", type=int, default=0,
                    help="window W of the prefill workload (256, 128 or 64; default 256)")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be at least 3")
    if args.eps_report:
        eps_report(args)
        return
    w = synth.CONFIGS[WORKLOADS[args.workload]]
    if args.n:
        w = w.with_(n=args.n, name=f"{w.name} (n overridden to {args.n})")
    if args.profile or args.n:
        args.workloads = False
    if args.profile:
        args.dense = False
        args.no_cpu_baseline = True
    if WORKLOADS[args.workload] == 3:
        w = w.with_(W=args.window or 256)
        if args.impl == "reference":
            world, rank, _ = dist_env()
            if rank == 0:
                x = synth.make(w)
                per = max(2.0, 120.0 / max(1, args.steps + args.warmup))
                rates = [prefill_oracle_rate(w, x, budget_s=per)
                         for _ in range(args.warmup + args.steps)][args.warmup:]
                value = sum(r["value"] for r in rates) / len(rates)
                cpu = dict(rates[-1], value=value)
                print(json.dumps({
                    "impl": "reference", "metric": PREFILL_METRIC, "value": value,
                    "unit": "TFLOP/s", "n_gpus": world, "steps": args.steps,
                    "warmup": args.warmup, "ms_per_step": None, "higher_is_better": True,
                    "scaling": "weak", "vs_baseline": None,
                    "dtype": "f64 (float32 ranking score)", "data": "synthetic",
                    "config": {"workload": workload_desc(w)}, "cpu_baseline": cpu,
                    "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0,
                            "d2h_bytes_per_step": 0}}), flush=True)
        else:
            bench_prefill(args, w)
        return
    if args.impl == "reference":
        bench_reference(args, w)
    else:
        bench_ours(args, w)


if __name__ == "__main__":
    main()
