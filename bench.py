#!/usr/bin/env python
"""Benchmark of the expert-slot-cache MoE decode step on GB300.

Workload: Qwen3-30B-A3B-shaped decode (48 MoE layers, 128 experts, top-8,
hidden 2048, expert intermediate 768, bf16 weights, batch 1), cache of 37% of
the 6144 (layer, expert) slots, Zipf(1.1) routing with 80% step-to-step reuse.
One bench step = one decode token through all 48 MoE layers: per layer the
control kernel, the slot fills on the side stream, the grouped SwiGLU GEMV
over resident and filled experts, and the combine with supplied CPU partial
sums.  Metric: MoE-layer decode steps per second (48 per bench step).

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

Under torchrun each rank runs an independent replica on its own GPU (the path
has no exchange step on one node: replicas only), the timed region is bracketed
by barriers, and rank 0 prints one JSON line with the max time over ranks.
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402

from workloads import (activations, config, default_max_fetch, make_blob, make_pool,  # noqa: E402
                       prefill_routing, routing_trace)

WORKLOAD = "qwen3_decode_b1"
METRIC = "MoE-layer decode steps/s"
UNIT = "layer-steps/s"
# DRAM bytes (read + write) of the resident-expert GEMV pair per layer-step, from
# one ncu capture of both grids (cache control off, all-resident layers of the
# qwen3 b1 shape, 8 resident experts each: the same work per layer-step as the
# roofline replay); see profiles/decode_gemv_pair_qwen3_b1.md.
TRAFFIC_PER_LAYER_STEP = 75_280_000
TRAFFIC_SOURCE = ("ncu dram__bytes_read.sum + dram__bytes_write.sum of the gate/up and down grids of one "
                  "layer-step, mean of 4 all-resident layer-steps of bench.py --mode profile-decode "
                  "(16-layer qwen3 b1 shape, 8 resident experts per layer); profiles/decode_gemv_pair_qwen3_b1.md")
# the same for the fused resident launch (MOE_DECODE_FUSED=1): one ncu capture of
# the launch, mean of 8 all-resident layer-steps; profiles/decode_fused_resident_qwen3_b1.md
FUSED_TRAFFIC_PER_LAYER_STEP = 80_870_000
FUSED_TRAFFIC_SOURCE = ("ncu dram__bytes_read.sum + dram__bytes_write.sum of the fused resident launch, mean of 8 "
                        "all-resident layer-steps of MOE_DECODE_FUSED=1 bench.py --mode profile-decode (16-layer "
                        "qwen3 b1 shape, 8 resident experts per layer); profiles/decode_fused_resident_qwen3_b1.md")


def parse_args(argv=None):
    p = argparse.ArgumentParser()
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=256)
    p.add_argument("--warmup", type=int, default=8)
    p.add_argument("--impl", default="ours", choices=["ours", "reference"])
    p.add_argument("--pool-blobs", type=int, default=64, help="distinct expert blobs in the host arena")
    p.add_argument("--no-graph", action="store_true", help="launch eagerly instead of replaying a CUDA graph")
    p.add_argument("--cpu-seconds", type=float, default=15.0, help="budget of the oracle CPU baseline")
    p.add_argument("--no-cpu-baseline", action="store_true")
    p.add_argument("--no-prefill", action="store_true")
    p.add_argument("--no-nvfp4", action="store_true",
                   help="skip the 4-bit-expert variants (NVFP4, MXFP4) of the decode workload")
    p.add_argument("--mode", default="all", choices=["all", "decode", "prefill", "profile-decode"],
                   help="prefill: only the prefill measurement (small profiling runs)")
    p.add_argument("--prefill-tokens", type=int, default=8192)
    p.add_argument("--no-prefill-ablation", action="store_true",
                   help="skip the prefill chunks without the second buffer (4k / 8k / 16k tokens)")
    p.add_argument("--capacity", type=int, default=0, help="override the slot count (small profiling runs)")
    p.add_argument("--profile-layers", type=int, default=16, help="profile-decode: MoE layers of the small case")
    p.add_argument("--profile-allhit", action="store_true",
                   help="profile-decode: replay one step so every routed expert is resident after the first")
    p.add_argument("--cpu-worker", action="store_true", help=argparse.SUPPRESS)
    p.add_argument("--cpu-samples", type=int, default=1, help=argparse.SUPPRESS)
    p.add_argument("--ref-seconds", type=float, default=0.0,
                   help="reference arm: oracle seconds per bench step (0: fit the run into about two minutes)")
    return p.parse_args(argv)


# ----------------------------------------------------------------------------
# measured peaks and clocks
# ----------------------------------------------------------------------------
def measured_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as fh:
            d = json.load(fh)
        hbm = d.get("hbm_gbs") or d.get("hbm_GBs")
        bf16 = d.get("bf16_tflops")
        bf16_s = d.get("bf16_tflops_sustained", bf16)
        if hbm:
            return float(hbm), float(bf16 or 1900.0), float(bf16_s or 1700.0), "of measured"
    return 6800.0, 1900.0, 1700.0, "of fallback"


class ClockSampler:
    """nvidia-smi clock / throttle sampling while the timed region runs."""

    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, device_index: int):
        self.dev = device_index
        self.proc = None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(["nvidia-smi", f"--id={self.dev}", f"--query-gpu={self.QUERY}",
                                          "--format=csv,noheader,nounits", "-lms", "200"],
                                         stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
        return self

    def __exit__(self, *a):
        self.lines = []
        if self.proc is not None:
            time.sleep(0.25)
            self.proc.terminate()
            try:
                out, _ = self.proc.communicate(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
                out, _ = self.proc.communicate()
            self.lines = [l for l in out.splitlines() if l.strip()]

    def summary(self):
        sm, mx, reasons = [], 0, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for l in getattr(self, "lines", []):
            f = [x.strip() for x in l.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                mx = max(mx, float(f[2]))
            except ValueError:
                continue
            for n, v in zip(names, f[5:9]):
                if v.lower() == "active":
                    reasons.add(n)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"], "samples": 0}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": mx, "reasons": sorted(reasons),
                "samples": len(sm)}


# ----------------------------------------------------------------------------
# the oracle as CPU baseline (runs in a fresh interpreter: no fork after CUDA init)
# ----------------------------------------------------------------------------
def cpu_worker(seconds: float, pool_blobs: int, bw, samples: int = 1):
    """Oracle control + float64 SwiGLU on successive layer-steps of the workload.

    Prints one JSON line per sample; each sample runs until `seconds` of oracle
    time are spent.  Generating the synthetic expert blobs (input synthesis) is
    not counted; parsing them to float64 is (the oracle reads its weights).
    """
    from oracle.cache import SlotCache
    from oracle.ffn import combine, swiglu_expert
    from oracle.formats import activations_to_f64, parse_blob
    cfg = config(WORKLOAD)
    s = cfg.shape
    ids, w = routing_trace(cfg)
    K = default_max_fetch(s, cfg.T)
    ora = SlotCache(s.L, s.E, cfg.capacity, K, bw[0], bw[1])
    raw = {}
    st, l = 0, 0
    for _ in range(samples):
        spent, n = 0.0, 0
        while spent < seconds:
            sid = st % cfg.steps
            need = {(l * s.E + int(e)) % pool_blobs for e in ids[sid, l].ravel()}
            for p in need - raw.keys():
                raw[p] = make_blob(s, cfg.seed, p)          # input synthesis, not timed
            xs = activations(cfg, sid, l)
            t0 = time.perf_counter()
            plan = ora.decode(l, ids[sid, l])
            x = activations_to_f64(xs, s.adtype)
            y = np.zeros((cfg.T, s.k, s.H))
            for t in range(cfg.T):
                for j in range(s.k):
                    p = (l * s.E + int(ids[sid, l, t, j])) % pool_blobs
                    y[t, j] = swiglu_expert(x[t], *parse_blob(raw[p], s.wdtype, s.H, s.I))
            combine(w[sid, l], y, plan.slot_map, y)
            spent += time.perf_counter() - t0
            n += 1
            l += 1
            if l == s.L:
                l, st = 0, st + 1
        print(json.dumps({"layer_steps": n, "seconds": spent}), flush=True)


def run_cpu_baseline(seconds: float, pool_blobs: int, bw, samples: int = 1):
    """Run the oracle in a fresh interpreter (no fork after CUDA init); one dict per sample."""
    env = dict(os.environ, OMP_NUM_THREADS="1", OPENBLAS_NUM_THREADS="1", MKL_NUM_THREADS="1")
    cmd = [sys.executable, os.path.abspath(__file__), "--cpu-worker", "--cpu-seconds", str(seconds),
           "--pool-blobs", str(pool_blobs), "--cpu-samples", str(samples)]
    env["BENCH_BW"] = f"{bw[0]},{bw[1]}"
    r = subprocess.run(cmd, capture_output=True, text=True, env=env, timeout=samples * (seconds * 4 + 60) + 120)
    lines = [json.loads(l) for l in r.stdout.splitlines() if l.startswith("{")]
    if r.returncode != 0 or not lines:
        return None
    out = []
    for d in lines:
        out.append({"value": d["layer_steps"] / d["seconds"], "unit": UNIT, "cores": 1, "kind": "oracle",
                    "sample": f"{d['layer_steps']} layer-steps of {WORKLOAD} (list-LRU control + float64 SwiGLU "
                              f"per routed pair from the host pool + fixed-order combine), one thread, "
                              f"{d['seconds']:.1f} s of oracle time"})
    return out if samples > 1 else out[0]


# ----------------------------------------------------------------------------
# GPU arm
# ----------------------------------------------------------------------------
def main(args):
    import torch
    import torch.distributed as dist

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        dist.init_process_group("nccl" if args.impl == "ours" else "gloo")
    if args.impl == "reference":
        return reference_arm(args, world, rank)
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    if args.mode == "prefill":
        if rank == 0:
            print(json.dumps({"prefill": prefill_measure(args, dev, local)}))
        return
    if args.mode == "profile-decode":
        return profile_case(args, dev)

    from serving_layer_moe_gb300 import MoECache, bench_bw

    cfg = config(WORKLOAD)
    if args.capacity:
        cfg = cfg.with_(capacity=args.capacity)
    s = cfg.shape
    # calibration: B_P through the fill path, B_H host read; B_cpu = residual
    bp_gbs, bh_gbs, rec = bench_bw(local, s.blob_bytes)
    b_pcie = max(1, int(bp_gbs * 1000))
    b_cpu = max(0, int(bh_gbs * 1000) - b_pcie)

    arena, offs = make_pool(s, cfg.seed, n_phys=args.pool_blobs)
    pool = torch.from_numpy(arena).pin_memory()
    del arena
    K = default_max_fetch(s, cfg.T)
    cache = MoECache(L=s.L, E=s.E, H=s.H, I=s.I, top_k=s.k, max_tokens=cfg.T, wdtype=s.wdtype,
                     adtype=s.adtype, host_pool=pool, blob_offsets=offs, n_slots=cfg.capacity,
                     max_fetch=K, bw_pcie_mbps=b_pcie, bw_cpu_mbps=b_cpu, device=local)

    ids, w = routing_trace(cfg)
    xs = np.stack([np.stack([activations(cfg, st, l) for l in range(s.L)]) for st in range(cfg.steps)])
    x_all = torch.from_numpy(xs.view(np.int16)).to(dev)            # [steps, L, T, H] bf16 bits
    ids_all = torch.from_numpy(ids).to(dev)                         # [steps, L, T, k]
    w_all = torch.from_numpy(w).to(dev)
    xb = torch.empty_like(x_all[0])
    ib = torch.empty_like(ids_all[0])
    wb = torch.empty_like(w_all[0])
    out = torch.empty(s.L, cfg.T, s.H, dtype=torch.float32, device=dev)
    cpu_part = torch.zeros(cfg.T, s.k, s.H, dtype=torch.float32, device=dev)
    stream = torch.cuda.Stream(device=dev)
    sp = stream.cuda_stream
    layer_bytes = [(xb[l].data_ptr(), ib[l].data_ptr(), wb[l].data_ptr(), out[l].data_ptr()) for l in range(s.L)]

    def enqueue_step():
        for l in range(s.L):
            xp, ip, wp, op = layer_bytes[l]
            cache.decode_ptrs(l, cfg.T, xp, ip, wp, cpu_part.data_ptr(), op, None, sp)

    def stage(st):
        xb.copy_(x_all[st % cfg.steps], non_blocking=True)
        ib.copy_(ids_all[st % cfg.steps], non_blocking=True)
        wb.copy_(w_all[st % cfg.steps], non_blocking=True)

    step = 0
    with torch.cuda.stream(stream):
        for _ in range(args.warmup):
            stage(step)
            enqueue_step()
            step += 1
    torch.cuda.synchronize(dev)
    graph = None
    if not args.no_graph:
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph, stream=stream):
            enqueue_step()
        torch.cuda.synchronize(dev)

    # control, fill (+ the filled experts' gate/up), the filled experts' down grid and
    # the resident experts' kernels (one launch, or a gate/up grid and a down +
    # combine grid), as the library reports
    launches_per_layer = int(cache.info()[6])
    resident_path = int(cache.info()[7])   # 0: two grids, 1: one launch with a grid barrier
    # ---- timed region: inputs resident in HBM ---------------------------------
    cnt0 = cache.state()[3].copy()
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize(dev)
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    with ClockSampler(local) as clk, torch.cuda.stream(stream):
        e0.record(stream)
        for _ in range(args.steps):
            stage(step)
            if graph is not None:
                graph.replay()
            else:
                enqueue_step()
            step += 1
        e1.record(stream)
        torch.cuda.synchronize(dev)
    ms = e0.elapsed_time(e1)
    if world > 1:
        t = torch.tensor([ms], device=dev)
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
        ms = float(t.item())
        dist.barrier()
    cnt1 = cache.state()[3].copy()
    layer_steps = args.steps * s.L * world
    value = layer_steps / (ms / 1e3)

    # ---- end to end: host buffers in, result out, every step ------------------------
    x_h = torch.from_numpy(xs.view(np.int16)).pin_memory()
    ids_h = torch.from_numpy(ids).pin_memory()
    w_h = torch.from_numpy(w).pin_memory()
    out_h = torch.empty(s.L, cfg.T, s.H, dtype=torch.float32).pin_memory()
    e2e_steps = max(8, args.steps // 2)
    torch.cuda.synchronize(dev)
    if world > 1:
        dist.barrier()
    e2 = torch.cuda.Event(enable_timing=True)
    e3 = torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(stream):
        e2.record(stream)
        for _ in range(e2e_steps):
            st = step % cfg.steps
            xb.copy_(x_h[st], non_blocking=True)
            ib.copy_(ids_h[st], non_blocking=True)
            wb.copy_(w_h[st], non_blocking=True)
            if graph is not None:
                graph.replay()
            else:
                enqueue_step()
            out_h.copy_(out, non_blocking=True)
            step += 1
        e3.record(stream)
        torch.cuda.synchronize(dev)
    ms_e2e = e2.elapsed_time(e3)
    if world > 1:
        t = torch.tensor([ms_e2e], device=dev)
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
        ms_e2e = float(t.item())
    h2d = xb.numel() * 2 + ib.numel() * 4 + wb.numel() * 4
    d2h = out.numel() * 4

    # ---- kernel timing for the roofline: library CUDA events captured into a graph ----
    # (a second graph of the same step with an event pair around each kernel group;
    # after each replay the pairs hold that replay's device times)
    prof_steps = 32
    cache.profile_start()
    pgraph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(pgraph, stream=stream):
        enqueue_step()
    cache.profile_pause()
    torch.cuda.synchronize(dev)
    cnt_p0 = cache.state()[3].copy()
    prof = {k: [0.0, 0] for k in cache.PROFILE_KINDS}
    with torch.cuda.stream(stream):
        for _ in range(prof_steps):
            stage(step)
            pgraph.replay()
            step += 1
            for k, (ms_k, n_k) in cache.profile_read().items():
                prof[k][0] += ms_k
                prof[k][1] += n_k
    cnt_p1 = cache.state()[3].copy()
    # ---- roofline of the dominant HBM kernels, the resident-expert GEMV pair
    # (gate/up grid, which also has L2 fetch the experts' W_down, then the down +
    # combine grid), with nothing beside them: one step's inputs are replayed
    # until every routed expert is resident (all hits, no fill), then the same
    # event pairs time the two grids on their stream.  Algorithmic bytes: each
    # resident expert's whole blob, read once.
    res_reps = 16
    with torch.cuda.stream(stream):
        stage(step)
        for _ in range(3):
            pgraph.replay()
            cache.profile_read()
    torch.cuda.synchronize(dev)
    cnt_r0 = cache.state()[3].copy()
    res_prof = {k: [0.0, 0] for k in cache.PROFILE_KINDS}
    with torch.cuda.stream(stream):
        for _ in range(res_reps):
            pgraph.replay()
            for k, (ms_k, n_k) in cache.profile_read().items():
                res_prof[k][0] += ms_k
                res_prof[k][1] += n_k
    cnt_r1 = cache.state()[3].copy()
    cache.profile_stop()
    e4 = torch.cuda.Event(enable_timing=True)
    e5 = torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(stream):   # the same all-hit step without event pairs: whole-layer time
        e4.record(stream)
        for _ in range(res_reps):
            if graph is not None:
                graph.replay()
            else:
                enqueue_step()
        e5.record(stream)
    torch.cuda.synchronize(dev)
    ms_res = e4.elapsed_time(e5)
    step += 1
    hbm_peak, bf16_peak, bf16_sust, peak_src = measured_peaks()
    res_hits = int(cnt_r1[0] - cnt_r0[0])
    res_fills = int(cnt_r1[2] - cnt_r0[2])
    gemv_kinds = ("gemv_resident", "down_combine")   # split: the pair is one group; down_combine stays 0
    res_ms = sum(res_prof[k][0] for k in gemv_kinds)
    res_launches = res_prof["gemv_resident"][1]
    res_bytes = res_hits * s.blob_bytes
    res_gbs = res_bytes / (res_ms / 1e3) / 1e9 if res_ms > 0 else None
    # the same pair inside the timed step's mix (concurrent fills, event pairs in the graph)
    resident = int(cnt_p1[0] - cnt_p0[0])
    gemv_bytes = resident * s.blob_bytes
    gemv_ms = sum(prof[k][0] for k in gemv_kinds)
    gemv_launches = prof["gemv_resident"][1]         # one per MoE-layer decode
    fill_bytes = int(cnt_p1[2] - cnt_p0[2]) * s.blob_bytes
    total_prof_ms = sum(v[0] for v in prof.values())
    # Distribution of whole MoE-layer decode times (median, p90), after the timed
    # region: eager calls, one event pair around each layer's call on its stream,
    # fills included where they occur.  Reported beside the means; a failure here
    # leaves the rest of the line intact.
    try:
        lat_steps = 8
        lat_ev = [[(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
                   for _ in range(s.L)] for _ in range(lat_steps)]
        with torch.cuda.stream(stream):
            for st_i in range(lat_steps):
                stage(step)
                step += 1
                for l in range(s.L):
                    xp, ip, wp, op = layer_bytes[l]
                    lat_ev[st_i][l][0].record(stream)
                    cache.decode_ptrs(l, cfg.T, xp, ip, wp, cpu_part.data_ptr(), op, None, sp)
                    lat_ev[st_i][l][1].record(stream)
        torch.cuda.synchronize(dev)
        lat_us = np.array([1e3 * a.elapsed_time(b) for row in lat_ev for a, b in row])
        layer_step_us = {"median": round(float(np.median(lat_us)), 2),
                         "p90": round(float(np.percentile(lat_us, 90)), 2),
                         "mean": round(float(lat_us.mean()), 2), "n": int(lat_us.size),
                         "note": "eager calls after the timed region, an event pair around each MoE-layer "
                                 "decode (launch gaps included, so above the graph-replayed mean)"}
    except Exception as exc:   # diagnostics only
        layer_step_us = {"error": repr(exc)[:200]}

    result = {
        "metric": METRIC, "value": round(value, 1), "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(ms / args.steps, 4), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": {"workload": f"{WORKLOAD}: Qwen3-30B-A3B-shaped decode, 48 MoE layers x 128 experts, "
                               f"top-8, H 2048, I 768, bf16 weights, batch 1, C={cfg.capacity} slots (37%), "
                               f"Zipf(1.1) routing with 80% reuse; one step = 48 MoE-layer decodes",
                   "global_batch": cfg.T * world, "parallelism": f"replicas x{world}",
                   "B_pcie_mbps": b_pcie, "B_cpu_mbps": b_cpu, "B_H_gbs": round(bh_gbs, 1),
                   "recommend_hybrid": rec, "K": K,
                   "host_pool": f"{args.pool_blobs} distinct seeded expert blobs in a page-locked arena, "
                                f"flat id f -> blob f mod {args.pool_blobs}",
                   "graph": graph is not None,
                   "l2": "inputs larger than L2: each step reads ~48 x 8 x 9.4 MB of expert weights"},
        "cache_stats": {"hits": int(cnt1[0] - cnt0[0]), "misses": int(cnt1[1] - cnt0[1]),
                        "fills": int(cnt1[2] - cnt0[2]), "cpu_assigned": int(cnt1[3] - cnt0[3]),
                        "read_miss_rate": round(float(cnt1[5] - cnt0[5]) / max(1, float(cnt1[4] + cnt1[5] - cnt0[4] - cnt0[5])), 4)},
        "e2e": {"value": round(e2e_steps * s.L * world / (ms_e2e / 1e3), 1), "unit": UNIT,
                "h2d_bytes_per_step": int(h2d), "d2h_bytes_per_step": int(d2h)},
        "gpu_launches": args.steps * s.L * launches_per_layer,
        "roofline": {"bound": "hbm",
                     "kernel": {
                         0: "resident-expert GEMV pair per layer-step: gate/up grid (with the L2 fetch of W_down) "
                            "+ down-projection grid fused with the combine; one step replayed with every routed "
                            "expert resident, event pairs around the two grids",
                         1: "resident-expert SwiGLU per layer-step, one launch: the gate/up stream (with the L2 "
                            "fetch of W_down), a grid-wide barrier, then the down projection fused with the "
                            "combine; one step replayed with every routed expert resident, an event pair around "
                            "the launch"}[resident_path],
                     "achieved": round(res_gbs, 1) if res_gbs else None, "peak": hbm_peak, "unit": "GB/s",
                     "frac": round(res_gbs / hbm_peak, 3) if res_gbs else None, "peak_source": peak_src,
                     "traffic": TRAFFIC_PER_LAYER_STEP if resident_path == 0 else FUSED_TRAFFIC_PER_LAYER_STEP,
                     "traffic_source": TRAFFIC_SOURCE if resident_path == 0 else FUSED_TRAFFIC_SOURCE,
                     "bytes_per_layer_step": round(res_bytes / max(1, res_launches)),
                     "us_per_layer_step": round(1e3 * res_ms / max(1, res_launches), 2),
                     "layer_steps_timed": res_launches, "fills_during": res_fills,
                     "all_resident_layer_us": round(1e3 * ms_res / (res_reps * s.L), 2)},
        "in_step_gemv": {"note": "the same resident-expert kernels inside the timed step's mix (fills beside "
                                 "them; the event pairs in the graph also drop their programmatic overlap)",
                         "achieved_gbs": round(gemv_bytes / (gemv_ms / 1e3) / 1e9, 1) if gemv_ms > 0 else None,
                         "bytes_per_layer_step": round(gemv_bytes / max(1, gemv_launches)),
                         "us_per_layer_step": round(1e3 * gemv_ms / max(1, gemv_launches), 2)},
        "kernel_ms_share": {k: round(v[0] / total_prof_ms, 3) for k, v in prof.items() if v[1]},
        "kernel_us_per_layer": {k: round(1e3 * v[0] / max(1, v[1]), 2) for k, v in prof.items() if v[1]},
        "fill": {"achieved_gbs": round(fill_bytes / (prof["fill"][0] / 1e3) / 1e9, 1) if prof["fill"][0] > 0 else None,
                 "bench_bw_B_P_gbs": round(bp_gbs, 1), "note": "fill kernel (with the filled experts' gate/up) "
                 "on the side stream, concurrent with the resident-expert GEMV; bytes = filled blobs"},
        "control_us": round(1e3 * prof["control"][0] / max(1, prof["control"][1]), 2),
        "layer_step_us": layer_step_us,
        "control_us_all_resident": round(1e3 * res_prof["control"][0] / max(1, res_prof["control"][1]), 2),
        "control_note": "event pair around the control kernel in the replayed graph (its launch and grid-"
                        "dependency wait included), in the timed step and in the all-resident replay",
        "clocks": clk.summary(),
    }
    if args.mode == "all" and not args.no_nvfp4:
        cache.close()
        result["nvfp4_decode"] = fp4_measure(args, dev, local, b_pcie, b_cpu, "nvfp4")
        result["mxfp4_decode"] = fp4_measure(args, dev, local, b_pcie, b_cpu, "mxfp4")
    if not args.no_prefill and args.mode == "all":
        result["prefill"] = prefill_measure(args, dev, local)
        if not args.no_nvfp4:
            result["prefill_mxfp4"] = prefill_fp4_measure(args, dev, local, "mxfp4")
    if rank == 0 and not args.no_cpu_baseline:
        result["cpu_baseline"] = run_cpu_baseline(args.cpu_seconds, args.pool_blobs, (b_pcie, b_cpu))
    if rank == 0:
        print(json.dumps(result))
    cache.close()
    if world > 1:
        dist.destroy_process_group()


def profile_case(args, dev):
    """A small decode case for ncu captures (a few GB on the device): the qwen3 b1
    shape with --profile-layers layers and 256 slots (--capacity to change),
    --steps eager steps of single decode calls, no graph, no timing."""
    import torch
    from serving_layer_moe_gb300 import MoECache
    base = config(WORKLOAD)
    cfg = base.with_(shape=base.shape.__class__(**{**base.shape.__dict__, "L": args.profile_layers}))
    s = cfg.shape
    arena, offs = make_pool(s, cfg.seed, n_phys=16)
    pool = torch.from_numpy(arena).pin_memory()
    cache = MoECache(L=s.L, E=s.E, H=s.H, I=s.I, top_k=s.k, max_tokens=1, wdtype=s.wdtype, adtype=s.adtype,
                     host_pool=pool, blob_offsets=offs, n_slots=args.capacity or 256, bw_pcie_mbps=192000,
                     bw_cpu_mbps=0, device=dev.index or 0)
    ids, w = routing_trace(cfg)
    out = torch.empty(1, s.H, device=dev)
    for st0 in range(args.steps):
        st = 0 if args.profile_allhit else st0 % cfg.steps
        for l in range(s.L):
            x = torch.from_numpy(activations(cfg, st, l).view(np.int16)).to(dev)
            cache.decode(l, x, torch.from_numpy(ids[st, l]).to(dev), torch.from_numpy(w[st, l]).to(dev), out)
    torch.cuda.synchronize(dev)
    c = cache.state()[3]
    print(json.dumps({"profile_case": f"{WORKLOAD} shape, {s.L} layers, {int(cache.info()[1])} slots",
                      "hits": int(c[0]), "misses": int(c[1]), "fills": int(c[2])}))
    cache.close()


FP4_DESC = {"nvfp4": "NVFP4 experts (e2m1 + e4m3 per 16 + fp32 per matrix)",
            "mxfp4": "MXFP4 experts (e2m1 + e8m0 per 32)"}


def fp4_measure(args, dev, local, b_pcie, b_cpu, fmt, steps=64, warmup=8):
    """The decode workload with 4-bit experts (same shape, routing and slot count):
    a blob is 2.65 MB (NVFP4) or 2.51 MB (MXFP4) instead of 9.44 MB, so fills
    and the resident GEMVs move 3.6x or 3.8x fewer bytes.  Graph replay of whole
    steps, inputs resident."""
    import torch
    from serving_layer_moe_gb300 import MoECache
    base = config(WORKLOAD)
    cfg = base.with_(shape=base.shape.__class__(**{**base.shape.__dict__, "wdtype": fmt}))
    s = cfg.shape
    arena, offs = make_pool(s, cfg.seed, n_phys=args.pool_blobs)
    pool = torch.from_numpy(arena).pin_memory()
    del arena
    K = default_max_fetch(s, cfg.T)
    cache = MoECache(L=s.L, E=s.E, H=s.H, I=s.I, top_k=s.k, max_tokens=cfg.T, wdtype=s.wdtype, adtype=s.adtype,
                     host_pool=pool, blob_offsets=offs, n_slots=cfg.capacity, max_fetch=K, bw_pcie_mbps=b_pcie,
                     bw_cpu_mbps=b_cpu, device=local)
    ids, w = routing_trace(cfg)
    xs = np.stack([np.stack([activations(cfg, st, l) for l in range(s.L)]) for st in range(cfg.steps)])
    x_all = torch.from_numpy(xs.view(np.int16)).to(dev)
    ids_all = torch.from_numpy(ids).to(dev)
    w_all = torch.from_numpy(w).to(dev)
    xb, ib, wb = torch.empty_like(x_all[0]), torch.empty_like(ids_all[0]), torch.empty_like(w_all[0])
    out = torch.empty(s.L, cfg.T, s.H, dtype=torch.float32, device=dev)
    cpu_part = torch.zeros(cfg.T, s.k, s.H, dtype=torch.float32, device=dev)
    stream = torch.cuda.Stream(device=dev)
    sp = stream.cuda_stream

    def enqueue_step():
        for l in range(s.L):
            cache.decode_ptrs(l, cfg.T, xb[l].data_ptr(), ib[l].data_ptr(), wb[l].data_ptr(), cpu_part.data_ptr(),
                              out[l].data_ptr(), None, sp)

    def stage(st):
        xb.copy_(x_all[st % cfg.steps], non_blocking=True)
        ib.copy_(ids_all[st % cfg.steps], non_blocking=True)
        wb.copy_(w_all[st % cfg.steps], non_blocking=True)

    with torch.cuda.stream(stream):
        for st in range(warmup):
            stage(st)
            enqueue_step()
    torch.cuda.synchronize(dev)
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=stream):
        enqueue_step()
    torch.cuda.synchronize(dev)
    cnt0 = cache.state()[3].copy()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(stream):
        e0.record(stream)
        for st in range(warmup, warmup + steps):
            stage(st)
            graph.replay()
        e1.record(stream)
    torch.cuda.synchronize(dev)
    ms = e0.elapsed_time(e1)
    cnt1 = cache.state()[3].copy()
    cache.close()
    return {"workload": f"{WORKLOAD} with {FP4_DESC[fmt]}, C={cfg.capacity} slots",
            "value": round(steps * s.L / (ms / 1e3), 1), "unit": UNIT, "steps": steps,
            "ms_per_step": round(ms / steps, 4), "blob_bytes": int(s.blob_bytes),
            "fills": int(cnt1[2] - cnt0[2]), "hits": int(cnt1[0] - cnt0[0])}


def prefill_measure(args, dev, local):
    """Prefill chunk: 8192 tokens through all 48 layers with full-layer double buffering.

    Reports the wall time of the chunk (bound by the host link: every layer's
    experts cross it once), the grouped-GEMM TFLOP/s inside that run, and the
    GEMM TFLOP/s of a layer whose experts are already resident (no concurrent
    loads).  One activation matrix x (N(0,1), bf16) serves every layer.
    """
    import torch
    from serving_layer_moe_gb300 import MoECache
    cfg = config("qwen3_prefill_8k").with_(T=args.prefill_tokens)
    if args.capacity:
        cfg = cfg.with_(capacity=args.capacity)
    s = cfg.shape
    arena, offs = make_pool(s, cfg.seed, n_phys=args.pool_blobs)
    pool = torch.from_numpy(arena).pin_memory()
    del arena
    ablation_T = [t for t in (4096, 8192, 16384) if not args.no_prefill_ablation]
    cache = MoECache(L=s.L, E=s.E, H=s.H, I=s.I, top_k=s.k, max_tokens=1, wdtype=s.wdtype, adtype=s.adtype,
                     host_pool=pool, blob_offsets=offs, n_slots=cfg.capacity, bw_pcie_mbps=1000, bw_cpu_mbps=0,
                     device=local, max_prefill_tokens=max([cfg.T] + ablation_T))
    x = torch.from_numpy(activations(cfg, 0, 0).view(np.int16)).to(dev)
    routes = [prefill_routing(cfg, l) for l in range(s.L)]
    ids = [torch.from_numpy(r[0]).to(dev) for r in routes]
    ws = [torch.from_numpy(r[1]).to(dev) for r in routes]
    out = torch.empty(cfg.T, s.H, dtype=torch.float32, device=dev)
    stream = torch.cuda.Stream(device=dev)
    flops_layer = 6.0 * s.H * s.I * cfg.T * s.k
    hbm_peak, bf16_peak, bf16_sust, src = measured_peaks()

    def chunk():
        for l in range(s.L):
            cache.prefill(l, x, ids[l], ws[l], out, stream=stream)

    with torch.cuda.stream(stream):
        chunk()                                   # warm-up (cold cache)
    torch.cuda.synchronize(dev)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(stream):
        e0.record(stream)
        chunk()
        e1.record(stream)
    torch.cuda.synchronize(dev)
    wall_ms = e0.elapsed_time(e1)
    cache.profile_start()
    with torch.cuda.stream(stream):
        chunk()
    prof = cache.profile_stop()
    gemm_ms = prof["prefill_gemm"][0]
    load_ms = prof["prefill_load"][0]
    # isolated: layer 0 again and again, its experts (and layer 1's) stay resident
    with torch.cuda.stream(stream):
        for _ in range(3):
            cache.prefill(0, x, ids[0], ws[0], out, stream=stream)
    torch.cuda.synchronize(dev)
    cnt0 = cache.state()[3].copy()
    cache.profile_start()
    reps = 10
    with torch.cuda.stream(stream):
        for _ in range(reps):
            cache.prefill(0, x, ids[0], ws[0], out, stream=stream)
    iso = cache.profile_stop()
    loads_iso = int(cache.state()[3][7] - cnt0[7])
    # The pages' comparison without the second buffer (ai.thesatyajit.com, "Prefill:
    # hide the pool behind the wire"; snackonai, "It In Action"): the same chunk
    # with each layer's loads and GEMMs one after the other.  Every timed chunk
    # starts with layers 0 and 1 evicted by the chunk before it, so both modes
    # move all L x E experts across the link.
    ablation = {}
    for Ta in ablation_T:
        ca = cfg.with_(T=Ta)
        xa = torch.from_numpy(activations(ca, 0, 0).view(np.int16)).to(dev)
        ra = [prefill_routing(ca, l) for l in range(s.L)]
        ida = [torch.from_numpy(r[0]).to(dev) for r in ra]
        wa = [torch.from_numpy(r[1]).to(dev) for r in ra]
        oa = torch.empty(Ta, s.H, dtype=torch.float32, device=dev)
        ms_mode = {}
        for on in (True, False):
            cache.set_prefill_prefetch(on)
            with torch.cuda.stream(stream):
                if on:
                    for l in range(s.L):   # warm-up chunk of this size
                        cache.prefill(l, xa, ida[l], wa[l], oa, stream=stream)
                a0, a1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                a0.record(stream)
                for l in range(s.L):
                    cache.prefill(l, xa, ida[l], wa[l], oa, stream=stream)
                a1.record(stream)
            torch.cuda.synchronize(dev)
            ms_mode[on] = a0.elapsed_time(a1)
        cache.set_prefill_prefetch(True)
        ablation[str(Ta)] = {"double_ms": round(ms_mode[True], 2), "single_ms": round(ms_mode[False], 2),
                             "double_tokens_per_s": round(Ta / (ms_mode[True] / 1e3), 1),
                             "single_tokens_per_s": round(Ta / (ms_mode[False] / 1e3), 1),
                             "throughput_loss": round(1.0 - ms_mode[True] / ms_mode[False], 3)}
    cache.close()
    iso_tf = reps * flops_layer / (iso["prefill_gemm"][0] / 1e3) / 1e12
    return {"workload": f"qwen3_prefill_8k: {cfg.T} tokens, top-8 of 128 (N(0,1) logits), 48 layers, "
                        f"C={cfg.capacity} slots, full-layer double buffering",
            "wall_ms": round(wall_ms, 2), "tokens_per_s": round(cfg.T / (wall_ms / 1e3), 1),
            "expert_bytes_per_chunk": int(s.L * s.E * s.blob_bytes),
            "link_gbs_wall": round(s.L * s.E * s.blob_bytes / (wall_ms / 1e3) / 1e9, 1),
            "gemm_ms_in_chunk": round(gemm_ms, 3),
            "gemm_tflops_in_chunk": round(s.L * flops_layer / (gemm_ms / 1e3) / 1e12, 1),
            "load_ms_in_chunk": round(load_ms, 2),
            "gemm_tflops_isolated": round(iso_tf, 1),
            "gemm_frac_isolated": round(iso_tf / bf16_peak, 3),
            "tensor_peak_tflops": bf16_peak, "peak_source": src,
            "loads_during_isolated": loads_iso,
            "flops_per_layer": flops_layer,
            "second_buffer_ablation": {
                "note": "the same chunk without the second buffer (each layer's loads, then its GEMMs); "
                        "throughput_loss = 1 - double/single wall time; the pages' 5090 figures: 0.19 at 4096, "
                        "0.25 at 8192, 0.26 at 16384 tokens",
                "by_tokens": ablation}}


def prefill_fp4_measure(args, dev, local, fmt):
    """The prefill chunk with 4-bit experts: the host link carries 4-bit blobs
    (2.51 MB for MXFP4 instead of 9.44 MB), and before its GEMMs each layer's
    routed experts are decoded to bf16 in HBM.  Wall time of one chunk after a
    warm-up chunk; the profile splits it into loads and decode + GEMMs."""
    import torch
    from serving_layer_moe_gb300 import MoECache
    base = config("qwen3_prefill_8k").with_(T=args.prefill_tokens)
    if args.capacity:
        base = base.with_(capacity=args.capacity)
    cfg = base.with_(shape=base.shape.__class__(**{**base.shape.__dict__, "wdtype": fmt}))
    s = cfg.shape
    arena, offs = make_pool(s, cfg.seed, n_phys=args.pool_blobs)
    pool = torch.from_numpy(arena).pin_memory()
    del arena
    cache = MoECache(L=s.L, E=s.E, H=s.H, I=s.I, top_k=s.k, max_tokens=1, wdtype=s.wdtype, adtype=s.adtype,
                     host_pool=pool, blob_offsets=offs, n_slots=cfg.capacity, bw_pcie_mbps=1000, bw_cpu_mbps=0,
                     device=local, max_prefill_tokens=cfg.T)
    x = torch.from_numpy(activations(cfg, 0, 0).view(np.int16)).to(dev)
    routes = [prefill_routing(cfg, l) for l in range(s.L)]
    ids = [torch.from_numpy(r[0]).to(dev) for r in routes]
    ws = [torch.from_numpy(r[1]).to(dev) for r in routes]
    out = torch.empty(cfg.T, s.H, dtype=torch.float32, device=dev)
    stream = torch.cuda.Stream(device=dev)

    def chunk():
        for l in range(s.L):
            cache.prefill(l, x, ids[l], ws[l], out, stream=stream)

    with torch.cuda.stream(stream):
        chunk()
    torch.cuda.synchronize(dev)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(stream):
        e0.record(stream)
        chunk()
        e1.record(stream)
    torch.cuda.synchronize(dev)
    wall_ms = e0.elapsed_time(e1)
    cache.profile_start()
    with torch.cuda.stream(stream):
        chunk()
    prof = cache.profile_stop()
    cache.close()
    return {"workload": f"qwen3_prefill_8k with {FP4_DESC[fmt]}: {cfg.T} tokens, 48 layers, C={cfg.capacity} slots",
            "wall_ms": round(wall_ms, 2), "tokens_per_s": round(cfg.T / (wall_ms / 1e3), 1),
            "blob_bytes": int(s.blob_bytes), "expert_bytes_per_chunk": int(s.L * s.E * s.blob_bytes),
            "link_gbs_wall": round(s.L * s.E * s.blob_bytes / (wall_ms / 1e3) / 1e9, 1),
            "decode_and_gemm_ms_in_chunk": round(prof["prefill_gemm"][0], 3),
            "load_ms_in_chunk": round(prof["prefill_load"][0], 2)}


def reference_arm(args, world, rank):
    """The oracle as the reference arm: bounded samples of the same workload on host cores."""
    if rank != 0:
        return
    b = os.environ.get("BENCH_BW", "200000,100000").split(",")
    bw = (int(b[0]), int(b[1]))
    per_step = args.ref_seconds or max(2.0, min(20.0, 120.0 / max(1, args.steps + args.warmup)))
    res = run_cpu_baseline(per_step, args.pool_blobs, bw, samples=args.warmup + args.steps)
    if isinstance(res, dict):
        res = [res]
    vals = [r["value"] for r in (res or [])[args.warmup:]]
    v = statistics.mean(vals) if vals else None
    line = {"impl": "reference", "metric": METRIC, "value": v, "unit": UNIT, "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": f"{WORKLOAD} (oracle: list-LRU control + float64 SwiGLU)"},
            "cpu_baseline": {"value": v, "unit": UNIT, "kind": "oracle", "cores": 1,
                             "sample": f"{per_step:.0f} s of oracle layer-steps per bench step, one thread"},
            "e2e": {"value": v, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line))


if __name__ == "__main__":
    a = parse_args()
    if a.cpu_worker:
        b = os.environ.get("BENCH_BW", "200000,100000").split(",")
        cpu_worker(a.cpu_seconds, a.pool_blobs, (int(b[0]), int(b[1])), samples=a.cpu_samples)
    else:
        main(a)
