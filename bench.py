#!/usr/bin/env python
"""Benchmark of the expert-slot-cache MoE decode step on GB300.

Workload: Qwen3-30B-A3B-shaped decode (48 MoE layers, 128 experts, top-8,
hidden 2048, expert intermediate 768, bf16 weights, batch 1), cache of 37% of
the 6144 (layer, expert) slots, Zipf(1.1) routing with 80% step-to-step reuse.
One bench step = one decode token through all 48 MoE layers: per layer the
control kernel, the slot fills on the side stream, the grouped SwiGLU GEMV
over resident and filled experts, and the combine with supplied CPU partial
sums.  Metric: MoE-layer decode steps per second (48 per bench step).

The timed window is trace steps [64, 64 + K) (mod the 256-step trace): the
first 64 steps run untimed, the last W of them as warm-up, so the window never
starts from a cold cache and does not move with --steps.  The end-to-end figure
replays the same prefix on a fresh cache, then times the same K steps with
host-resident inputs copied in and the outputs copied out every step.

Beside the headline line the run measures the other decode workloads (tiny,
Qwen3 shape at batch 16 across its mid-run resize, the DeepSeek-V3 fp8 slice),
the 4-bit-expert variants of the headline, and the prefill chunk.

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

from workloads import (activations, config, default_max_fetch, make_blob, make_pool, make_shared,  # noqa: E402
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


RESIDENT_TRAFFIC = {0: (TRAFFIC_PER_LAYER_STEP, TRAFFIC_SOURCE), 1: (FUSED_TRAFFIC_PER_LAYER_STEP, FUSED_TRAFFIC_SOURCE)}
# DRAM bytes per launch of the other workloads' dominant kernel group, from ncu
# captures (none yet: the roofline's traffic stays null).
WORKLOAD_TRAFFIC: dict = {}
WORKLOAD_TRAFFIC_SOURCE: dict = {}
# The all-resident replays' pair (every routed expert + the shared one resident): DRAM
# bytes per layer-step from ncu; the windows' launches mix hits and fills, so their
# per-launch bytes vary and carry no ncu figure.
ALL_RESIDENT_TRAFFIC = {
    "dsv3_decode_slice": (399_100_000,
                          "ncu dram__bytes_read.sum + dram__bytes_write.sum of gate_up_bulk_kernel + down_bulk_kernel "
                          "pass 0, mean of the three all-resident layer-steps (9 experts, 396.4 MB algorithmic) in "
                          "bench.py --mode profile-decode --steps 4 --profile-workload dsv3_decode_slice "
                          "--profile-layers 4 --capacity 64; profiles/decode_dsv3_fp8_slice.md"),
}


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
    p.add_argument("--mode", default="all", choices=["all", "decode", "prefill", "profile-decode", "workloads",
                                                     "cpu-branch", "fill-step"],
                   help="prefill: only the prefill measurement; workloads: only the tiny, batch-16 and "
                        "DeepSeek-V3 decode workloads; fill-step: a layer-step with one fill against its floor")
    p.add_argument("--no-workloads", action="store_true",
                   help="skip the tiny, batch-16 and DeepSeek-V3 decode workloads")
    p.add_argument("--cpu-workload", default=WORKLOAD, help=argparse.SUPPRESS)
    p.add_argument("--prefill-tokens", type=int, default=8192)
    p.add_argument("--no-prefill-ablation", action="store_true",
                   help="skip the prefill chunks without the second buffer (4k / 8k / 16k tokens)")
    p.add_argument("--capacity", type=int, default=0, help="override the slot count (small profiling runs)")
    p.add_argument("--profile-layers", type=int, default=16, help="profile-decode: MoE layers of the small case")
    p.add_argument("--profile-workload", default=WORKLOAD, help="profile-decode: the workload whose shape to use")
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
def cpu_worker(seconds: float, pool_blobs: int, bw, samples: int = 1, workload: str = WORKLOAD):
    """Oracle control + float64 SwiGLU on successive layer-steps of a workload.

    Prints one JSON line per sample; each sample runs until `seconds` of oracle
    time are spent.  Generating the synthetic expert blobs (input synthesis) is
    not counted; parsing them to float64 is (the oracle reads its weights).
    """
    from oracle.cache import SlotCache
    from oracle.ffn import combine, swiglu_expert
    from oracle.formats import activations_to_f64, parse_blob
    cfg = config(workload)
    s = cfg.shape
    n_phys = min(pool_blobs, s.n_flat)
    ids, w = routing_trace(cfg)
    K = default_max_fetch(s, cfg.T)
    ora = SlotCache(s.L, s.E, cfg.capacity, K, bw[0], bw[1])
    raw, shared_raw = {}, {}
    st, l = 0, 0
    for _ in range(samples):
        spent, n = 0.0, 0
        while spent < seconds:
            sid = st % cfg.steps
            need = {(l * s.E + int(e)) % n_phys for e in ids[sid, l].ravel()}
            for p in need - raw.keys():
                raw[p] = make_blob(s, cfg.seed, p)          # input synthesis, not timed
            if s.n_shared and l not in shared_raw:
                shared_raw[l] = make_blob(s, cfg.seed, l, tag=0x5AED)
            xs = activations(cfg, sid, l)
            t0 = time.perf_counter()
            plan = ora.decode(l, ids[sid, l])
            x = activations_to_f64(xs, s.adtype)
            y = np.zeros((cfg.T, s.k, s.H))
            for t in range(cfg.T):
                for j in range(s.k):
                    p = (l * s.E + int(ids[sid, l, t, j])) % n_phys
                    y[t, j] = swiglu_expert(x[t], *parse_blob(raw[p], s.wdtype, s.H, s.I))
            sh_y = swiglu_expert(x, *parse_blob(shared_raw[l], s.wdtype, s.H, s.I)) if s.n_shared else None
            combine(w[sid, l], y, plan.slot_map, y, shared_y=sh_y)
            spent += time.perf_counter() - t0
            n += 1
            l += 1
            if l == s.L:
                l, st = 0, st + 1
        print(json.dumps({"layer_steps": n, "seconds": spent}), flush=True)


def run_cpu_baseline(seconds: float, pool_blobs: int, bw, samples: int = 1, workload: str = WORKLOAD,
                     threads: int = 1):
    """Run the oracle in a fresh interpreter (no fork after CUDA init); one dict per sample.

    threads = 1 is the oracle alone; more threads let NumPy's BLAS spread the
    float64 matrix-vector products of the SwiGLU over that many host cores.
    """
    env = dict(os.environ, OMP_NUM_THREADS=str(threads), OPENBLAS_NUM_THREADS=str(threads),
               MKL_NUM_THREADS=str(threads))
    cmd = [sys.executable, os.path.abspath(__file__), "--cpu-worker", "--cpu-seconds", str(seconds),
           "--pool-blobs", str(pool_blobs), "--cpu-samples", str(samples), "--cpu-workload", workload]
    env["BENCH_BW"] = f"{bw[0]},{bw[1]}"
    r = subprocess.run(cmd, capture_output=True, text=True, env=env, timeout=samples * (seconds * 4 + 120) + 180)
    lines = [json.loads(l) for l in r.stdout.splitlines() if l.startswith("{")]
    if r.returncode != 0 or not lines:
        return None
    out = []
    how = "one thread" if threads == 1 else f"BLAS on {threads} threads"
    for d in lines:
        out.append({"value": d["layer_steps"] / d["seconds"], "unit": UNIT, "cores": threads, "kind": "oracle",
                    "sample": f"{d['layer_steps']} layer-steps of {workload} from its first step (list-LRU control "
                              f"+ float64 SwiGLU per routed pair from the host pool + fixed-order combine), {how}, "
                              f"{d['seconds']:.1f} s of oracle time"})
    return out if samples > 1 else out[0]


def host_cores() -> int:
    try:
        return len(os.sched_getaffinity(0))
    except (AttributeError, OSError):
        return os.cpu_count() or 1


# ----------------------------------------------------------------------------
# a decode workload on one cache, replayed step by step
# ----------------------------------------------------------------------------
# Trace steps replayed untimed before a timed window, so the window never starts
# from a cold cache and does not move with --steps (the warm-up steps are the
# last of these).
PREFIX_STEPS = 64


def expert_bytes(s) -> tuple[int, int]:
    """(gate/up bytes, down bytes) of one expert blob, each with its scales (they sum to S)."""
    H, I = s.H, s.I
    if s.wdtype == "f32":
        return 8 * I * H, 4 * I * H
    if s.wdtype == "bf16":
        return 4 * I * H, 2 * I * H
    if s.wdtype == "fp8":
        return 2 * I * H + 4 * (2 * I // 128) * (H // 128), H * I + 4 * (H // 128) * (I // 128)
    if s.wdtype == "nvfp4":
        return I * H + 2 * I * H // 16 + 8, H * I // 2 + H * I // 16 + 8
    return I * H + 2 * I * H // 32, H * I // 2 + H * I // 32   # mxfp4


class DecodeRunner:
    """One decode workload on one cache: the inputs of the trace steps it runs in
    HBM, one whole decode step (L MoE-layer calls) captured in a CUDA graph and
    replayed per step.  Run step n uses trace step n mod steps.  A workload with a
    mid-run resize resizes once, before run step resize_step, and re-captures the
    graph (the slot pool moves)."""

    def __init__(self, cfg, pool, offs, shared, bw, dev, need_steps, K=None):
        import torch
        from serving_layer_moe_gb300 import MoECache
        s = cfg.shape
        self.torch = torch
        self.cfg, self.s, self.dev = cfg, s, dev
        self.K = default_max_fetch(s, cfg.T) if K is None else K
        self.cache = MoECache(L=s.L, E=s.E, H=s.H, I=s.I, top_k=s.k, max_tokens=cfg.T, wdtype=s.wdtype,
                              adtype=s.adtype, host_pool=pool, blob_offsets=offs, shared=shared,
                              n_slots=cfg.capacity, max_fetch=self.K, bw_pcie_mbps=bw[0], bw_cpu_mbps=bw[1],
                              device=dev.index or 0)
        self.n_trace = min(cfg.steps, need_steps)
        ids, w = routing_trace(cfg)
        acts = np.stack([np.stack([activations(cfg, st, l) for l in range(s.L)]) for st in range(self.n_trace)])
        self.acts = acts.view(np.int16) if acts.dtype == np.uint16 else acts
        self.ids, self.w = ids[:self.n_trace], w[:self.n_trace]
        self.x_all = torch.from_numpy(self.acts).to(dev)            # [steps, L, T, H]
        self.ids_all = torch.from_numpy(self.ids).to(dev)           # [steps, L, T, k]
        self.w_all = torch.from_numpy(self.w).to(dev)
        self.xb = torch.empty_like(self.x_all[0])
        self.ib = torch.empty_like(self.ids_all[0])
        self.wb = torch.empty_like(self.w_all[0])
        self.out = torch.empty(s.L, cfg.T, s.H, dtype=torch.float32, device=dev)
        # caller-supplied CPU partial sums: the combine reads them where a pair is CPU-assigned
        self.cpu_part = torch.zeros(cfg.T, s.k, s.H, dtype=torch.float32, device=dev)
        self.stream = torch.cuda.Stream(device=dev)
        self.ptrs = [(self.xb[l].data_ptr(), self.ib[l].data_ptr(), self.wb[l].data_ptr(), self.out[l].data_ptr())
                     for l in range(s.L)]
        self.step = 0
        self.graph = None
        self.resized = cfg.resize_step is None
        self.resize_ms = None

    def trace_index(self, n: int) -> int:
        st = n % self.cfg.steps
        assert st < self.n_trace, "run step beyond the trace steps held on the device"
        return st

    def enqueue(self):
        sp = self.stream.cuda_stream
        for l in range(self.s.L):
            xp, ip, wp, op = self.ptrs[l]
            self.cache.decode_ptrs(l, self.cfg.T, xp, ip, wp, self.cpu_part.data_ptr(), op, None, sp)

    def stage(self, n: int):
        st = self.trace_index(n)
        self.xb.copy_(self.x_all[st], non_blocking=True)
        self.ib.copy_(self.ids_all[st], non_blocking=True)
        self.wb.copy_(self.w_all[st], non_blocking=True)

    def sync(self):
        """Wait for the device through the library (its call releases the interpreter lock,
        which a registered CPU branch's host function takes on a driver thread)."""
        self.cache.plan()

    def capture(self):
        torch = self.torch
        self.sync()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=self.stream):
            self.enqueue()
        self.sync()
        self.graph = g

    def _maybe_resize(self):
        if not self.resized and self.step == self.cfg.resize_step:
            self.sync()   # the steps queued so far are not part of the resize
            t0 = time.perf_counter()
            self.cache.resize(self.cfg.resize_to)     # a safe point: synchronises the device
            if self.graph is not None:
                self.capture()
            self.resize_ms = 1e3 * (time.perf_counter() - t0)
            self.resized = True

    def warm(self, prefix: int):
        """Run steps 0 .. prefix-1 untimed: two eager steps, then graph replays."""
        with self.torch.cuda.stream(self.stream):
            for _ in range(min(2, prefix)):
                self._maybe_resize()
                self.stage(self.step)
                self.enqueue()
                self.step += 1
        self.capture()
        self.advance(prefix - self.step)

    def advance(self, n: int):
        with self.torch.cuda.stream(self.stream):
            for _ in range(n):
                self._maybe_resize()
                self.stage(self.step)
                self.graph.replay()
                self.step += 1

    def advance_host(self, n: int, x_h, ids_h, w_h, out_h):
        """n steps from page-locked host inputs, the outputs copied back every step."""
        with self.torch.cuda.stream(self.stream):
            for _ in range(n):
                self._maybe_resize()
                st = self.trace_index(self.step)
                self.xb.copy_(x_h[st], non_blocking=True)
                self.ib.copy_(ids_h[st], non_blocking=True)
                self.wb.copy_(w_h[st], non_blocking=True)
                self.graph.replay()
                out_h.copy_(self.out, non_blocking=True)
                self.step += 1

    def timed(self, n: int, clocks=None):
        """(milliseconds, counter delta) of n steps between two events on the stream."""
        torch = self.torch
        cnt0 = self.cache.state()[3].copy()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(self.stream)
        self.advance(n)
        e1.record(self.stream)
        self.sync()
        return e0.elapsed_time(e1), self.cache.state()[3].copy() - cnt0

    def profiled(self, n: int, same_step: bool = False):
        """Kernel-group times over n replays of a second graph of the step with the
        library's event pair around each kernel group: ({kind: [ms, launches]},
        counter delta).  same_step replays the current step's inputs every time."""
        torch = self.torch
        cache = self.cache
        cache.profile_start()
        pgraph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(pgraph, stream=self.stream):
            self.enqueue()
        cache.profile_pause()
        torch.cuda.synchronize(self.dev)
        prof = {k: [0.0, 0] for k in cache.PROFILE_KINDS}
        cnt0 = cache.state()[3].copy()
        with torch.cuda.stream(self.stream):
            if same_step:
                self.stage(self.step)
            for _ in range(n):
                if not same_step:
                    assert self.resized or self.step + 1 < self.cfg.resize_step, "profiled replays across the resize"
                    self.stage(self.step)
                    self.step += 1
                pgraph.replay()
                for k, (ms_k, n_k) in cache.profile_read().items():
                    prof[k][0] += ms_k
                    prof[k][1] += n_k
        cnt1 = cache.state()[3].copy()
        cache.profile_stop()
        return prof, cnt1 - cnt0

    def close(self):
        self.cache.close()


def kernel_groups(s, prof, dcnt):
    """Algorithmic HBM bytes and event time of the decode kernel groups over profiled
    replays: {kind: (bytes, ms, launches)}.  Resident experts are this window's
    unique hits (+ the shared expert of every launch); each weight byte counts
    once.  Split path ("down_filled" present): the resident gate/up + down +
    combine is one group over whole blobs.  Otherwise the resident gate/up grid
    reads W_gu and the down + combine grid reads W_down of every GPU expert."""
    gu, wd = expert_bytes(s)
    hits, fills = int(dcnt[0]), int(dcnt[2])
    launches = prof["gemv_resident"][1]
    shared = s.n_shared * launches
    out = {}
    if prof["down_filled"][1]:
        out["gemv_resident"] = ((hits + shared) * s.blob_bytes, prof["gemv_resident"][0], launches)
        out["down_filled"] = (fills * wd, prof["down_filled"][0], prof["down_filled"][1])
    else:
        out["gemv_resident"] = ((hits + shared) * gu, prof["gemv_resident"][0], launches)
        out["down_combine"] = ((hits + fills + shared) * wd, prof["down_combine"][0], prof["down_combine"][1])
    return out


KERNEL_NAMES = {
    "gemv_resident_split": "resident-expert GEMV pair: gate_up_bulk_kernel (with the L2 fetch of W_down) + "
                           "down_bulk_kernel pass 0 fused with the combine",
    "gemv_resident": "resident-expert gate/up grid (gate_up_bulk_kernel)",
    "down_combine": "down projection of every GPU expert fused with the combine, one grid after the fills "
                    "(down_bulk_kernel over all GPU experts, each item's h read through L1)",
}


def roofline_from_groups(groups, hbm_peak, peak_src, traffic=None, traffic_source=None, split=None):
    """The roofline object of the group with the most event time (all are HBM-bound)
    among those that move bytes: a grid whose expert set is empty (the resident
    gate/up grid when every read misses) only waits for SMs and has no roofline.
    split: the call took the split down grids (the resident group is the whole pair);
    by default read from the groups (a "down_filled" group exists)."""
    moving = {k: v for k, v in groups.items() if v[0] > 0} or groups
    kind, (b, ms, n) = max(moving.items(), key=lambda kv: kv[1][1])
    if ms <= 0 or n == 0:
        return None
    if split is None:
        split = "down_filled" in groups
    achieved = b / (ms / 1e3) / 1e9
    return {"bound": "hbm",
            "kernel": KERNEL_NAMES["gemv_resident_split" if (split and kind == "gemv_resident") else kind],
            "achieved": round(achieved, 1), "peak": hbm_peak, "unit": "GB/s", "frac": round(achieved / hbm_peak, 3),
            "peak_source": peak_src, "traffic": traffic, "traffic_source": traffic_source,
            "bytes_per_launch": round(b / n), "us_per_launch": round(1e3 * ms / n, 2), "launches_timed": n}


def cache_stats(dcnt):
    reads = float(dcnt[4] + dcnt[5])
    return {"hits": int(dcnt[0]), "misses": int(dcnt[1]), "fills": int(dcnt[2]), "cpu_assigned": int(dcnt[3]),
            "read_miss_rate": round(float(dcnt[5]) / max(1.0, reads), 4)}


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
            res = {"prefill": prefill_measure(args, dev, local)}
            if not args.no_nvfp4:
                res["prefill_mxfp4"] = prefill_fp4_measure(args, dev, local, "mxfp4")
            print(json.dumps(res))
        return
    if args.mode == "profile-decode":
        return profile_case(args, dev)

    from serving_layer_moe_gb300 import bench_bw

    cfg = config(WORKLOAD)
    if args.capacity:
        cfg = cfg.with_(capacity=args.capacity)
    s = cfg.shape
    # calibration: B_P through the fill path, B_H host read; B_cpu = residual
    bp_gbs, bh_gbs, rec = bench_bw(local, s.blob_bytes)
    b_pcie = max(1, int(bp_gbs * 1000))
    b_cpu = max(0, int(bh_gbs * 1000) - b_pcie)
    hbm_peak, bf16_peak, bf16_sust, peak_src = measured_peaks()

    if args.mode == "cpu-branch":
        if rank == 0:
            print(json.dumps({"cpu_branch": cpu_branch_measure(args, dev)}))
        return
    if args.mode == "fill-step":
        if rank == 0:
            print(json.dumps({"fill_step": fill_step_measure(args, dev, bp_gbs)}))
        return
    if args.mode == "workloads":
        res = {n: decode_workload_measure(n, args, dev, (b_pcie, b_cpu), hbm_peak, peak_src,
                                          rank == 0 and not args.no_cpu_baseline, bp_gbs)
               for n in EXTRA_WORKLOADS}
        if rank == 0:
            print(json.dumps({"workloads": res}))
        return

    arena, offs = make_pool(s, cfg.seed, n_phys=args.pool_blobs)
    pool = torch.from_numpy(arena).pin_memory()
    del arena
    prefix = max(PREFIX_STEPS, args.warmup + 2)
    need = prefix + args.steps + 64
    run = DecodeRunner(cfg, pool, offs, None, (b_pcie, b_cpu), dev, need)
    K = run.K
    run.warm(prefix)
    # control, fill (+ the filled experts' gate/up), the filled experts' down grid and
    # the resident experts' kernels (one launch, or a gate/up grid and a down +
    # combine grid), as the library reports
    launches_per_layer = int(run.cache.info()[6])
    resident_path = int(run.cache.info()[7])   # 0: two grids, 1: one launch with a grid barrier

    # ---- timed region: inputs resident in HBM; trace steps [prefix, prefix + steps) ----
    if world > 1:
        dist.barrier()
    with ClockSampler(local) as clk:
        ms, dcnt = run.timed(args.steps)
    if world > 1:
        t = torch.tensor([ms], device=dev)
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
        ms = float(t.item())
        dist.barrier()
    layer_steps = args.steps * s.L * world
    value = layer_steps / (ms / 1e3)
    window = {"trace_steps": f"[{prefix}, {prefix + args.steps}) mod {cfg.steps}",
              "untimed_prefix_steps": prefix, **cache_stats(dcnt)}

    # ---- kernel timing inside the step's mix: a second graph of the step with the
    # library's event pair around each kernel group, over the next 32 steps ----------
    prof, dcnt_p = run.profiled(32)
    groups = kernel_groups(s, prof, dcnt_p)
    total_prof_ms = sum(v[0] for v in prof.values())
    gb, gms, gn = groups["gemv_resident"]
    fill_bytes = int(dcnt_p[2]) * s.blob_bytes
    # ---- roofline of the dominant HBM kernels, the resident-expert GEMV pair, with
    # nothing beside them: one step's inputs replayed until every routed expert is
    # resident (all hits, no fill), the same event pairs around the resident grids.
    # Algorithmic bytes: each resident expert's whole blob, read once.
    res_reps = 16
    run.profiled(3, same_step=True)
    res_prof, dcnt_r = run.profiled(res_reps, same_step=True)
    with torch.cuda.stream(run.stream):   # the same all-hit step without event pairs: whole-layer time
        e4, e5 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e4.record(run.stream)
        for _ in range(res_reps):
            run.graph.replay()
        e5.record(run.stream)
    torch.cuda.synchronize(dev)
    ms_res = e4.elapsed_time(e5)
    res_hits, res_fills = int(dcnt_r[0]), int(dcnt_r[2])
    gemv_kinds = ("gemv_resident", "down_combine")   # split: the pair is one group; down_combine stays 0
    res_ms = sum(res_prof[k][0] for k in gemv_kinds)
    res_launches = res_prof["gemv_resident"][1]
    res_bytes = res_hits * s.blob_bytes
    res_gbs = res_bytes / (res_ms / 1e3) / 1e9 if res_ms > 0 else None
    run.step += 1
    # Distribution of whole MoE-layer decode times (median, p90): eager calls, one
    # event pair around each layer's call on its stream, fills included where they
    # occur.  Reported beside the means; a failure here leaves the rest of the line intact.
    try:
        lat_steps = 8
        lat_ev = [[(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
                   for _ in range(s.L)] for _ in range(lat_steps)]
        with torch.cuda.stream(run.stream):
            for st_i in range(lat_steps):
                run.stage(run.step)
                run.step += 1
                for l in range(s.L):
                    xp, ip, wp, op = run.ptrs[l]
                    lat_ev[st_i][l][0].record(run.stream)
                    run.cache.decode_ptrs(l, cfg.T, xp, ip, wp, run.cpu_part.data_ptr(), op, None,
                                          run.stream.cuda_stream)
                    lat_ev[st_i][l][1].record(run.stream)
        torch.cuda.synchronize(dev)
        lat_us = np.array([1e3 * a.elapsed_time(b) for row in lat_ev for a, b in row])
        layer_step_us = {"median": round(float(np.median(lat_us)), 2),
                         "p90": round(float(np.percentile(lat_us, 90)), 2),
                         "mean": round(float(lat_us.mean()), 2), "n": int(lat_us.size),
                         "note": "eager calls after the timed region, an event pair around each MoE-layer "
                                 "decode (launch gaps included, so above the graph-replayed mean)"}
    except Exception as exc:   # diagnostics only
        layer_step_us = {"error": repr(exc)[:200]}
    run.close()

    # ---- end to end: a fresh cache, the same untimed prefix, then the same trace
    # steps as the timed region with host buffers in and the result out every step ----
    run2 = DecodeRunner(cfg, pool, offs, None, (b_pcie, b_cpu), dev, need)
    run2.warm(prefix)
    x_h = torch.from_numpy(run2.acts).pin_memory()
    ids_h = torch.from_numpy(run2.ids).pin_memory()
    w_h = torch.from_numpy(run2.w).pin_memory()
    out_h = torch.empty(s.L, cfg.T, s.H, dtype=torch.float32).pin_memory()
    torch.cuda.synchronize(dev)
    if world > 1:
        dist.barrier()
    cnt_e0 = run2.cache.state()[3].copy()
    e2, e3 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e2.record(run2.stream)
    run2.advance_host(args.steps, x_h, ids_h, w_h, out_h)
    e3.record(run2.stream)
    torch.cuda.synchronize(dev)
    ms_e2e = e2.elapsed_time(e3)
    dcnt_e = run2.cache.state()[3].copy() - cnt_e0
    if world > 1:
        t = torch.tensor([ms_e2e], device=dev)
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
        ms_e2e = float(t.item())
    h2d = run2.xb.numel() * run2.xb.element_size() + run2.ib.numel() * 4 + run2.wb.numel() * 4
    d2h = run2.out.numel() * 4
    run2.close()
    del pool

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
                   "graph": True,
                   "l2": "inputs larger than L2: each step reads ~48 x 8 x 9.4 MB of expert weights"},
        "window": window,
        "cache_stats": cache_stats(dcnt),
        "e2e": {"value": round(args.steps * s.L * world / (ms_e2e / 1e3), 1), "unit": UNIT,
                "h2d_bytes_per_step": int(h2d), "d2h_bytes_per_step": int(d2h),
                "window": f"the timed region's trace steps on a fresh cache after the same untimed prefix "
                          f"(fills {int(dcnt_e[2])} vs {int(dcnt[2])} in the timed region)"},
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
                     "traffic": RESIDENT_TRAFFIC[resident_path][0],
                     "traffic_source": RESIDENT_TRAFFIC[resident_path][1],
                     "bytes_per_layer_step": round(res_bytes / max(1, res_launches)),
                     "us_per_layer_step": round(1e3 * res_ms / max(1, res_launches), 2),
                     "layer_steps_timed": res_launches, "fills_during": res_fills,
                     "all_resident_layer_us": round(1e3 * ms_res / (res_reps * s.L), 2)},
        "in_step_gemv": {"note": "the same resident-expert kernels inside the step's mix (fills beside them; the "
                                 "event pairs in the graph also drop their programmatic overlap), 32 steps after "
                                 "the timed region",
                         "achieved_gbs": round(gb / (gms / 1e3) / 1e9, 1) if gms > 0 else None,
                         "frac": round(gb / (gms / 1e3) / 1e9 / hbm_peak, 3) if gms > 0 else None,
                         "bytes_per_layer_step": round(gb / max(1, gn)),
                         "us_per_layer_step": round(1e3 * gms / max(1, gn), 2)},
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
    if args.mode == "all" and not args.no_workloads:
        result["workloads"] = {n: decode_workload_measure(n, args, dev, (b_pcie, b_cpu), hbm_peak, peak_src,
                                                          rank == 0 and not args.no_cpu_baseline, bp_gbs)
                               for n in EXTRA_WORKLOADS}
    if args.mode == "all" and not args.no_nvfp4:
        result["nvfp4_decode"] = fp4_measure(args, dev, local, b_pcie, b_cpu, "nvfp4")
        result["mxfp4_decode"] = fp4_measure(args, dev, local, b_pcie, b_cpu, "mxfp4")
    if not args.no_prefill and args.mode == "all":
        result["prefill"] = prefill_measure(args, dev, local)
        if not args.no_nvfp4:
            result["prefill_mxfp4"] = prefill_fp4_measure(args, dev, local, "mxfp4")
    if rank == 0 and not args.no_cpu_baseline:
        result["cpu_baseline"] = run_cpu_baseline(args.cpu_seconds, args.pool_blobs, (b_pcie, b_cpu))
        cores = host_cores()
        if cores > 1:
            result["cpu_baseline_all_cores"] = run_cpu_baseline(args.cpu_seconds / 2, args.pool_blobs,
                                                                (b_pcie, b_cpu), threads=cores)
    if rank == 0:
        print(json.dumps(result))
    if world > 1:
        dist.destroy_process_group()


def cpu_branch_measure(args, dev, steps=32):
    """The CPU branch of the decode step (moe_cache_set_cpu_branch), on the headline
    shape with B_pcie = B_cpu, so about half the misses go to the CPU: the same
    trace steps with the CPU partial sums supplied by the caller, then computed
    by a registered host function from the page-locked copies of x, the ids and
    the slot map (a host node in the replayed step graph).  The host function
    here does the least a CPU branch can (it writes zeros for its pairs): the
    difference is the branch's own cost (the copies, the host node, the combine
    kernel after both branches) where it does not overlap the GPU path."""
    import torch
    cfg = config(WORKLOAD)
    s = cfg.shape
    arena, offs = make_pool(s, cfg.seed, n_phys=args.pool_blobs)
    pool = torch.from_numpy(arena).pin_memory()
    del arena
    bw = (100000, 100000)
    out = {"workload": f"{WORKLOAD} with B_pcie = B_cpu (hybrid: about half the misses to the CPU), "
                       f"C={cfg.capacity} slots", "steps": steps,
           "window": f"trace steps [{PREFIX_STEPS}, {PREFIX_STEPS + steps})"}
    for mode in ("supplied", "branch"):
        run = DecodeRunner(cfg, pool, offs, None, bw, dev, PREFIX_STEPS + steps + 8)
        host = {"calls": 0, "s": 0.0, "pairs": 0}
        if mode == "branch":
            def fn(layer, T, x, ids, sm, cp, host=host):
                t0 = time.perf_counter()
                cpu = sm < 0
                cp[cpu] = 0.0
                host["calls"] += 1
                host["pairs"] += int(cpu.sum())
                host["s"] += time.perf_counter() - t0
            run.cache.set_cpu_branch(fn)
        run.warm(PREFIX_STEPS)
        run.sync()
        host.update(calls=0, s=0.0, pairs=0)
        ms, dcnt = run.timed(steps)
        out[mode] = {"value": round(steps * s.L / (ms / 1e3), 1), "unit": UNIT, "ms_per_step": round(ms / steps, 4),
                     "cpu_assigned": int(dcnt[3]), "fills": int(dcnt[2]),
                     "kernels_per_layer": int(run.cache.info()[6])}
        if mode == "branch":
            out[mode]["host_calls"] = host["calls"]
            out[mode]["host_pairs"] = host["pairs"]
            out[mode]["host_us_per_call"] = round(1e6 * host["s"] / max(1, host["calls"]), 2)
            run.cache.set_cpu_branch(None)
        run.close()
    out["branch_cost_us_per_layer"] = round(1e3 * (out["branch"]["ms_per_step"] - out["supplied"]["ms_per_step"]) / s.L, 2)
    return out


def fill_step_measure(args, dev, b_p, calls=96, reps=6):
    """The link-bound layer-step against its floor.  One Qwen3-shaped layer with
    C = 8 slots and B_cpu = 0: every call routes the same 7 hot experts (resident
    after the first call) and one expert that no call of the last 96 routed, so
    each call fills exactly one 9.44 MB blob over the host link while the 7
    resident experts stream from HBM.  The calls are graph-replayed back to back;
    the same calls with the 8th expert hot too give the all-resident layer-step.
    A fill step cannot be shorter than its fill, which cannot start before the
    control kernel has picked the victim: the line reports the fill kernel's own
    event time beside one blob at bench_bw's B_P, and what the step spends
    outside the fill (control, the filled expert's down grid, the combine)."""
    import torch
    from dataclasses import replace
    from serving_layer_moe_gb300 import MoECache
    base = config(WORKLOAD)
    s = replace(base.shape, L=1)
    arena, offs = make_pool(s, base.seed, n_phys=32)
    pool = torch.from_numpy(arena).pin_memory()
    del arena
    rng = np.random.default_rng(base.seed)
    x = torch.from_numpy(rng.standard_normal((1, s.H)).astype(np.float32)).to(dev).to(torch.bfloat16).view(torch.int16)
    w_d = torch.full((calls, 1, s.k), 1.0 / s.k, dtype=torch.float32, device=dev)
    cpu = torch.zeros(1, s.k, s.H, dtype=torch.float32, device=dev)
    out_all = torch.empty(calls, 1, s.H, dtype=torch.float32, device=dev)
    stream = torch.cuda.Stream(device=dev)
    res = {"workload": f"{WORKLOAD} shape, one layer, C = {s.k} slots, B_cpu = 0: 7 hot experts + one expert "
                       f"not routed in the last {calls} calls (exactly one fill per call)",
           "calls_timed": calls * reps, "B_P_gbs": round(b_p, 1), "blob_bytes": s.blob_bytes}
    for mode in ("one_fill", "all_resident"):
        cache = MoECache(L=1, E=s.E, H=s.H, I=s.I, top_k=s.k, max_tokens=1, wdtype=s.wdtype, adtype=s.adtype,
                         host_pool=pool, blob_offsets=offs, n_slots=s.k, max_fetch=s.k,
                         bw_pcie_mbps=int(b_p * 1000), bw_cpu_mbps=0, device=dev.index or 0)
        ids = np.empty((calls, 1, s.k), np.int32)
        for c in range(calls):
            ids[c, 0, :s.k - 1] = np.arange(s.k - 1)
            ids[c, 0, s.k - 1] = s.k - 1 + (c % (s.E - s.k + 1) if mode == "one_fill" else 0)
        i_d = torch.from_numpy(ids).to(dev)

        def enqueue():
            for c in range(calls):
                cache.decode_ptrs(0, 1, x.data_ptr(), i_d[c].data_ptr(), w_d[c].data_ptr(), cpu.data_ptr(),
                                  out_all[c].data_ptr(), None, stream.cuda_stream)

        with torch.cuda.stream(stream):
            enqueue()                       # eager: fills the hot experts
        cache.plan()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            enqueue()
        cache.plan()
        with torch.cuda.stream(stream):
            g.replay()
        cache.plan()
        cnt0 = cache.state()[3].copy()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        with torch.cuda.stream(stream):
            e0.record(stream)
            for _ in range(reps):
                g.replay()
            e1.record(stream)
        cache.plan()
        ms = e0.elapsed_time(e1)
        dcnt = cache.state()[3].copy() - cnt0
        # kernel groups: event pairs in a second graph of the same calls
        cache.profile_start()
        pg = torch.cuda.CUDAGraph()
        with torch.cuda.graph(pg, stream=stream):
            enqueue()
        cache.profile_pause()
        cache.plan()
        prof = {k: [0.0, 0] for k in cache.PROFILE_KINDS}
        with torch.cuda.stream(stream):
            for _ in range(2):
                pg.replay()
                for k, (ms_k, n_k) in cache.profile_read().items():
                    prof[k][0] += ms_k
                    prof[k][1] += n_k
        cache.profile_stop()
        cache.close()
        r = {"us_per_call": round(1e3 * ms / (calls * reps), 2), "fills": int(dcnt[2]), "hits": int(dcnt[0]),
             "cpu_assigned": int(dcnt[3]),
             "group_us_per_call": {k: round(1e3 * v[0] / max(1, v[1]), 2) for k, v in prof.items() if v[1]}}
        res[mode] = r
    fill_ev = res["one_fill"]["group_us_per_call"].get("fill", 0.0)
    res["blob_at_B_P_us"] = round(s.blob_bytes / (b_p * 1e9) * 1e6, 2)
    res["fill_kernel_us"] = fill_ev
    res["outside_fill_us"] = round(res["one_fill"]["us_per_call"] - fill_ev, 2)
    res["note"] = ("fill_kernel_us: event pair around the fill kernel in a profiling graph of the same calls; "
                   "B_P is a long-transfer rate, one blob alone takes longer (first-byte latency and ramp); "
                   "outside_fill_us: control kernel + filled-expert down grid + combine + launch gaps")
    return res


# The other decode workloads, measured beside the headline: (untimed prefix, timed
# steps, distinct host-pool blobs, all-resident roofline possible).
EXTRA_WORKLOADS = {
    # 32-step trace of one layer: the window wraps around it
    "tiny": (8, 256, None, False),
    # the window spans the resize from 1228 to 737 slots before step 128
    "qwen3_decode_b16": (96, 64, 64, False),
    # 4 layers x (8 routed + 1 shared) fp8 experts; 32 routed experts fit C = 112
    "dsv3_decode_slice": (32, 64, 8, True),
}
WORKLOAD_DESC = {
    "tiny": "tiny single MoE layer: E=8, top-2, H 256, I 512, fp32 weights and activations, T=4, C=4 slots, "
            "B_pcie:B_cpu = 2:1",
    "qwen3_decode_b16": "Qwen3-30B-A3B-shaped decode at batch 16: 48 layers x 128 experts, top-8, bf16, "
                        "N(0,1) logits + per-expert bias N(0,0.5), B_pcie:B_cpu = 1:1, C = 1228 slots (20%) "
                        "resized to 737 (12%) before step 128",
    "dsv3_decode_slice": "DeepSeek-V3-shaped decode slice: 4 layers x 256 routed + 1 shared expert, top-8, "
                         "H 7168, I 2048, fp8 e4m3 with 128x128 fp32 scales (44 MB blobs), batch 1, C = 112 "
                         "slots (11%), Zipf(1.0) routing with 80% reuse",
}


def decode_workload_measure(name, args, dev, bw_measured, hbm_peak, peak_src, with_cpu, bw_link_gbs=None):
    """One of the other decode workloads: graph-replayed steps after an untimed
    prefix, the kernel groups' event times over profiled replays after the
    window, and a bounded oracle sample of the same workload."""
    import torch
    prefix, steps, n_phys, all_resident = EXTRA_WORKLOADS[name]
    cfg = config(name)
    s = cfg.shape
    bw = cfg.bw_mbps or bw_measured
    arena, offs = make_pool(s, cfg.seed, n_phys=n_phys)
    pool = torch.from_numpy(arena).pin_memory()
    del arena
    shared = make_shared(s, cfg.seed) if s.n_shared else None
    prof_steps = 16
    run = DecodeRunner(cfg, pool, offs, shared, bw, dev, prefix + steps + prof_steps + 8)
    run.warm(prefix)
    ms, dcnt = run.timed(steps)
    launches = int(run.cache.info()[6])
    prof, dcnt_p = run.profiled(prof_steps)
    groups = kernel_groups(s, prof, dcnt_p)
    total_prof_ms = sum(v[0] for v in prof.values())
    res = {"workload": WORKLOAD_DESC[name],
           "value": round(steps * s.L / (ms / 1e3), 1), "unit": UNIT, "steps": steps,
           "ms_per_step": round(ms / steps, 4),
           "window": {"trace_steps": f"[{prefix}, {prefix + steps}) mod {cfg.steps}", "untimed_prefix_steps": prefix},
           "cache_stats": cache_stats(dcnt), "gpu_launches": steps * s.L * launches,
           "B_pcie_mbps": bw[0], "B_cpu_mbps": bw[1], "blob_bytes": int(s.blob_bytes),
           "host_pool": f"{n_phys or s.n_flat} distinct seeded expert blobs, flat id f -> blob f mod "
                        f"{n_phys or s.n_flat}",
           "roofline": roofline_from_groups(groups, hbm_peak, peak_src, WORKLOAD_TRAFFIC.get(name),
                                            WORKLOAD_TRAFFIC_SOURCE.get(name)),
           # the fills' bytes over the window's wall time, against the calibrated host link
           "link": {"fill_bytes_per_step": round(int(dcnt[2]) * s.blob_bytes / steps),
                    "achieved_gbs": round(int(dcnt[2]) * s.blob_bytes / (ms / 1e3) / 1e9, 1),
                    "B_P_gbs": round(bw_link_gbs, 1),
                    "frac": round(int(dcnt[2]) * s.blob_bytes / (ms / 1e3) / 1e9 / bw_link_gbs, 3) if bw_link_gbs else None,
                    "note": "fill bytes of the timed window over its whole wall time (a lower bound of the fill "
                            "rate), against bench_bw's B_P"},
           "roofline_note": "the kernel group with the most event time, over profiled replays of the "
                            f"{prof_steps} steps after the timed window (fills and CPU-assigned pairs as they occur)",
           "kernel_groups": {k: {"bytes_per_launch": round(b / max(1, n)), "us_per_launch": round(1e3 * m / max(1, n), 2),
                                 "gbs": round(b / (m / 1e3) / 1e9, 1) if m > 0 else None}
                             for k, (b, m, n) in groups.items()},
           "kernel_ms_share": {k: round(v[0] / total_prof_ms, 3) for k, v in prof.items() if v[1]},
           "control_us": round(1e3 * prof["control"][0] / max(1, prof["control"][1]), 2)}
    if run.resize_ms is not None:
        res["resize_ms"] = round(run.resize_ms, 2)
        res["resize_note"] = "moe_cache_resize (a safe point that synchronises) plus the graph re-capture, inside " \
                             "the timed window"
    if all_resident:
        run.profiled(3, same_step=True)
        rp, dr = run.profiled(16, same_step=True)
        rg = kernel_groups(s, rp, dr)
        tr, trs = ALL_RESIDENT_TRAFFIC.get(name, (None, None))
        res["roofline_all_resident"] = roofline_from_groups({"gemv_resident": rg["gemv_resident"]}, hbm_peak, peak_src,
                                                            tr, trs, split="down_filled" in rg)
        res["roofline_all_resident_note"] = "one step's inputs replayed until every routed expert is resident; " \
                                            f"{int(dr[2])} fills during the 16 replays"
    run.close()
    if with_cpu:
        res["cpu_baseline"] = run_cpu_baseline(min(args.cpu_seconds, 6.0), n_phys or s.n_flat, bw, workload=name)
    return res


def profile_case(args, dev):
    """A small decode case for ncu captures (a few GB on the device): the shape of
    --profile-workload (default the qwen3 b1 one) with --profile-layers layers and
    256 slots (--capacity to change), the workload's bandwidth split if it fixes
    one (else every miss fills), --steps eager steps of single decode calls, no
    graph, no timing.  With --profile-allhit every step replays step 0, so all
    routed experts are resident after the first."""
    import torch
    from serving_layer_moe_gb300 import MoECache
    name = args.profile_workload
    base = config(name)
    cfg = base.with_(shape=base.shape.__class__(**{**base.shape.__dict__, "L": min(args.profile_layers, base.shape.L)}),
                     resize_step=None, resize_to=None)
    s = cfg.shape
    arena, offs = make_pool(s, cfg.seed, n_phys=min(16, s.n_flat))
    pool = torch.from_numpy(arena).pin_memory()
    shared = make_shared(s, cfg.seed) if s.n_shared else None
    bw = cfg.bw_mbps or (192000, 0)   # the workload's split where it fixes one, else every miss fills
    cache = MoECache(L=s.L, E=s.E, H=s.H, I=s.I, top_k=s.k, max_tokens=cfg.T, wdtype=s.wdtype, adtype=s.adtype,
                     host_pool=pool, blob_offsets=offs, shared=shared, n_slots=args.capacity or 256,
                     bw_pcie_mbps=bw[0], bw_cpu_mbps=bw[1], device=dev.index or 0)
    ids, w = routing_trace(cfg)
    out = torch.empty(cfg.T, s.H, device=dev)
    cpu = torch.zeros(cfg.T, s.k, s.H, device=dev)   # the CPU-assigned pairs' partial sums (zeros)
    for st0 in range(args.steps):
        st = 0 if args.profile_allhit else st0 % cfg.steps
        for l in range(s.L):
            xa = activations(cfg, st, l)
            x = torch.from_numpy(xa.view(np.int16) if xa.dtype == np.uint16 else xa).to(dev)
            cache.decode(l, x, torch.from_numpy(ids[st, l]).to(dev), torch.from_numpy(w[st, l]).to(dev), out,
                         cpu_part=cpu)
    torch.cuda.synchronize(dev)
    c = cache.state()[3]
    print(json.dumps({"profile_case": f"{name} shape, {s.L} layers, {int(cache.info()[1])} slots",
                      "hits": int(c[0]), "misses": int(c[1]), "fills": int(c[2]), "cpu_assigned": int(c[3])}))
    cache.close()


FP4_DESC = {"nvfp4": "NVFP4 experts (e2m1 + e4m3 per 16 + fp32 per matrix)",
            "mxfp4": "MXFP4 experts (e2m1 + e8m0 per 32)"}


def fp4_measure(args, dev, local, b_pcie, b_cpu, fmt, steps=64):
    """The decode workload with 4-bit experts (same shape, routing and slot count):
    a blob is 2.65 MB (NVFP4) or 2.51 MB (MXFP4) instead of 9.44 MB, so fills
    and the resident GEMVs move 3.6x or 3.8x fewer bytes.  Graph replay of whole
    steps after the same untimed prefix as the headline, inputs resident."""
    import torch
    base = config(WORKLOAD)
    cfg = base.with_(shape=base.shape.__class__(**{**base.shape.__dict__, "wdtype": fmt}))
    s = cfg.shape
    arena, offs = make_pool(s, cfg.seed, n_phys=args.pool_blobs)
    pool = torch.from_numpy(arena).pin_memory()
    del arena
    run = DecodeRunner(cfg, pool, offs, None, (b_pcie, b_cpu), dev, PREFIX_STEPS + steps)
    run.warm(PREFIX_STEPS)
    ms, dcnt = run.timed(steps)
    run.close()
    return {"workload": f"{WORKLOAD} with {FP4_DESC[fmt]}, C={cfg.capacity} slots",
            "value": round(steps * s.L / (ms / 1e3), 1), "unit": UNIT, "steps": steps,
            "window": f"trace steps [{PREFIX_STEPS}, {PREFIX_STEPS + steps})",
            "ms_per_step": round(ms / steps, 4), "blob_bytes": int(s.blob_bytes),
            "fills": int(dcnt[2]), "hits": int(dcnt[0])}


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
        cpu_worker(a.cpu_seconds, a.pool_blobs, (int(b[0]), int(b[1])), samples=a.cpu_samples,
                   workload=a.cpu_workload)
    else:
        main(a)
