"""Shared driver for GPU parity tests: run a workload through libmoecache.so and the oracle side by side.

Importable without a GPU; the functions that run need CUDA.
"""
from __future__ import annotations

from dataclasses import dataclass, field

import numpy as np

from oracle.cache import SlotCache
from oracle.ffn import ExpertStore, combine, pair_outputs, relative_max_error, shared_outputs
from workloads import (Config, activations, default_max_fetch, make_pool, make_shared,
                       routing_trace)

TOL = 2e-2   # max |y - y_ref| / max |y_ref| for bf16 / fp8 weights with fp32 accumulation


def torch_act(x: np.ndarray, dev):
    import torch
    if x.dtype == np.uint16:
        return torch.from_numpy(x.view(np.int16)).to(dev)
    return torch.from_numpy(np.ascontiguousarray(x)).to(dev)


@dataclass
class DecodeRun:
    max_err: float = 0.0
    fp_checked: int = 0
    calls: int = 0
    cpu_pairs: int = 0
    fills: int = 0
    mismatches: list = field(default_factory=list)


def build_pool(cfg: Config, n_phys=None, pinned=True):
    import torch
    s = cfg.shape
    arena, offs = make_pool(s, cfg.seed, n_phys=n_phys)
    pool = torch.from_numpy(arena).pin_memory() if pinned else arena
    return arena, offs, pool


def make_cache(cfg: Config, pool, offs, shared, bw, max_prefill_tokens=0, n_slots=None, device=0):
    from serving_layer_moe_gb300 import MoECache
    s = cfg.shape
    K = cfg.max_fetch if cfg.max_fetch is not None else default_max_fetch(s, cfg.T)
    return MoECache(L=s.L, E=s.E, H=s.H, I=s.I, top_k=s.k, max_tokens=cfg.T, wdtype=s.wdtype,
                    adtype=s.adtype, host_pool=pool, blob_offsets=offs, shared=shared,
                    n_slots=n_slots or cfg.capacity, max_fetch=K, bw_pcie_mbps=bw[0], bw_cpu_mbps=bw[1],
                    device=device, max_prefill_tokens=max_prefill_tokens), K


def run_decode_parity(cfg: Config, bw, n_phys=None, fp_every=1, fp_limit=None, check_plan=True,
                      pinned=True, state_every=1, fp_steps=(), memo=16, trace=None) -> DecodeRun:
    """Replay cfg's decode trace on the GPU and in the oracle; compare control state bit for bit.

    Every call: slot map (bit-exact) and, with check_plan, q / victims / fills.
    Every `state_every` steps: slot table, stamps, flat-id table, counters, clock.
    Every `fp_every`-th layer-step (up to fp_limit), and every layer-step of the
    steps in `fp_steps`: the layer output within TOL, with the CPU-assigned
    pairs' partial sums supplied from the oracle and NaN planted in every entry
    the combine must not read.  `memo`: parsed experts the oracle keeps.
    `trace`: (ids, gates) replacing cfg's generated routing.
    """
    import torch
    s = cfg.shape
    dev = torch.device("cuda", 0)
    arena, offs, pool = build_pool(cfg, n_phys=n_phys, pinned=pinned)
    shared = make_shared(s, cfg.seed) if s.n_shared else None
    cache, K = make_cache(cfg, pool, offs, shared, bw)
    ora = SlotCache(s.L, s.E, cfg.capacity, K, bw[0], bw[1])
    store = ExpertStore(arena, offs, s.wdtype, s.H, s.I, s.blob_bytes, memo=memo)
    fp_steps = set(fp_steps)
    ids, w = routing_trace(cfg) if trace is None else trace
    res = DecodeRun()
    out = torch.empty(cfg.T, s.H, device=dev)
    sm = torch.empty(cfg.T, s.k, dtype=torch.int32, device=dev)
    zeros_cpu = torch.zeros(cfg.T, s.k, s.H, device=dev)
    n = 0
    for st in range(cfg.steps):
        if cfg.resize_step is not None and st == cfg.resize_step:
            ora.resize(cfg.resize_to)
            cache.resize(cfg.resize_to)
        for l in range(s.L):
            plan = ora.decode(l, ids[st, l])
            x = activations(cfg, st, l)
            check_fp = (st in fp_steps) or ((n % fp_every == 0) and (fp_limit is None or res.fp_checked < fp_limit))
            n += 1
            if check_fp:
                y = pair_outputs(store, l, s.E, x, s.adtype, ids[st, l])
                sh_y = shared_outputs(shared, l, s.wdtype, s.H, s.I, s.blob_bytes, x, s.adtype) \
                    if shared is not None else None
                ref = combine(w[st, l], y, plan.slot_map, y, shared_y=sh_y)
                cpu = torch.from_numpy(np.where(plan.slot_map[..., None] < 0, y, np.nan)
                                       .astype(np.float32)).to(dev)
            else:
                cpu = zeros_cpu
            cache.decode(l, torch_act(x, dev), torch.from_numpy(ids[st, l]).to(dev),
                         torch.from_numpy(w[st, l]).to(dev), out, cpu_part=cpu, slot_map=sm)
            res.calls += 1
            got_sm = sm.cpu().numpy()
            if not np.array_equal(got_sm, plan.slot_map):
                res.mismatches.append(("slot_map", st, l, got_sm.tolist(), plan.slot_map.tolist()))
                return res
            if check_plan:
                p = cache.plan()
                if p["q"] != plan.q or p["victims"] != plan.victims or p["fills"] != plan.fills \
                        or p["h"] != len(plan.hits) or p["m"] != len(plan.misses):
                    res.mismatches.append(("plan", st, l, p, (plan.q, plan.victims, plan.fills)))
                    return res
            res.cpu_pairs += int((plan.slot_map < 0).sum())
            res.fills += plan.q
            if check_fp:
                got = out.cpu().numpy()
                if not np.all(np.isfinite(got)):
                    res.mismatches.append(("nonfinite", st, l))
                    return res
                err = relative_max_error(got, ref)
                res.max_err = max(res.max_err, err)
                res.fp_checked += 1
        if (st + 1) % state_every == 0 or st == cfg.steps - 1:
            g = cache.state()
            o = ora.state()
            for name, a, b in zip(["s2e", "stamps", "e2s", "counters"], g[:4], o[:4]):
                if not np.array_equal(a, b):
                    res.mismatches.append(("state", st, name))
                    return res
            if g[4] != o[4]:
                res.mismatches.append(("clock", st, g[4], o[4]))
                return res
    cache.close()
    return res


POOL_SHORT_STEP = 7


def pool_short_trace(tail_steps=8, seed=95):
    """A one-layer trace on which the kept pool of the 64 least-recent slots holds
    fewer evictable slots than the call needs, even after a rebuild.

    100 slots, 128 experts, top-8 over 16 tokens (128 routed pairs), K = 16, so
    the pool keeps min(C, max(64, 4K)) = 64 keys.  Steps 0-6 fill every slot
    (experts 0-95 in groups of 16, then 84-99); step POOL_SHORT_STEP routes
    experts 0-59 (60 hits, all among the 64 least recent) and 100-115 (16
    misses): 4 evictable pool entries for 16 victims, so the victims come from
    the selection over all slots.  `tail_steps` steps of random routing follow.
    Returns (cfg, ids [steps, 1, 16, 8], gates).
    """
    from workloads import Shape
    shape = Shape(L=1, E=128, k=8, H=256, I=128, wdtype="bf16", adtype="bf16")
    T, k = 16, 8
    groups = [list(range(b, b + 16)) for b in (0, 16, 32, 48, 64, 80, 84)]
    groups.append(list(range(60)) + list(range(100, 116)))
    steps = len(groups) + tail_steps
    ids = np.empty((steps, 1, T, k), np.int32)
    for st, grp in enumerate(groups):
        for t in range(T):
            ids[st, 0, t] = [grp[(k * t + i) % len(grp)] for i in range(k)]
    g = np.random.default_rng(seed)
    for st in range(len(groups), steps):
        for t in range(T):
            ids[st, 0, t] = g.choice(shape.E, size=k, replace=False)
    w = g.dirichlet(np.ones(k), size=(steps, 1, T)).astype(np.float32)
    cfg = Config("pool_short", shape, T=T, steps=steps, capacity=100, routing="softmax", seed=seed,
                 max_fetch=16)
    return cfg, ids, w
