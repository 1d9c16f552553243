"""The CPU branch of the decode step (moe_cache_set_cpu_branch), against the oracle.

The pages run the CPU-assigned experts on the host from a host-function node of
the captured step, between a copy of what they read to the host and a copy of
their partial sums back, beside the GPU path; the exact merge waits for both.
Here the registered host function computes the CPU-assigned pairs with the
oracle's float64 expert, so the layer output must match the oracle's combine
within the tolerance and the slot maps bit for bit, eagerly and when a whole
step is captured in a CUDA graph and replayed.

The host function runs on a CUDA driver thread and takes the interpreter lock,
so these tests wait for the device only through the library (plan() and
state() release the lock) before touching tensors.
"""
from dataclasses import replace

import numpy as np
import pytest

from oracle.cache import SlotCache
from oracle.ffn import ExpertStore, combine, pair_outputs, relative_max_error
from oracle.formats import activations_to_f64
from tests.harness import TOL, build_pool, make_cache, torch_act
from workloads import QWEN3, activations, config, routing_trace

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import serving_layer_moe_gb300 as m
    m.load_library()


def _cfg(layers=4, steps=6, T=1):
    shape = replace(QWEN3, L=layers)
    return config("qwen3_decode_b1").with_(shape=shape, T=T, steps=steps, capacity=int(0.2 * layers * shape.E))


class OracleBranch:
    """The host function: the CPU-assigned pairs through the oracle's float64 expert."""

    def __init__(self, store, cfg):
        self.store, self.cfg, self.calls, self.pairs = store, cfg, [], 0

    def __call__(self, layer, T, x, ids, sm, cpu_part):
        s = self.cfg.shape
        xf = activations_to_f64(np.array(x), s.adtype)
        self.calls.append((layer, T))
        for t in range(T):
            for j in range(s.k):
                if sm[t, j] < 0:
                    cpu_part[t, j] = self.store.expert(layer * s.E + int(ids[t, j]), xf[t]).astype(np.float32)
                    self.pairs += 1


@pytest.mark.parametrize("T", [1, 4])
def test_cpu_branch_matches_the_oracle(T):
    import torch
    cfg = _cfg(T=T)
    s = cfg.shape
    dev = torch.device("cuda", 0)
    bw = (100000, 100000)   # half the misses go to the CPU
    arena, offs, pool = build_pool(cfg, n_phys=24)
    cache, K = make_cache(cfg, pool, offs, None, bw)
    store = ExpertStore(arena, offs, s.wdtype, s.H, s.I, s.blob_bytes, memo=32)
    branch = OracleBranch(store, cfg)
    cache.set_cpu_branch(branch)
    ora = SlotCache(s.L, s.E, cfg.capacity, K, bw[0], bw[1])
    ids, w = routing_trace(cfg)
    out = torch.empty(cfg.T, s.H, device=dev)
    sm = torch.empty(cfg.T, s.k, dtype=torch.int32, device=dev)
    worst, cpu_pairs = 0.0, 0
    for st in range(cfg.steps):
        for l in range(s.L):
            plan = ora.decode(l, ids[st, l])
            x = activations(cfg, st, l)
            cache.decode(l, torch_act(x, dev), torch.from_numpy(ids[st, l]).to(dev),
                         torch.from_numpy(w[st, l]).to(dev), out, slot_map=sm)
            cache.plan()   # waits for the device through the library
            assert np.array_equal(sm.cpu().numpy(), plan.slot_map), (st, l)
            y = pair_outputs(store, l, s.E, x, s.adtype, ids[st, l])
            ref = combine(w[st, l], y, plan.slot_map, y)
            got = out.cpu().numpy()
            assert np.all(np.isfinite(got))
            worst = max(worst, relative_max_error(got, ref))
            cpu_pairs += int((plan.slot_map < 0).sum())
    assert worst <= TOL, worst
    assert cpu_pairs > 0 and branch.pairs == cpu_pairs
    assert len(branch.calls) == cfg.steps * s.L and all(c[1] == T for c in branch.calls)
    g, o = cache.state(), ora.state()
    assert all(np.array_equal(a, b) for a, b in zip(g[:4], o[:4])) and g[4] == o[4]
    # removed again: the caller's cpu_part is read once more
    cache.set_cpu_branch(None)
    plan = ora.decode(0, ids[0, 0])
    x = activations(cfg, 0, 0)
    y = pair_outputs(store, 0, s.E, x, s.adtype, ids[0, 0])
    cpu = torch.from_numpy(np.where(plan.slot_map[..., None] < 0, y, np.nan).astype(np.float32)).to(dev)
    cache.decode(0, torch_act(x, dev), torch.from_numpy(ids[0, 0]).to(dev), torch.from_numpy(w[0, 0]).to(dev),
                 out, cpu_part=cpu, slot_map=sm)
    cache.plan()
    assert relative_max_error(out.cpu().numpy(), combine(w[0, 0], y, plan.slot_map, y)) <= TOL
    cache.close()


def test_cpu_branch_in_a_captured_step_graph():
    import torch
    cfg = _cfg(layers=3, steps=6)
    s = cfg.shape
    dev = torch.device("cuda", 0)
    bw = (100000, 100000)
    arena, offs, pool = build_pool(cfg, n_phys=24)
    cache, K = make_cache(cfg, pool, offs, None, bw)
    store = ExpertStore(arena, offs, s.wdtype, s.H, s.I, s.blob_bytes, memo=32)
    branch = OracleBranch(store, cfg)
    cache.set_cpu_branch(branch)
    ora = SlotCache(s.L, s.E, cfg.capacity, K, bw[0], bw[1])
    ids, w = routing_trace(cfg)
    xs = torch.stack([torch.stack([torch_act(activations(cfg, st, l), dev) for l in range(s.L)])
                      for st in range(cfg.steps)])
    ids_d, w_d = torch.from_numpy(ids).to(dev), torch.from_numpy(w).to(dev)
    xb, ib, wb = torch.empty_like(xs[0]), torch.empty_like(ids_d[0]), torch.empty_like(w_d[0])
    out = torch.empty(s.L, cfg.T, s.H, device=dev)
    stream = torch.cuda.Stream(device=dev)
    with torch.cuda.stream(stream):   # one eager step first (fills the cache like any step)
        xb.copy_(xs[0]); ib.copy_(ids_d[0]); wb.copy_(w_d[0])
        for l in range(s.L):
            cache.decode(l, xb[l], ib[l], wb[l], out[l], stream=stream)
    cache.plan()
    for l in range(s.L):
        ora.decode(l, ids[0, l])
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=stream):
        for l in range(s.L):
            cache.decode(l, xb[l], ib[l], wb[l], out[l], stream=stream)
    cache.plan()
    n_calls = len(branch.calls)
    worst = 0.0
    for st in range(1, cfg.steps):
        with torch.cuda.stream(stream):
            xb.copy_(xs[st]); ib.copy_(ids_d[st]); wb.copy_(w_d[st])
            graph.replay()
        cache.plan()
        got = out.cpu().numpy()
        for l in range(s.L):
            plan = ora.decode(l, ids[st, l])
            x = activations(cfg, st, l)
            y = pair_outputs(store, l, s.E, x, s.adtype, ids[st, l])
            worst = max(worst, relative_max_error(got[l], combine(w[st, l], y, plan.slot_map, y)))
    assert worst <= TOL, worst
    assert len(branch.calls) == n_calls + (cfg.steps - 1) * s.L   # the host node ran in every replay
    assert branch.pairs > 0
    g, o = cache.state(), ora.state()
    assert all(np.array_equal(a, b) for a, b in zip(g[:4], o[:4])) and g[4] == o[4]
    cache.close()
