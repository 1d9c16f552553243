"""Failure handling, made to happen from the host (no GPU fault, trap or hang).

* Allocation failures: MOE_INJECT_ALLOC_FAILURE=n makes the n-th device or
  page-locked allocation (or host-pool registration) of one moe_cache_create
  or moe_cache_resize call report out of memory.  Create must return
  MOE_ENOMEM at every such point and leave nothing behind; a failed resize
  must return MOE_ENOMEM and keep the old pool, so decode goes on matching the
  oracle bit for bit.
* A bounded device wait that runs out: with MOE_TEST_UNSET_WAIT=1 when the
  cache is created, the resident experts' down kernel also waits for a word
  nothing writes.  It gives up after 20 ms, flags the timeout and returns; the next
  call on the cache reports MOE_EDEVICE, and a fresh cache afterwards computes
  correctly.
"""
import os
from dataclasses import replace

import numpy as np
import pytest

from tests.harness import TOL, build_pool, make_cache, run_decode_parity, torch_act
from workloads import QWEN3, activations, config, routing_trace

pytestmark = pytest.mark.gpu

ENOMEM, EDEVICE = 2, 6


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import serving_layer_moe_gb300 as m
    m.load_library()


def _qwen3_small(T=1, steps=8, layers=4, **kw):
    shape = replace(QWEN3, L=layers)
    return config("qwen3_decode_b1").with_(shape=shape, T=T, steps=steps,
                                           capacity=int(0.37 * layers * shape.E), **kw)


def test_create_fails_cleanly_at_every_allocation(monkeypatch):
    from serving_layer_moe_gb300 import MoEError
    cfg = config("tiny")
    arena, offs, _ = build_pool(cfg, pinned=False)   # pageable: the library registers it (one more point)
    failed = 0
    for n in range(1, 40):
        monkeypatch.setenv("MOE_INJECT_ALLOC_FAILURE", str(n))
        try:
            c, _ = make_cache(cfg, arena, offs, None, cfg.bw_mbps, max_prefill_tokens=0)
        except MoEError as e:
            assert e.status == ENOMEM, (n, str(e))
            failed += 1
            continue
        c.close()
        break
    else:
        pytest.fail("create never succeeded")
    assert failed >= 10, failed   # registration, offsets, slots, tables, work buffers, error word ...
    monkeypatch.delenv("MOE_INJECT_ALLOC_FAILURE")
    res = run_decode_parity(cfg.with_(steps=6), cfg.bw_mbps, pinned=False)
    assert not res.mismatches and res.max_err <= TOL


def test_failed_resize_keeps_the_old_pool(monkeypatch):
    import torch
    from oracle.cache import SlotCache
    from serving_layer_moe_gb300 import MoEError
    cfg = _qwen3_small(steps=10)
    s = cfg.shape
    dev = torch.device("cuda", 0)
    arena, offs, pool = build_pool(cfg, n_phys=16)
    bw = (100000, 100000)
    cache, K = make_cache(cfg, pool, offs, None, bw)
    ora = SlotCache(s.L, s.E, cfg.capacity, K, bw[0], bw[1])
    ids, w = routing_trace(cfg)
    out = torch.empty(cfg.T, s.H, device=dev)
    sm = torch.empty(cfg.T, s.k, dtype=torch.int32, device=dev)
    cpu = torch.zeros(cfg.T, s.k, s.H, device=dev)

    def step(st):
        for l in range(s.L):
            plan = ora.decode(l, ids[st, l])
            cache.decode(l, torch_act(activations(cfg, st, l), dev), torch.from_numpy(ids[st, l]).to(dev),
                         torch.from_numpy(w[st, l]).to(dev), out, cpu_part=cpu, slot_map=sm)
            assert np.array_equal(sm.cpu().numpy(), plan.slot_map), (st, l)

    def same_state():
        g, o = cache.state(), ora.state()
        return all(np.array_equal(a, b) for a, b in zip(g[:4], o[:4])) and g[4] == o[4]

    for st in range(4):
        step(st)
    assert same_state()
    for n in (1, 2, 3, 4):          # each of the resize's four allocations
        monkeypatch.setenv("MOE_INJECT_ALLOC_FAILURE", str(n))
        with pytest.raises(MoEError) as ei:
            cache.resize(cfg.capacity // 2)
        assert ei.value.status == ENOMEM
        assert cache.C == cfg.capacity and same_state()
    monkeypatch.delenv("MOE_INJECT_ALLOC_FAILURE")
    for st in range(4, 7):
        step(st)
    assert same_state()
    cache.resize(cfg.capacity // 2)   # and a resize that succeeds still matches the oracle's
    ora.resize(cfg.capacity // 2)
    assert same_state()
    for st in range(7, 10):
        step(st)
    assert same_state()
    cache.close()


@pytest.mark.parametrize("mode,path", [("grids", 0)])
def test_bounded_wait_runs_out_and_is_reported(monkeypatch, mode, path):
    import torch
    from serving_layer_moe_gb300 import MoEError
    cfg = _qwen3_small(steps=2, layers=2)
    s = cfg.shape
    dev = torch.device("cuda", 0)
    arena, offs, pool = build_pool(cfg, n_phys=8)
    monkeypatch.delenv("MOE_DECODE_FUSED", raising=False)
    monkeypatch.setenv("MOE_DECODE_RESIDENT", mode)
    monkeypatch.setenv("MOE_TEST_UNSET_WAIT", "1")
    cache, _ = make_cache(cfg, pool, offs, None, (100000, 0))
    monkeypatch.delenv("MOE_TEST_UNSET_WAIT")
    monkeypatch.delenv("MOE_DECODE_RESIDENT")
    assert int(cache.info()[7]) == path          # how the resident experts run
    ids, w = routing_trace(cfg)
    out = torch.empty(cfg.T, s.H, device=dev)
    x = torch_act(activations(cfg, 0, 0), dev)
    i_d, w_d = torch.from_numpy(ids[0, 0]).to(dev), torch.from_numpy(w[0, 0]).to(dev)
    cache.decode(0, x, i_d, w_d, out)           # cold: fills only
    cache.decode(0, x, i_d, w_d, out)           # every expert resident: the test wait runs out
    torch.cuda.synchronize()                    # the kernel returned (bounded waits)
    with pytest.raises(MoEError) as ei:
        cache.state()
    assert ei.value.status == EDEVICE and "timed out" in str(ei.value)
    cache.state()                               # the error was reported once and cleared
    cache.close()
    res = run_decode_parity(_qwen3_small(steps=4, layers=2), (100000, 0), n_phys=8)
    assert not res.mismatches and res.max_err <= TOL
