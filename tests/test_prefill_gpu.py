"""Prefill parity on the GPU: full-layer double buffering and on-demand groups vs the oracle.

Residency state after every layer must be bit-exact; outputs within 2e-2
relative max error (h is stored as bf16 between the two GEMMs).
"""
import numpy as np
import pytest

from oracle.cache import SlotCache
from oracle.ffn import ExpertStore, combine, pair_outputs, relative_max_error
from tests.harness import TOL, torch_act
from workloads import Config, Shape, activations, config, make_pool, prefill_routing, routing_trace

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")


def _make(cfg, C, n_phys=None, max_tokens=None):
    import torch
    from serving_layer_moe_gb300 import MoECache
    s = cfg.shape
    arena, offs = make_pool(s, cfg.seed, n_phys=n_phys)
    pool = torch.from_numpy(arena).pin_memory()
    if max_tokens is None:
        max_tokens = 16
    cache = MoECache(L=s.L, E=s.E, H=s.H, I=s.I, top_k=s.k, max_tokens=max_tokens, wdtype=s.wdtype,
                     adtype=s.adtype, host_pool=pool, blob_offsets=offs, n_slots=C, bw_pcie_mbps=1000,
                     bw_cpu_mbps=0, device=0, max_prefill_tokens=cfg.T)
    store = ExpertStore(arena, offs, s.wdtype, s.H, s.I, s.blob_bytes, memo=2 * s.E + 4)
    return cache, store


def _check_state(cache, ora):
    g = cache.state()
    o = ora.state()
    for name, a, b in zip(["s2e", "stamps", "e2s", "counters"], g[:4], o[:4]):
        assert np.array_equal(a, b), name
    assert g[4] == o[4]


def _run_prefill(cfg, C, layers, n_phys=None, sample=None, seed=0, prefetch_next=True):
    """prefetch_next: the second buffer on or off, for every call or per call (a list)."""
    import torch
    s = cfg.shape
    dev = torch.device("cuda", 0)
    cache, store = _make(cfg, C, n_phys=n_phys)
    ora = SlotCache(s.L, s.E, C, K=s.E, b_pcie=1000, b_cpu=0)
    out = torch.empty(cfg.T, s.H, device=dev)
    worst = 0.0
    g = np.random.default_rng(seed)
    modes = prefetch_next if isinstance(prefetch_next, list) else [prefetch_next] * len(layers)
    for l, nxt in zip(layers, modes):
        ids, w = prefill_routing(cfg, l)
        x = activations(cfg, 0, l)
        cache.set_prefill_prefetch(nxt)
        plan = ora.prefill(l, ids, prefetch_next=nxt)
        cache.prefill(l, torch_act(x, dev), torch.from_numpy(ids).to(dev), torch.from_numpy(w).to(dev), out)
        torch.cuda.synchronize()
        _check_state(cache, ora)
        got = out.cpu().numpy()
        assert np.all(np.isfinite(got))
        toks = np.arange(cfg.T) if sample is None else np.sort(g.choice(cfg.T, size=sample, replace=False))
        mask = np.zeros(ids.shape, bool)
        mask[toks] = True
        y = pair_outputs(store, l, s.E, x, s.adtype, ids, mask=mask)
        ref = combine(w[toks], y[toks], np.zeros((len(toks), s.k), np.int32), None)
        err = relative_max_error(got[toks], ref)
        worst = max(worst, err)
        assert err <= TOL, (l, err)
    cache.close()
    return worst, ora


SMALL = Config("prefill_small", Shape(L=3, E=8, k=2, H=256, I=128, wdtype="bf16", adtype="bf16"),
               T=300, steps=1, capacity=16, routing="softmax", seed=4321, prefill=True)


def test_small_full_layer_double_buffer():
    worst, ora = _run_prefill(SMALL, C=16, layers=[0, 1, 2])
    assert worst < 5e-3


def test_small_repeat_and_out_of_order_layers():
    _run_prefill(SMALL, C=17, layers=[2, 0, 1, 1, 0])


def test_small_without_second_buffer():
    # each call loads only its own layer (the pages' no-second-buffer comparison)
    worst, ora = _run_prefill(SMALL, C=16, layers=[0, 1, 2, 1], prefetch_next=False)
    assert worst < 5e-3


def test_second_buffer_switch_midway_and_bad_values():
    import serving_layer_moe_gb300 as m
    # on, off (layer 1 is already resident: nothing to load), on, off
    _run_prefill(SMALL, C=17, layers=[0, 1, 2, 0, 1], prefetch_next=[True, False, True, False, False])
    cache, _ = _make(SMALL, 16)
    lib = m.load_library()
    assert lib.moe_cache_set_prefill_prefetch(cache._h, 2) == 1
    assert lib.moe_cache_set_prefill_prefetch(None, 1) == 1
    cache.close()


def test_small_on_demand_one_group():
    _run_prefill(SMALL, C=12, layers=[0, 1, 2, 0])      # E <= C < 2E


def test_small_on_demand_several_groups():
    _run_prefill(SMALL, C=3, layers=[0, 1, 2])          # C < E: groups of 3 routed experts


def test_ragged_tokens_and_tiny_chunk():
    for T in (1, 7, 129):
        _run_prefill(SMALL.with_(T=T), C=16, layers=[0, 1])


def test_qwen3_shape_1k_tokens():
    cfg = config("qwen3_prefill_8k").with_(T=1024)
    _run_prefill(cfg, C=300, layers=[0, 1, 2], n_phys=64, sample=256)


def test_qwen3_prefill_8k_every_token_of_two_layers():
    # the whole 8192-token chunk's outputs, every token, for a layer loaded in full and
    # the one prefetched beside its GEMMs
    cfg = config("qwen3_prefill_8k")
    worst, _ = _run_prefill(cfg, C=cfg.capacity, layers=[0, 1], n_phys=64, sample=None)
    assert worst <= TOL


def test_qwen3_prefill_8k_all_layers_state_and_sampled_outputs():
    import torch
    cfg = config("qwen3_prefill_8k")
    s = cfg.shape
    dev = torch.device("cuda", 0)
    cache, store = _make(cfg, cfg.capacity, n_phys=64)
    ora = SlotCache(s.L, s.E, cfg.capacity, K=s.E, b_pcie=1000, b_cpu=0)
    out = torch.empty(cfg.T, s.H, device=dev)
    g = np.random.default_rng(7)
    for l in range(s.L):
        ids, w = prefill_routing(cfg, l)
        x = activations(cfg, 0, l)
        ora.prefill(l, ids)
        cache.prefill(l, torch_act(x, dev), torch.from_numpy(ids).to(dev), torch.from_numpy(w).to(dev), out)
        if l in (0, 23, 47):
            torch.cuda.synchronize()
            _check_state(cache, ora)
            toks = np.sort(g.choice(cfg.T, size=48, replace=False))
            mask = np.zeros(ids.shape, bool)
            mask[toks] = True
            y = pair_outputs(store, l, s.E, x, s.adtype, ids, mask=mask)
            ref = combine(w[toks], y[toks], np.zeros((len(toks), s.k), np.int32), None)
            err = relative_max_error(out.cpu().numpy()[toks], ref)
            assert err <= TOL, (l, err)
    torch.cuda.synchronize()
    _check_state(cache, ora)
    cache.close()


def test_prefill_survivors_seed_decode():
    # prefill and decode share one pool: decode after prefill starts from the survivors
    import torch
    cfg = SMALL
    s = cfg.shape
    dev = torch.device("cuda", 0)
    cache, store = _make(cfg, 16, max_tokens=4)
    ora = SlotCache(s.L, s.E, 16, K=s.E if False else min(s.E, 4 * s.k), b_pcie=1000, b_cpu=0)
    out = torch.empty(cfg.T, s.H, device=dev)
    for l in range(s.L):
        ids, w = prefill_routing(cfg, l)
        ora.prefill(l, ids)
        cache.prefill(l, torch_act(activations(cfg, 0, l), dev), torch.from_numpy(ids).to(dev),
                      torch.from_numpy(w).to(dev), out)
    dcfg = cfg.with_(T=4, steps=6, prefill=False)
    ids, w = routing_trace(dcfg)
    sm = torch.empty(4, s.k, dtype=torch.int32, device=dev)
    o4 = torch.empty(4, s.H, device=dev)
    hits = 0
    for st in range(dcfg.steps):
        for l in range(s.L):
            plan = ora.decode(l, ids[st, l])
            hits += len(plan.hits)
            cache.decode(l, torch_act(activations(dcfg, st, l), dev), torch.from_numpy(ids[st, l]).to(dev),
                         torch.from_numpy(w[st, l]).to(dev), o4, slot_map=sm)
            torch.cuda.synchronize()
            assert np.array_equal(sm.cpu().numpy(), plan.slot_map)
    _check_state(cache, ora)
    assert hits > 0
    cache.close()


def test_decode_prefill_decode_interleaved():
    # decode keeps victim candidates between calls; a prefill in between rewrites
    # slots and stamps, and the decode calls after it must still match the oracle
    import torch
    cfg = SMALL.with_(shape=Shape(L=3, E=24, k=2, H=256, I=128, wdtype="bf16", adtype="bf16"))
    s = cfg.shape
    dev = torch.device("cuda", 0)
    C = 20
    cache, store = _make(cfg, C, max_tokens=4)
    K = min(s.E, 4 * s.k)
    ora = SlotCache(s.L, s.E, C, K=K, b_pcie=1000, b_cpu=0)
    dcfg = cfg.with_(T=4, steps=12, prefill=False)
    ids, w = routing_trace(dcfg)
    sm = torch.empty(4, s.k, dtype=torch.int32, device=dev)
    o4 = torch.empty(4, s.H, device=dev)
    out = torch.empty(cfg.T, s.H, device=dev)
    for st in range(dcfg.steps):
        if st in (4, 9):   # a prefill of one layer between decode steps
            l = st % s.L
            pids, pw = prefill_routing(cfg, l)
            ora.prefill(l, pids)
            cache.prefill(l, torch_act(activations(cfg, 0, l), dev), torch.from_numpy(pids).to(dev),
                          torch.from_numpy(pw).to(dev), out)
            torch.cuda.synchronize()
            _check_state(cache, ora)
        for l in range(s.L):
            plan = ora.decode(l, ids[st, l])
            cache.decode(l, torch_act(activations(dcfg, st, l), dev), torch.from_numpy(ids[st, l]).to(dev),
                         torch.from_numpy(w[st, l]).to(dev), o4, slot_map=sm)
            torch.cuda.synchronize()
            assert np.array_equal(sm.cpu().numpy(), plan.slot_map), (st, l)
            assert np.array_equal(cache.plan(T=4)["victims"], plan.victims), (st, l)
    _check_state(cache, ora)
    cache.close()


def test_prefill_rejects_bad_config():
    import torch
    from serving_layer_moe_gb300 import MoECache, MoEError
    cfg = config("tiny")
    s = cfg.shape
    arena, offs = make_pool(s, cfg.seed)
    with pytest.raises(MoEError):   # fp32 weights cannot run the bf16 tensor-core prefill
        MoECache(L=s.L, E=s.E, H=s.H, I=s.I, top_k=s.k, max_tokens=4, wdtype="f32", adtype="f32",
                 host_pool=arena, blob_offsets=offs, n_slots=4, max_prefill_tokens=64)


# ---- 4-bit experts: the slots and the host link carry NVFP4 / MXFP4 blobs; the
# grouped GEMMs read each routed expert decoded to bf16 ----

FP4 = ["nvfp4", "mxfp4"]


def _fp4(cfg, fmt):
    return cfg.with_(shape=Shape(**{**cfg.shape.__dict__, "wdtype": fmt}))


@pytest.mark.parametrize("fmt", FP4)
def test_fp4_small_full_layer_on_demand_and_ragged(fmt):
    cfg = _fp4(SMALL, fmt)
    worst, _ = _run_prefill(cfg, C=16, layers=[0, 1, 2])
    assert worst <= (5e-3 if fmt == "mxfp4" else TOL)     # MXFP4 weights are exact in bf16
    _run_prefill(cfg, C=3, layers=[0, 1, 2])               # on demand, groups of 3 routed experts
    _run_prefill(cfg.with_(T=7), C=12, layers=[1, 0, 1])   # ragged chunk, one on-demand group
    _run_prefill(cfg, C=17, layers=[2, 0, 1], prefetch_next=[True, False, True])


@pytest.mark.parametrize("fmt", FP4)
def test_fp4_qwen3_shape_1k_tokens(fmt):
    cfg = _fp4(config("qwen3_prefill_8k").with_(T=1024), fmt)
    _run_prefill(cfg, C=300, layers=[0, 1, 2], n_phys=64, sample=128)


@pytest.mark.parametrize("fmt", FP4)
def test_fp4_qwen3_prefill_8k_every_token(fmt):
    # the bench's 4-bit chunk size: every token of two layers, full-layer double buffering
    cfg = _fp4(config("qwen3_prefill_8k"), fmt)
    _run_prefill(cfg, C=cfg.capacity, layers=[0, 1], n_phys=64, sample=None)


def test_mxfp4_prefill_survivors_seed_decode():
    # the 4-bit slots a prefill loads are the ones decode then reads
    import torch
    cfg = _fp4(SMALL, "mxfp4")
    s = cfg.shape
    dev = torch.device("cuda", 0)
    cache, store = _make(cfg, 16, max_tokens=2)
    ora = SlotCache(s.L, s.E, 16, K=min(s.E, 2 * s.k), b_pcie=1000, b_cpu=0)
    out = torch.empty(cfg.T, s.H, device=dev)
    for l in range(s.L):
        ids, w = prefill_routing(cfg, l)
        ora.prefill(l, ids)
        cache.prefill(l, torch_act(activations(cfg, 0, l), dev), torch.from_numpy(ids).to(dev),
                      torch.from_numpy(w).to(dev), out)
    dcfg = cfg.with_(T=2, steps=6, prefill=False)
    ids, w = routing_trace(dcfg)
    sm = torch.empty(2, s.k, dtype=torch.int32, device=dev)
    o2 = torch.empty(2, s.H, device=dev)
    hits = 0
    for st in range(dcfg.steps):
        for l in range(s.L):
            plan = ora.decode(l, ids[st, l])
            hits += len(plan.hits)
            x = activations(dcfg, st, l)
            cache.decode(l, torch_act(x, dev), torch.from_numpy(ids[st, l]).to(dev),
                         torch.from_numpy(w[st, l]).to(dev), o2, slot_map=sm)
            torch.cuda.synchronize()
            assert np.array_equal(sm.cpu().numpy(), plan.slot_map)
            if (plan.slot_map >= 0).all():
                y = pair_outputs(store, l, s.E, x, s.adtype, ids[st, l])
                ref = combine(w[st, l], y, plan.slot_map, None)
                assert relative_max_error(o2.cpu().numpy(), ref) <= TOL
    _check_state(cache, ora)
    assert hits > 0
    cache.close()
