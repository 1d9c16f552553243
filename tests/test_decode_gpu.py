"""Decode parity on the GPU: libmoecache.so through its C ABI vs the CPU oracle.

Control state (slot maps, q, victims, fills, residency tables, stamps, clock,
counters) must be bit-exact; layer outputs within 2e-2 relative max error.
"""
import numpy as np
import pytest

from tests.harness import TOL, build_pool, make_cache, run_decode_parity, torch_act
from workloads import activations, config, routing_trace

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import serving_layer_moe_gb300 as m
    m.load_library()


def _ok(res):
    assert not res.mismatches, res.mismatches[:1]
    assert res.max_err <= TOL, res.max_err


def test_tiny_all_steps():
    cfg = config("tiny")
    res = run_decode_parity(cfg, cfg.bw_mbps, fp_every=1)
    _ok(res)
    assert res.fp_checked == 32 and res.cpu_pairs > 0 and res.fills > 0


def test_tiny_registered_pageable_pool_and_offload_mode():
    # pool handed over as pageable numpy memory (the library registers it); B_cpu = 0
    cfg = config("tiny").with_(steps=12)
    res = run_decode_parity(cfg, (1000, 0), fp_every=1, pinned=False)
    _ok(res)


def test_tiny_fetch_cap_and_cpu_heavy_split():
    cfg = config("tiny").with_(steps=16, max_fetch=1)
    res = run_decode_parity(cfg, (100, 900), fp_every=2)
    _ok(res)
    assert res.cpu_pairs > 0


def test_tiny_zero_fetch_is_all_cpu():
    cfg = config("tiny").with_(steps=4, max_fetch=0)
    res = run_decode_parity(cfg, (1000, 1000), fp_every=1)
    _ok(res)
    assert res.fills == 0


def test_qwen3_b1_full_trace():
    cfg = config("qwen3_decode_b1")
    res = run_decode_parity(cfg, (200000, 100000), n_phys=48, fp_every=997, state_every=16)
    _ok(res)
    assert res.calls == 256 * 48 and res.fp_checked >= 10


def test_qwen3_b16_with_resize():
    # outputs on every layer-step of the 8 steps around the resize (1228 -> 737 slots before step 128)
    cfg = config("qwen3_decode_b16")
    res = run_decode_parity(cfg, cfg.bw_mbps, n_phys=48, fp_every=1499, state_every=8, check_plan=True,
                            fp_steps=range(124, 132), memo=48)
    _ok(res)
    assert res.calls == 256 * 48 and res.cpu_pairs > 0 and res.fp_checked >= 8 * 48


def test_dsv3_fp8_shared_expert():
    # outputs on every layer-step of the first 16 steps (cold start: fills, hits, CPU pairs and the
    # shared expert mixed), then every 97th
    cfg = config("dsv3_decode_slice")
    res = run_decode_parity(cfg, (150000, 150000), n_phys=6, fp_every=97, state_every=4, fp_steps=range(16))
    _ok(res)
    assert res.fp_checked >= 16 * 4 and res.cpu_pairs > 0 and res.fills > 0


def test_control_one_warp_path_at_its_limit():
    # The control kernel takes calls of at most 32 routed pairs (and K <= 16) in
    # one warp: 4 tokens x top-8 is exactly 32; 5 tokens (40 pairs) take the
    # block-wide path.  Both against the oracle, with CPU-assigned pairs.
    from dataclasses import replace
    from workloads import QWEN3
    for T in (4, 5):
        cfg = config("qwen3_decode_b1").with_(shape=replace(QWEN3, L=4), T=T, steps=12,
                                              capacity=int(0.3 * 4 * 128), max_fetch=8)
        res = run_decode_parity(cfg, (100000, 100000), n_phys=16, fp_every=5, state_every=2)
        _ok(res)
        assert res.cpu_pairs > 0 and res.fills > 0


def test_ragged_T_and_empty_call():
    import torch
    cfg = config("qwen3_decode_b16").with_(steps=3)
    s = cfg.shape
    arena, offs, pool = build_pool(cfg, n_phys=16)
    cache, K = make_cache(cfg, pool, offs, None, (1000, 0))
    dev = torch.device("cuda", 0)
    ids, w = routing_trace(cfg)
    out = torch.full((16, s.H), 7.0, device=dev)
    # T = 0 is a no-op
    cache.decode(0, torch.empty(0, s.H, dtype=torch.int16, device=dev), torch.empty(0, s.k, dtype=torch.int32, device=dev),
                 torch.empty(0, s.k, device=dev), out)
    torch.cuda.synchronize()
    assert float(out[0, 0]) == 7.0
    # T = 3 of max 16
    x = activations(cfg, 0, 0)[:3]
    cache.decode(0, torch_act(x, dev), torch.from_numpy(ids[0, 0, :3].copy()).to(dev),
                 torch.from_numpy(w[0, 0, :3].copy()).to(dev), out[:3])
    torch.cuda.synchronize()
    assert np.all(np.isfinite(out[:3].cpu().numpy()))
    assert float(out[3, 0]) == 7.0
    cache.close()


def test_exact_merge_split_equals_all_gpu():
    # The combine merges exactly: supplying, as CPU partial sums, the very fp32
    # values the GPU computes for those experts gives a bit-identical output.
    import torch
    cfg = config("tiny").with_(steps=1)
    s = cfg.shape
    arena, offs, pool = build_pool(cfg)
    dev = torch.device("cuda", 0)
    ids, w = routing_trace(cfg)
    x = torch_act(activations(cfg, 0, 0), dev)
    i_d, w_d = torch.from_numpy(ids[0, 0]).to(dev), torch.from_numpy(w[0, 0]).to(dev)
    big, _ = make_cache(cfg, pool, offs, None, (1000, 0), n_slots=8)      # everything fits
    out_all = torch.empty(cfg.T, s.H, device=dev)
    big.decode(0, x, i_d, w_d, out_all)
    y_all = big.plan(T=cfg.T)["y"]
    small, _ = make_cache(cfg.with_(max_fetch=1), pool, offs, None, (100, 900), n_slots=4)
    sm = torch.empty(cfg.T, s.k, dtype=torch.int32, device=dev)
    out_split = torch.empty(cfg.T, s.H, device=dev)
    cpu = torch.from_numpy(y_all).to(dev)
    small.decode(0, x, i_d, w_d, out_split, cpu_part=cpu, slot_map=sm)
    torch.cuda.synchronize()
    assert (sm < 0).any()
    assert torch.equal(out_split, out_all)
    big.close()
    small.close()


def test_device_errors_are_reported_on_the_next_call():
    import torch
    from serving_layer_moe_gb300 import MoEError
    cfg = config("tiny").with_(steps=1)
    s = cfg.shape
    arena, offs, pool = build_pool(cfg)
    cache, _ = make_cache(cfg.with_(max_fetch=1), pool, offs, None, (100, 900))
    dev = torch.device("cuda", 0)
    x = torch_act(activations(cfg, 0, 0), dev)
    w = torch.full((cfg.T, s.k), 0.5, device=dev)
    out = torch.empty(cfg.T, s.H, device=dev)
    bad = torch.tensor([[0, 9]] * cfg.T, dtype=torch.int32, device=dev)        # 9 >= E
    cache.decode(0, x, bad, w, out, cpu_part=torch.zeros(cfg.T, s.k, s.H, device=dev))
    torch.cuda.synchronize()
    good = torch.tensor([[0, 1], [2, 3], [4, 5], [6, 7]], dtype=torch.int32, device=dev)
    with pytest.raises(MoEError) as ei:
        cache.decode(0, x, good, w, out)
    assert ei.value.status == 6
    # CPU-assigned pairs but no CPU partial sums: flagged, outputs stay finite
    cache.decode(0, x, good, w, out)
    torch.cuda.synchronize()
    assert torch.isfinite(out).all()
    with pytest.raises(MoEError) as ei:
        cache.decode(0, x, good, w, out)
    assert ei.value.status == 6
    cache.close()


def test_bench_bw_reports_two_bandwidths():
    from serving_layer_moe_gb300 import bench_bw
    bp, bh, rec = bench_bw(0, 9437184)
    assert bp > 1.0 and bh > 1.0
    assert rec == (bh > 2.0 * bp)


def _small_shape(E, k, wdtype="bf16", H=256, I=128):
    from workloads import Shape
    return Shape(L=3, E=E, k=k, H=H, I=I, wdtype=wdtype, adtype="bf16" if wdtype != "f32" else "f32")


def test_odd_expert_count_and_top3():
    # E = 40 (bitmap words partly used), k = 3, K <= 32 victim path
    from workloads import Config
    cfg = Config("odd", _small_shape(40, 3), T=5, steps=20, capacity=17, routing="softmax", seed=91)
    res = run_decode_parity(cfg, (3000, 2000), fp_every=3)
    _ok(res)
    assert res.cpu_pairs > 0 and res.fills > 0


def test_radix_victim_path_small():
    # K = min(E, T*k) = 64: the block-wide path with the kept pool of 256 candidates,
    # rebuilt by radix select whenever it runs short
    from workloads import Config
    cfg = Config("radix", _small_shape(64, 4), T=16, steps=12, capacity=40, routing="softmax_bias", bias_std=0.5,
                 seed=92)
    res = run_decode_parity(cfg, (1000, 1000), fp_every=5)
    _ok(res)


def test_exact_select_path_above_the_pool():
    # K = min(E, T*k) = 192 > 128: the radix select over all slots on every call
    from workloads import Config
    cfg = Config("radix_k192", _small_shape(256, 8), T=24, steps=10, capacity=150, routing="softmax_bias",
                 bias_std=0.5, seed=93)
    res = run_decode_parity(cfg, (1000, 1000), fp_every=7)
    _ok(res)
    assert res.fills > 0 and res.cpu_pairs > 0


@pytest.mark.parametrize("bw", [(1000, 0), (1000, 1000)])
def test_pool_short_falls_back_to_selection_over_all_slots(bw):
    # 60 of the call's hits among the 64 least-recent slots, K = 16: the pool (also
    # after its rebuild) holds 4 victims, the other 12 come from all slots
    from tests.harness import pool_short_trace
    cfg, ids, w = pool_short_trace()
    res = run_decode_parity(cfg, bw, fp_every=1, trace=(ids, w))
    _ok(res)
    assert res.calls == cfg.steps and res.fp_checked == cfg.steps and res.fills > 100


def test_random_resizes_grow_and_shrink():
    import torch
    from oracle.cache import SlotCache
    from workloads import Config
    cfg = Config("resz", _small_shape(16, 2), T=3, steps=40, capacity=10, routing="softmax", seed=93)
    s = cfg.shape
    arena, offs, pool = build_pool(cfg)
    cache, K = make_cache(cfg, pool, offs, None, (500, 500))
    ora = SlotCache(s.L, s.E, cfg.capacity, K, 500, 500)
    dev = torch.device("cuda", 0)
    ids, w = routing_trace(cfg)
    g = np.random.default_rng(0)
    sm = torch.empty(cfg.T, s.k, dtype=torch.int32, device=dev)
    out = torch.empty(cfg.T, s.H, device=dev)
    cpu = torch.zeros(cfg.T, s.k, s.H, device=dev)
    for st in range(cfg.steps):
        if st % 5 == 4:
            newC = int(g.integers(1, 40))
            ora.resize(newC)
            cache.resize(newC)
        for l in range(s.L):
            plan = ora.decode(l, ids[st, l])
            cache.decode(l, torch_act(activations(cfg, st, l), dev), torch.from_numpy(ids[st, l]).to(dev),
                         torch.from_numpy(w[st, l]).to(dev), out, cpu_part=cpu, slot_map=sm)
            torch.cuda.synchronize()
            assert np.array_equal(sm.cpu().numpy(), plan.slot_map), (st, l)
        gs, os_ = cache.state(), ora.state()
        for a, b in zip(gs[:4], os_[:4]):
            assert np.array_equal(a, b), st
        assert gs[4] == os_[4]
    cache.close()


def test_varying_T_on_one_cache():
    import torch
    from oracle.cache import SlotCache
    from oracle.ffn import ExpertStore, combine, pair_outputs, relative_max_error
    from workloads import Config
    cfg = Config("varT", _small_shape(24, 4), T=12, steps=16, capacity=30, routing="softmax", seed=94)
    s = cfg.shape
    arena, offs, pool = build_pool(cfg)
    cache, K = make_cache(cfg, pool, offs, None, (1000, 400))
    ora = SlotCache(s.L, s.E, cfg.capacity, K, 1000, 400)
    store = ExpertStore(arena, offs, s.wdtype, s.H, s.I, s.blob_bytes, memo=64)
    dev = torch.device("cuda", 0)
    ids, w = routing_trace(cfg)
    g = np.random.default_rng(1)
    for st in range(cfg.steps):
        for l in range(s.L):
            T = int(g.integers(1, cfg.T + 1))
            i_t, w_t = ids[st, l, :T].copy(), w[st, l, :T].copy()
            x = activations(cfg, st, l)[:T].copy()
            plan = ora.decode(l, i_t)
            y = pair_outputs(store, l, s.E, x, s.adtype, i_t)
            ref = combine(w_t, y, plan.slot_map, y)
            cpu = torch.from_numpy(np.where(plan.slot_map[..., None] < 0, y, np.nan).astype(np.float32)).to(dev)
            out = torch.empty(T, s.H, device=dev)
            sm = torch.empty(T, s.k, dtype=torch.int32, device=dev)
            cache.decode(l, torch_act(x, dev), torch.from_numpy(i_t).to(dev), torch.from_numpy(w_t).to(dev), out,
                         cpu_part=cpu, slot_map=sm)
            torch.cuda.synchronize()
            assert np.array_equal(sm.cpu().numpy(), plan.slot_map)
            assert relative_max_error(out.cpu().numpy(), ref) <= TOL
    cache.close()


# ---- 4-bit experts: NVFP4 (e2m1 codes, e4m3 scales per 16 row elements, fp32 per
# matrix) and MXFP4 (e2m1 codes, e8m0 scales per 32 row elements) ----

@pytest.mark.parametrize("I,T", [(1536, 1), (2048, 1), (1536, 2), (2048, 2)])
def test_fp8_straight_line_shapes(I, T):
    # fp8 rows of 96 and 128 16-byte chunks take the straight-line down paths (the
    # 8-row ring items of the resident grid, the 4-row items of the filled-expert
    # grid) and the unrolled gate/up loop; B_pcie = B_cpu gives fills, hits and
    # CPU-assigned pairs in the same calls
    from workloads import Config, Shape
    cfg = Config(f"fp8_I{I}_T{T}", Shape(L=3, E=24, k=4, H=1024, I=I, wdtype="fp8", adtype="bf16"), T=T,
                 steps=16, capacity=24, routing="softmax", seed=97)
    res = run_decode_parity(cfg, (1000, 1000), n_phys=12, fp_every=1)
    _ok(res)
    assert res.fills > 0 and res.cpu_pairs > 0 and res.fp_checked == 16 * 3


@pytest.mark.parametrize("wdtype", ["bf16", "fp8", "f32"])
def test_h_through_l1_above_two_tokens(wdtype):
    # 12 tokens x top-8 at I = 512: 96 pairs' h (196 KB in fp32) do not fit in shared
    # memory, so the bulk down kernel reads each item's h through L1; CPU pairs mixed in
    from workloads import Config, Shape
    cfg = Config(f"hl1_{wdtype}", Shape(L=2, E=32, k=8, H=256, I=512, wdtype=wdtype,
                                        adtype="f32" if wdtype == "f32" else "bf16"),
                 T=12, steps=10, capacity=40, routing="softmax_bias", bias_std=0.5, seed=98)
    res = run_decode_parity(cfg, (1000, 1000), fp_every=1)
    _ok(res)
    assert res.fills > 0 and res.cpu_pairs > 0 and res.fp_checked == 10 * 2


@pytest.mark.parametrize("T,wdtype", [(128, "bf16"), (160, "bf16"), (128, "nvfp4")])
def test_down_fallbacks_when_the_ring_does_not_fit(T, wdtype):
    # H = 8192 gives each down CTA 54 rows; with 1024 or more routed pairs their
    # partial sums no longer fit in shared memory beside a ring, so the down
    # projection takes the register-staged kernels: down_combine_kernel up to 1024
    # pairs, down_kernel + combine_kernel above (and for 4-bit experts)
    from workloads import Config, Shape
    cfg = Config(f"fallback_{T}_{wdtype}", Shape(L=1, E=16, k=8, H=8192, I=256, wdtype=wdtype, adtype="bf16"),
                 T=T, steps=2, capacity=16, routing="softmax", seed=99)
    res = run_decode_parity(cfg, (1000, 1000), fp_every=1)
    _ok(res)
    assert res.fills > 0 and res.cpu_pairs > 0 and res.fp_checked == 2


FP4 = ["nvfp4", "mxfp4"]

@pytest.mark.parametrize("fmt,adtype", [("nvfp4", "bf16"), ("mxfp4", "bf16"), ("mxfp4", "f32")])
def test_fp4_small_decode_two_tokens(fmt, adtype):
    from workloads import Config, Shape
    cfg = Config(f"{fmt}_small", Shape(L=3, E=24, k=4, H=256, I=128, wdtype=fmt, adtype=adtype), T=2, steps=24,
                 capacity=20, routing="softmax", seed=95)
    res = run_decode_parity(cfg, (1000, 0), fp_every=1)
    _ok(res)
    assert res.fills > 0 and res.fp_checked == 24 * 3


@pytest.mark.parametrize("fmt", FP4)
def test_fp4_qwen3_shape_batch1(fmt):
    cfg = config("qwen3_decode_b1")
    cfg = cfg.with_(shape=cfg.shape.__class__(**{**cfg.shape.__dict__, "wdtype": fmt}), steps=24)
    res = run_decode_parity(cfg, (200000, 0), n_phys=24, fp_every=37, state_every=8)
    _ok(res)
    assert res.calls == 24 * 48 and res.fp_checked >= 20


@pytest.mark.parametrize("fmt", FP4)
def test_fp4_split_merges_exactly(fmt):
    # resident and filled experts give the same y bits, so CPU partials equal to the
    # GPU's own values merge into a bit-identical output (see test_exact_merge_...)
    import torch
    from workloads import Config, Shape
    cfg = Config(f"{fmt}_merge", Shape(L=1, E=8, k=2, H=256, I=128, wdtype=fmt, adtype="bf16"), T=2, steps=1,
                 capacity=8, routing="softmax", seed=96)
    s = cfg.shape
    arena, offs, pool = build_pool(cfg)
    dev = torch.device("cuda", 0)
    ids, w = routing_trace(cfg)
    x = torch_act(activations(cfg, 0, 0), dev)
    i_d, w_d = torch.from_numpy(ids[0, 0]).to(dev), torch.from_numpy(w[0, 0]).to(dev)
    big, _ = make_cache(cfg, pool, offs, None, (1000, 0), n_slots=8)
    out_all = torch.empty(cfg.T, s.H, device=dev)
    big.decode(0, x, i_d, w_d, out_all)                 # fills every expert
    big.decode(0, x, i_d, w_d, out_all)                 # every expert resident now
    y_all = big.plan(T=cfg.T)["y"]
    small, _ = make_cache(cfg.with_(max_fetch=1), pool, offs, None, (100, 900), n_slots=2)
    sm = torch.empty(cfg.T, s.k, dtype=torch.int32, device=dev)
    out_split = torch.empty(cfg.T, s.H, device=dev)
    small.decode(0, x, i_d, w_d, out_split, cpu_part=torch.from_numpy(y_all).to(dev), slot_map=sm)
    torch.cuda.synchronize()
    assert (sm < 0).any()
    assert torch.equal(out_split, out_all)
    big.close()
    small.close()


@pytest.mark.parametrize("fmt,adtype", [("nvfp4", "bf16"), ("mxfp4", "bf16"), ("mxfp4", "f32")])
def test_fp4_small_decode_sixteen_tokens(fmt, adtype):
    # batches above 2 tokens: the register-staged gate/up and down kernels with 4-bit
    # chunks, then the separate combine; ragged batches from one cache
    from workloads import Config, Shape
    cfg = Config(f"{fmt}_t16", Shape(L=3, E=24, k=4, H=256, I=128, wdtype=fmt, adtype=adtype), T=16, steps=16,
                 capacity=30, routing="softmax_bias", bias_std=0.5, seed=97)
    res = run_decode_parity(cfg, (1000, 1000), fp_every=1)
    _ok(res)
    assert res.fills > 0 and res.cpu_pairs > 0 and res.fp_checked == 16 * 3


@pytest.mark.parametrize("fmt", FP4)
def test_fp4_qwen3_shape_batch16(fmt):
    # the batch-16 decode shape (top-8 of 128 with per-expert bias, 1:1 bandwidths) with 4-bit experts
    cfg = config("qwen3_decode_b16")
    cfg = cfg.with_(shape=cfg.shape.__class__(**{**cfg.shape.__dict__, "wdtype": fmt, "L": 6}), steps=10,
                    capacity=150, resize_step=None, resize_to=None)
    res = run_decode_parity(cfg, cfg.bw_mbps, n_phys=32, fp_every=2, state_every=2, memo=32)
    _ok(res)
    assert res.calls == 10 * 6 and res.fp_checked >= 30 and res.cpu_pairs > 0


@pytest.mark.parametrize("fmt", FP4)
def test_fp4_rejects_misshaped_prefill(fmt):
    import torch
    from serving_layer_moe_gb300 import MoECache, MoEError
    from workloads import Shape
    s = Shape(L=1, E=8, k=2, H=256, I=128, wdtype=fmt, adtype="bf16")
    pool = torch.zeros(8 * s.blob_bytes, dtype=torch.uint8).pin_memory()
    # prefill with fp32 activations or H not a multiple of 256
    for kw in ({"max_tokens": 1, "max_prefill_tokens": 64, "adtype": "f32"},
               {"max_tokens": 1, "max_prefill_tokens": 64, "H": 160}):
        args = dict(L=1, E=8, H=256, I=128, top_k=2, wdtype=fmt, adtype="bf16", host_pool=pool, n_slots=4,
                    bw_pcie_mbps=1000, bw_cpu_mbps=0)
        args.update(kw)
        with pytest.raises(MoEError) as ei:
            MoECache(**args)
        assert ei.value.status == 1
    # a 16-token decode cache with prefill is fine
    c = MoECache(L=1, E=8, H=256, I=128, top_k=2, wdtype=fmt, adtype="bf16", host_pool=pool, n_slots=4,
                 bw_pcie_mbps=1000, bw_cpu_mbps=0, max_tokens=16, max_prefill_tokens=64)
    c.close()


@pytest.mark.parametrize("name,fmt", [("qwen3_decode_b1", None), ("dsv3_decode_slice", None),
                                      ("qwen3_decode_b1", "nvfp4"), ("qwen3_decode_b1", "mxfp4")])
def test_a_pair_is_the_same_filled_or_resident(name, fmt):
    # One layer twice on the same input: first every routed expert is filled (the
    # fill computes gate/up on the way, the filled-expert grid the down rows), then
    # every one is resident (the resident grids).  Both form each pair's y in the
    # same per-lane order and butterfly, so y and the layer output match bit for bit.
    import torch
    from dataclasses import replace
    from workloads import make_shared
    base = config(name)
    shape = replace(base.shape, L=1, **({"wdtype": fmt} if fmt else {}))
    cfg = base.with_(shape=shape, steps=1, capacity=2 * shape.k, max_fetch=shape.k,
                     resize_step=None, resize_to=None)
    s = cfg.shape
    dev = torch.device("cuda", 0)
    arena, offs, pool = build_pool(cfg, n_phys=16)
    shared = make_shared(s, cfg.seed) if s.n_shared else None
    cache, _ = make_cache(cfg, pool, offs, shared, (100000, 0))
    ids, w = routing_trace(cfg)
    x = torch_act(activations(cfg, 0, 0), dev)
    i_d, w_d = torch.from_numpy(ids[0, 0]).to(dev), torch.from_numpy(w[0, 0]).to(dev)
    outs, ys = [], []
    for call in range(2):
        out = torch.empty(cfg.T, s.H, device=dev)
        sm = torch.empty(cfg.T, s.k, dtype=torch.int32, device=dev)
        cache.decode(0, x, i_d, w_d, out, slot_map=sm)
        torch.cuda.synchronize()
        p = cache.plan(T=cfg.T)
        assert (p["q"], p["h"]) == ((s.k, 0) if call == 0 else (0, s.k)), p
        assert bool((sm >= 0).all())
        outs.append(out.cpu().numpy())
        ys.append(p["y"])
    cache.close()
    assert np.all(np.isfinite(outs[0]))
    assert np.array_equal(ys[0].view(np.uint32), ys[1].view(np.uint32))
    assert np.array_equal(outs[0].view(np.uint32), outs[1].view(np.uint32))
