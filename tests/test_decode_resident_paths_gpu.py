"""The two ways a decode call can run its resident experts, against each other.

By default a gate/up grid then a down + combine grid ("grids"); with
MOE_DECODE_RESIDENT=fused (or MOE_DECODE_FUSED=1) set when the cache is
created, one-token bf16 calls run both in one launch with a grid-wide barrier
between them.  Both compute each resident expert's gate/up rows, down rows and
the combine in the same arithmetic order, so on the same trace they give
bit-identical layer outputs; the fused launch is also held to the oracle (slot
maps bit-exact, outputs within 2e-2).  The traces start cold, so they also
cover calls with fills but no resident expert, and calls whose pairs all go to
the CPU.
"""
import os
from dataclasses import replace

import pytest

from tests.harness import TOL, build_pool, make_cache, run_decode_parity, torch_act
from workloads import QWEN3, activations, config, routing_trace

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import serving_layer_moe_gb300 as m
    m.load_library()


def _qwen3_small(T, steps, layers=6, **kw):
    shape = replace(QWEN3, L=layers)
    return config("qwen3_decode_b1").with_(shape=shape, T=T, steps=steps,
                                           capacity=int(0.37 * layers * shape.E), **kw)


MODE_PATH = {"grids": 0, "fused": 1}


def _cache(cfg, pool, offs, bw, mode):
    saved = {k: os.environ.get(k) for k in ("MOE_DECODE_FUSED", "MOE_DECODE_RESIDENT")}
    os.environ.pop("MOE_DECODE_FUSED", None)
    os.environ["MOE_DECODE_RESIDENT"] = mode
    try:
        return make_cache(cfg, pool, offs, None, bw)[0]
    finally:
        for k, v in saved.items():
            if v is None:
                os.environ.pop(k, None)
            else:
                os.environ[k] = v


def _path_equals_two_grids(cfg, bw, mode):
    import torch
    s = cfg.shape
    dev = torch.device("cuda", 0)
    arena, offs, pool = build_pool(cfg, n_phys=16)
    one = _cache(cfg, pool, offs, bw, mode)
    two = _cache(cfg, pool, offs, bw, "grids")
    assert int(one.info()[6]) == 4 and int(two.info()[6]) == 5   # kernels per decode call
    assert int(one.info()[7]) == MODE_PATH[mode] and int(two.info()[7]) == 0   # how the resident experts run
    ids, w = routing_trace(cfg)
    gen = torch.Generator(device="cpu").manual_seed(7)
    cpu = torch.randn(cfg.T, s.k, s.H, generator=gen).to(dev)     # read only where a pair goes to the CPU
    out1 = torch.empty(cfg.T, s.H, device=dev)
    out2 = torch.empty(cfg.T, s.H, device=dev)
    sm1 = torch.empty(cfg.T, s.k, dtype=torch.int32, device=dev)
    sm2 = torch.empty_like(sm1)
    n_cpu = n_fill_only = 0
    for st in range(cfg.steps):
        for l in range(s.L):
            x = torch_act(activations(cfg, st, l), dev)
            i_d = torch.from_numpy(ids[st, l]).to(dev)
            w_d = torch.from_numpy(w[st, l]).to(dev)
            one.decode(l, x, i_d, w_d, out1, cpu_part=cpu, slot_map=sm1)
            two.decode(l, x, i_d, w_d, out2, cpu_part=cpu, slot_map=sm2)
            torch.cuda.synchronize()
            assert torch.equal(sm1, sm2), (st, l)
            assert torch.equal(out1, out2), (st, l, float((out1 - out2).abs().max()))
            p = one.plan()
            n_cpu += int((sm1 < 0).sum())
            n_fill_only += int(p["h"] == 0 and p["q"] > 0)
    one.close()
    two.close()
    return n_cpu, n_fill_only


@pytest.mark.parametrize("mode", ["fused"])
def test_bit_identical_to_two_grids_offload(mode):
    n_cpu, n_fill_only = _path_equals_two_grids(_qwen3_small(T=1, steps=20), (100000, 0), mode)
    assert n_cpu == 0 and n_fill_only > 0


@pytest.mark.parametrize("mode", ["fused"])
def test_bit_identical_to_two_grids_hybrid(mode):
    n_cpu, _ = _path_equals_two_grids(_qwen3_small(T=1, steps=20), (100000, 900000), mode)
    assert n_cpu > 0


@pytest.mark.parametrize("mode", ["fused"])
def test_bit_identical_all_cpu_calls(mode):
    # K = 0: no fill ever; cold calls send every pair to the CPU
    n_cpu, _ = _path_equals_two_grids(_qwen3_small(T=1, steps=4, layers=3, max_fetch=0), (1000, 1000), mode)
    assert n_cpu > 0


@pytest.mark.parametrize("mode", ["fused"])
def test_oracle_parity_one_token(monkeypatch, mode):
    monkeypatch.delenv("MOE_DECODE_FUSED", raising=False)
    monkeypatch.setenv("MOE_DECODE_RESIDENT", mode)
    cfg = _qwen3_small(T=1, steps=40)
    res = run_decode_parity(cfg, (100000, 100000), n_phys=24, fp_every=5, state_every=8)
    assert not res.mismatches, res.mismatches[:1]
    assert res.max_err <= TOL, res.max_err
    assert res.fp_checked >= 40 and res.cpu_pairs > 0 and res.fills > 0


@pytest.mark.parametrize("mode", ["fused"])
def test_one_token_paths_fall_back_where_they_do_not_apply(monkeypatch, mode):
    # two tokens per call: the fused launch does not apply and the two grids run
    monkeypatch.delenv("MOE_DECODE_FUSED", raising=False)
    monkeypatch.setenv("MOE_DECODE_RESIDENT", mode)
    cfg = _qwen3_small(T=2, steps=6, layers=3)
    arena, offs, pool = build_pool(cfg, n_phys=8)
    c, _ = make_cache(cfg, pool, offs, None, (100000, 100000))
    assert int(c.info()[7]) == 0 and int(c.info()[6]) == 5
    c.close()
    res = run_decode_parity(cfg, (100000, 100000), n_phys=8, fp_every=3, state_every=3)
    assert not res.mismatches and res.max_err <= TOL


def test_bad_resident_mode_is_refused(monkeypatch):
    from serving_layer_moe_gb300 import MoEError
    monkeypatch.setenv("MOE_DECODE_RESIDENT", "bogus")
    cfg = _qwen3_small(T=1, steps=2, layers=2)
    arena, offs, pool = build_pool(cfg, n_phys=4)
    with pytest.raises(MoEError) as ei:
        make_cache(cfg, pool, offs, None, (1000, 0))
    assert ei.value.status == 1
