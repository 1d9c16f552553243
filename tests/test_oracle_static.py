"""Pins of the static-split comparator and of the locality claim on synthetic traces."""
import numpy as np

from oracle.cache import SlotCache
from oracle.static_split import lru_miss_rate, static_split_expected, static_split_miss_rate
from tests.conftest import read_golden
from workloads import config, routing_trace


def test_static_split_closed_form():
    for L, E, C in [(48, 128, 2273), (48, 128, 1228), (4, 256, 112), (10, 8, 33)]:
        trace = np.zeros((3, L, 2, 4), np.int32)
        assert static_split_miss_rate(trace, C, E) == static_split_expected(C, E, L)
    assert static_split_expected(2273, 128, 48) == 31 / 48      # 17 of 48 layers resident


def test_static_split_is_close_to_one_minus_capacity():
    # The pages' prediction: routing-blind placement misses ~ 1 - capacity.
    for cap, predicted, measured in read_golden("locality.txt"):
        cap = int(cap) / 100
        L, E = 48, 128
        C = int(cap * L * E)
        rate = static_split_expected(C, E, L)
        assert abs(rate - (1 - cap)) <= 1.0 / L + 1e-9          # within one layer's share
        assert abs(round(100 * (1 - cap)) - int(predicted)) == 0


def test_random_static_placement_misses_one_minus_capacity():
    # Expert-granular random placement: each read hits with probability C/(L*E).
    g = np.random.default_rng(0)
    L, E, C = 8, 32, 64
    cfg = config("qwen3_decode_b1").with_(steps=60, shape=config("qwen3_decode_b1").shape.__class__(
        L=L, E=E, k=4, H=8, I=8, wdtype="bf16", adtype="bf16"))
    ids, _ = routing_trace(cfg)
    rates = []
    for _ in range(200):
        resident = set(g.choice(L * E, size=C, replace=False).tolist())
        flat = ids + (np.arange(L)[None, :, None, None] * E)
        rates.append(np.mean([f not in resident for f in flat.ravel()]))
    assert abs(np.mean(rates) - (1 - C / (L * E))) < 0.01


def test_global_lru_beats_static_split_on_zipf_trace():
    cfg = config("qwen3_decode_b1").with_(steps=64)
    ids, _ = routing_trace(cfg)
    s = cfg.shape
    c = SlotCache(s.L, s.E, cfg.capacity, K=8, b_pcie=1, b_cpu=0)
    for st in range(cfg.steps):
        for l in range(s.L):
            c.decode(l, ids[st, l])
    lru = lru_miss_rate(c.counters)
    static = static_split_miss_rate(ids, cfg.capacity, s.E)
    assert lru < static
