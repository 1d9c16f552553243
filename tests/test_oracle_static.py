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


# ---- prefill-pinned hot subset (the KTransformers-style comparator) ----

def test_prefill_pinned_hand_example():
    from oracle.static_split import pinned_misses, prefill_pinned_placement
    # reads during prefill: expert 0 three times, 1 twice, 2 once, 3 never
    pre = [np.array([[0, 1], [0, 2], [0, 1]], np.int32)]
    assert prefill_pinned_placement(pre, 2, 4) == {0, 1}
    assert prefill_pinned_placement(pre, 0, 4) == set()
    assert prefill_pinned_placement(pre, 9, 4) == {0, 1, 2, 3}
    assert pinned_misses(np.array([[[[2, 3]]]], np.int32), {0, 1}, 4) == (2, 2)
    assert pinned_misses(np.array([[[[0, 2]]]], np.int32), {0, 1}, 4) == (1, 2)
    # layer 1's ids are flat ids 4..7: its reads count apart from layer 0's
    pre2 = [np.array([[3, 2]], np.int32), np.array([[0, 1], [0, 2]], np.int32)]
    assert prefill_pinned_placement(pre2, 2, 4) == {4, 2}     # flat 4 read twice; ties 2, 3, 5, 6 -> 2


def test_prefill_pinned_is_a_maximum_coverage_subset_brute_force():
    # Brute force over every C-subset of a tiny pool: the pinned set covers the
    # most prefill reads of any subset, and swapping any pinned pair for an
    # unpinned one never gains (the tie rule: lower flat id first).
    import itertools
    from oracle.static_split import prefill_pinned_placement
    g = np.random.default_rng(11)
    for trial in range(30):
        L, E = int(g.integers(1, 3)), int(g.integers(2, 5))
        k = int(g.integers(1, E + 1))
        pre = [np.stack([g.choice(E, size=k, replace=False) for _ in range(int(g.integers(1, 6)))])
               for _ in range(L)]
        reads = np.zeros(L * E, int)
        for l, ids in enumerate(pre):
            for e in ids.ravel():
                reads[l * E + e] += 1
        for C in range(0, L * E + 1):
            pin = prefill_pinned_placement(pre, C, E)
            assert len(pin) == C
            best = max(sum(reads[f] for f in sub) for sub in itertools.combinations(range(L * E), C))
            assert sum(reads[f] for f in pin) == best
            for f in pin:
                for h in set(range(L * E)) - pin:
                    assert reads[f] > reads[h] or (reads[f] == reads[h] and f < h)


def test_prefill_pinned_is_the_best_static_placement_when_routing_does_not_shift():
    # Decode that replays the prefill's own routing: no static placement of the
    # same size misses fewer reads (brute force on a tiny pool).
    import itertools
    from oracle.static_split import pinned_misses, prefill_pinned_placement
    g = np.random.default_rng(12)
    L, E, k, T = 2, 4, 2, 5
    pre = [np.stack([g.choice(E, size=k, replace=False, p=[0.5, 0.3, 0.15, 0.05]) for _ in range(T)])
           for _ in range(L)]
    trace = np.stack(pre, axis=0)[None]                      # [1, L, T, k]
    for C in range(L * E + 1):
        pin = prefill_pinned_placement(pre, C, E)
        m, r = pinned_misses(trace, pin, E)
        best = min(pinned_misses(trace, set(sub), E)[0] for sub in itertools.combinations(range(L * E), C))
        assert m == best and r == L * T * k
    assert pinned_misses(trace, prefill_pinned_placement(pre, L * E, E), E)[0] == 0


def test_prefill_updated_placement_follows_each_turn():
    # Two turns whose prefills favour disjoint experts: the second turn's decode
    # hits only because its prefill replaced the placement.
    from oracle.static_split import prefill_updated_miss_rate
    E = 4
    turn1 = ([np.array([[0, 1]] * 3, np.int32)], np.array([[[[0, 1]]]], np.int32))
    turn2 = ([np.array([[2, 3]] * 3, np.int32)], np.array([[[[2, 3]]]], np.int32))
    assert prefill_updated_miss_rate([turn1, turn2], 2, E) == 0.0
    frozen = ([np.array([[0, 1]] * 3, np.int32)], turn2[1])          # placement never updated
    assert prefill_updated_miss_rate([turn1, frozen], 2, E) == 0.5


def test_lru_beats_a_prefill_pinned_subset_when_routing_shifts():
    # The decode routing (Zipf popularity over a per-layer permutation, step-to-
    # step reuse) is independent of the prefill's (N(0,1) logits): the pinned
    # subset is then no better informed than a random placement and misses about
    # 1 - capacity of the decode reads, while the global LRU follows the router.
    from oracle.static_split import prefill_updated_miss_rate
    from workloads import prefill_routing
    cfg = config("qwen3_decode_b1").with_(steps=32)
    s = cfg.shape
    ids, _ = routing_trace(cfg)
    pre_cfg = config("qwen3_prefill_8k").with_(T=2048)
    pre = [prefill_routing(pre_cfg, l)[0] for l in range(s.L)]
    pinned = prefill_updated_miss_rate([(pre, ids)], cfg.capacity, s.E)
    assert abs(pinned - (1 - cfg.capacity / (s.L * s.E))) < 0.03
    c = SlotCache(s.L, s.E, cfg.capacity, K=8, b_pcie=1, b_cpu=0)
    for st in range(cfg.steps):
        for l in range(s.L):
            c.decode(l, ids[st, l])
    assert lru_miss_rate(c.counters) < pinned


def test_lru_beats_the_static_placements_at_eleven_percent_capacity():
    # The pages' second capacity point (about 11%: the DeepSeek-V3-shaped slice,
    # C = 112 of 4 x 256 slots).  The layer-granular split cannot hold even one
    # whole layer (it misses every read), the prefill-pinned subset misses about
    # 1 - capacity of the decode reads (its prefill's routing is independent of the
    # decode's), and the global LRU misses far fewer.
    from oracle.static_split import prefill_updated_miss_rate, static_split_miss_rate
    from workloads import Config, prefill_routing
    cfg = config("dsv3_decode_slice").with_(steps=32)
    s = cfg.shape
    cap = cfg.capacity / (s.L * s.E)
    assert abs(cap - 0.11) < 0.005
    ids, _ = routing_trace(cfg)
    pre_cfg = Config("dsv3_prefill", s, T=2048, steps=1, capacity=cfg.capacity, routing="softmax",
                     seed=cfg.seed + 100, prefill=True)
    pre = [prefill_routing(pre_cfg, l)[0] for l in range(s.L)]
    pinned = prefill_updated_miss_rate([(pre, ids)], cfg.capacity, s.E)
    assert abs(pinned - (1 - cap)) < 0.06   # 1024 decode reads of a Zipf(1.0) trace: a few points of noise
    assert static_split_miss_rate(ids, cfg.capacity, s.E) == 1.0
    c = SlotCache(s.L, s.E, cfg.capacity, K=8, b_pcie=1, b_cpu=0)
    for st in range(cfg.steps):
        for l in range(s.L):
            c.decode(l, ids[st, l])
    lru = lru_miss_rate(c.counters)
    assert lru < 0.5 * pinned
