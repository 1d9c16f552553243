"""Pins of the oracle's list-based LRU slot cache.

Checked against (a) a definition-level model that keeps only slot contents and
a log of every touch, and takes each slot's recency by scanning that log; (b)
functools.lru_cache in the special case where the policy is a textbook LRU
(one expert per call, every miss fills); (c) invariants.
"""
import functools
from fractions import Fraction

import numpy as np
import pytest

from oracle.cache import SlotCache


class HistoryModel:
    def __init__(self, L, E, C, K, bp, bc):
        self.L, self.E, self.C, self.K, self.bp, self.bc = L, E, C, K, bp, bc
        self.content = [None] * C
        self.log = []            # flat ids in touch order; touch i has clock value i + 1

    def last_touch(self, s):
        f = self.content[s]
        if f is None:
            return 0
        for i in range(len(self.log) - 1, -1, -1):
            if self.log[i] == f:
                return i + 1
        raise AssertionError("resident expert never touched")

    def order(self, protected):
        return [s for _, s in sorted((self.last_touch(s), s) for s in range(self.C) if s not in protected)]

    def decode(self, layer, ids):
        flat = [[layer * self.E + int(e) for e in row] for row in ids]
        uniq = sorted({f for row in flat for f in row})
        where = {f: s for s, f in enumerate(self.content) if f is not None}
        hits = [f for f in uniq if f in where]
        misses = [f for f in uniq if f not in where]
        order = self.order({where[f] for f in hits})
        victims = (order + [-1] * self.K)[: self.K]
        m = len(misses)
        q = 0
        if m:
            q = max(1, min(round(Fraction(m * self.bp, self.bp + self.bc)), m))
            q = min(q, self.K, len(order))
        for i in range(q):
            self.content[order[i]] = misses[i]
        touched = sorted(hits + misses[:q])
        self.log.extend(touched)
        where = {f: s for s, f in enumerate(self.content) if f is not None}
        sm = [[where[f] if f in touched else -1 for f in row] for row in flat]
        return q, victims, np.array(sm, np.int32)

    def prefill(self, layer, ids, prefetch_next=True):
        E = self.E
        where = {f: s for s, f in enumerate(self.content) if f is not None}
        if self.C >= 2 * E:
            cur = list(range(layer * E, layer * E + E))
            nxt = list(range(layer * E + E, layer * E + 2 * E)) if prefetch_next and layer + 1 < self.L else []
            need = [f for f in cur if f not in where] + [f for f in nxt if f not in where]
            order = self.order({where[f] for f in cur + nxt if f in where})
            for f, s in zip(need, order):
                self.content[s] = f
            self.log.extend(cur)
            self.log.extend([f for f in nxt if f in need])
        else:
            routed = sorted({layer * E + int(e) for e in np.asarray(ids).ravel()})
            for g0 in range(0, len(routed), self.C):
                where = {f: s for s, f in enumerate(self.content) if f is not None}
                grp = routed[g0:g0 + self.C]
                miss = [f for f in grp if f not in where]
                order = self.order({where[f] for f in grp if f in where})
                for f, s in zip(miss, order):
                    self.content[s] = f
                self.log.extend(grp)

    def resize(self, new_C):
        res = [(self.last_touch(s), s) for s in range(self.C) if self.content[s] is not None]
        keep = sorted(s for _, s in sorted(res, reverse=True)[:new_C])
        self.content = [self.content[s] for s in keep] + [None] * (new_C - len(keep))
        self.C = new_C

    def stamps(self):
        return np.array([self.last_touch(s) for s in range(self.C)], np.uint64)


def _check_invariants(c: SlotCache):
    s2e, st, e2s, counters, clock = c.state()
    # maps are inverse
    for s, f in enumerate(s2e):
        if f >= 0:
            assert e2s[f] == s
    assert (e2s >= 0).sum() == (s2e >= 0).sum() <= c.C
    # list order == stamp order, stamps unique, empty slots stamp 0
    stamps_in_list = [int(st[c.slot_of[f]]) for f in c.lru]
    assert stamps_in_list == sorted(stamps_in_list)
    assert len(set(stamps_in_list)) == len(stamps_in_list)
    assert all(st[s] == 0 for s in range(c.C) if s2e[s] < 0)
    assert clock >= max(stamps_in_list, default=0)


def _random_ids(g, T, k, E):
    return np.stack([g.choice(E, size=k, replace=False) for _ in range(T)]).astype(np.int32)


@pytest.mark.parametrize("seed", range(40))
def test_decode_matches_history_model(seed):
    g = np.random.default_rng(seed)
    L, E = int(g.integers(1, 4)), int(g.integers(2, 9))
    k = int(g.integers(1, min(E, 3) + 1))
    T = int(g.integers(1, 4))
    C = int(g.integers(1, 2 * E + 2))
    K = int(g.integers(0, 6))
    bp, bc = int(g.integers(1, 5)), int(g.integers(0, 5))
    o = SlotCache(L, E, C, K, bp, bc)
    h = HistoryModel(L, E, C, K, bp, bc)
    for step in range(30):
        layer = int(g.integers(0, L))
        ids = _random_ids(g, T, k, E)
        p = o.decode(layer, ids)
        q, victims, sm = h.decode(layer, ids)
        assert p.q == q and p.victims == victims
        assert np.array_equal(p.slot_map, sm)
        s2e, st, e2s, _, _ = o.state()
        assert [(-1 if x is None else x) for x in h.content] == list(s2e)
        assert np.array_equal(st, h.stamps())
        _check_invariants(o)
        # slot map points at the right expert
        for (t, j), s in np.ndenumerate(p.slot_map):
            if s >= 0:
                assert s2e[s] == layer * E + ids[t, j]


@pytest.mark.parametrize("seed", range(20))
def test_prefill_and_resize_match_history_model(seed):
    g = np.random.default_rng(100 + seed)
    L, E = int(g.integers(2, 5)), int(g.integers(2, 6))
    k = int(g.integers(1, min(E, 3) + 1))
    C = int(g.integers(1, 3 * E + 1))
    o = SlotCache(L, E, C, K=E, b_pcie=1, b_cpu=1)
    h = HistoryModel(L, E, C, E, 1, 1)
    for op in range(25):
        r = g.random()
        if r < 0.35:
            layer = int(g.integers(0, L))
            ids = _random_ids(g, int(g.integers(1, 6)), k, E)
            nxt = bool(g.random() < 0.7)   # with or without the second buffer
            o.prefill(layer, ids, prefetch_next=nxt)
            h.prefill(layer, ids, prefetch_next=nxt)
        elif r < 0.85:
            layer = int(g.integers(0, L))
            ids = _random_ids(g, int(g.integers(1, 3)), k, E)
            p = o.decode(layer, ids)
            q, victims, sm = h.decode(layer, ids)
            assert p.q == q and p.victims == victims and np.array_equal(p.slot_map, sm)
        else:
            newC = int(g.integers(1, 3 * E + 1))
            o.resize(newC)
            h.resize(newC)
        s2e, st, _, _, _ = o.state()
        assert [(-1 if x is None else x) for x in h.content] == list(s2e)
        assert np.array_equal(st, h.stamps())
        _check_invariants(o)


def test_full_layer_prefill_leaves_layer_and_next_resident():
    o = SlotCache(L=4, E=3, C=6, K=3, b_pcie=1, b_cpu=0)
    for l in range(4):
        p = o.prefill(l, np.array([[0, 1], [2, 0]], np.int32))
        assert p.full_layer
        for f in range(l * 3, min(4, l + 2) * 3):
            assert f in o.slot_of
        assert np.all(p.slot_map >= 0)


def test_prefill_without_second_buffer_loads_only_its_layer():
    # Cold cache, C >= 2E: with the second buffer each call after the first
    # finds its layer resident (loaded ahead by the call before); without it,
    # every call loads its own E experts and nothing of the next layer.
    L, E = 4, 3
    ids = np.array([[0, 1], [2, 0]], np.int32)
    two = SlotCache(L, E, C=2 * E, K=E, b_pcie=1, b_cpu=0)
    one = SlotCache(L, E, C=2 * E, K=E, b_pcie=1, b_cpu=0)
    for l in range(L):
        p2 = two.prefill(l, ids)
        p1 = one.prefill(l, ids, prefetch_next=False)
        assert len(p2.loads) == (E if l == 0 else 0)
        assert len(p2.prefetch) == (E if l + 1 < L else 0)
        assert sorted(f for f, _ in p1.loads) == list(range(l * E, (l + 1) * E)) and p1.prefetch == []
        assert all(f not in one.slot_of for f in range((l + 1) * E, L * E))
    # both moved every expert across the link once
    assert two.counters[7] == one.counters[7] == L * E


def test_single_expert_offload_is_a_textbook_lru():
    # One routed expert per call and every miss fills: the policy is plain LRU,
    # so its hit/miss sequence equals functools.lru_cache of the same size.
    g = np.random.default_rng(3)
    E, C = 40, 7
    seq = [int(x) for x in np.minimum(g.zipf(1.3, size=3000) - 1, E - 1)]
    o = SlotCache(L=1, E=E, C=C, K=1, b_pcie=1, b_cpu=0)

    @functools.lru_cache(maxsize=C)
    def fetch(e):
        return e

    for e in seq:
        before = fetch.cache_info().hits
        fetch(e)
        lib_hit = fetch.cache_info().hits > before
        p = o.decode(0, np.array([[e]], np.int32))
        assert (len(p.hits) == 1) == lib_hit
    assert o.counters[0] == fetch.cache_info().hits


def test_cpu_assigned_experts_do_not_enter_the_cache():
    o = SlotCache(L=1, E=8, C=4, K=8, b_pcie=1, b_cpu=3)
    p = o.decode(0, np.array([[0, 1], [2, 3]], np.int32))   # m = 4 -> q* = 1
    assert p.q == 1 and p.fills == [(0, 0)] and p.cpu == [1, 2, 3]
    assert set(o.slot_of) == {0}
    assert p.slot_map.tolist() == [[0, -1], [-1, -1]]


def test_pool_short_trace_needs_victims_beyond_the_pool():
    # The scripted trace must put more of its hits among the 64 least-recent slots
    # than 64 - K, so that the GPU test of it reaches the selection over all slots.
    from tests.harness import POOL_SHORT_STEP, pool_short_trace
    cfg, ids, _ = pool_short_trace()
    ora = SlotCache(1, cfg.shape.E, cfg.capacity, cfg.max_fetch, 1000, 0)
    for st in range(POOL_SHORT_STEP):
        ora.decode(0, ids[st, 0])
    assert len(ora.expert_in) == cfg.capacity
    s2e, stamps, _, _, _ = ora.state()
    n_pool = min(cfg.capacity, max(64, 4 * cfg.max_fetch))
    oldest = sorted(range(cfg.capacity), key=lambda s: (int(stamps[s]), s))[:n_pool]
    routed = set(ids[POOL_SHORT_STEP, 0].ravel().tolist())
    hits_in_pool = sum(int(s2e[s]) in routed for s in oldest)
    assert n_pool - hits_in_pool < cfg.max_fetch
    plan = ora.decode(0, ids[POOL_SHORT_STEP, 0])
    assert len(plan.hits) == 60 and len(plan.misses) == 16 and plan.q == 16
    assert len(set(plan.victims) - set(oldest)) == cfg.max_fetch - (n_pool - hits_in_pool)
