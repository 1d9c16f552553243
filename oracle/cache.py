"""One LRU cache of whole experts, one slot per resident (layer, expert) (oracle, test infrastructure).

Passages followed:
  * snackonai deep dive "FreeToken, or why your laptop was never the
    bottleneck", section "The Architecture, Unpacked": all tables use the flat
    id l*E+e; the prefill and the decode draw on the same slots; for each MoE
    layer one kernel removes duplicate routed ids, looks them up, computes q,
    chooses victims and maps every id to a slot or to the CPU; the victims
    are the K slots used longest ago, found in a single pass.
  * same page, "The split policy itself": the first q misses fill, the rest
    run on the CPU; and "Resizing the cache without a restart".
  * ai.thesatyajit.com "FreeToken: a 753B model on one GPU ...", sections
    "Residency that follows the router" (a hit makes an expert the most
    recent, a fill brings one in, an eviction drops the one whose last use is
    oldest), "Prefill: hide the pool behind the wire" (the pool lends room for
    two whole layers; layer l+1 loads while layer l computes; experts load as
    needed when two layers do not fit; with the second buffer off, loading
    and computing take turns) and "Elastic memory ..." (rebuild the cache for
    a new budget; cold start).

The LRU order is an explicit Python list (least recent first).  Slots are
dicts.  Stamps are kept alongside only because they are part of the state the
CUDA library exposes; victim order here comes from the list, and the test
suite checks that list order and stamp order agree.

Readings taken where the pages are silent:
  * dedup order and fill order: ascending flat id; the i-th fill takes the
    i-th victim.
  * victims: empty slots first by slot index, then resident slots least
    recent first; slots holding one of this call's hits are never victims.
    In stamp form the key is (stamp, slot) ascending with empty slots at 0.
  * recency within one call: after the rewrite every touched expert (hits
    and fills, not CPU-assigned ones) moves to the most-recent end in
    ascending flat id, each taking the next value of one global clock.
  * prefill (full-layer mode, C >= 2E): the call for layer l loads whatever
    of layer l is missing, then all missing experts of layer l+1, into
    victims that exclude every slot holding an expert of l or l+1; it then
    touches all E experts of l (ascending e) and then the experts of l+1 it
    just loaded (ascending e).  When C < 2E: on-demand, the routed experts of
    l in ascending order in groups of at most C, each group loaded into
    victims that exclude the group's own resident slots, then touched.
  * prefill without the second buffer (prefetch_next=False, C >= 2E): the
    call for layer l loads only what is missing of l, into victims that
    exclude the slots of l, and touches the E experts of l; nothing of l+1
    is loaded ahead.
  * resize: keep the min(C_new, resident) most recent entries, packed into
    slots 0.. in ascending old-slot order with their recency kept.
"""
from __future__ import annotations

from dataclasses import dataclass, field

import numpy as np

from .policy import fill_count

# counter indices, as exposed in the state readout
C_HITS, C_MISSES, C_FILLS, C_CPU, C_READ_HITS, C_READ_MISSES, C_DECODE_CALLS, C_PREFILL_LOADS = range(8)


@dataclass
class DecodePlan:
    """What one decode call decided (snackonai "The Architecture, Unpacked":
    dedup, classify, split, victims, rewrite)."""
    layer: int
    uniq: list            # unique flat ids, ascending
    hits: list            # resident unique flat ids, ascending
    misses: list          # non-resident unique flat ids, ascending
    q: int                # misses that fill
    victims: list         # K slots in eviction order, -1 padded
    fills: list           # [(flat id, slot)] in fill order
    cpu: list             # CPU-assigned flat ids, ascending
    slot_map: np.ndarray  # [T, k] int32: slot, or -1 = CPU


@dataclass
class PrefillPlan:
    """What one prefill call loaded and computed (ai.thesatyajit.com "Prefill:
    hide the pool behind the wire")."""
    layer: int
    loads: list           # [(flat id, slot)]: missing experts of this layer (or group) first
    prefetch: list        # [(flat id, slot)]: experts of layer+1 loaded ahead (full-layer mode)
    groups: list          # on-demand mode: list of flat-id groups computed in turn
    full_layer: bool
    slot_map: np.ndarray  # [T, k] slot of every routed pair at the time it is computed


@dataclass
class SlotCache:
    """C slots shared by every layer, indexed by flat id l*E+e, with one LRU
    list (snackonai "The Architecture, Unpacked"; ai.thesatyajit.com
    "Residency that follows the router").  b_pcie / b_cpu are the two
    bandwidths of the split rule, K the fetch cap."""
    L: int
    E: int
    C: int
    K: int
    b_pcie: int
    b_cpu: int
    slot_of: dict = field(default_factory=dict)     # flat id -> slot
    expert_in: dict = field(default_factory=dict)   # slot -> flat id
    lru: list = field(default_factory=list)         # flat ids, least recent first
    stamp: dict = field(default_factory=dict)       # slot -> stamp (absent = 0)
    clock: int = 0
    counters: list = field(default_factory=lambda: [0] * 8)

    # -- eviction order ------------------------------------------------------
    def candidates(self, protected: set) -> list:
        """All slots this call may evict, in eviction order."""
        empties = [s for s in range(self.C) if s not in self.expert_in and s not in protected]
        used = [self.slot_of[f] for f in self.lru if self.slot_of[f] not in protected]
        return empties + used

    def _admit(self, f: int, s: int) -> None:
        old = self.expert_in.get(s)
        if old is not None:
            del self.slot_of[old]
            self.lru.remove(old)
        self.expert_in[s] = f
        self.slot_of[f] = s

    def _touch(self, f: int) -> None:
        if f in self.lru:
            self.lru.remove(f)
        self.lru.append(f)
        self.clock += 1
        self.stamp[self.slot_of[f]] = self.clock

    # -- decode: one MoE layer -------------------------------------------------
    def decode(self, layer: int, topk_ids: np.ndarray) -> DecodePlan:
        """One MoE layer's decode control (snackonai "The Architecture, Unpacked",
        "The split policy itself"): dedup the routed flat ids, classify them,
        fill the first q misses into the K least-recent victims, send the rest
        to the CPU, and refresh the recency of every GPU-run expert."""
        ids = np.asarray(topk_ids)
        assert ids.ndim == 2
        assert 0 <= layer < self.L
        if ids.size and (ids.min() < 0 or ids.max() >= self.E):
            raise ValueError("expert id out of range")
        flat = [[layer * self.E + int(e) for e in row] for row in ids]
        uniq = sorted({f for row in flat for f in row})
        hits = [f for f in uniq if f in self.slot_of]
        misses = [f for f in uniq if f not in self.slot_of]
        m = len(misses)
        protected = {self.slot_of[f] for f in hits}
        cands = self.candidates(protected)
        victims = (cands[: self.K] + [-1] * self.K)[: self.K]
        q = fill_count(m, self.b_pcie, self.b_cpu, self.K, len(cands))
        fills = []
        for i in range(q):
            self._admit(misses[i], cands[i])
            fills.append((misses[i], cands[i]))
        cpu = misses[q:]
        on_gpu = set(hits) | {f for f, _ in fills}
        for f in sorted(on_gpu):
            self._touch(f)
        slot_map = np.array([[self.slot_of[f] if f in on_gpu else -1 for f in row] for row in flat],
                            dtype=np.int32).reshape(ids.shape)
        c = self.counters
        c[C_HITS] += len(hits)
        c[C_MISSES] += m
        c[C_FILLS] += q
        c[C_CPU] += m - q
        hit_set = set(hits)
        c[C_READ_HITS] += sum(f in hit_set for row in flat for f in row)
        c[C_READ_MISSES] += sum(f not in hit_set for row in flat for f in row)
        c[C_DECODE_CALLS] += 1
        return DecodePlan(layer, uniq, hits, misses, q, victims, fills, cpu, slot_map)

    # -- prefill: one MoE layer of a chunk ------------------------------------
    def prefill(self, layer: int, topk_ids: np.ndarray, prefetch_next: bool = True) -> PrefillPlan:
        """One MoE layer of a prefill chunk (ai.thesatyajit.com "Prefill: hide the
        pool behind the wire"): full-layer residency of l (and of l+1 when
        prefetch_next) if C >= 2E, else the routed experts of l on demand in
        groups of at most C."""
        ids = np.asarray(topk_ids)
        E = self.E
        if ids.size and (ids.min() < 0 or ids.max() >= E):
            raise ValueError("expert id out of range")
        flat = np.asarray(ids, dtype=np.int64) + layer * E
        if self.C >= 2 * E:
            cur = list(range(layer * E, (layer + 1) * E))
            nxt = list(range((layer + 1) * E, (layer + 2) * E)) if prefetch_next and layer + 1 < self.L else []
            need_cur = [f for f in cur if f not in self.slot_of]
            need_nxt = [f for f in nxt if f not in self.slot_of]
            protected = {self.slot_of[f] for f in cur + nxt if f in self.slot_of}
            cands = self.candidates(protected)
            assert len(cands) >= len(need_cur) + len(need_nxt)
            loads = list(zip(need_cur, cands))
            prefetch = list(zip(need_nxt, cands[len(need_cur):]))
            for f, s in loads + prefetch:
                self._admit(f, s)
            slot_map = np.vectorize(lambda f: self.slot_of[int(f)])(flat).astype(np.int32) \
                if flat.size else np.zeros(ids.shape, np.int32)
            for f in cur:
                self._touch(f)
            for f, _ in prefetch:
                self._touch(f)
            self.counters[C_PREFILL_LOADS] += len(loads) + len(prefetch)
            return PrefillPlan(layer, loads, prefetch, [cur], True, slot_map.reshape(ids.shape))
        # on-demand fallback
        routed = sorted({int(f) for f in flat.ravel()})
        loads, groups = [], []
        slot_map = np.full(ids.shape, -1, np.int32)
        for g0 in range(0, len(routed), self.C):
            grp = routed[g0:g0 + self.C]
            hits = [f for f in grp if f in self.slot_of]
            misses = [f for f in grp if f not in self.slot_of]
            cands = self.candidates({self.slot_of[f] for f in hits})
            assert len(cands) >= len(misses)
            for f, s in zip(misses, cands):
                self._admit(f, s)
                loads.append((f, s))
            gset = set(grp)
            for idx in np.ndindex(ids.shape):
                if int(flat[idx]) in gset:
                    slot_map[idx] = self.slot_of[int(flat[idx])]
            for f in grp:
                self._touch(f)
            groups.append(grp)
        self.counters[C_PREFILL_LOADS] += len(loads)
        return PrefillPlan(layer, loads, [], groups, False, slot_map)

    # -- resize ---------------------------------------------------------------
    def resize(self, new_C: int) -> list:
        """Rebuild for new_C slots; returns [(old slot, new slot, flat id)] of the survivors."""
        keep_n = min(new_C, len(self.lru))
        keep = set(self.lru[len(self.lru) - keep_n:]) if keep_n else set()
        survivors = sorted((s, f) for s, f in self.expert_in.items() if f in keep)
        moves = [(s_old, s_new, f) for s_new, (s_old, f) in enumerate(survivors)]
        new_stamp = {s_new: self.stamp[s_old] for s_old, s_new, _ in moves}
        self.expert_in = {s_new: f for _, s_new, f in moves}
        self.slot_of = {f: s_new for _, s_new, f in moves}
        self.lru = [f for f in self.lru if f in keep]
        self.stamp = new_stamp
        self.C = new_C
        return moves

    # -- state readout --------------------------------------------------------
    def state(self):
        """(slot -> flat id, slot stamps, flat id -> slot, counters, clock): the
        state the CUDA library reads out, in the same layout."""
        s2e = np.full(self.C, -1, np.int32)
        st = np.zeros(self.C, np.uint64)
        e2s = np.full(self.L * self.E, -1, np.int32)
        for s, f in self.expert_in.items():
            s2e[s] = f
            e2s[f] = s
            st[s] = self.stamp.get(s, 0)
        return s2e, st, e2s, np.array(self.counters, np.uint64), self.clock
