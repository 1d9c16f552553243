"""Static placements, the comparators of the locality result (oracle, test infrastructure):
the routing-blind split and the prefill-pinned hot subset.

Passage followed: snackonai deep dive "FreeToken, or why your laptop was never
the bottleneck", section "The Locality Result Nobody Is Quoting": a placement
uncorrelated with routing misses about 1 - capacity of the expert reads; the
layer-granular static split (llama.cpp style) measures at that rate.

Reading taken: the static split keeps the first floor(C / E) layers fully
resident for the whole run; every other routed read is a miss.
"""
from __future__ import annotations

from fractions import Fraction

import numpy as np


def static_split_miss_rate(ids_trace: np.ndarray, C: int, E: int) -> float:
    """ids_trace [steps, L, T, k] -> fraction of routed reads that miss the static split."""
    steps, L, T, k = ids_trace.shape
    resident_layers = min(L, C // E)
    reads = steps * L * T * k
    misses = steps * (L - resident_layers) * T * k
    return float(Fraction(misses, reads)) if reads else 0.0


def static_split_expected(C: int, E: int, L: int) -> float:
    """Closed form when every layer gets the same number of reads: 1 - floor(C/E)/L."""
    return float(1 - Fraction(min(L, C // E), L))


def lru_miss_rate(counters) -> float:
    """Miss rate over routed reads from a cache's counters (read hits, read misses)."""
    from .cache import C_READ_HITS, C_READ_MISSES
    h, m = int(counters[C_READ_HITS]), int(counters[C_READ_MISSES])
    return m / (h + m) if h + m else 0.0


# ---- prefill-pinned placement (the KTransformers-style comparator) -----------
#
# Passage followed: "FreeToken: a 753B model on one GPU, and the two bandwidths
# that decide everything" (ai.thesatyajit.com), section "Residency that follows
# the router": the comparator engine decides, when a prompt is prefilled, which
# frequently used experts stay on the GPU, keeps that choice fixed while it
# decodes, and runs every other expert on the CPU.  On identical routing and
# capacity, that placement loses more decode reads to misses than the global
# LRU and fewer than the routing-blind split.
#
# Readings taken (the pages name the policy but give no rule):
#   * the hot subset is the C (layer, expert) pairs read most often by the
#     prefill's tokens, ties to the lower flat id l*E + e;
#   * it stays fixed through the decode that follows, and each new prefill
#     (one per turn) replaces it;
#   * a decode read misses when its pair is not in the subset.

def prefill_pinned_placement(prefill_ids, C: int, E: int) -> set[int]:
    """prefill_ids: one [T, k] id array per layer (layer l = index l) -> the
    pinned set of flat ids, of size min(C, L*E)."""
    L = len(prefill_ids)
    reads = np.zeros(L * E, np.int64)
    for l, ids in enumerate(prefill_ids):
        for e in np.asarray(ids).ravel():
            reads[l * E + int(e)] += 1
    order = sorted(range(L * E), key=lambda f: (-int(reads[f]), f))
    return set(order[:max(0, min(C, L * E))])


def pinned_misses(ids_trace: np.ndarray, placement: set[int], E: int) -> tuple[int, int]:
    """ids_trace [steps, L, T, k] -> (decode reads that miss the placement, all reads)."""
    steps, L, T, k = ids_trace.shape
    misses = 0
    for l in range(L):
        flat = ids_trace[:, l].ravel().astype(np.int64) + l * E
        misses += sum(1 for f in flat if int(f) not in placement)
    return misses, steps * L * T * k


def prefill_updated_miss_rate(turns, C: int, E: int) -> float:
    """turns: a sequence of (prefill_ids per layer, decode ids_trace) pairs, one per
    turn -> the fraction of all decode reads that miss the placement that turn's
    prefill pinned."""
    miss = reads = 0
    for prefill_ids, trace in turns:
        m, r = pinned_misses(np.asarray(trace), prefill_pinned_placement(prefill_ids, C, E), E)
        miss += m
        reads += r
    return miss / reads if reads else 0.0
