"""Routing-blind static placement, the comparator of the locality result (oracle, test infrastructure).

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
