"""GB300-native expert-slot cache for MoE layers (FreeToken's decode hot path).

The work runs in libmoecache.so (hand-written CUDA for sm_103a, C ABI in
include/moe_cache.h); this package is its thin Python binding.
"""
from .binding import (DTYPES, SYMBOLS, MoECache, MoEError, bench_bw, load_library)  # noqa: F401

__all__ = ["MoECache", "MoEError", "bench_bw", "load_library", "DTYPES", "SYMBOLS"]
