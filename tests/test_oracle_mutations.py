"""Plant plausible mistakes in the oracle (on the CPU) and check that its pins catch each one."""
from fractions import Fraction

import numpy as np
import pytest

import oracle.cache as cache_mod
import oracle.ffn as ffn_mod
import oracle.policy as policy_mod
from tests import test_oracle_cache as tc
from tests import test_oracle_ffn as tf
from tests import test_oracle_policy as tp


def _fails(fn, *a):
    with pytest.raises(AssertionError):
        fn(*a)


def test_floor_instead_of_round_is_caught(monkeypatch):
    monkeypatch.setattr(policy_mod, "round_half_even", lambda x: Fraction(x).numerator // Fraction(x).denominator)
    _fails(tp.test_worked_examples_from_the_pages)


def test_half_up_rounding_is_caught(monkeypatch):
    def half_up(x):
        x = Fraction(x)
        return int((x + Fraction(1, 2)).numerator // (x + Fraction(1, 2)).denominator)
    monkeypatch.setattr(policy_mod, "round_half_even", half_up)
    _fails(tp.test_rounding_is_half_to_even_and_exact)


def test_ratio_over_cpu_bandwidth_is_caught(monkeypatch):
    # q* = round(m * B_p / B_c): forgets that the CPU branch has only the residual
    monkeypatch.setattr(policy_mod, "q_star",
                        lambda m, bp, bc: policy_mod.round_half_even(Fraction(m * bp, max(bc, 1))))
    _fails(tp.test_worked_examples_from_the_pages)


def test_missing_clamp_is_caught(monkeypatch):
    def no_clamp(m, bp, bc, K, V):
        return 0 if m == 0 else min(policy_mod.q_star(m, bp, bc), K, V)
    monkeypatch.setattr(cache_mod, "fill_count", no_clamp)
    failures = 0
    for seed in range(40):
        try:
            tc.test_decode_matches_history_model(seed)
        except AssertionError:
            failures += 1
    assert failures > 0


def test_most_recent_first_eviction_is_caught(monkeypatch):
    orig = cache_mod.SlotCache.candidates

    def mru_first(self, protected):
        empties = [s for s in range(self.C) if s not in self.expert_in and s not in protected]
        used = [self.slot_of[f] for f in reversed(self.lru) if self.slot_of[f] not in protected]
        return empties + used
    monkeypatch.setattr(cache_mod.SlotCache, "candidates", mru_first)
    failures = 0
    for seed in range(10):
        try:
            tc.test_decode_matches_history_model(seed)
        except AssertionError:
            failures += 1
    assert failures > 0


def test_hits_not_refreshed_is_caught(monkeypatch):
    orig = cache_mod.SlotCache._touch

    def touch_fills_only(self, f):
        if f in self.lru:
            return
        orig(self, f)
    monkeypatch.setattr(cache_mod.SlotCache, "_touch", touch_fills_only)
    _fails(tc.test_single_expert_offload_is_a_textbook_lru)


def test_swapped_gate_and_up_is_caught(monkeypatch):
    def swapped(x, wg, wu, wd):
        x = np.asarray(x, dtype=np.float64)
        return (ffn_mod.silu(x @ wu.T) * (x @ wg.T)) @ wd.T
    monkeypatch.setattr(tf, "swiglu_expert", swapped)
    _fails(tf.test_hand_derived_expert)


def test_transposed_down_projection_is_caught(monkeypatch):
    def transposed(x, wg, wu, wd):
        x = np.asarray(x, dtype=np.float64)
        return (ffn_mod.silu(x @ wg.T) * (x @ wu.T)) @ wd
    monkeypatch.setattr(tf, "swiglu_expert", transposed)
    _fails(tf.test_hand_derived_expert)


def test_e8m0_bias_off_by_one_is_caught(monkeypatch):
    import oracle.formats as formats_mod
    from tests import test_oracle_formats as tfm
    monkeypatch.setattr(formats_mod, "e8m0_codes_to_f64",
                        lambda c: np.ldexp(1.0, np.asarray(c, np.uint8).astype(np.int64) - 126))
    _fails(tfm.test_e8m0_closed_form_values)
    _fails(tfm.test_mxfp4_hand_built_blob_indexes_scales_by_row_and_32_block)


def test_mxfp4_nibble_order_swapped_is_caught(monkeypatch):
    import oracle.formats as formats_mod
    from tests import test_oracle_formats as tfm
    orig = formats_mod.mxfp4_dequant

    def swapped(packed, scales):
        p = np.asarray(packed, np.uint8)
        return orig(((p >> 4) | (p << 4)).astype(np.uint8), scales)
    monkeypatch.setattr(formats_mod, "mxfp4_dequant", swapped)
    _fails(tfm.test_mxfp4_hand_built_blob_indexes_scales_by_row_and_32_block)
    _fails(tfm.test_mxfp4_blob_follows_the_mx_conversion)


def test_pinning_the_least_read_experts_is_caught(monkeypatch):
    import oracle.static_split as ss_mod
    from tests import test_oracle_static as ts

    def coldest(prefill_ids, C, E):
        L = len(prefill_ids)
        reads = np.zeros(L * E, np.int64)
        for l, ids in enumerate(prefill_ids):
            for e in np.asarray(ids).ravel():
                reads[l * E + int(e)] += 1
        return set(sorted(range(L * E), key=lambda f: (int(reads[f]), f))[:max(0, min(C, L * E))])
    monkeypatch.setattr(ss_mod, "prefill_pinned_placement", coldest)
    _fails(ts.test_prefill_pinned_hand_example)
    _fails(ts.test_prefill_pinned_is_a_maximum_coverage_subset_brute_force)


def test_pinned_counts_merged_across_layers_is_caught(monkeypatch):
    # counts reads per expert index, not per (layer, expert)
    import oracle.static_split as ss_mod
    from tests import test_oracle_static as ts

    def merged(prefill_ids, C, E):
        L = len(prefill_ids)
        reads = np.zeros(E, np.int64)
        for ids in prefill_ids:
            for e in np.asarray(ids).ravel():
                reads[int(e)] += 1
        order = sorted(range(L * E), key=lambda f: (-int(reads[f % E]), f))
        return set(order[:max(0, min(C, L * E))])
    monkeypatch.setattr(ss_mod, "prefill_pinned_placement", merged)
    _fails(ts.test_prefill_pinned_hand_example)
