"""Pins of the miss-split rule against the pages' worked numbers and closed forms."""
from fractions import Fraction

import pytest

from oracle.policy import (branch_times, fill_count, q_star, q_star_pages, recommend_hybrid,
                           round_half_even)
from tests.conftest import read_golden


def mbps(gbs: str) -> int:
    """GB/s as printed -> integer MB/s (the quantisation the library takes)."""
    return int(round(float(gbs) * 1000))


def test_worked_examples_from_the_pages():
    for m, bp, bh, approx, q in read_golden("q_split_worked.txt"):
        m, q = int(m), int(q)
        b_p, b_h = mbps(bp), mbps(bh)
        b_c = b_h - b_p                      # the residual host bandwidth
        assert q_star(m, b_p, b_c) == q
        assert q_star_pages(m, Fraction(bp), Fraction(bh)) == q
        assert fill_count(m, b_p, b_c, max_fetch=8, evictable=100) == q
        # the unrounded value the page prints, to its 2 decimals
        assert abs(float(Fraction(m * b_p, b_h)) - float(approx)) < 0.005


def test_branch_times_from_the_pages():
    g = {row[0]: float(row[1]) for row in read_golden("branch_times.txt")}
    B_P, B_H = Fraction("11.8"), Fraction("47.5")
    t_fill, t_cpu = branch_times(1, 4, B_P, B_H)
    assert round(float(t_fill), 4) == g["t_fill"]
    assert round(float(t_cpu), 4) == g["t_cpu"]
    assert round(float(max(t_fill, t_cpu)), 4) == g["exposed"]
    assert round(float(branch_times(4, 4, B_P, B_H)[0]), 4) == g["naive"]
    assert round(float(Fraction(4) / B_H), 4) == g["pure_cpu"]


def test_calibration_table_cpu_share_and_backend():
    # For large m the CPU share (m - q)/m tends to 1 - B_P/B_H; the table prints it in percent.
    for name, bp, bh, ratio, backend, share in read_golden("calibration_table.txt"):
        b_p, b_h = mbps(bp), mbps(bh)
        m = 10 ** 6
        q = q_star(m, b_p, b_h - b_p)
        assert round(100 * (m - q) / m) == int(share), name
        assert round(float(bh) / float(bp), 2) == float(ratio), name
        assert recommend_hybrid(Fraction(bp), Fraction(bh)) == (backend == "hybrid"), name


def test_balanced_point_closed_form():
    # At the unrounded balance point both branch times equal m / B_H (the expert size cancels).
    for m in range(1, 40):
        for b_p, b_c in [(1, 1), (2, 1), (11800, 35700), (52700, 24600), (3, 7)]:
            x = Fraction(m * b_p, b_p + b_c)
            assert x / b_p == (m - x) / b_c == Fraction(m, b_p + b_c)


def test_rounding_is_half_to_even_and_exact():
    assert round_half_even(Fraction(5, 2)) == 2
    assert round_half_even(Fraction(7, 2)) == 4
    assert round_half_even(Fraction(1, 2)) == 0
    assert round_half_even(Fraction(3, 2)) == 2
    assert round_half_even(Fraction(249999, 100000)) == 2
    assert round_half_even(Fraction(250001, 100000)) == 3
    # 1:1 bandwidths, odd m: exactly half, ties to even (Python round semantics)
    assert [q_star(m, 100, 100) for m in range(1, 8)] == [0, 1, 2, 2, 2, 3, 4]
    for m in range(0, 60):
        for b in [(3, 5), (7, 2), (1, 1), (11800, 35700)]:
            assert q_star(m, *b) == round(Fraction(m * b[0], b[0] + b[1]))


def test_q_is_one_of_the_two_integer_neighbours_of_the_balance_point():
    # Brute force over integers: the minimiser of the exposed time max(q/B_p, (m-q)/B_c)
    # is floor or ceil of the balance point, and round() picks one of those two.
    for m in range(1, 64):
        for b_p, b_c in [(1, 3), (3, 1), (2, 5), (11800, 35700), (52700, 24600)]:
            x = Fraction(m * b_p, b_p + b_c)
            best = min(range(m + 1), key=lambda q: max(Fraction(q, b_p), Fraction(m - q, b_c)))
            lo, hi = x.numerator // x.denominator, -((-x.numerator) // x.denominator)
            assert best in (lo, hi)
            assert q_star(m, b_p, b_c) in (lo, hi)
            assert abs(q_star(m, b_p, b_c) - x) <= Fraction(1, 2)


def test_clamp_and_caps():
    assert fill_count(0, 100, 100, 8, 8) == 0                 # nothing missed
    assert fill_count(1, 1, 1000, 8, 8) == 1                  # q* = 0 -> always >= 1 fill
    assert fill_count(4, 11800, 35700, 8, 8) == 1
    assert fill_count(10, 1000, 0, 8, 100) == 8               # offload mode, capped by K
    assert fill_count(10, 1000, 0, 20, 3) == 3                # capped by evictable slots
    assert fill_count(10, 1000, 0, 0, 3) == 0                 # K = 0: every miss on the CPU
    assert fill_count(5, 1000, 1000, 8, 0) == 0               # nothing evictable
    # degenerate case of the pages: B_H -> B_P (B_cpu -> 0) gives q -> m
    for m in range(1, 30):
        assert q_star(m, 1000, 0) == m
    with pytest.raises(ValueError):
        q_star(3, 0, 0)
