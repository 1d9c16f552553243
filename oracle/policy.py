"""The miss split q* (oracle, test infrastructure).

Passages followed:
  * snackonai deep dive "FreeToken, or why your laptop was never the
    bottleneck", section "The split policy itself": balance the two
    concurrent branch times q*S/B_P and (m-q)*S/(B_H-B_P); S cancels; round
    to an integer with Python's round; clamp to max(1, min(q, m)); the first
    q misses fill, the rest run on the CPU.
  * ai.thesatyajit.com "FreeToken: a 753B model on one GPU ...", section
    "Decode: the one equation": the CPU branch works with the residual host
    bandwidth B_H - B_P; the balanced time is m*S/B_H; as B_H -> B_P, q* -> m.
  * same article, section "Four backends ...": --moe-hybrid-max-fetch caps
    fills per layer per step (the K of the victim selection).

Reading taken (the article's equations are lost in extraction):
  B_cpu := B_H - B_P, so the rule is q* = round(m * B_pcie / (B_pcie + B_cpu)),
  computed exactly on integer bandwidths (MB/s) and rounded half to even
  (Python's `round`).  The clamp applies only when m > 0 (m = 0 gives q = 0).
  After the clamp, q is capped by the fetch cap K and by V, the number of
  slots this call may evict; if either is 0 every miss goes to the CPU.
"""
from __future__ import annotations

from fractions import Fraction


def round_half_even(x: Fraction) -> int:
    """Nearest integer to a non-negative rational, ties to the even neighbour."""
    x = Fraction(x)
    assert x >= 0
    fl = x.numerator // x.denominator
    rem = x - fl
    half = Fraction(1, 2)
    if rem > half:
        return fl + 1
    if rem < half:
        return fl
    return fl if fl % 2 == 0 else fl + 1


def q_star(m: int, b_pcie: int, b_cpu: int) -> int:
    """Unclamped balanced fill count round(m * B_pcie / (B_pcie + B_cpu))."""
    if b_pcie < 0 or b_cpu < 0 or b_pcie + b_cpu == 0:
        raise ValueError("bandwidths must be non-negative and not both zero")
    return round_half_even(Fraction(m * b_pcie, b_pcie + b_cpu))


def q_star_pages(m: int, B_P: Fraction | float, B_H: Fraction | float) -> int:
    """The pages' own form round(m * B_P / B_H) in exact arithmetic (B_H = B_P + B_cpu)."""
    return round_half_even(Fraction(m) * Fraction(B_P) / Fraction(B_H))


def fill_count(m: int, b_pcie: int, b_cpu: int, max_fetch: int, evictable: int) -> int:
    """q for one call: clamp max(1, min(q*, m)) when m > 0, then cap by K and V."""
    if m == 0:
        return 0
    q = max(1, min(q_star(m, b_pcie, b_cpu), m))
    return max(0, min(q, max_fetch, evictable))


def branch_times(q: int, m: int, B_P: Fraction | float, B_H: Fraction | float):
    """(T_fill, T_cpu) in units of one expert's bytes S: q/B_P and (m-q)/(B_H-B_P).

    The fill branch moves q experts over the link at B_P; the CPU branch runs
    m-q experts in place on the residual host bandwidth B_H - B_P.
    """
    B_P = Fraction(B_P)
    B_H = Fraction(B_H)
    t_fill = Fraction(q) / B_P
    t_cpu = Fraction(m - q) / (B_H - B_P) if m > q else Fraction(0)
    return t_fill, t_cpu


def recommend_hybrid(B_P, B_H, threshold: Fraction = Fraction(2)) -> bool:
    """Calibration rule: recommend the hybrid backend iff B_H > threshold * B_P (threshold 2.0)."""
    return Fraction(B_H) > Fraction(threshold) * Fraction(B_P)
