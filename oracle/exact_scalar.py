"""Exact rational evaluation of the K = V = 1 KDA case -- TEST INFRASTRUCTURE ONLY.

With one key channel and one value channel the recurrence
S_t = (1 - beta_t k^_t^2) a_t S_{t-1} + beta_t k^_t v_t (a_t = e^{g_t}, k^ = k/|k|
so k^2 = 1) has the explicit solution

    S_t = sum_{j <= t} beta_j k^_j v_j  prod_{i=j+1..t} (1 - beta_i) a_i,
    o_t = scale * S_t * q^_t,

which this module evaluates term by term in ``fractions.Fraction`` -- a
different computation from the oracle's token loop, with no rounding at all.
The decay factors a_t are given as rationals; the oracle receives g_t = ln a_t.
"""
from __future__ import annotations

from fractions import Fraction
from typing import List, Sequence, Tuple


def _sign(x: Fraction) -> int:
    if x == 0:
        raise ValueError("a zero key/query has no direction")
    return 1 if x > 0 else -1


def explicit_sum(q: Sequence[Fraction], k: Sequence[Fraction], v: Sequence[Fraction],
                 a: Sequence[Fraction], beta: Sequence[Fraction], cu_seqlens: Sequence[int],
                 scale: Fraction) -> Tuple[List[Fraction], List[Fraction]]:
    """Outputs o_t (one per token) and the final S of each sequence."""
    o: List[Fraction] = [Fraction(0)] * len(q)
    finals: List[Fraction] = []
    for n in range(len(cu_seqlens) - 1):
        bos, eos = cu_seqlens[n], cu_seqlens[n + 1]
        S_t = Fraction(0)
        for t in range(bos, eos):
            S_t = Fraction(0)
            for j in range(bos, t + 1):
                term = beta[j] * _sign(k[j]) * v[j]
                for i in range(j + 1, t + 1):
                    term *= (1 - beta[i]) * a[i]
                S_t += term
            o[t] = scale * S_t * _sign(q[t])
        finals.append(S_t if eos > bos else Fraction(0))
    return o, finals
