"""The KDA recurrence in exact rational arithmetic -- TEST INFRASTRUCTURE.

For tiny inputs only (a few tokens, d <= 4).  Decay gates are given directly
as rationals alpha (not log alpha) so that nothing is rounded.  Same steps
and order as the recurrence in the deep dive, section 03:
S' = Diag(alpha) S; e = v - S'^T k; S = S' + beta k e^T; o = S^T q.
"""
from __future__ import annotations

from fractions import Fraction as F


def prefill(q, k, v, alpha, beta, s0):
    """q, k, alpha: [T][dk]; v: [T][dv]; beta: [T]; s0: [dk][dv] (Fractions).

    Returns (out [T][dv], final state [dk][dv]) as lists of Fractions.
    """
    dk, dv = len(s0), len(s0[0])
    S = [[F(x) for x in row] for row in s0]
    out = []
    for t in range(len(q)):
        S = [[F(alpha[t][i]) * S[i][j] for j in range(dv)] for i in range(dk)]
        e = [F(v[t][j]) - sum(F(k[t][i]) * S[i][j] for i in range(dk)) for j in range(dv)]
        S = [[S[i][j] + F(beta[t]) * F(k[t][i]) * e[j] for j in range(dv)] for i in range(dk)]
        out.append([sum(F(q[t][i]) * S[i][j] for i in range(dk)) for j in range(dv)])
    return out, S
