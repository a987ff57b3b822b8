"""Exact rational brute force of the gated delta rule.  TEST INFRASTRUCTURE.

For tiny cases (d <= 4, a handful of tokens) with dyadic inputs, this runs
the recurrence of Gated DeltaNet (Yang, Kautz and Hatamizadeh, ICLR 2025, the
gated delta rule) in ``fractions.Fraction`` arithmetic, with no rounding at
all:

    S_t = alpha_t S_{t-1} - beta_t k_t (k_t^T (alpha_t S_{t-1})) + beta_t k_t v_t^T
    o_t = scale * S_t^T q_t

``alpha`` is given directly (as an exact rational or as the exact value of a
double), so the only rounding on the fp64 side is its own arithmetic.
"""
from __future__ import annotations

from fractions import Fraction


def run(q, k, v, alpha, beta, S0, scale=Fraction(1)):
    """q, k: [T][d_k]; v: [T][d_v]; alpha, beta: [T]; S0: [d_k][d_v].

    All entries are converted with ``Fraction(x)`` (exact for floats).
    Returns (o [T][d_v], S_T [d_k][d_v]) as nested lists of Fractions.
    """
    F = Fraction
    d_k, d_v = len(S0), len(S0[0])
    S = [[F(S0[i][j]) for j in range(d_v)] for i in range(d_k)]
    outs = []
    for t in range(len(q)):
        a, b = F(alpha[t]), F(beta[t])
        kt = [F(x) for x in k[t]]
        qt = [F(x) for x in q[t]]
        vt = [F(x) for x in v[t]]
        aS = [[a * S[i][j] for j in range(d_v)] for i in range(d_k)]
        kaS = [sum(kt[i] * aS[i][j] for i in range(d_k)) for j in range(d_v)]
        S = [[aS[i][j] - b * kt[i] * kaS[j] + b * kt[i] * vt[j] for j in range(d_v)]
             for i in range(d_k)]
        outs.append([F(scale) * sum(S[i][j] * qt[i] for i in range(d_k)) for j in range(d_v)])
    return outs, S
