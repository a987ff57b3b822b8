"""Chunked (UT / WY) fp64 form of the gated delta rule.  TEST INFRASTRUCTURE.

A second, independent CPU form used only to check the token oracle.  It
follows the chunkwise parallel form of the delta rule (Yang, Wang, Zhang,
Shen and Kim, "Parallelizing Linear Transformers with the Delta Rule over
Sequence Length", NeurIPS 2024, the WY / UT representation) with the gating
of Gated DeltaNet (Yang, Kautz and Hatamizadeh, ICLR 2025), derived here from
the recurrence

    S_t = alpha_t (I - beta_t k_t k_t^T) S_{t-1} + beta_t k_t v_t^T,
    o_t = scale * S_t^T q_t.

For a chunk of C tokens entering with state S0, with local index i:

    G_i   = sum_{s<=i} log(alpha_s),      gamma_i = exp(G_i)
    write S_i = gamma_i S0 + sum_{j<=i} (gamma_i/gamma_j) k_j u_j^T.
    Substituting into the recurrence gives, for the rows u_i,
        u_i + beta_i sum_{j<i} (gamma_i/gamma_j) (k_i.k_j) u_j
            = beta_i (v_i - gamma_i S0^T k_i)
    i.e. (I + A) U = diag(beta) V - diag(beta gamma) K S0 with
        A_ij = beta_i (gamma_i/gamma_j) k_i.k_j  for j < i, else 0.
    With T = (I + A)^{-1}:  W = T diag(beta gamma) K,  U' = T diag(beta) V,
        U   = U' - W S0
        O   = scale * [diag(gamma) Q S0 + (M o Q K^T) U],
              M_ij = gamma_i/gamma_j for j <= i, else 0
        S_C = gamma_C S0 + (diag(gamma_C/gamma) K)^T U.

C = 1 reduces to the token recurrence.  The inverse is taken with scipy's
triangular solve.
"""
from __future__ import annotations

import numpy as np
from scipy.linalg import solve_triangular


def chunk_step(Q, K, V, g, beta, S0, scale=1.0):
    """One chunk: returns (O [C][d_v], S_C [d_k][d_v]); all fp64."""
    C = Q.shape[0]
    G = np.cumsum(g)
    gam = np.exp(G)
    ratio = np.exp(G[:, None] - G[None, :])           # gamma_i / gamma_j
    A = np.tril(beta[:, None] * ratio * (K @ K.T), -1)
    T = solve_triangular(np.eye(C) + A, np.eye(C), lower=True, unit_diagonal=True)
    W = T @ ((beta * gam)[:, None] * K)
    Up = T @ (beta[:, None] * V)
    U = Up - W @ S0
    M = np.tril(ratio)
    O = scale * (gam[:, None] * (Q @ S0) + (M * (Q @ K.T)) @ U)
    decay_to_end = np.exp(G[-1] - G)                   # gamma_C / gamma_i
    S_C = gam[-1] * S0 + (decay_to_end[:, None] * K).T @ U
    return O, S_C


def chunked_chain(Q, K, V, g, beta, S0, C=64, scale=1.0, emit_every_chunks=0):
    """Whole chain in chunks of C (last chunk may be partial).

    Returns (O [T][d_v], S_T, emitted states after every ``emit_every_chunks``
    full chunks)."""
    T = Q.shape[0]
    S = np.array(S0, dtype=np.float64, copy=True)
    O = np.zeros((T, V.shape[1]))
    emits = []
    for c, t0 in enumerate(range(0, T, C)):
        t1 = min(t0 + C, T)
        O[t0:t1], S = chunk_step(Q[t0:t1], K[t0:t1], V[t0:t1], g[t0:t1], beta[t0:t1], S, scale)
        if emit_every_chunks and t1 - t0 == C and (c + 1) % emit_every_chunks == 0:
            emits.append(S.copy())
    return O, S, emits
