"""Input preparation of a Gated DeltaNet layer, in fp64.  TEST INFRASTRUCTURE.

The pages give no formula for this step ("parity unpinned" against the
pages).  Reading, from the Gated DeltaNet layer (Yang, Kautz, Hatamizadeh,
ICLR 2025) as used by the Qwen3-Next models the pages serve:

    q_hat = q / sqrt(sum(q^2) + eps),  k_hat likewise   (per token and key head)
    g     = -exp(A_log[h]) * softplus(a + dt_bias[h])   (log decay, alpha = exp(g))
    beta  = sigmoid(b)

with softplus(x) = log(1 + exp(x)).  The normalised q, k are then rounded to
bf16 (round to nearest even) and g, beta to fp32: the storage types the
recurrence consumes.  Pinned in tests/test_oracle_prep_pins.py by closed
forms (unit norms, softplus(0) = ln 2, sigmoid(0) = 1/2, the large-argument
limits, scale invariance of the normalisation).
"""
from __future__ import annotations

import numpy as np

import gdn_inputs as gi


def l2_normalize(x: np.ndarray, eps: float) -> np.ndarray:
    x = np.asarray(x, np.float64)
    return x / np.sqrt(np.sum(x * x, axis=-1, keepdims=True) + eps)


def softplus(x: np.ndarray) -> np.ndarray:
    x = np.asarray(x, np.float64)
    return np.log1p(np.exp(-np.abs(x))) + np.maximum(x, 0.0)


def sigmoid(x: np.ndarray) -> np.ndarray:
    x = np.asarray(x, np.float64)
    return 1.0 / (1.0 + np.exp(-x))


def gates(a, b, A_log, dt_bias):
    """(g, beta) in fp64 for a, b [T][h_v] and per-head A_log, dt_bias [h_v]."""
    g = -np.exp(np.asarray(A_log, np.float64)) * softplus(np.asarray(a, np.float64) + np.asarray(dt_bias, np.float64))
    return g, sigmoid(b)


def prep(raw: gi.RawInputs, eps: float = 1e-6):
    """(q_bits, k_bits, g, beta): normalised q, k as bf16 bits, g and beta as
    fp32, ready for the recurrence."""
    q = l2_normalize(gi.bf16_to_f32(raw.q), eps)
    k = l2_normalize(gi.bf16_to_f32(raw.k), eps)
    g, beta = gates(raw.a, raw.b, raw.A_log, raw.dt_bias)
    return (gi.bf16_bits(q.astype(np.float32)), gi.bf16_bits(k.astype(np.float32)),
            g.astype(np.float32), beta.astype(np.float32))
