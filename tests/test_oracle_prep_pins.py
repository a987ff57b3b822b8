"""Pins of the fp64 input-preparation oracle (oracle/prep.py) against closed
forms.  The formula itself is a reading (the pages give none); these tests
check that the oracle computes that reading, not that the reading is the
pages'."""
import math

import numpy as np

import gdn_inputs as gi
from oracle import prep


def test_normalised_rows_have_unit_norm_and_keep_direction():
    rng = np.random.default_rng(0)
    x = rng.standard_normal((50, 3, 128)) * rng.uniform(0.1, 10, (50, 3, 1))
    y = prep.l2_normalize(x, 0.0)
    assert np.allclose(np.linalg.norm(y, axis=-1), 1.0, atol=1e-14)
    cos = np.sum(x * y, axis=-1) / np.linalg.norm(x, axis=-1)
    assert np.allclose(cos, 1.0, atol=1e-14)
    # scale invariance, and eps only matters for tiny rows
    assert np.allclose(prep.l2_normalize(7.5 * x, 0.0), y, atol=1e-14)
    z = prep.l2_normalize(np.full((1, 4), 1e-4), 1e-6)   # |x|^2 = 4e-8 << eps
    assert np.allclose(z, 1e-4 / math.sqrt(4e-8 + 1e-6))


def test_softplus_and_sigmoid_closed_forms():
    assert prep.softplus(0.0) == math.log(2.0)
    assert abs(prep.softplus(50.0) - 50.0) < 1e-15
    assert abs(prep.softplus(-50.0) - math.exp(-50.0)) < 1e-30
    x = np.linspace(-5, 5, 11)
    assert np.allclose(prep.softplus(x) - prep.softplus(-x), x, atol=1e-14)     # softplus(x) - softplus(-x) = x
    assert prep.sigmoid(0.0) == 0.5
    assert np.allclose(prep.sigmoid(x) + prep.sigmoid(-x), 1.0, atol=1e-15)
    assert np.allclose(np.exp(-prep.softplus(-x)), prep.sigmoid(x), atol=1e-15)  # sigmoid = exp(-softplus(-x))


def test_gates_special_values():
    A_log = np.log(np.array([0.1, 0.5]))
    dt_bias = np.array([0.25, -1.0])
    a = -dt_bias[None, :] * np.ones((3, 2))          # a + dt_bias = 0
    b = np.zeros((3, 2))
    g, beta = prep.gates(a, b, A_log, dt_bias)
    assert np.allclose(g, -np.array([0.1, 0.5]) * math.log(2.0))
    assert np.all(beta == 0.5)
    g2, _ = prep.gates(np.full((1, 2), 40.0), b[:1], A_log, dt_bias)
    assert np.allclose(g2, -np.array([0.1, 0.5]) * (40.0 + dt_bias), rtol=1e-15)
    assert np.all(g < 0)


def test_prep_outputs_are_the_storage_types():
    raw = gi.raw_inputs(16, 2, 4, 64, seed=3)
    qb, kb, g, beta = prep.prep(raw)
    assert qb.dtype == np.uint16 and kb.dtype == np.uint16
    assert g.dtype == np.float32 and beta.dtype == np.float32
    qn = np.linalg.norm(gi.bf16_to_f32(qb).astype(np.float64), axis=-1)
    assert np.allclose(qn, 1.0, atol=2 ** -7)        # bf16 rounding of unit rows
    assert np.all((beta > 0) & (beta < 1)) and np.all(g < 0)
