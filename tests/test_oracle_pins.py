"""Pins of the fp64 oracle against facts other than itself.

Each test ties the token oracle (oracle/gdn_oracle.c) to something it does
not share code with: a hand-worked example, exact rational arithmetic, closed
forms of special cases, invariants of the delta rule, library routines
(scipy.signal.lfilter, torch.autograd) and the independent chunked form.
Together they catch a dropped term, a wrong sign, a wrong index or a
transposed operand anywhere in the recurrence (see test_oracle_mutations.py).
"""
import json
import math
import os
from fractions import Fraction

import numpy as np
import pytest

import gdn_inputs as gi
import oracle
from oracle import chunked, exact_tiny

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _batch_from_float(q, k, v, g, beta, s0=None, h_k=1, h_v=1):
    """Single-sequence batch from exactly-bf16-representable float arrays
    shaped [T][h][d]; raises if a value is not exact in bf16."""
    q = np.asarray(q, np.float32)
    k = np.asarray(k, np.float32)
    v = np.asarray(v, np.float32)
    for a in (q, k, v):
        assert np.array_equal(gi.bf16_to_f32(gi.bf16_bits(a)), a), "not bf16-exact"
    T = q.shape[0]
    d = q.shape[-1]
    b = gi.TokenBatch(h_k, h_v, d, np.array([0, T], np.int32),
                      gi.bf16_bits(q), gi.bf16_bits(k), gi.bf16_bits(v),
                      np.asarray(g, np.float32).reshape(T, h_v),
                      np.asarray(beta, np.float32).reshape(T, h_v), None)
    if s0 is not None:
        b.init_state = np.asarray(s0, np.float32).reshape(1, h_v, d, v.shape[-1])
    return b


def _dyadic(rng, shape, scale_pow=3, lo=-8, hi=8):
    return rng.integers(lo, hi + 1, size=shape).astype(np.float32) / np.float32(2 ** scale_pow)


# ---------------------------------------------------------------------------
# 1. Hand-worked example (tests/golden/worked_example_3tok.json)
# ---------------------------------------------------------------------------

def test_worked_example_by_hand():
    ex = json.load(open(os.path.join(GOLDEN, "worked_example_3tok.json")))
    fr = lambda m: np.array([[float(Fraction(x)) for x in r] for r in m])
    q, k, v = fr(ex["q"]), fr(ex["k"]), fr(ex["v"])
    alpha = np.array([float(Fraction(a)) for a in ex["alpha"]])
    beta = np.array([float(Fraction(b)) for b in ex["beta"]])
    g = np.log(alpha).astype(np.float32)
    b = _batch_from_float(q[:, None], k[:, None], v[:, None], g, beta, fr(ex["S0"]))
    r = oracle.run_chains(b)
    # g is stored in fp32, so alpha = exp(g) carries a relative error <= 2^-24 |g|.
    np.testing.assert_allclose(r["o"][0], fr(ex["o"]), rtol=0, atol=1e-6)
    np.testing.assert_allclose(r["s_final"][0], fr(ex["S_final"]), rtol=0, atol=1e-6)
    # The same example through the exact rational brute force is exact.
    o_ex, S_ex = exact_tiny.run(
        [[Fraction(x) for x in row] for row in ex["q"]],
        [[Fraction(x) for x in row] for row in ex["k"]],
        [[Fraction(x) for x in row] for row in ex["v"]],
        [Fraction(a) for a in ex["alpha"]], [Fraction(x) for x in ex["beta"]],
        [[Fraction(x) for x in row] for row in ex["S0"]])
    assert [[str(x) for x in row] for row in o_ex] == ex["o"]
    assert [[str(x) for x in row] for row in S_ex] == ex["S_final"]


# ---------------------------------------------------------------------------
# 2. Exact rational brute force on tiny dyadic inputs
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("seed", range(6))
def test_exact_rational_bruteforce(seed):
    rng = np.random.default_rng(seed)
    T, d_k, d_v = 6, 3, 4
    d = max(d_k, d_v)
    # The oracle takes d_k == d_v per batch; embed a 3x4 problem by zero padding
    # the key dimension (zero key components change nothing).
    q = np.zeros((T, 1, d), np.float32)
    k = np.zeros((T, 1, d), np.float32)
    q[:, 0, :d_k] = _dyadic(rng, (T, d_k))
    k[:, 0, :d_k] = _dyadic(rng, (T, d_k))
    v = _dyadic(rng, (T, 1, d_v))
    g = -rng.integers(0, 5, size=T).astype(np.float32) / np.float32(8)
    beta = rng.integers(0, 9, size=T).astype(np.float32) / np.float32(8)
    s0 = np.zeros((d, d_v), np.float32)
    s0[:d_k] = _dyadic(rng, (d_k, d_v))
    scale = 0.5
    b = _batch_from_float(q, k, v, g, beta, s0)
    r = oracle.run_chains(b, scale=scale)
    alpha = [Fraction(math.exp(float(x))) for x in g]   # the double the C oracle uses
    o_ex, S_ex = exact_tiny.run(q[:, 0].tolist(), k[:, 0].tolist(), v[:, 0].tolist(),
                                alpha, beta.tolist(), s0.tolist(), Fraction(scale))
    np.testing.assert_allclose(r["o"][0], np.array(o_ex, dtype=float), rtol=0, atol=1e-13)
    np.testing.assert_allclose(r["s_final"][0], np.array(S_ex, dtype=float), rtol=0, atol=1e-13)


# ---------------------------------------------------------------------------
# 3. Closed forms and invariants of special cases
# ---------------------------------------------------------------------------

def test_beta_zero_is_pure_decay():
    """beta = 0: S_t = (prod alpha) S_0 and o_t = (prod_{s<=t} alpha_s) S_0^T q_t."""
    b = gi.token_batch([37], 2, 2, 16, seed=3, init_state=True)
    b.beta[:] = 0.0
    r = oracle.run_chains(b)
    for p, (s, h) in enumerate(r["pairs"]):
        S0 = b.init_state[s, h].astype(np.float64)
        G = np.cumsum(b.g[:, h].astype(np.float64))
        q = gi.bf16_to_f32(b.q[:, h // (b.h_v // b.h_k)]).astype(np.float64)
        o_ref = np.exp(G)[:, None] * (q @ S0)
        np.testing.assert_allclose(r["o"][p], o_ref, rtol=1e-12, atol=1e-14)
        np.testing.assert_allclose(r["s_final"][p], np.exp(G[-1]) * S0, rtol=1e-12, atol=1e-14)


def test_delta_rule_overwrites_along_unit_key():
    """beta = 1 and |k| = 1: S_t^T k_t = v_t for any alpha and S_{t-1}; with
    q_t = k_t the post-update output therefore equals v_t exactly."""
    rng = np.random.default_rng(1)
    T, d = 9, 4
    signs = rng.choice([-0.5, 0.5], size=(T, 1, d)).astype(np.float32)  # |k| = 1 exactly
    v = _dyadic(rng, (T, 1, d))
    g = rng.uniform(-1.0, 0.0, size=T).astype(np.float32)
    b = _batch_from_float(signs, signs, v, g, np.ones(T, np.float32), _dyadic(rng, (d, d)))
    r = oracle.run_chains(b)
    np.testing.assert_allclose(r["o"][0], v[:, 0].astype(np.float64), rtol=0, atol=1e-12)
    np.testing.assert_allclose(r["s_final"][0].T @ signs[-1, 0], v[-1, 0], rtol=0, atol=1e-12)


def test_orthonormal_keys_store_and_retrieve():
    """alpha = beta = 1, S_0 = 0, orthonormal keys: S = sum_i k_i v_i^T, and a
    read-only query (beta = 0) with q = k_j returns v_j."""
    H = np.array([[1, 1, 1, 1], [1, -1, 1, -1], [1, 1, -1, -1], [1, -1, -1, 1]], np.float32) / 2
    rng = np.random.default_rng(2)
    v = _dyadic(rng, (4, 4))
    order = [2, 0, 3, 1]
    keys = H[order]
    qs = np.concatenate([keys, H], 0)           # 4 writes, then 4 read-only queries
    ks = np.concatenate([keys, H], 0)
    vs = np.concatenate([v, np.zeros((4, 4), np.float32)], 0)
    beta = np.array([1] * 4 + [0] * 4, np.float32)
    b = _batch_from_float(qs[:, None], ks[:, None], vs[:, None], np.zeros(8, np.float32), beta)
    r = oracle.run_chains(b)
    S_ref = keys.T.astype(np.float64) @ v.astype(np.float64)
    np.testing.assert_allclose(r["s_final"][0], S_ref, rtol=0, atol=1e-14)
    for j in range(4):
        np.testing.assert_allclose(r["o"][0][4 + j], v[order.index(j)], rtol=0, atol=1e-14)


def test_update_is_a_gradient_step_on_the_regression_loss():
    """The gated delta rule is one gradient step, size beta, on
    L(X) = 1/2 |X^T k - v|^2 taken at the decayed state X = alpha S:
    S_t = X - beta dL/dX.  The gradient comes from torch.autograd."""
    torch = pytest.importorskip("torch")
    b = gi.token_batch([1], 1, 1, 32, seed=5, init_state=True)
    r = oracle.run_chains(b)
    alpha = math.exp(float(b.g[0, 0]))
    beta = float(b.beta[0, 0])
    S = torch.tensor(b.init_state[0, 0], dtype=torch.float64)
    k = torch.tensor(gi.bf16_to_f32(b.k[0, 0]), dtype=torch.float64)
    v = torch.tensor(gi.bf16_to_f32(b.v[0, 0]), dtype=torch.float64)
    X = (alpha * S).requires_grad_(True)
    loss = 0.5 * torch.sum((X.T @ k - v) ** 2)
    loss.backward()
    S_ref = (X - beta * X.grad).detach().numpy()
    np.testing.assert_allclose(r["s_final"][0], S_ref, rtol=1e-12, atol=1e-13)


def test_beta_two_is_a_householder_reflection():
    """alpha = 1, beta = 2, v = 0, |k| = 1: S_t = (I - 2kk^T) S_{t-1}, an
    orthogonal reflection: the Frobenius norm is kept and applying the same
    key twice returns the start state."""
    rng = np.random.default_rng(4)
    d = 4
    kk = rng.choice([-0.5, 0.5], size=(1, 1, d)).astype(np.float32)
    ks = np.concatenate([kk, kk], 0)
    s0 = _dyadic(rng, (d, d))
    b1 = _batch_from_float(ks[:1], ks[:1], np.zeros((1, 1, d), np.float32), [0.0], [2.0], s0)
    r1 = oracle.run_chains(b1)
    assert abs(np.linalg.norm(r1["s_final"][0]) - np.linalg.norm(s0.astype(np.float64))) < 1e-13
    b2 = _batch_from_float(ks, ks, np.zeros((2, 1, d), np.float32), [0.0, 0.0], [2.0, 2.0], s0)
    r2 = oracle.run_chains(b2)
    np.testing.assert_allclose(r2["s_final"][0], s0, rtol=0, atol=1e-14)


def test_scalar_case_is_a_first_order_linear_filter():
    """d_k = d_v = 1 with constant alpha, beta, k: s_t = c s_{t-1} + beta k v_t
    with c = alpha (1 - beta k^2); scipy.signal.lfilter computes the same
    recursion, and o_t = scale q_t s_t."""
    signal = pytest.importorskip("scipy.signal")
    rng = np.random.default_rng(6)
    T = 50
    kval, alpha, beta, s0 = 0.75, 0.875, 0.625, 0.5
    v = _dyadic(rng, (T, 1, 1))
    q = _dyadic(rng, (T, 1, 1))
    g = np.full(T, math.log(alpha), np.float32)
    alpha_d = math.exp(float(g[0]))
    b = _batch_from_float(q, np.full((T, 1, 1), kval, np.float32), v, g,
                          np.full(T, beta, np.float32), [[s0]])
    r = oracle.run_chains(b, scale=0.5)
    c = alpha_d * (1 - beta * kval * kval)
    s_ref, _ = signal.lfilter([beta * kval], [1.0, -c], v[:, 0, 0].astype(np.float64), zi=[c * s0])
    np.testing.assert_allclose(r["o"][0][:, 0], 0.5 * q[:, 0, 0] * s_ref, rtol=1e-12, atol=1e-14)
    np.testing.assert_allclose(r["s_final"][0][0, 0], s_ref[-1], rtol=1e-12)


def test_linear_in_initial_state_and_values():
    """F(S0, V) = F(S0, 0) + F(0, V) for outputs and states."""
    b = gi.token_batch([70], 2, 2, 32, seed=8, init_state=True)
    r_full = oracle.run_chains(b)
    b_s0 = gi.token_batch([70], 2, 2, 32, seed=8, init_state=True)
    b_s0.v[:] = 0
    r_s0 = oracle.run_chains(b_s0)
    b_v = gi.token_batch([70], 2, 2, 32, seed=8, init_state=False)
    r_v = oracle.run_chains(b_v)
    for p in range(len(r_full["pairs"])):
        np.testing.assert_allclose(r_full["o"][p], r_s0["o"][p] + r_v["o"][p], rtol=1e-11, atol=1e-12)
        np.testing.assert_allclose(r_full["s_final"][p], r_s0["s_final"][p] + r_v["s_final"][p],
                                   rtol=1e-11, atol=1e-12)


# ---------------------------------------------------------------------------
# 4. Structural properties: GVA mapping, resume, emission
# ---------------------------------------------------------------------------

def test_gva_equals_repeated_key_heads():
    """Value head h reads key head h // (h_v / h_k): a GVA batch equals an
    h_k = h_v batch whose key heads are repeated in contiguous groups."""
    b = gi.token_batch([40, 23], 2, 6, 16, seed=9, init_state=True)
    r = oracle.run_chains(b)
    rep = gi.TokenBatch(6, 6, 16, b.cu_seqlens, np.repeat(b.q, 3, axis=1), np.repeat(b.k, 3, axis=1),
                        b.v, b.g, b.beta, b.init_state)
    r2 = oracle.run_chains(rep)
    for p in range(len(r["pairs"])):
        np.testing.assert_array_equal(r["o"][p], r2["o"][p])
        np.testing.assert_array_equal(r["s_final"][p], r2["s_final"][p])


def _slice_batch(b, t0, t1, s0=None):
    return gi.TokenBatch(b.h_k, b.h_v, b.d, np.array([0, t1 - t0], np.int32), b.q[t0:t1], b.k[t0:t1],
                         b.v[t0:t1], b.g[t0:t1], b.beta[t0:t1], s0)


def test_resume_from_a_split_is_exact():
    """Stopping after token t and resuming from the fp64 state reproduces the
    uninterrupted outputs and final state bit for bit (same operations)."""
    b = gi.token_batch([150], 1, 2, 16, seed=10, init_state=True)
    full = oracle.run_chains(b)
    for t in (1, 64, 100):
        a = oracle.run_chains(_slice_batch(b, 0, t, b.init_state))
        rest = oracle.run_chains(_slice_batch(b, t, 150), init_state=a["s_final"])
        for p in range(len(full["pairs"])):
            np.testing.assert_array_equal(full["o"][p][:t], a["o"][p])
            np.testing.assert_array_equal(full["o"][p][t:], rest["o"][p])
            np.testing.assert_array_equal(full["s_final"][p], rest["s_final"][p])


def test_emitted_states_equal_truncated_runs():
    b = gi.token_batch([200, 130], 1, 2, 16, seed=11, init_state=True)
    r = oracle.run_chains(b, emit_every=64)
    for p, (s, h) in enumerate(r["pairs"]):
        L = b.seqlens[s]
        assert len(r["emits"][p]) == L // 64
        t0 = int(b.cu_seqlens[s])
        for e in range(L // 64):
            bb = _slice_batch(b, t0, t0 + 64 * (e + 1), b.init_state[s:s + 1])
            rr = oracle.run_chains(bb, pairs=[(0, h)])
            np.testing.assert_array_equal(r["emits"][p][e], rr["s_final"][0])


# ---------------------------------------------------------------------------
# 5. The independent chunked (UT / WY) form agrees with the token oracle
# ---------------------------------------------------------------------------

def _chain_arrays(b, s, h):
    t0, t1 = int(b.cu_seqlens[s]), int(b.cu_seqlens[s + 1])
    kh = h // (b.h_v // b.h_k)
    f = lambda x: gi.bf16_to_f32(x).astype(np.float64)
    return (f(b.q[t0:t1, kh]), f(b.k[t0:t1, kh]), f(b.v[t0:t1, h]),
            b.g[t0:t1, h].astype(np.float64), b.beta[t0:t1, h].astype(np.float64))


@pytest.mark.parametrize("C", [1, 16, 64])
def test_chunked_form_matches_token_oracle(C):
    b = gi.token_batch([64, 100, 157], 2, 4, 32, seed=12, init_state=True)
    r = oracle.run_chains(b, scale=0.25, emit_every=64)
    for p, (s, h) in enumerate(r["pairs"]):
        Q, K, V, g, beta = _chain_arrays(b, s, h)
        O, S, emits = chunked.chunked_chain(Q, K, V, g, beta, b.init_state[s, h].astype(np.float64), C=C,
                                            scale=0.25, emit_every_chunks=64 // C)
        rel = np.linalg.norm(O - r["o"][p]) / np.linalg.norm(r["o"][p])
        assert rel < 1e-10, rel
        rel_s = np.linalg.norm(S - r["s_final"][p]) / np.linalg.norm(r["s_final"][p])
        assert rel_s < 1e-10, rel_s
        assert len(emits) == len(r["emits"][p])
        for e1, e2 in zip(emits, r["emits"][p]):
            assert np.linalg.norm(e1 - e2) < 1e-10 * np.linalg.norm(e2)


def test_chunked_form_with_gates_from_the_workload_recipe():
    """Strong decay (g ~ -0.1 softplus(N(0,1))) and d = 128 as in the serving
    workloads; the two forms still agree."""
    b = gi.token_batch([130], 1, 1, 128, seed=13, init_state=True)
    r = oracle.run_chains(b)
    Q, K, V, g, beta = _chain_arrays(b, 0, 0)
    O, S, _ = chunked.chunked_chain(Q, K, V, g, beta, b.init_state[0, 0].astype(np.float64))
    assert np.linalg.norm(O - r["o"][0]) / np.linalg.norm(r["o"][0]) < 1e-10
    assert np.linalg.norm(S - r["s_final"][0]) / np.linalg.norm(r["s_final"][0]) < 1e-10


# ---------------------------------------------------------------------------
# 6. Prefix-cache grid rules against the values printed on the page
# ---------------------------------------------------------------------------

def test_prefix_grid_rules_match_the_page():
    from oracle import grid
    ex = json.load(open(os.path.join(GOLDEN, "prefix_grid.json")))
    assert grid.align_block_size(ex["block_size_in"]) == ex["block_size_aligned"]
    assert grid.grid_tokens(ex["block_size_in"]) == ex["grid"]
    for h in ex["hits"]:
        assert grid.floor_hit(h["hit"], h["prompt"], ex["block_size_in"]) == h["floored"]
    # a hit covering the full prompt is not floored
    assert grid.floor_hit(2000, 2000, ex["block_size_in"]) == 2000
    # the emission stride of the 1088-token grid is 17 chunks of 64
    assert ex["grid"] // ex["chunk"] == 17
