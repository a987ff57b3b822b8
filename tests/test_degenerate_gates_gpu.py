"""Degenerate gates through the C ABI against the fp64 oracle.

Gated DeltaNet (Yang, Kautz, Hatamizadeh, ICLR 2025; the gating the vLLM
pages' GDN layer uses) has boundary values of its two gates where the
recurrence reduces to a simpler one: alpha_t = exp(g_t) = 1 is the plain
delta rule with nothing forgotten, alpha_t -> 0 (g_t very negative) erases
the state, beta_t = 0 leaves it to decay without a write, beta_t = 1 replaces
the value stored along the key.  The chunked prefill forms exp(G_t - G_s)
over a whole 64-token chunk, so these cases stress its decay factors: no
decay at all across many chunks (rounding is not damped), and factors that
underflow to zero inside a chunk (the masked upper triangle must stay out of
the products).  Same bars as the other parity tests.
"""
import dataclasses

import numpy as np
import pytest
import torch

import gdn_inputs as gi
import oracle
from tests import gpu_util as gu
from tests.test_parity_gpu import _prefill_vs_oracle

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def gdn():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from linear_attention_serving_gdn_gb300 import _build
    _build.build()
    import linear_attention_serving_gdn_gb300 as m
    return m


def _f32(x):
    return np.ascontiguousarray(x, dtype=np.float32)


# pattern -> (g, beta) from a seeded generator and the recipe's own gates
PATTERNS = {
    "no_decay": lambda rng, g, b: (np.zeros_like(g), b),
    "no_decay_full_write": lambda rng, g, b: (np.zeros_like(g), np.ones_like(b)),
    "weak_decay": lambda rng, g, b: (np.full_like(g, -1e-3), b),
    "erase_one_token_in_ten": lambda rng, g, b: (np.where(rng.random(g.shape) < 0.1, -30.0, 0.0), b),
    "mostly_no_write": lambda rng, g, b: (g, np.where(rng.random(b.shape) < 0.9, 0.0, b)),
}


def _with_pattern(b: gi.TokenBatch, name: str, seed: int) -> gi.TokenBatch:
    g, beta = PATTERNS[name](np.random.default_rng(seed), b.g, b.beta)
    return dataclasses.replace(b, g=_f32(g), beta=_f32(beta))


@pytest.mark.parametrize("pattern", list(PATTERNS))
@pytest.mark.parametrize("d,h_k,h_v", [(128, 2, 4), (64, 2, 6)])
def test_prefill_degenerate_gates(gdn, pattern, d, h_k, h_v):
    """Sequences of 1, 64, 130 and 700 tokens from given initial states,
    every chunk's state emitted (E = 1): outputs, final and emitted states."""
    b = gi.token_batch([1, 64, 130, 700], h_k, h_v, d, seed=61, init_state=True)
    b = _with_pattern(b, pattern, 62)
    _prefill_vs_oracle(gdn, b, E=1, init_slots=[1, 1, 1, 1], scale=d ** -0.5)


@pytest.mark.parametrize("pattern", list(PATTERNS))
def test_decode_degenerate_gates(gdn, pattern):
    """64 cached rows, H = 16, d = 128, four in-place decode steps."""
    rows, h, d, steps = 64, 16, 128, 4
    seqs = _with_pattern(gi.token_batch([steps] * rows, h, h, d, 71, init_state=True), pattern, 72)
    src, n_slots = gi.slots(rows, 71)
    cache = gu.empty_cache(n_slots, h, d)
    gu.put_states(cache, src, seqs.init_state)
    src_t = torch.from_numpy(src).cuda()
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    outs = []
    for t in range(steps):
        idx = seqs.cu_seqlens[:-1] + t
        x = gu.arrays_to_device({n: getattr(seqs, n)[idx] for n in ("q", "k", "v", "g", "beta")})
        o = torch.empty((rows, h, d), dtype=torch.bfloat16, device="cuda")
        gdn.gdn_decode_packed(x["q"], x["k"], x["v"], x["g"], x["beta"], cache, src_t, o, dev_status=st)
        outs.append(gu.o_to_numpy(o))
    torch.cuda.synchronize()
    assert st.item() == 0
    ref = oracle.run_chains(seqs)
    gu.assert_o_close(np.stack(outs, 1).reshape(rows * steps, h, d), gu.o_ref_dense(seqs, ref))
    gu.assert_state_close(gu.get_states_math(cache, src), ref["s_final"].reshape(rows, h, d, d))
