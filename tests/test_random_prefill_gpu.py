"""Seeded random large prefill batches through the C ABI: up to 48
sequences of 1..3000 tokens (tens of thousands of tokens per call), four
head layouts, emission every 1 or 17 chunks or none, from random fp32
states.  Each batch runs twice and must repeat bit for bit (every output,
final and emitted state); two sampled sequences are checked against the
fp64 oracle."""
import numpy as np
import pytest
import torch

import gdn_inputs as gi
import oracle
from tests import gpu_util as gu

pytestmark = pytest.mark.gpu

HEADS = ((16, 32, 128), (4, 8, 64), (16, 16, 128), (2, 6, 64))


@pytest.fixture(scope="module")
def gdn():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from linear_attention_serving_gdn_gb300 import _build
    _build.build()
    import linear_attention_serving_gdn_gb300 as m
    return m


def _run(gdn, b, E, S0):
    n = b.num_seqs
    cache = gu.empty_cache(2 * n, b.h_v, b.d)
    cache[:n] = S0
    src = torch.arange(n, dtype=torch.int32, device="cuda")
    dst = torch.arange(n, 2 * n, dtype=torch.int32, device="cuda")
    dv = gu.batch_to_device(b)
    o = torch.empty((b.total_tokens, b.h_v, b.d), dtype=torch.bfloat16, device="cuda")
    n_emit = gdn.gdn_prefill_num_emits(dv["cu_host"], E) if E else 0
    cs = torch.zeros((max(n_emit, 1), b.h_v, b.d, b.d), device="cuda") if E else None
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    gdn.gdn_prefill_varlen(dv["q"], dv["k"], dv["v"], dv["g"], dv["beta"], dv["cu"], dv["cu_host"], o,
                           state=cache, src_slot=src, dst_slot=dst, chunk_states=cs, emit_every_chunks=E,
                           dev_status=st)
    torch.cuda.synchronize()
    assert st.item() == 0
    return o, cache[n:].clone(), cs


@pytest.mark.parametrize("case", range(8))
def test_random_large_prefill_repeats_and_matches_oracle(gdn, case):
    rng = np.random.default_rng(7000 + case)
    h_k, h_v, d = HEADS[case % len(HEADS)]
    ns = int(rng.integers(1, 48))
    lens = [int(x) for x in rng.integers(1, 3000, size=ns)]
    E = int(rng.choice([0, 1, 17]))
    b = gi.token_batch(lens, h_k, h_v, d, 8000 + case, init_state=True)
    S0 = torch.from_numpy(np.swapaxes(b.init_state, -1, -2).copy()).cuda()
    o1, s1, c1 = _run(gdn, b, E, S0)
    o2, s2, c2 = _run(gdn, b, E, S0)
    assert torch.equal(o1.view(torch.int16), o2.view(torch.int16))
    assert torch.equal(s1, s2)
    if E:
        assert torch.equal(c1, c2)
    pick = sorted(rng.choice(ns, size=min(2, ns), replace=False).tolist())
    cu = b.cu_seqlens
    idx = np.concatenate([np.arange(cu[s], cu[s + 1]) for s in pick])
    sub_cu = np.concatenate([[0], np.cumsum([lens[s] for s in pick])]).astype(np.int32)
    sub = gi.TokenBatch(h_k, h_v, d, sub_cu, b.q[idx], b.k[idx], b.v[idx], b.g[idx], b.beta[idx],
                        b.init_state[pick])
    ref = oracle.run_chains(sub)
    gu.assert_o_close(gu.o_to_numpy(o1)[idx], gu.o_ref_dense(sub, ref))
    S = gu.get_states_math(s1, np.array(pick))
    gu.assert_state_close(np.stack([S[i, hh] for i in range(len(pick)) for hh in range(h_v)]), ref["s_final"])
