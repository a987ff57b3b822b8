"""Seeded random mixed steps through the C ABI against the fp64 oracle:
random decode-row counts, prefill lengths around the chunk edges, head
layouts, emission periods and slot assignments, each checked in full
(every output, every final and emitted state)."""
import numpy as np
import pytest
import torch

import gdn_inputs as gi
import oracle
from tests import gpu_util as gu

pytestmark = pytest.mark.gpu

LENGTHS = (0, 1, 2, 63, 64, 65, 127, 128, 129, 200, 700, 1100)
HEADS = ((4, 4, 64), (2, 6, 64), (4, 8, 128), (8, 8, 128))


@pytest.fixture(scope="module")
def gdn():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from linear_attention_serving_gdn_gb300 import _build
    _build.build()
    import linear_attention_serving_gdn_gb300 as m
    return m


@pytest.mark.parametrize("case", range(40))
def test_random_mixed_step_vs_oracle(gdn, case):
    rng = np.random.default_rng(1000 + case)
    h_k, h_v, d = HEADS[case % len(HEADS)]
    nd = int(rng.integers(0, 24))
    lens = [int(x) for x in rng.choice(LENGTHS, size=int(rng.integers(1, 6)))]
    E = int(rng.choice([0, 1, 17]))
    scale = float(rng.choice([1.0, d ** -0.5]))
    dec = gi.token_batch([1] * max(nd, 1), h_k, h_v, d, 2000 + case, init_state=True)
    pre = gi.token_batch(lens, h_k, h_v, d, 3000 + case, init_state=True)
    n_slots = 2 * (nd + len(lens)) + 1
    perm = rng.permutation(n_slots).astype(np.int32)
    dsrc, psrc = perm[:nd], perm[nd:nd + len(lens)]
    pdst = perm[nd + len(lens):nd + 2 * len(lens)]
    cache = gu.empty_cache(n_slots, h_v, d)
    if nd:
        gu.put_states(cache, dsrc, dec.init_state[:nd])
    gu.put_states(cache, psrc, pre.init_state)
    decs = {n: getattr(dec, n)[:nd] for n in ("q", "k", "v", "g", "beta")}
    arrs = gu.arrays_to_device({n: np.concatenate([decs[n], getattr(pre, n)]) for n in decs})
    T = nd + pre.total_tokens
    o = torch.full((T, h_v, d), 9.0, dtype=torch.bfloat16, device="cuda")
    n_emit = gdn.gdn_prefill_num_emits(pre.cu_seqlens, E) if E else 0
    cs = torch.zeros((max(n_emit, 1), h_v, d, d), device="cuda") if E else None
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    t = lambda x: torch.from_numpy(np.ascontiguousarray(x)).cuda()
    gdn.gdn_mixed_step(nd, arrs["q"], arrs["k"], arrs["v"], arrs["g"], arrs["beta"],
                       t(pre.cu_seqlens.astype(np.int32)), [int(x) for x in pre.cu_seqlens], cache,
                       t(dsrc) if nd else None, o, pre_src_slot=t(psrc), pre_dst_slot=t(pdst),
                       chunk_states=cs, emit_every_chunks=E, dev_status=st, scale=scale)
    torch.cuda.synchronize()
    assert st.item() == 0
    o_np = gu.o_to_numpy(o)
    if nd:
        b_dec = gi.TokenBatch(h_k, h_v, d, np.arange(nd + 1, dtype=np.int32), decs["q"], decs["k"], decs["v"],
                              decs["g"], decs["beta"], dec.init_state[:nd])
        r_dec = oracle.run_chains(b_dec, scale=scale)
        gu.assert_o_close(o_np[:nd], gu.o_ref_dense(b_dec, r_dec), "decode o")
        gu.assert_state_close(gu.get_states_math(cache, dsrc), r_dec["s_final"].reshape(nd, h_v, d, d),
                              "decode state")
    r_pre = oracle.run_chains(pre, scale=scale, emit_every=64 * E)
    gu.assert_o_close(o_np[nd:], gu.o_ref_dense(pre, r_pre), "prefill o")
    gu.assert_state_close(gu.get_states_math(cache, pdst), r_pre["s_final"].reshape(len(lens), h_v, d, d),
                          "prefill state")
    if E and n_emit:
        offs = gdn.gdn_prefill_emit_offsets(pre.cu_seqlens, E)
        per_pair = {pair: np.asarray(e).reshape(-1, d, d) for pair, e in zip(r_pre["pairs"], r_pre["emits"])}
        want = np.stack([np.stack([per_pair[(s, hh)][kk] for hh in range(h_v)])
                         for s in range(len(lens)) for kk in range(offs[s + 1] - offs[s])])
        gu.assert_state_close(gu.get_states_math(cs, list(range(n_emit))), want, "emitted states")
