"""Size limits of the C ABI against the fp64 oracle.

- More prefill sequences than the launch orders by length (2048): the rest
  keep their own order and must still run, each on its own chain.
- A state cache past 2^31 floats (8,200 slots x 16 heads x 128 x 128 fp32,
  8.6 GB): slots at its far end must be read and written at the right
  place by decode and prefill (64-bit state offsets).
"""
import numpy as np
import pytest
import torch

import gdn_inputs as gi
import oracle
from tests import gpu_util as gu

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def gdn():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from linear_attention_serving_gdn_gb300 import _build
    _build.build()
    import linear_attention_serving_gdn_gb300 as m
    return m


def test_prefill_more_sequences_than_the_length_order(gdn):
    n = 2100
    rng = np.random.default_rng(81)
    lens = [int(x) for x in rng.choice([1, 2, 64, 65, 130], size=n)]
    b = gi.token_batch(lens, 1, 2, 64, seed=81)
    x = gu.batch_to_device(b)
    cache = gu.empty_cache(n, b.h_v, b.d)
    dst = torch.arange(n, dtype=torch.int32, device="cuda")
    o = torch.empty((b.total_tokens, b.h_v, b.d), dtype=torch.bfloat16, device="cuda")
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    gdn.gdn_prefill_varlen(x["q"], x["k"], x["v"], x["g"], x["beta"], x["cu"], x["cu_host"], o,
                           state=cache, dst_slot=dst, dev_status=st, scale=0.125)
    torch.cuda.synchronize()
    assert st.item() == 0
    ref = oracle.run_chains(b, scale=0.125)
    gu.assert_o_close(gu.o_to_numpy(o), gu.o_ref_dense(b, ref))
    gu.assert_state_close(gu.get_states_math(cache, np.arange(n)), ref["s_final"].reshape(n, b.h_v, b.d, b.d))


def test_state_cache_past_2_31_floats(gdn):
    h, d, n_slots = 16, 128, 8200
    assert n_slots * h * d * d > 2 ** 31
    cache = gu.empty_cache(n_slots, h, d)
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    # decode: 4 rows from slots 8195..8198 into 8199, 8194, 8193, 8192 (one step)
    rows = 4
    dec = gi.token_batch([1] * rows, h, h, d, seed=91, init_state=True)
    src = np.array([8195, 8196, 8197, 8198], np.int32)
    dst = np.array([8199, 8194, 8193, 8192], np.int32)
    gu.put_states(cache, src, dec.init_state)
    xd = gu.batch_to_device(dec)
    o = torch.empty((rows, h, d), dtype=torch.bfloat16, device="cuda")
    gdn.gdn_decode_packed(xd["q"], xd["k"], xd["v"], xd["g"], xd["beta"], cache, torch.from_numpy(src).cuda(), o,
                          dst_slot=torch.from_numpy(dst).cuda(), dev_status=st)
    # prefill: 2 sequences from slots 8190, 8191 into 8188, 8189, every chunk's state emitted
    pre = gi.token_batch([130, 64], h, h, d, seed=92, init_state=True)
    psrc = np.array([8190, 8191], np.int32)
    pdst = np.array([8188, 8189], np.int32)
    gu.put_states(cache, psrc, pre.init_state)
    xp = gu.batch_to_device(pre)
    op = torch.empty((pre.total_tokens, h, d), dtype=torch.bfloat16, device="cuda")
    n_emit = gdn.gdn_prefill_num_emits(xp["cu_host"], 1)
    cs = torch.zeros((n_emit, h, d, d), device="cuda")
    gdn.gdn_prefill_varlen(xp["q"], xp["k"], xp["v"], xp["g"], xp["beta"], xp["cu"], xp["cu_host"], op,
                           state=cache, src_slot=torch.from_numpy(psrc).cuda(),
                           dst_slot=torch.from_numpy(pdst).cuda(), chunk_states=cs, emit_every_chunks=1,
                           dev_status=st)
    torch.cuda.synchronize()
    assert st.item() == 0
    ref = oracle.run_chains(dec)
    gu.assert_o_close(gu.o_to_numpy(o), gu.o_ref_dense(dec, ref))
    gu.assert_state_close(gu.get_states_math(cache, dst), ref["s_final"].reshape(rows, h, d, d))
    gu.assert_state_close(gu.get_states_math(cache, src), dec.init_state.astype(np.float64), "decode src slots")
    refp = oracle.run_chains(pre, emit_every=64)
    gu.assert_o_close(gu.o_to_numpy(op), gu.o_ref_dense(pre, refp))
    gu.assert_state_close(gu.get_states_math(cache, pdst), refp["s_final"].reshape(2, h, d, d))
    assert n_emit == 2 + 1
    # no other slot was written
    touched = set(src.tolist()) | set(dst.tolist()) | set(psrc.tolist()) | set(pdst.tolist())
    lo, hi = cache.view(n_slots, -1).aminmax(dim=1)   # per-slot reduction, no 8.6 GB temporary
    untouched = np.setdiff1d(np.arange(n_slots), sorted(touched))
    assert not lo.cpu().numpy()[untouched].any() and not hi.cpu().numpy()[untouched].any()
