"""Slot routing under the library's aliasing rule: within one call the slots
written must be disjoint from the slots other rows read.  A shift of states
along the slots (row r's state moves to the slot next to it) therefore runs
as two calls, each with disjoint read and write sets, and must equal the
oracle's two-token chains."""
import numpy as np
import pytest
import torch

import gdn_inputs as gi
import oracle
from tests import gpu_util as gu

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def gdn():
    import linear_attention_serving_gdn_gb300 as g
    g.load_library()
    return g


def test_slot_shift_as_two_calls_matches_oracle(gdn):
    R, H, d = 8, 16, 128
    b = gi.token_batch([2] * R, H, H, d, 41, init_state=True)   # two tokens per row
    cache = gu.empty_cache(2 * R, H, d)
    gu.put_states(cache, np.arange(R), b.init_state)
    dv = gu.batch_to_device(b)
    first = torch.arange(R, device="cuda") * 2      # token 0 of each row
    second = first + 1
    src1 = torch.arange(R, dtype=torch.int32, device="cuda")
    dst1 = (R + (src1 + 1) % R).to(torch.int32)                # into the spare slots, shifted by one
    src2 = dst1.clone()
    dst2 = ((src1 + 2) % R).to(torch.int32)                    # back, shifted by two
    o = torch.empty((2 * R, H, d), dtype=torch.bfloat16, device="cuda")
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    for tok, src, dst in ((first, src1, dst1), (second, src2, dst2)):
        out = torch.empty((R, H, d), dtype=torch.bfloat16, device="cuda")
        gdn.gdn_decode_packed(dv["q"][tok].contiguous(), dv["k"][tok].contiguous(), dv["v"][tok].contiguous(),
                              dv["g"][tok].contiguous(), dv["beta"][tok].contiguous(), cache, src, out,
                              dst_slot=dst, dev_status=st)
        o[tok] = out
    torch.cuda.synchronize()
    assert st.item() == 0
    ref = oracle.run_chains(b)
    gu.assert_o_close(gu.o_to_numpy(o), gu.o_ref_dense(b, ref))
    S = gu.get_states_math(cache, ((np.arange(R) + 2) % R))
    gu.assert_state_close(np.stack([S[r, h] for r, h in ref["pairs"]]), ref["s_final"])
