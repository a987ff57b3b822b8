"""The prefill's bounded waits, exercised on the GPU without a fault.

A variant of the library is built with the handshake waits between the
prefill's warp groups limited to a single clock cycle (the waits for work
already in flight keep their normal limit).  The first handshake that is not
complete at once runs out, so the kernel must take its failure path: set
GDN_DEV_TIMEOUT in the device status word, drain the copies and tensor-core
products it has in flight, release its tensor memory and return.  The context
must stay usable: a normal call afterwards on the same device matches the
oracle.
"""
import ctypes

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


@pytest.fixture(scope="module")
def short_wait_lib():
    import linear_attention_serving_gdn_gb300 as g
    from linear_attention_serving_gdn_gb300 import _build
    path = _build.build_variant("waittest", ["GDN_WAIT_CYCLES=1LL"])
    return g._configure(ctypes.CDLL(path))


def _run_prefill(gdn, b, lib=None):
    """One prefill of batch b through the Python binding, optionally routed to
    another build of the library; returns (o, states, device status word)."""
    n = b.num_seqs
    cache = gu.empty_cache(n, b.h_v, b.d)
    dv = gu.batch_to_device(b)
    o = torch.zeros((b.total_tokens, b.h_v, b.d), dtype=torch.bfloat16, device="cuda")
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    saved = gdn._lib
    try:
        if lib is not None:
            gdn._lib = lib
        gdn.gdn_prefill_varlen(dv["q"], dv["k"], dv["v"], dv["g"], dv["beta"], dv["cu"], dv["cu_host"], o,
                               state=cache, dst_slot=torch.arange(n, dtype=torch.int32, device="cuda"),
                               dev_status=st)
    finally:
        gdn._lib = saved
    torch.cuda.synchronize()
    return o, cache, int(st.item())


def test_prefill_handshake_timeout_reports_and_context_survives(gdn, short_wait_lib):
    b = gi.token_batch([300, 129, 64], 4, 8, 128, 31)
    _, _, word = _run_prefill(gdn, b, lib=short_wait_lib)
    assert word & gdn.GDN_DEV_TIMEOUT, f"no timeout reported (status {word:#x})"
    assert gdn.gdn_status_from_device(word) == 5  # GDN_ERR_TIMEOUT
    # Twice more, to show that a kernel which timed out left nothing behind
    # (tensor memory released, no copy still landing).
    for _ in range(2):
        _, _, w = _run_prefill(gdn, b, lib=short_wait_lib)
        assert w & gdn.GDN_DEV_TIMEOUT
    # The same context still runs the normal build correctly.
    o, cache, word = _run_prefill(gdn, b)
    assert word == 0
    ref = oracle.run_chains(b)
    gu.assert_o_close(gu.o_to_numpy(o), gu.o_ref_dense(b, ref))
    S = gu.get_states_math(cache, np.arange(b.num_seqs))
    gu.assert_state_close(np.stack([S[s, h] for s, h in ref["pairs"]]), ref["s_final"])
