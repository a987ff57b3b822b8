"""Input preparation (q/k normalisation, decay and write-strength gating)
through the C ABI: the standalone kernel against the fp64 oracle of the same
reading (oracle/prep.py), and the fused decode against prep + decode (bit
for bit) and against the oracle end to end."""
import numpy as np
import pytest
import torch

import gdn_inputs as gi
import oracle
from oracle import prep as oprep
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


def _raw_to_device(raw):
    t = lambda x: torch.from_numpy(np.ascontiguousarray(x)).cuda()
    return {"q_raw": gu.bf16_tensor(raw.q), "k_raw": gu.bf16_tensor(raw.k), "v": gu.bf16_tensor(raw.v),
            "a": t(raw.a), "b": t(raw.b), "A_log": t(raw.A_log), "dt_bias": t(raw.dt_bias)}


def _prep(gdn, x, eps=1e-6, in_place=False):
    T, h_v = x["a"].shape
    q = x["q_raw"].clone() if in_place else torch.empty_like(x["q_raw"])
    k = x["k_raw"].clone() if in_place else torch.empty_like(x["k_raw"])
    g = torch.empty((T, h_v), dtype=torch.float32, device="cuda")
    beta = torch.empty_like(g)
    gdn.gdn_prep_inputs(q if in_place else x["q_raw"], k if in_place else x["k_raw"], x["a"], x["b"],
                        x["A_log"], x["dt_bias"], q, k, g, beta, eps=eps)
    return q, k, g, beta


@pytest.mark.parametrize("T,h_k,h_v,d", [(300, 16, 32, 128), (77, 2, 6, 64)])
def test_prep_kernel_vs_oracle(gdn, T, h_k, h_v, d):
    raw = gi.raw_inputs(T, h_k, h_v, d, seed=8)
    x = _raw_to_device(raw)
    q, k, g, beta = _prep(gdn, x)
    qi = _prep(gdn, x, in_place=True)[0]
    torch.cuda.synchronize()
    assert torch.equal(q.view(torch.int16), qi.view(torch.int16))      # in place == out of place
    qb, kb, g_ref, b_ref = oprep.prep(raw)
    for got, ref in ((q, qb), (k, kb)):
        gf = got.float().cpu().numpy().astype(np.float64)
        rf = gi.bf16_to_f32(ref).astype(np.float64)
        # bf16 results of fp32 vs fp64 arithmetic: at most one bf16 step apart
        ulp = np.exp2(np.floor(np.log2(np.maximum(np.abs(rf), 1e-30))) - 7)
        assert np.all(np.abs(gf - rf) <= ulp)
        assert np.mean(gf == rf) > 0.99
    assert np.allclose(g.cpu().numpy(), g_ref, rtol=2e-6, atol=1e-9)
    assert np.allclose(beta.cpu().numpy(), b_ref, rtol=2e-6, atol=1e-9)


def _at_offset(t):
    """A contiguous copy of t starting 4 bytes past a 16-byte boundary."""
    buf = torch.empty(t.numel() + 1, dtype=t.dtype, device="cuda")
    v = buf[1:].view(t.shape)
    v.copy_(t)
    return v


@pytest.mark.parametrize("T,h_k,h_v,d", [(4099, 1, 66, 64), (20001, 16, 32, 128)])
def test_prep_gate_vector_and_scalar_paths_bitwise(gdn, T, h_k, h_v, d):
    """The gates of 16-byte aligned arrays go through float4 runs of four
    (two runs at a time while whole sets remain, then single runs) and the
    last n_gate % 4 elements one by one (4099 x 66 leaves 2); the same arrays
    at a 4-byte offset go element by element.  Both give the same bits, and
    both match the oracle."""
    raw = gi.raw_inputs(T, h_k, h_v, d, seed=14)
    x = _raw_to_device(raw)
    q, k, g, beta = _prep(gdn, x)
    g_s = _at_offset(torch.zeros_like(g))
    beta_s = _at_offset(torch.zeros_like(beta))
    q_s, k_s = torch.empty_like(q), torch.empty_like(k)
    gdn.gdn_prep_inputs(x["q_raw"], x["k_raw"], _at_offset(x["a"]), _at_offset(x["b"]), x["A_log"],
                        x["dt_bias"], q_s, k_s, g_s, beta_s)
    torch.cuda.synchronize()
    assert torch.equal(g, g_s) and torch.equal(beta, beta_s)
    assert torch.equal(q.view(torch.int16), q_s.view(torch.int16))
    _, _, g_ref, b_ref = oprep.prep(raw)
    assert np.allclose(g.cpu().numpy(), g_ref, rtol=2e-6, atol=1e-9)
    assert np.allclose(beta.cpu().numpy(), b_ref, rtol=2e-6, atol=1e-9)


def test_fused_decode_equals_prep_then_decode_bitwise(gdn):
    rows, h, d = 256, 16, 128
    raw = gi.raw_inputs(rows, h, h, d, seed=12)
    x = _raw_to_device(raw)
    init = gi.token_batch([1] * rows, h, h, d, 12, init_state=True).init_state
    src, n_slots = gi.slots(rows, 12)
    cache_f = gu.empty_cache(n_slots, h, d)
    gu.put_states(cache_f, src, init)
    cache_u = cache_f.clone()
    src_t = torch.from_numpy(src).cuda()
    o_f = torch.empty((rows, h, d), dtype=torch.bfloat16, device="cuda")
    o_u = torch.empty_like(o_f)
    gdn.gdn_decode_packed_raw(x["q_raw"], x["k_raw"], x["v"], x["a"], x["b"], x["A_log"], x["dt_bias"],
                              cache_f, src_t, o_f)
    q, k, g, beta = _prep(gdn, x)
    gdn.gdn_decode_packed(q, k, x["v"], g, beta, cache_u, src_t, o_u)
    torch.cuda.synchronize()
    assert torch.equal(o_f.view(torch.int16), o_u.view(torch.int16))
    assert torch.equal(cache_f, cache_u)


@pytest.mark.parametrize("h_k,h,d", [(16, 16, 128), (2, 6, 64)])
def test_fused_decode_vs_oracle(gdn, h_k, h, d):
    rows, steps = 24, 3
    raws = [gi.raw_inputs(rows, h_k, h, d, seed=40 + t) for t in range(steps)]
    init = gi.token_batch([1] * rows, h_k, h, d, 40, init_state=True).init_state
    src, n_slots = gi.slots(rows, 40)
    cache = gu.empty_cache(n_slots, h, d)
    gu.put_states(cache, src, init)
    src_t = torch.from_numpy(src).cuda()
    outs = []
    for raw in raws:
        x = _raw_to_device(raw)
        o = torch.empty((rows, h, d), dtype=torch.bfloat16, device="cuda")
        gdn.gdn_decode_packed_raw(x["q_raw"], x["k_raw"], x["v"], x["a"], x["b"], x["A_log"],
                                  x["dt_bias"], cache, src_t, o)
        outs.append(gu.o_to_numpy(o))
    torch.cuda.synchronize()
    # oracle: prepare each step in fp64 (rounded to the storage types), then
    # run every row as a `steps`-token sequence
    preps = [oprep.prep(r) for r in raws]
    order = lambda arr_list: np.stack(arr_list, 1).reshape((rows * steps,) + arr_list[0].shape[1:])
    b = gi.TokenBatch(h_k, h, d, np.arange(rows + 1, dtype=np.int32) * steps,
                      order([p[0] for p in preps]), order([p[1] for p in preps]),
                      order([r.v for r in raws]), order([p[2] for p in preps]), order([p[3] for p in preps]),
                      init)
    ref = oracle.run_chains(b)
    gu.assert_o_close(np.stack(outs, 1).reshape(rows * steps, h, d), gu.o_ref_dense(b, ref))
    gu.assert_state_close(gu.get_states_math(cache, src), ref["s_final"].reshape(rows, h, d, d))
