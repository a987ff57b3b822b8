"""GPU parity: the CUDA path (through the C ABI) against the fp64 oracle on
the same seeded inputs, for the five serving workloads and the edge cases.

Bars: bf16 o within max |err| <= 2e-2 of the oracle; fp32 states within 1e-3
relative Frobenius error (tests/gpu_util.py).
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


def _status():
    return torch.zeros(1, dtype=torch.int32, device="cuda")


# ---------------------------------------------------------------------------
# decode
# ---------------------------------------------------------------------------

def _decode_steps(gdn, rows, h, d, steps, seed, n_slots=None, scale=1.0, h_k=None):
    """Run `steps` in-place decode steps of `rows` rows; returns GPU o per step,
    final states, and the oracle's results for the same token sequences."""
    h_k = h if h_k is None else h_k
    seqs = gi.token_batch([steps] * rows, h_k, h, d, seed, init_state=True)
    src, n_slots = gi.slots(rows, seed, n_slots)
    cache = gu.empty_cache(n_slots, h, d)
    gu.put_states(cache, src, seqs.init_state)
    src_t = torch.from_numpy(src).cuda()
    st = _status()
    outs = []
    for t in range(steps):
        idx = seqs.cu_seqlens[:-1] + t
        sub = {n: getattr(seqs, n)[idx] for n in ("q", "k", "v", "g", "beta")}
        dv = gu.arrays_to_device(sub)
        o = torch.empty((rows, h, d), dtype=torch.bfloat16, device="cuda")
        gdn.gdn_decode_packed(dv["q"], dv["k"], dv["v"], dv["g"], dv["beta"], cache, src_t, o,
                              dev_status=st, scale=scale)
        outs.append(gu.o_to_numpy(o))
    torch.cuda.synchronize()
    assert st.item() == 0
    ref = oracle.run_chains(seqs, scale=scale)
    o_ref = gu.o_ref_dense(seqs, ref)          # [rows*steps][h][d], row-major by row then step
    o_gpu = np.stack(outs, 1).reshape(rows * steps, h, d)
    S_gpu = gu.get_states_math(cache, src)
    S_ref = ref["s_final"].reshape(rows, h, d, d)
    return o_gpu, o_ref, S_gpu, S_ref


def test_decode_qwen35_08b_layer_full_size(gdn):
    """256 rows, H=16, d=128, slot cache of 512, 8 in-place steps."""
    o_gpu, o_ref, S_gpu, S_ref = _decode_steps(gdn, 256, 16, 128, steps=8, seed=0)
    gu.assert_o_close(o_gpu, o_ref)
    gu.assert_state_close(S_gpu, S_ref)


@pytest.mark.parametrize("d,h,h_k,scale", [(64, 4, 4, 1.0), (64, 6, 2, 0.125), (128, 4, 1, 0.0883883)])
def test_decode_small_shapes(gdn, d, h, h_k, scale):
    o_gpu, o_ref, S_gpu, S_ref = _decode_steps(gdn, 5, h, d, steps=3, seed=3, scale=scale, h_k=h_k)
    gu.assert_o_close(o_gpu, o_ref)
    gu.assert_state_close(S_gpu, S_ref)


def test_decode_padded_rows_bad_slots_and_slot_copy(gdn):
    """src < 0: row skipped, o zeroed; src >= num_slots: status bit, o
    zeroed, nothing written; src != dst: state recycled into a new slot."""
    b = gi.token_batch([1] * 4, 2, 2, 64, seed=5, init_state=True)
    cache = gu.empty_cache(6, 2, 64)
    gu.put_states(cache, [0, 1, 2, 3], b.init_state)
    before = cache.clone()
    dv = gu.batch_to_device(b)
    src = torch.tensor([0, -1, 9, 2], dtype=torch.int32, device="cuda")
    dst = torch.tensor([0, -1, 4, 5], dtype=torch.int32, device="cuda")
    o = torch.full((4, 2, 64), 7.0, dtype=torch.bfloat16, device="cuda")
    st = _status()
    gdn.gdn_decode_packed(dv["q"], dv["k"], dv["v"], dv["g"], dv["beta"], cache, src, o, dst_slot=dst,
                          dev_status=st)
    torch.cuda.synchronize()
    assert st.item() & gdn.GDN_DEV_BAD_SLOT
    assert torch.all(o[1] == 0) and torch.all(o[2] == 0)
    # row 3 reads slot 2, which holds init_state[2]
    init = np.stack([b.init_state[0, 0], b.init_state[0, 1], b.init_state[2, 0], b.init_state[2, 1]])
    ref = oracle.run_chains(b, pairs=[(0, 0), (0, 1), (3, 0), (3, 1)], init_state=init)
    o_np = gu.o_to_numpy(o)
    gu.assert_o_close(o_np[0], np.stack([ref["o"][0][0], ref["o"][1][0]]))
    gu.assert_o_close(o_np[3], np.stack([ref["o"][2][0], ref["o"][3][0]]))
    gu.assert_state_close(gu.get_states_math(cache, [0])[0], ref["s_final"][:2])
    gu.assert_state_close(gu.get_states_math(cache, [5])[0], ref["s_final"][2:])
    # slot 2 (src of row 3, not its dst), slot 1 (padded) and slot 3 are untouched
    for s in (1, 2, 3):
        assert torch.equal(cache[s], before[s])
    assert torch.equal(cache[4], before[4])   # bad-slot row wrote nothing


# ---------------------------------------------------------------------------
# prefill
# ---------------------------------------------------------------------------

def _prefill(gdn, b, E=0, init_slots=None, scale=1.0, n_slots=None):
    n = b.num_seqs
    n_slots = n_slots or 2 * n + 2
    cache = gu.empty_cache(n_slots, b.h_v, b.d)
    dst = np.arange(n, dtype=np.int32) + n   # final states in slots [n, 2n)
    src = np.full(n, -1, np.int32)
    if init_slots is not None:
        for s in range(n):
            if init_slots[s]:
                src[s] = s
        gu.put_states(cache, np.arange(n), b.init_state)
    dv = gu.batch_to_device(b)
    o = torch.empty((b.total_tokens, b.h_v, b.d), dtype=torch.bfloat16, device="cuda")
    n_emit = gdn.gdn_prefill_num_emits(dv["cu_host"], E) if E else 0
    cs = torch.full((max(n_emit, 1), b.h_v, b.d, b.d), float("nan"), device="cuda") if E else None
    st = _status()
    gdn.gdn_prefill_varlen(dv["q"], dv["k"], dv["v"], dv["g"], dv["beta"], dv["cu"], dv["cu_host"], o,
                           state=cache, src_slot=torch.from_numpy(src).cuda(),
                           dst_slot=torch.from_numpy(dst).cuda(), chunk_states=cs,
                           emit_every_chunks=E, dev_status=st, scale=scale)
    torch.cuda.synchronize()
    assert st.item() == 0
    return o, cache, dst, cs, src


def _prefill_vs_oracle(gdn, b, E=0, init_slots=None, scale=1.0, pairs=None):
    o, cache, dst, cs, src = _prefill(gdn, b, E, init_slots, scale)
    init = None
    if pairs is None:
        pairs = [(s, h) for s in range(b.num_seqs) for h in range(b.h_v)]
    if init_slots is not None:
        init = np.stack([b.init_state[s, h] if init_slots[s] else np.zeros((b.d, b.d), np.float32)
                         for s, h in pairs])
    else:
        init = np.zeros((len(pairs), b.d, b.d), np.float32)
    ref = oracle.run_chains(b, pairs=pairs, init_state=init, scale=scale, emit_every=64 * E)
    o_np = gu.o_to_numpy(o)
    S_all = gu.get_states_math(cache, dst)
    for p, (s, h) in enumerate(pairs):
        t0, t1 = int(b.cu_seqlens[s]), int(b.cu_seqlens[s + 1])
        gu.assert_o_close(o_np[t0:t1, h], ref["o"][p], f"o seq {s} head {h}")
    S_gpu = np.stack([S_all[s, h] for s, h in pairs])
    rel = gu.assert_state_close(S_gpu, ref["s_final"])
    if E:
        offs = gdn.gdn_prefill_emit_offsets([int(x) for x in b.cu_seqlens], E)
        cs_np = cs.cpu().numpy()
        for p, (s, h) in enumerate(pairs):
            got = np.swapaxes(cs_np[offs[s]:offs[s + 1], h], -1, -2).astype(np.float64)
            assert got.shape[0] == len(ref["emits"][p])
            if got.shape[0]:
                gu.assert_state_close(got, ref["emits"][p], f"emits seq {s} head {h}")
    return rel


def test_prefill_qwen3next_gva_full_size(gdn):
    """8 sequences drawn from {116, 321, 1059, 2000}; H_k=16, H_v=32, d=128;
    every chunk's state emitted (E=1)."""
    wl = gi.prefill_qwen3next_gva(0)
    _prefill_vs_oracle(gdn, wl["prefill"], E=1)


def test_prefill_prefix_cache_full_size_sampled_chains(gdn):
    """4 x 32768 tokens, H_k=16, H_v=32, d=128, states on the 1088-token grid
    (E=17).  The oracle checks 4 sampled (sequence, head) chains."""
    wl = gi.prefix_cache_prefill(0)
    _prefill_vs_oracle(gdn, wl["prefill"], E=17, pairs=[(0, 0), (1, 17), (2, 31), (3, 6)])


@pytest.mark.parametrize("d", [64, 128])
def test_prefill_edge_lengths_gva_scale_and_initial_states(gdn, d):
    lens = [0, 1, 63, 64, 65, 130, 200]
    b = gi.token_batch(lens, 2, 4, d, seed=21, init_state=True)
    _prefill_vs_oracle(gdn, b, E=1, init_slots=[1, 0, 1, 0, 1, 1, 0], scale=0.125)


def test_prefill_bad_slot_sets_status(gdn):
    b = gi.token_batch([70, 5], 1, 1, 64, seed=22)
    dv = gu.batch_to_device(b)
    cache = gu.empty_cache(2, 1, 64)
    o = torch.full((75, 1, 64), 3.0, dtype=torch.bfloat16, device="cuda")
    st = _status()
    gdn.gdn_prefill_varlen(dv["q"], dv["k"], dv["v"], dv["g"], dv["beta"], dv["cu"], dv["cu_host"], o,
                           state=cache, src_slot=torch.tensor([-1, 7], dtype=torch.int32, device="cuda"),
                           dst_slot=torch.tensor([0, 1], dtype=torch.int32, device="cuda"), dev_status=st)
    torch.cuda.synchronize()
    assert st.item() & gdn.GDN_DEV_BAD_SLOT
    assert torch.all(o[70:] == 0)
    ref = oracle.run_chains(b, pairs=[(0, 0)])
    gu.assert_o_close(gu.o_to_numpy(o[:70, 0]), ref["o"][0])


# ---------------------------------------------------------------------------
# mixed step
# ---------------------------------------------------------------------------

def _mixed(gdn, wl, E=0):
    dec, pre = wl["decode"], wl["prefill"]
    nd, npf = dec.num_seqs, pre.num_seqs
    n_slots = 2 * (nd + npf)
    src = gi.slots(nd + npf, 1, n_slots)[0]
    cache = gu.empty_cache(n_slots, dec.h_v, dec.d)
    gu.put_states(cache, src[:nd], dec.init_state)
    arrs = gu.arrays_to_device(gu.concat_batches(dec, pre))
    T = nd + pre.total_tokens
    o = torch.empty((T, dec.h_v, dec.d), dtype=torch.bfloat16, device="cuda")
    cu_p = torch.from_numpy(pre.cu_seqlens.astype(np.int32)).cuda()
    n_emit = gdn.gdn_prefill_num_emits(pre.cu_seqlens, E) if E else 0
    cs = torch.zeros((max(n_emit, 1), dec.h_v, dec.d, dec.d), device="cuda") if E else None
    st = _status()
    dsrc = torch.from_numpy(src[:nd]).cuda()
    pdst = torch.from_numpy(src[nd:]).cuda()
    gdn.gdn_mixed_step(nd, arrs["q"], arrs["k"], arrs["v"], arrs["g"], arrs["beta"], cu_p,
                       [int(x) for x in pre.cu_seqlens], cache, dsrc, o, pre_dst_slot=pdst,
                       chunk_states=cs, emit_every_chunks=E, dev_status=st)
    torch.cuda.synchronize()
    assert st.item() == 0
    return o, cache, src, cs


def _check_mixed(gdn, wl, E=0):
    dec, pre = wl["decode"], wl["prefill"]
    nd = dec.num_seqs
    o, cache, src, cs = _mixed(gdn, wl, E)
    r_dec = oracle.run_chains(dec)
    r_pre = oracle.run_chains(pre, emit_every=64 * E)
    o_np = gu.o_to_numpy(o)
    gu.assert_o_close(o_np[:nd], gu.o_ref_dense(dec, r_dec), "decode o")
    gu.assert_o_close(o_np[nd:], gu.o_ref_dense(pre, r_pre), "prefill o")
    gu.assert_state_close(gu.get_states_math(cache, src[:nd]),
                          r_dec["s_final"].reshape(nd, dec.h_v, dec.d, dec.d), "decode state")
    gu.assert_state_close(gu.get_states_math(cache, src[nd:]),
                          r_pre["s_final"].reshape(pre.num_seqs, pre.h_v, pre.d, pre.d), "prefill state")
    return o, cache, src


def test_mixed_tiny_h4_d64(gdn):
    """2 cached decode rows + prefills of 64 and 100 tokens, then 8 more
    decode-only steps on the two rows."""
    wl = gi.tiny_mixed(0)
    o, cache, src = _check_mixed(gdn, wl, E=1)
    dec = wl["decode"]
    more = gi.token_batch([8, 8], 4, 4, 64, seed=99)
    src_t = torch.from_numpy(src[:2]).cuda()
    outs = []
    for t in range(8):
        idx = more.cu_seqlens[:-1] + t
        dv = gu.arrays_to_device({n: getattr(more, n)[idx] for n in ("q", "k", "v", "g", "beta")})
        ot = torch.empty((2, 4, 64), dtype=torch.bfloat16, device="cuda")
        gdn.gdn_decode_packed(dv["q"], dv["k"], dv["v"], dv["g"], dv["beta"], cache, src_t, ot)
        outs.append(gu.o_to_numpy(ot))
    # oracle: each row is the 9-token sequence [mixed-step token, 8 decode tokens]
    seqs = {}
    for n in ("q", "k", "v", "g", "beta"):
        seqs[n] = np.concatenate([np.concatenate([getattr(dec, n)[r:r + 1], getattr(more, n)[8 * r:8 * r + 8]])
                                  for r in range(2)])
    full = gi.TokenBatch(4, 4, 64, np.array([0, 9, 18], np.int32), seqs["q"], seqs["k"], seqs["v"],
                         seqs["g"], seqs["beta"], dec.init_state)
    ref = oracle.run_chains(full)
    o_ref = gu.o_ref_dense(full, ref).reshape(2, 9, 4, 64)
    o_gpu = np.stack(outs, 1)
    gu.assert_o_close(o_gpu, o_ref[:, 1:])
    gu.assert_state_close(gu.get_states_math(cache, src[:2]), ref["s_final"].reshape(2, 4, 64, 64))


def test_mixed_step_64_decodes_4_prefills_full_size(gdn):
    _check_mixed(gdn, gi.mixed_step(0))
