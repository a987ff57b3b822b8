"""Multi-token decode (rows carrying several speculative tokens) through the
C ABI, against the fp64 oracle and against the packed single-token decode.

The oracle has no separate arithmetic for this: a row of T tokens is the
token recurrence over those T tokens, and the snapshot after token t is the
oracle's final state of the row's first t + 1 tokens.
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


def _prefix_batch(b: gi.TokenBatch, n: int) -> gi.TokenBatch:
    """The first n tokens of every sequence of a uniform-length batch."""
    L = int(b.cu_seqlens[1] - b.cu_seqlens[0])
    idx = np.concatenate([np.arange(r * L, r * L + n) for r in range(b.num_seqs)])
    cu = np.arange(b.num_seqs + 1, dtype=np.int32) * n
    return gi.TokenBatch(b.h_k, b.h_v, b.d, cu, b.q[idx], b.k[idx], b.v[idx], b.g[idx], b.beta[idx],
                         b.init_state)


def _setup(rows, T, h_k, h, d, seed):
    b = gi.token_batch([T] * rows, h_k, h, d, seed, init_state=True)
    n_slots = rows * (T + 1) + 3
    perm = np.random.default_rng(seed + 5).permutation(n_slots).astype(np.int32)
    src = perm[:rows]
    dst = perm[rows:rows * (T + 1)].reshape(rows, T)
    cache = gu.empty_cache(n_slots, h, d)
    gu.put_states(cache, src, b.init_state)
    x = gu.batch_to_device(b)
    return b, src, dst, cache, x


@pytest.mark.parametrize("rows,T,h_k,h,d,scale", [(16, 4, 4, 16, 128, 1.0), (5, 7, 2, 6, 64, 0.125),
                                                 (3, 1, 4, 4, 128, 1.0),
                                                 (4, 11, 4, 8, 128, 1.0)])  # more tokens than the stage holds
def test_multi_decode_outputs_and_snapshots_vs_oracle(gdn, rows, T, h_k, h, d, scale):
    b, src, dst, cache, x = _setup(rows, T, h_k, h, d, seed=21)
    o = torch.empty((rows * T, h, d), dtype=torch.bfloat16, device="cuda")
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    gdn.gdn_decode_multi(T, x["q"], x["k"], x["v"], x["g"], x["beta"], cache,
                         torch.from_numpy(src).cuda(), o, dst_slots=torch.from_numpy(dst.reshape(-1)).cuda(),
                         dev_status=st, scale=scale)
    torch.cuda.synchronize()
    assert st.item() == 0
    ref = oracle.run_chains(b, scale=scale)
    gu.assert_o_close(gu.o_to_numpy(o), gu.o_ref_dense(b, ref))
    for t in range(T):
        snap = oracle.run_chains(_prefix_batch(b, t + 1), scale=scale)["s_final"].reshape(rows, h, d, d)
        gu.assert_state_close(gu.get_states_math(cache, dst[:, t]), snap, f"snapshot after token {t}")
    # the entering states are untouched
    gu.assert_state_close(gu.get_states_math(cache, src), b.init_state.astype(np.float64), "src slots")


@pytest.mark.parametrize("T", [4, 5])  # 4: the kernel that prefetches the next item; 5: the other one
def test_multi_decode_equals_packed_decode_steps_bitwise(gdn, T):
    """T tokens in one call == T packed-decode calls chained through the same
    snapshot slots, bit for bit (outputs and every snapshot)."""
    rows, h, d = 32, 16, 128
    b, src, dst, cache_m, x = _setup(rows, T, 16, h, d, seed=4)
    cache_p = cache_m.clone()
    o_m = torch.empty((rows * T, h, d), dtype=torch.bfloat16, device="cuda")
    gdn.gdn_decode_multi(T, x["q"], x["k"], x["v"], x["g"], x["beta"], cache_m,
                         torch.from_numpy(src).cuda(), o_m, dst_slots=torch.from_numpy(dst.reshape(-1)).cuda())
    o_p = torch.empty((rows, T, h, d), dtype=torch.bfloat16, device="cuda")
    prev = src
    for t in range(T):
        idx = torch.from_numpy(np.arange(rows) * T + t).cuda()
        step = {n: x[n].index_select(0, idx).contiguous() for n in ("q", "k", "v", "g", "beta")}
        ot = torch.empty((rows, h, d), dtype=torch.bfloat16, device="cuda")
        gdn.gdn_decode_packed(step["q"], step["k"], step["v"], step["g"], step["beta"], cache_p,
                              torch.from_numpy(prev).cuda(), ot, dst_slot=torch.from_numpy(dst[:, t].copy()).cuda())
        o_p[:, t] = ot
        prev = dst[:, t].copy()
    torch.cuda.synchronize()
    assert torch.equal(o_m.view(torch.int16), o_p.reshape(rows * T, h, d).view(torch.int16))
    assert torch.equal(cache_m, cache_p)


def test_multi_decode_in_place_padded_rows_and_bad_snapshot_slot(gdn):
    rows, T, h, d = 6, 3, 4, 64
    b, src, dst, cache, x = _setup(rows, T, 4, h, d, seed=9)
    # dst_slots == NULL: the state after the last token goes back to src.
    c_inplace = cache.clone()
    o1 = torch.empty((rows * T, h, d), dtype=torch.bfloat16, device="cuda")
    gdn.gdn_decode_multi(T, x["q"], x["k"], x["v"], x["g"], x["beta"], c_inplace,
                         torch.from_numpy(src).cuda(), o1)
    torch.cuda.synchronize()
    ref = oracle.run_chains(b)
    gu.assert_state_close(gu.get_states_math(c_inplace, src), ref["s_final"].reshape(rows, h, d, d))
    gu.assert_o_close(gu.o_to_numpy(o1), gu.o_ref_dense(b, ref))
    # padded row 1 (src < 0) and an out-of-range snapshot slot on row 2, token 1
    src2 = src.copy()
    src2[1] = -1
    dst2 = dst.copy()
    dst2[2, 1] = cache.shape[0] + 5
    c2 = cache.clone()
    sentinel = c2[dst[1]].clone()
    o2 = torch.full((rows * T, h, d), 3.0, dtype=torch.bfloat16, device="cuda")
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    gdn.gdn_decode_multi(T, x["q"], x["k"], x["v"], x["g"], x["beta"], c2, torch.from_numpy(src2).cuda(), o2,
                         dst_slots=torch.from_numpy(dst2.reshape(-1)).cuda(), dev_status=st)
    torch.cuda.synchronize()
    assert st.item() & gdn.GDN_DEV_BAD_SLOT
    assert o2[T:2 * T].float().abs().max().item() == 0.0           # padded row: o zeroed
    assert torch.equal(c2[dst[1]], sentinel)                        # padded row: no snapshot written
    o2n, o1n = gu.o_to_numpy(o2), gu.o_to_numpy(o1)
    for r in (0, 2, 3, 4, 5):                                       # other rows unaffected
        assert np.array_equal(o2n[r * T:(r + 1) * T], o1n[r * T:(r + 1) * T])
    snap_last = gu.get_states_math(c2, dst[[0, 2, 3, 4, 5], T - 1])
    assert np.array_equal(snap_last, gu.get_states_math(c_inplace, src[[0, 2, 3, 4, 5]]))


def test_multi_decode_final_only_with_next_item_prefetch(gdn):
    """Final state only, T >= 3 and more items than the grid has warps: each
    warp prefetches its next item's state into L2.  Outputs and final states
    equal T in-place packed-decode calls bit for bit and match the oracle; a
    padded row (src < 0) is skipped by both, its prefetch included."""
    rows, T, h, d = 48, 4, 16, 128  # 48 x 16 x 8 = 6144 items, more than 2 x 8 warps per SM on 152 SMs
    b, src, _, cache_m, x = _setup(rows, T, 16, h, d, seed=13)
    src = src.copy()
    src[5] = -1
    cache_p = cache_m.clone()
    src_t = torch.from_numpy(src).cuda()
    o_m = torch.empty((rows * T, h, d), dtype=torch.bfloat16, device="cuda")
    gdn.gdn_decode_multi(T, x["q"], x["k"], x["v"], x["g"], x["beta"], cache_m, src_t, o_m)
    o_p = torch.empty((rows, T, h, d), dtype=torch.bfloat16, device="cuda")
    for t in range(T):
        idx = torch.from_numpy(np.arange(rows) * T + t).cuda()
        step = {n: x[n].index_select(0, idx).contiguous() for n in ("q", "k", "v", "g", "beta")}
        ot = torch.empty((rows, h, d), dtype=torch.bfloat16, device="cuda")
        gdn.gdn_decode_packed(step["q"], step["k"], step["v"], step["g"], step["beta"], cache_p, src_t, ot)
        o_p[:, t] = ot
    torch.cuda.synchronize()
    assert torch.equal(o_m.view(torch.int16), o_p.reshape(rows * T, h, d).view(torch.int16))
    assert torch.equal(cache_m, cache_p)
    live = np.array([r for r in range(rows) if src[r] >= 0])
    ref = oracle.run_chains(b)
    o_ref = gu.o_ref_dense(b, ref).reshape(rows, T, h, d)
    gu.assert_o_close(gu.o_to_numpy(o_m).reshape(rows, T, h, d)[live], o_ref[live])
    assert o_m.reshape(rows, T, h, d)[5].float().abs().max().item() == 0.0
    gu.assert_state_close(gu.get_states_math(cache_m, src[live]),
                          ref["s_final"].reshape(rows, h, d, d)[live], "final states")


@pytest.mark.parametrize("T,d,snapshots", [(4, 128, False), (6, 128, True), (4, 64, False), (11, 128, False)])
def test_multi_decode_many_items_with_padded_row_bitwise(gdn, T, d, snapshots):
    """More items than resident warps (5120 of them on 152 SMs, so warps take
    a second and third item, the last round partly filled), with a padded row
    whose skipped item is followed by live ones in the same warps (T = 11:
    more tokens than the stage holds, read directly): outputs and states
    equal T packed-decode calls bit for bit, the padded row writes zeros and
    leaves every state untouched."""
    h = 16
    rows = 40 if d == 128 else 80
    b, src, dst, cache_m, x = _setup(rows, T, 16, h, d, seed=31)
    src = src.copy()
    src[1] = -1
    cache_p = cache_m.clone()
    src_t = torch.from_numpy(src).cuda()
    o_m = torch.empty((rows * T, h, d), dtype=torch.bfloat16, device="cuda")
    dst_t = torch.from_numpy(dst.reshape(-1).copy()).cuda() if snapshots else None
    gdn.gdn_decode_multi(T, x["q"], x["k"], x["v"], x["g"], x["beta"], cache_m, src_t, o_m, dst_slots=dst_t)
    o_p = torch.empty((rows, T, h, d), dtype=torch.bfloat16, device="cuda")
    prev = src
    for t in range(T):
        idx = torch.from_numpy(np.arange(rows) * T + t).cuda()
        step = {n: x[n].index_select(0, idx).contiguous() for n in ("q", "k", "v", "g", "beta")}
        ot = torch.empty((rows, h, d), dtype=torch.bfloat16, device="cuda")
        nxt = dst[:, t].copy() if snapshots else prev
        if snapshots:
            nxt[1] = -1
        gdn.gdn_decode_packed(step["q"], step["k"], step["v"], step["g"], step["beta"], cache_p,
                              torch.from_numpy(prev).cuda(), ot, dst_slot=torch.from_numpy(nxt).cuda())
        o_p[:, t] = ot
        prev = nxt
    torch.cuda.synchronize()
    assert torch.equal(o_m.view(torch.int16), o_p.reshape(rows * T, h, d).view(torch.int16))
    assert torch.equal(cache_m, cache_p)
    assert o_m.reshape(rows, T, h, d)[1].float().abs().max().item() == 0.0
