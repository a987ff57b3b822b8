"""Bitwise GPU-vs-GPU invariances (atol = 0, rtol = 0).

I1  A decode row's output and updated state are identical whether it runs in
    a decode-only call or at the front of a mixed decode+prefill step, with 0,
    1, 4 or 8 co-scheduled prefills (vLLM page "Enable batch-invariant mixed
    decode and prefill for Qwen GDN", section "Test plan", route regression).
I2  A prefill sequence gives identical results alone or inside a batch of N
    (vLLM page "Enable GDN batch-invariant prefix caching", section "Test
    Result": BS=1 vs BS=N bitwise).
I3  Resuming a prefill from the state emitted at a 64-token (E=1) or
    1088-token (E=17) boundary reproduces the uninterrupted outputs and final
    state (same page, section "Purpose": one shared grid for chunks and hits).
I4  Two identical calls give identical bits.
"""
import numpy as np
import pytest
import torch

import gdn_inputs as gi
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


def _decode_only(gdn, dec, cache, slots):
    dv = gu.arrays_to_device({n: getattr(dec, n) for n in ("q", "k", "v", "g", "beta")})
    o = torch.empty((dec.num_seqs, dec.h_v, dec.d), dtype=torch.bfloat16, device="cuda")
    gdn.gdn_decode_packed(dv["q"], dv["k"], dv["v"], dv["g"], dv["beta"], cache,
                          torch.from_numpy(slots).cuda(), o)
    torch.cuda.synchronize()
    return o


def _mixed(gdn, dec, pre, cache, dslots, pslots):
    arrs = gu.arrays_to_device(gu.concat_batches(dec, pre) if pre is not None else
                               {n: getattr(dec, n) for n in ("q", "k", "v", "g", "beta")})
    nd = dec.num_seqs
    T = nd + (pre.total_tokens if pre is not None else 0)
    o = torch.empty((T, dec.h_v, dec.d), dtype=torch.bfloat16, device="cuda")
    if pre is not None:
        cu = torch.from_numpy(pre.cu_seqlens.astype(np.int32)).cuda()
        cu_h = [int(x) for x in pre.cu_seqlens]
        pdst = torch.from_numpy(pslots).cuda()
    else:
        cu, cu_h, pdst = None, None, None
    gdn.gdn_mixed_step(nd, arrs["q"], arrs["k"], arrs["v"], arrs["g"], arrs["beta"], cu, cu_h, cache,
                       torch.from_numpy(dslots).cuda(), o, pre_dst_slot=pdst)
    torch.cuda.synchronize()
    return o


@pytest.mark.parametrize("n_prefills", [0, 1, 4, 8])
def test_I1_decode_rows_alone_vs_front_of_mixed_batch(gdn, n_prefills):
    wl = gi.mixed_step(0)
    dec = wl["decode"]
    nd = dec.num_seqs
    lens = (list(gi.PROMPT_CLASSES) * 2)[:n_prefills]
    pre = gi.token_batch(lens, 16, 16, 128, seed=5) if n_prefills else None
    n_slots = 2 * (nd + 8)
    dslots = gi.slots(nd, 3, n_slots)[0]
    pslots = np.array([s for s in range(n_slots) if s not in set(dslots.tolist())][:max(n_prefills, 1)],
                      np.int32)
    c1 = gu.empty_cache(n_slots, 16, 128)
    gu.put_states(c1, dslots, dec.init_state)
    c2 = c1.clone()
    o_alone = _decode_only(gdn, dec, c1, dslots)
    o_mixed = _mixed(gdn, dec, pre, c2, dslots, pslots[:n_prefills])
    idx = torch.from_numpy(dslots.astype(np.int64)).cuda()
    assert torch.equal(o_alone.view(torch.int16), o_mixed[:nd].view(torch.int16))
    assert torch.equal(c1[idx].view(torch.int32), c2[idx].view(torch.int32))


def _prefill(gdn, b, src_states=None, E=0):
    """Run a batch; src_states: optional fp32 S^T [n][h_v][d][d] initial
    states.  Returns (o, final S^T [n][h_v][d][d], chunk_states)."""
    n = b.num_seqs
    cache = gu.empty_cache(2 * n, b.h_v, b.d)
    src = None
    if src_states is not None:
        cache[:n] = src_states
        src = torch.arange(n, dtype=torch.int32, device="cuda")
    dst = torch.arange(n, 2 * n, dtype=torch.int32, device="cuda")
    dv = gu.batch_to_device(b)
    o = torch.empty((b.total_tokens, b.h_v, b.d), dtype=torch.bfloat16, device="cuda")
    n_emit = gdn.gdn_prefill_num_emits(dv["cu_host"], E) if E else 0
    cs = torch.zeros((max(n_emit, 1), b.h_v, b.d, b.d), device="cuda") if E else None
    gdn.gdn_prefill_varlen(dv["q"], dv["k"], dv["v"], dv["g"], dv["beta"], dv["cu"], dv["cu_host"], o,
                           state=cache, src_slot=src, dst_slot=dst, chunk_states=cs, emit_every_chunks=E)
    torch.cuda.synchronize()
    return o, cache[n:].clone(), cs


def _sub_batch(b, seqs, t_from=None):
    """Batch of the given sequences of b (optionally starting each at token t_from)."""
    parts = []
    for s in seqs:
        t0, t1 = int(b.cu_seqlens[s]), int(b.cu_seqlens[s + 1])
        if t_from is not None:
            t0 += t_from
        parts.append((t0, t1))
    lens = [t1 - t0 for t0, t1 in parts]
    cu = np.zeros(len(lens) + 1, np.int32)
    cu[1:] = np.cumsum(lens)
    take = lambda a: np.concatenate([a[t0:t1] for t0, t1 in parts])
    return gi.TokenBatch(b.h_k, b.h_v, b.d, cu, take(b.q), take(b.k), take(b.v), take(b.g), take(b.beta))


def _bits(t):
    return t.contiguous().view(torch.int16 if t.dtype == torch.bfloat16 else torch.int32)


def test_I2_prefill_sequence_alone_vs_in_batch(gdn):
    b = gi.prefill_qwen3next_gva(0)["prefill"]
    o_all, S_all, _ = _prefill(gdn, b)
    for s in (0, 3, b.num_seqs - 1):
        one = _sub_batch(b, [s])
        o1, S1, _ = _prefill(gdn, one)
        t0, t1 = int(b.cu_seqlens[s]), int(b.cu_seqlens[s + 1])
        assert torch.equal(_bits(o1), _bits(o_all[t0:t1]))
        assert torch.equal(_bits(S1[0]), _bits(S_all[s]))


@pytest.mark.parametrize("E,ks", [(1, [1, 5, 31]), (17, [1])])
def test_I3_resume_from_emitted_state_on_the_grid(gdn, E, ks):
    b = gi.token_batch([2000, 1500], 16, 32, 128, seed=7)
    o_full, S_full, cs = _prefill(gdn, b, E=E)
    offs = gdn.gdn_prefill_emit_offsets([int(x) for x in b.cu_seqlens], E)
    for s in range(b.num_seqs):
        L = b.seqlens[s]
        for k in ks:
            if 64 * E * k > L:
                continue
            t = 64 * E * k
            part = _sub_batch(b, [s], t_from=t)
            st = cs[offs[s] + k - 1:offs[s] + k].clone()
            o_r, S_r, _ = _prefill(gdn, part, src_states=st)
            t0 = int(b.cu_seqlens[s])
            assert torch.equal(_bits(o_r), _bits(o_full[t0 + t:t0 + L])), (s, k)
            assert torch.equal(_bits(S_r[0]), _bits(S_full[s])), (s, k)


def test_I3_resume_prefix_cache_workload_at_1088_multiples(gdn):
    """4 x 32768 tokens, E=17: resume sequence 1 at 1088 * {1, 15, 30}."""
    b = gi.prefix_cache_prefill(0)["prefill"]
    o_full, S_full, cs = _prefill(gdn, b, E=17)
    offs = gdn.gdn_prefill_emit_offsets([int(x) for x in b.cu_seqlens], 17)
    s = 1
    t0 = int(b.cu_seqlens[s])
    for k in (1, 15, 30):
        t = 1088 * k
        part = _sub_batch(b, [s], t_from=t)
        o_r, S_r, _ = _prefill(gdn, part, src_states=cs[offs[s] + k - 1:offs[s] + k].clone())
        assert torch.equal(_bits(o_r), _bits(o_full[t0 + t:t0 + 32768])), k
        assert torch.equal(_bits(S_r[0]), _bits(S_full[s])), k


def test_I4_run_to_run_determinism(gdn):
    wl = gi.mixed_step(0)
    dec, pre = wl["decode"], wl["prefill"]
    nd = dec.num_seqs
    dslots = np.arange(nd, dtype=np.int32)
    pslots = np.arange(nd, nd + pre.num_seqs, dtype=np.int32)
    outs = []
    for _ in range(2):
        c = gu.empty_cache(nd + pre.num_seqs, 16, 128)
        gu.put_states(c, dslots, dec.init_state)
        o = _mixed(gdn, dec, pre, c, dslots, pslots)
        outs.append((o, c))
    assert torch.equal(_bits(outs[0][0]), _bits(outs[1][0]))
    assert torch.equal(_bits(outs[0][1]), _bits(outs[1][1]))


@pytest.mark.parametrize("which", ["gva_d128", "tiny_d64"])
def test_I4_prefill_repeatable_under_concurrent_load(gdn, which):
    """The prefill kernel's two warp groups hand work to each other through
    shared memory, TMEM and barriers; a missing barrier shows up as results
    that change with timing.  Six runs of the same prefill (with emission),
    three of them while decode launches on another stream compete for the
    SMs, must give the same o, final states and emitted states bit for bit."""
    if which == "gva_d128":
        b = gi.prefill_qwen3next_gva(0)["prefill"]
    else:
        b = gi.token_batch([64, 100, 1, 130, 700], 4, 4, 64, 17)
    rows = 256
    dec = gi.token_batch([1] * rows, 16, 16, 128, 3, init_state=True)
    dcache = gu.empty_cache(rows, 16, 128)
    dx = gu.batch_to_device(dec)
    dsrc = torch.arange(rows, dtype=torch.int32, device="cuda")
    do = torch.empty((rows, 16, 128), dtype=torch.bfloat16, device="cuda")
    side = torch.cuda.Stream()
    ref = None
    for run in range(6):
        if run % 2:
            with torch.cuda.stream(side):
                for _ in range(4):
                    gdn.gdn_decode_packed(dx["q"], dx["k"], dx["v"], dx["g"], dx["beta"], dcache, dsrc, do)
        res = _prefill(gdn, b, E=1)
        torch.cuda.synchronize()
        if ref is None:
            ref = res
            continue
        assert torch.equal(_bits(res[0]), _bits(ref[0])), run
        assert torch.equal(res[1], ref[1]), run
        assert torch.equal(res[2], ref[2]), run
