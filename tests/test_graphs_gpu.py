"""CUDA-graph capture and co-launch of the hot path.

vLLM page "Enable batch-invariant mixed decode and prefill for Qwen GDN":
decode batches run as full CUDA graphs per padded batch size, mixed batches
piecewise; the page asks that a row's result not depend on how it is
launched.  These tests capture the C-ABI calls into CUDA graphs and replay
them with new inputs in the static buffers, and run the decode and prefill
parts of a mixed step on two streams at once; every result must equal the
eager single-stream run bit for bit.
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


def _bits(t):
    return t.view(torch.int16) if t.dtype == torch.bfloat16 else t


def _step_inputs(seqs, t):
    idx = seqs.cu_seqlens[:-1] + t
    return gu.arrays_to_device({n: getattr(seqs, n)[idx] for n in ("q", "k", "v", "g", "beta")})


@pytest.mark.parametrize("rows,padded", [(1, 0), (8, 3), (64, 0), (256, 0)])
def test_decode_graph_replay_matches_eager(gdn, rows, padded):
    """One decode step captured per padded batch size; 3 replays with new
    inputs copied into the static buffers.  Padded rows (src < 0) keep o = 0."""
    h, d, steps = 16, 128, 3
    seqs = gi.token_batch([steps] * rows, h, h, d, seed=11, init_state=True)
    src, n_slots = gi.slots(rows, 11)
    src = src.copy()
    if padded:
        src[-padded:] = -1
    live = src[src >= 0]
    cache_e = gu.empty_cache(n_slots, h, d)
    gu.put_states(cache_e, live, seqs.init_state[:rows - padded])
    cache_g = cache_e.clone()
    src_t = torch.from_numpy(src).cuda()
    st_e = torch.zeros(1, dtype=torch.int32, device="cuda")
    st_g = torch.zeros(1, dtype=torch.int32, device="cuda")
    static = {k: torch.zeros_like(v) for k, v in _step_inputs(seqs, 0).items()}
    o_g = torch.full((rows, h, d), 7.0, dtype=torch.bfloat16, device="cuda")
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        gdn.gdn_decode_packed(static["q"], static["k"], static["v"], static["g"], static["beta"],
                              cache_g, src_t, o_g, dev_status=st_g)
    for t in range(steps):
        x = _step_inputs(seqs, t)
        for name in static:
            static[name].copy_(x[name])
        graph.replay()
        o_e = torch.full((rows, h, d), 7.0, dtype=torch.bfloat16, device="cuda")
        gdn.gdn_decode_packed(x["q"], x["k"], x["v"], x["g"], x["beta"], cache_e, src_t, o_e,
                              dev_status=st_e)
        torch.cuda.synchronize()
        assert torch.equal(_bits(o_g), _bits(o_e)), f"step {t}: graph o differs from eager"
        if padded:
            assert not o_g[-padded:].float().abs().max().item()
    assert torch.equal(cache_g, cache_e)
    assert st_g.item() == 0 and st_e.item() == 0


def _mixed_buffers(wl):
    dec, pre = wl["decode"], wl["prefill"]
    nd, npf = dec.num_seqs, pre.num_seqs
    n_slots = 2 * (nd + npf)
    src = gi.slots(nd + npf, 1, n_slots)[0]
    cache = gu.empty_cache(n_slots, dec.h_v, dec.d)
    gu.put_states(cache, src[:nd], dec.init_state)
    arrs = gu.arrays_to_device(gu.concat_batches(dec, pre))
    return {"nd": nd, "src": src, "cache": cache, "arrs": arrs,
            "cu_p": torch.from_numpy(pre.cu_seqlens.astype(np.int32)).cuda(),
            "cu_h": [int(x) for x in pre.cu_seqlens],
            "dsrc": torch.from_numpy(src[:nd]).cuda(), "pdst": torch.from_numpy(src[nd:]).cuda(),
            "T": nd + pre.total_tokens, "h": dec.h_v, "d": dec.d}


def _run_mixed(gdn, b, cache, arrs, o, st, stream=None):
    gdn.gdn_mixed_step(b["nd"], arrs["q"], arrs["k"], arrs["v"], arrs["g"], arrs["beta"], b["cu_p"],
                       b["cu_h"], cache, b["dsrc"], o, pre_dst_slot=b["pdst"], dev_status=st,
                       stream=stream)


@pytest.mark.parametrize("which", ["tiny", "full"])
def test_mixed_step_graph_replay_matches_eager(gdn, which):
    """The mixed step (decode launch + prefill launch) captured once and
    replayed twice; the second replay runs on the states the first wrote."""
    wl = gi.tiny_mixed(0) if which == "tiny" else gi.mixed_step(0)
    b = _mixed_buffers(wl)
    cache_e, cache_g = b["cache"], b["cache"].clone()
    o_e = torch.empty((b["T"], b["h"], b["d"]), dtype=torch.bfloat16, device="cuda")
    o_g = torch.empty_like(o_e)
    st_e = torch.zeros(1, dtype=torch.int32, device="cuda")
    st_g = torch.zeros(1, dtype=torch.int32, device="cuda")
    static = {k: torch.zeros_like(v) for k, v in b["arrs"].items()}
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        _run_mixed(gdn, b, cache_g, static, o_g, st_g)
    for rep in range(2):
        for name in static:
            static[name].copy_(b["arrs"][name])
        graph.replay()
        _run_mixed(gdn, b, cache_e, b["arrs"], o_e, st_e)
        torch.cuda.synchronize()
        assert torch.equal(_bits(o_g), _bits(o_e)), f"replay {rep}: o differs"
        assert torch.equal(cache_g, cache_e), f"replay {rep}: states differ"
    assert st_g.item() == 0 and st_e.item() == 0


def test_decode_prefill_colaunch_on_two_streams(gdn):
    """Decode rows on one stream and the prefills on another, at the same
    time (the prefill grid leaves most SMs free), eager and captured as one
    fork/join graph: both equal the single-stream mixed step bit for bit."""
    wl = gi.mixed_step(0)
    b = _mixed_buffers(wl)
    nd, arrs = b["nd"], b["arrs"]
    cache_ref = b["cache"]
    o_ref = torch.empty((b["T"], b["h"], b["d"]), dtype=torch.bfloat16, device="cuda")
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    cache_2s, cache_gr = cache_ref.clone(), cache_ref.clone()
    _run_mixed(gdn, b, cache_ref, arrs, o_ref, st)

    dec = {n: arrs[n][:nd] for n in arrs}
    pre = {n: arrs[n][nd:] for n in arrs}

    def colaunch(cache, o, s_dec, s_pre):
        main = torch.cuda.current_stream()
        s_dec.wait_stream(main)
        s_pre.wait_stream(main)
        with torch.cuda.stream(s_dec):
            gdn.gdn_decode_packed(dec["q"], dec["k"], dec["v"], dec["g"], dec["beta"], cache,
                                  b["dsrc"], o[:nd], dev_status=st)
        with torch.cuda.stream(s_pre):
            gdn.gdn_prefill_varlen(pre["q"], pre["k"], pre["v"], pre["g"], pre["beta"], b["cu_p"],
                                   b["cu_h"], o[nd:], state=cache, dst_slot=b["pdst"], dev_status=st)
        main.wait_stream(s_dec)
        main.wait_stream(s_pre)

    s_dec, s_pre = torch.cuda.Stream(), torch.cuda.Stream()
    o_2s = torch.empty_like(o_ref)
    colaunch(cache_2s, o_2s, s_dec, s_pre)
    torch.cuda.synchronize()
    assert torch.equal(_bits(o_2s), _bits(o_ref)) and torch.equal(cache_2s, cache_ref)

    o_gr = torch.empty_like(o_ref)
    graph = torch.cuda.CUDAGraph()
    g_dec, g_pre = torch.cuda.Stream(), torch.cuda.Stream()
    with torch.cuda.graph(graph):
        colaunch(cache_gr, o_gr, g_dec, g_pre)
    graph.replay()
    torch.cuda.synchronize()
    assert torch.equal(_bits(o_gr), _bits(o_ref)) and torch.equal(cache_gr, cache_ref)
    assert st.item() == 0


@pytest.mark.parametrize("which", ["tiny", "full"])
def test_mixed_step_colaunch_entry_point(gdn, which):
    """gdn_mixed_step_colaunch (decode on an aux stream, prefill on the
    caller's, fork/join through the caller's events): eager, captured in a
    CUDA graph and replayed twice, and with no aux stream; each equals the
    single-stream mixed step bit for bit, step after step."""
    wl = gi.tiny_mixed(0) if which == "tiny" else gi.mixed_step(0)
    b = _mixed_buffers(wl)
    arrs = b["arrs"]
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    caches = {n: b["cache"].clone() for n in ("ref", "eager", "noaux")}
    outs = {n: torch.empty((b["T"], b["h"], b["d"]), dtype=torch.bfloat16, device="cuda")
            for n in ("ref", "eager", "noaux", "graph")}
    aux, fork, join = torch.cuda.Stream(), torch.cuda.Event(), torch.cuda.Event()

    def co(cache, o, aux_stream):
        gdn.gdn_mixed_step_colaunch(b["nd"], arrs["q"], arrs["k"], arrs["v"], arrs["g"], arrs["beta"],
                                    b["cu_p"], b["cu_h"], cache, b["dsrc"], o, aux_stream, fork, join,
                                    pre_dst_slot=b["pdst"], dev_status=st)

    graph = torch.cuda.CUDAGraph()
    g_aux = torch.cuda.Stream()
    graph_cache = b["cache"].clone()
    with torch.cuda.graph(graph):
        co(graph_cache, outs["graph"], g_aux)
    # capture does not run the work; restore the states for the replays
    graph_cache.copy_(b["cache"])
    torch.cuda.synchronize()
    for rep in range(2):
        _run_mixed(gdn, b, caches["ref"], arrs, outs["ref"], st)
        co(caches["eager"], outs["eager"], aux)
        co(caches["noaux"], outs["noaux"], None)
        graph.replay()
        torch.cuda.synchronize()
        for n in ("eager", "noaux"):
            assert torch.equal(_bits(outs[n]), _bits(outs["ref"])), f"{n} rep {rep}: o differs"
            assert torch.equal(caches[n], caches["ref"]), f"{n} rep {rep}: states differ"
        assert torch.equal(_bits(outs["graph"]), _bits(outs["ref"])), f"graph rep {rep}: o differs"
        assert torch.equal(graph_cache, caches["ref"]), f"graph rep {rep}: states differ"
    assert st.item() == 0


@pytest.mark.parametrize("E", [1, 17])
def test_mixed_step_colaunch_with_emitted_states(gdn, E):
    """The co-launched step with the prefills emitting their states every E
    chunks: outputs, final states and every emitted state equal the
    single-stream mixed step's bit for bit."""
    b = _mixed_buffers(gi.mixed_step(0))
    arrs = b["arrs"]
    n_emit = gdn.gdn_prefill_num_emits(b["cu_h"], E)
    assert n_emit > 0
    res = []
    for colaunch in (False, True):
        cache = b["cache"].clone()
        o = torch.empty((b["T"], b["h"], b["d"]), dtype=torch.bfloat16, device="cuda")
        cs = torch.full((n_emit, b["h"], b["d"], b["d"]), 7.0, device="cuda")
        st = torch.zeros(1, dtype=torch.int32, device="cuda")
        kw = dict(pre_dst_slot=b["pdst"], chunk_states=cs, emit_every_chunks=E, dev_status=st)
        if colaunch:
            gdn.gdn_mixed_step_colaunch(b["nd"], arrs["q"], arrs["k"], arrs["v"], arrs["g"], arrs["beta"],
                                        b["cu_p"], b["cu_h"], cache, b["dsrc"], o, torch.cuda.Stream(),
                                        torch.cuda.Event(), torch.cuda.Event(), **kw)
        else:
            gdn.gdn_mixed_step(b["nd"], arrs["q"], arrs["k"], arrs["v"], arrs["g"], arrs["beta"], b["cu_p"],
                               b["cu_h"], cache, b["dsrc"], o, **kw)
        torch.cuda.synchronize()
        assert st.item() == 0
        res.append((o, cache, cs))
    (o1, c1, s1), (o2, c2, s2) = res
    assert torch.equal(_bits(o1), _bits(o2))
    assert torch.equal(c1, c2)
    assert torch.equal(s1, s2)


@pytest.mark.parametrize("parts", [2, 4, [32, 224]], ids=["2", "4", "32+224"])
def test_end_to_end_step_in_row_groups_matches_single_call(gdn, parts):
    """The benchmark's end-to-end decode step with its rows split into groups
    (host copies of one group overlapping the decode of another, on three
    streams, captured as a CUDA graph) gives the o and the states of the
    single-group step bit for bit, over two replays."""
    import bench
    res = []
    for p in (1, parts):
        _, t = bench.decode_setup(torch, seed=0, dev="cuda")
        graphs, h2d, d2h, o_host = bench.decode_e2e_graphs(torch, gdn, t, p)
        graphs[0].replay()
        graphs[1].replay()
        torch.cuda.synchronize()
        res.append((o_host.clone(), t["cache"].clone(), h2d, d2h))
    (o1, s1, i1, d1), (o2, s2, i2, d2) = res
    assert (i1, d1) == (i2, d2)
    assert torch.equal(_bits(o1), _bits(o2))
    assert torch.equal(s1, s2)


def test_prepared_decode_call_matches_checked_call(gdn):
    """prepare_decode_packed: the buffers checked once, then three steps with
    new inputs copied into them in place; outputs and states equal the
    checked call's bit for bit."""
    rows, h, d, steps = 24, 16, 128, 3
    seqs = gi.token_batch([steps] * rows, h, h, d, seed=12, init_state=True)
    src, n_slots = gi.slots(rows, 12)
    cache_c = gu.empty_cache(n_slots, h, d)
    gu.put_states(cache_c, src, seqs.init_state)
    cache_p = cache_c.clone()
    src_t = torch.from_numpy(src).cuda()
    static = {k: torch.zeros_like(v) for k, v in _step_inputs(seqs, 0).items()}
    o_p = torch.empty((rows, h, d), dtype=torch.bfloat16, device="cuda")
    step = gdn.prepare_decode_packed(static["q"], static["k"], static["v"], static["g"], static["beta"],
                                     cache_p, src_t, o_p)
    for t in range(steps):
        x = _step_inputs(seqs, t)
        for n in static:
            static[n].copy_(x[n])
        step()
        o_c = torch.empty_like(o_p)
        gdn.gdn_decode_packed(x["q"], x["k"], x["v"], x["g"], x["beta"], cache_c, src_t, o_c)
        torch.cuda.synchronize()
        assert torch.equal(_bits(o_p), _bits(o_c)), t
        assert torch.equal(cache_p, cache_c), t
