"""Benchmark of the Gated DeltaNet hot path on GB300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl gdn|reference]
                    [--no-extra] [--no-cpu-baseline]

Headline workload: packed recurrent decode of a Qwen3.5-0.8B-like GDN layer
(256 cached rows, 16 heads, d = 128, fp32 states in a slot cache of 512
slots, updated in place).  A step is one decode call over the 256 rows; the
metric is decode rows per second.  The JSON line also carries the prefill
workloads (varlen GVA prefill, 4 x 32768 prefix-cache prefill with state
emission, one mixed continuous-batching step) in prefill tokens/s.

Under torchrun each rank runs its own replica of the workload on its own GPU
(weak scaling, no collective on the data path); the timed region is bracketed
by barriers and the slowest rank's time is used.

--impl reference times the fp64 CPU oracle on the host cores on a bounded
sample of the same workload (the only other implementation of this path).
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import gdn_inputs as gi  # noqa: E402

DECODE_ROWS, H, D = 256, 16, 128
# Algorithmic bytes per decode row: state read + write, q, k, v, o, g, beta, slot index.
DECODE_BYTES_PER_ROW = 2 * H * D * D * 4 + 2 * H * D * 2 + 2 * H * D * 2 + 2 * H * 4 + 4
DECODE_BYTES_PER_ROW_H16 = DECODE_BYTES_PER_ROW  # the mixed step's decode rows have the same shape
# Algorithmic flops per prefill token (GVA H_k=16, H_v=32, d=128, C=64):
# shared K K^T and Q K^T per key head, then per value head the WY products,
# W S0, Q S0, (M o QK^T) U and K~^T U.
C = 64


def prefill_flops_per_token(h_k, h_v, d):
    return h_k * 4 * C * d + h_v * (2 * C * d + 4 * C * d + 6 * d * d)


def prefill_bytes_per_token(h_k, h_v, d):
    return 2 * h_k * d * 2 + 2 * h_v * d * 2 + 2 * h_v * 4


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        j = json.load(open(p))
        return {"hbm_gbs": j["hbm_gbs"], "bf16_tflops": j["bf16_tflops"],
                "bf16_tflops_sustained": j.get("bf16_tflops_sustained", j["bf16_tflops"]),
                "source": "measured"}
    return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0, "source": "fallback"}


# ---------------------------------------------------------------------------
# clocks sampler
# ---------------------------------------------------------------------------

class Clocks:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.gpu = gpu_index
        self.proc = None
        self.path = None

    def __enter__(self):
        fd, self.path = tempfile.mkstemp(suffix=".csv")
        os.close(fd)
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "100", "-f", self.path], stdout=subprocess.DEVNULL, stderr=subprocess.DEVNULL)
            time.sleep(0.3)
        except OSError:
            self.proc = None
        return self

    def __exit__(self, *exc):
        if self.proc is not None:
            time.sleep(0.25)
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self):
        if self.proc is None or not os.path.exists(self.path):
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        rows = []
        for line in open(self.path):
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                rows.append((float(parts[1]), float(parts[2]), parts[5:9]))
            except ValueError:
                continue
        os.unlink(self.path)
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"]}
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for _, _, r in rows for i, v in enumerate(r) if v.lower() == "active"})
        return {"sm_mhz": statistics.median(r[0] for r in rows), "sm_max_mhz": max(r[1] for r in rows),
                "samples": len(rows), "reasons": reasons}


# ---------------------------------------------------------------------------
# distributed plumbing (timing only; no data-path collective)
# ---------------------------------------------------------------------------

def dist_setup(torch):
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        backend = "nccl" if torch.cuda.is_available() else "gloo"
        if backend == "nccl":
            torch.cuda.set_device(local)
        dist.init_process_group(backend)
    elif torch.cuda.is_available():
        torch.cuda.set_device(local)
    return world, rank, local


def barrier(torch, world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(torch, world, x: float) -> float:
    if world == 1:
        return x
    import torch.distributed as dist
    dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([x], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


# ---------------------------------------------------------------------------
# GPU arm
# ---------------------------------------------------------------------------

def bf16(torch, bits, dev):
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16).to(dev)


def decode_setup(torch, seed, dev):
    wl = gi.decode_qwen35_08b(seed)
    b = wl["decode"]
    cache = torch.zeros((wl["n_slots"], H, D, D), dtype=torch.float32, device=dev)
    idx = torch.from_numpy(wl["src_slot"].astype(np.int64)).to(dev)
    cache[idx] = torch.from_numpy(np.swapaxes(b.init_state, -1, -2).copy()).to(dev)
    t = {"q": bf16(torch, b.q, dev), "k": bf16(torch, b.k, dev), "v": bf16(torch, b.v, dev),
         "g": torch.from_numpy(b.g).to(dev), "beta": torch.from_numpy(b.beta).to(dev),
         "src": torch.from_numpy(wl["src_slot"]).to(dev), "cache": cache,
         "o": torch.empty((DECODE_ROWS, H, D), dtype=torch.bfloat16, device=dev)}
    return wl, t


def run_decode(gdn, t):
    gdn.gdn_decode_packed(t["q"], t["k"], t["v"], t["g"], t["beta"], t["cache"], t["src"], t["o"])


def time_decode(torch, gdn, t, steps, warmup, world):
    for _ in range(warmup):
        run_decode(gdn, t)
    torch.cuda.synchronize()
    barrier(torch, world)
    torch.cuda.synchronize()
    # The timed region holds exactly `steps` decode launches back to back on
    # this stream, so the average launch duration is total / steps.
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    start.record()
    for _ in range(steps):
        run_decode(gdn, t)
    end.record()
    torch.cuda.synchronize()
    barrier(torch, world)
    total_ms = start.elapsed_time(end)
    return total_ms, [total_ms / steps] * steps


# Row groups of the end-to-end decode step (measured on the GB300, us per
# 256-row step: 1 group 120, 2 groups 116, 4 groups 127, 8 groups 143: each
# group adds graph-node dependencies of a few us; host copies run at
# ~180 GB/s H2D and ~145 GB/s D2H).
E2E_PARTS = 2


def decode_e2e_graphs(torch, gdn, t, parts):
    """The end-to-end decode step as CUDA graphs (two, for two alternating
    device input buffers), captured from the public entry point: the step's
    q, k, v, g, beta go from pinned host memory to the device, the decode
    runs, o comes back to pinned host memory.  The step's rows are split into
    `parts` equal groups, or groups of the row counts `parts` lists (parts =
    1: one copy, one call, one copy): group i's inputs
    are copied on an input stream, its decode runs on the capturing stream
    once they have landed, and its o is copied back on an output stream once
    its decode has finished, so the copies of one group overlap the decode of
    the others.  A row's result does not depend on the rows sharing its
    launch, so the groups compute exactly what one call over all rows does.
    Returns (graphs, h2d bytes per step, d2h bytes per step, o_host)."""
    names = ("q", "k", "v", "g", "beta")
    rows = t["q"].shape[0]
    if isinstance(parts, int):
        if rows % parts:
            raise ValueError(f"{rows} rows do not split into {parts} equal groups")
        counts = [rows // parts] * parts
    else:  # explicit row counts of the groups
        counts = [int(c) for c in parts]
        if sum(counts) != rows or min(counts) <= 0:
            raise ValueError(f"group sizes {counts} do not partition {rows} rows")
    first = [sum(counts[:p]) for p in range(len(counts))]
    # each group's inputs packed one after the other, every tensor 256-byte aligned
    layout, pos = [], 0
    for p, c in enumerate(counts):
        ent = []
        for n in names:
            sz = t[n][:c].numel() * t[n].element_size()
            ent.append((n, pos, sz))
            pos += (sz + 255) // 256 * 256
        layout.append(ent)
    starts = [ent[0][1] for ent in layout] + [pos]
    host = torch.empty(pos, dtype=torch.uint8).pin_memory()
    for p, c in enumerate(counts):
        for n, o0, sz in layout[p]:
            src = t[n][first[p]:first[p] + c].contiguous().view(torch.uint8).reshape(-1).cpu()
            host[o0:o0 + sz].copy_(src)
    o_host = torch.empty(t["o"].shape, dtype=t["o"].dtype).pin_memory()
    h2d = sum(sz for ent in layout for _, _, sz in ent)
    d2h = o_host.numel() * o_host.element_size()
    dev = t["q"].device
    dev_in = [torch.empty(pos, dtype=torch.uint8, device=dev) for _ in range(2)]
    outs = [torch.empty_like(t["o"]) for _ in range(2)]
    s_in, s_out = torch.cuda.Stream(device=dev), torch.cuda.Stream(device=dev)
    graphs = []
    for b in range(2):
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            main = torch.cuda.current_stream()
            s_in.wait_stream(main)
            s_out.wait_stream(main)
            landed = []
            with torch.cuda.stream(s_in):
                for p in range(len(counts)):
                    dev_in[b][starts[p]:starts[p + 1]].copy_(host[starts[p]:starts[p + 1]], non_blocking=True)
                    ev = torch.cuda.Event()
                    ev.record(s_in)
                    landed.append(ev)
            for p, c in enumerate(counts):
                main.wait_event(landed[p])
                x = {n: dev_in[b][o0:o0 + sz].view(t[n].dtype).view((c,) + tuple(t[n].shape[1:]))
                     for n, o0, sz in layout[p]}
                rs = slice(first[p], first[p] + c)
                gdn.gdn_decode_packed(x["q"], x["k"], x["v"], x["g"], x["beta"], t["cache"], t["src"][rs], outs[b][rs])
                done = torch.cuda.Event()
                done.record(main)
                with torch.cuda.stream(s_out):
                    s_out.wait_event(done)
                    o_host[rs].copy_(outs[b][rs], non_blocking=True)
            main.wait_stream(s_in)
            main.wait_stream(s_out)
        graphs.append(g)
    return graphs, h2d, d2h, o_host


def time_decode_e2e(torch, gdn, t, steps, warmup, world, parts=1):
    """End to end, as a serving loop runs decode: each step is one replay of
    the graphs of decode_e2e_graphs (alternating input buffers).  The state
    cache stays resident on the device; every step moves all of its input and
    output bytes inside the timed region.  Replays run back to back on one
    stream, so no step's copies overlap another step's decode (a decode
    step's inputs depend on the previous step's outputs)."""
    graphs, h2d, d2h, _ = decode_e2e_graphs(torch, gdn, t, parts)
    for k in range(warmup):
        graphs[k & 1].replay()
    torch.cuda.synchronize()
    barrier(torch, world)
    s, e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    s.record()
    for k in range(steps):
        graphs[k & 1].replay()
    e.record()
    torch.cuda.synchronize()
    barrier(torch, world)
    return s.elapsed_time(e), h2d, d2h


def time_decode_e2e_eager(torch, gdn, t, steps, warmup, world):
    """The same step issued from Python each time: pinned host -> device
    copies of q, k, v, g, beta, the decode call, device -> host copy of o,
    one after the other on one stream."""
    host = {n: t[n].cpu().pin_memory() for n in ("q", "k", "v", "g", "beta")}
    o_host = torch.empty(t["o"].shape, dtype=t["o"].dtype).pin_memory()
    h2d = sum(x.numel() * x.element_size() for x in host.values())
    d2h = o_host.numel() * o_host.element_size()

    def step():
        for n, x in host.items():
            t[n].copy_(x, non_blocking=True)
        run_decode(gdn, t)
        o_host.copy_(t["o"], non_blocking=True)

    for _ in range(warmup):
        step()
    torch.cuda.synchronize()
    barrier(torch, world)
    s, e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    s.record()
    for _ in range(steps):
        step()
    e.record()
    torch.cuda.synchronize()
    barrier(torch, world)
    return s.elapsed_time(e), h2d, d2h


_FLUSH = {}
FLUSH_NOTE = "each call preceded by a 256 MiB read on its stream (L2 flushed, host issue hidden)"


def l2_flush(torch):
    """Read 256 MiB on the current stream (a max-reduction).  It evicts the
    129 MB L2 before a timed call without leaving dirty lines to write back,
    and it keeps the device busy for ~40 us while the host issues the call
    (binding checks, C-ABI validation, launch), so that host time does not
    fall between the call's events."""
    dev = torch.cuda.current_device()
    buf = _FLUSH.get(dev)
    if buf is None:
        buf = _FLUSH[dev] = torch.ones(64 << 20, dtype=torch.float32, device=f"cuda:{dev}")
    buf.amax()


def timed_median(torch, fn, reps=20, warm=10):
    """Median device time (ms) of `reps` calls after `warm` untimed ones, each
    bracketed by CUDA events on the current stream after an L2 flush; clocks
    sampled meanwhile."""
    for _ in range(warm):
        fn()
    torch.cuda.synchronize()
    with Clocks(torch.cuda.current_device()) as clk:
        ev = []
        for _ in range(reps):
            l2_flush(torch)
            a, z = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record()
            fn()
            z.record()
            ev.append((a, z))
        torch.cuda.synchronize()
    return statistics.median(a.elapsed_time(z) for a, z in ev), clk.summary()


def prefill_case(torch, gdn, wl, dev, reps, E=0):
    b = wl["prefill"]
    q, k, v = bf16(torch, b.q, dev), bf16(torch, b.k, dev), bf16(torch, b.v, dev)
    g, beta = torch.from_numpy(b.g).to(dev), torch.from_numpy(b.beta).to(dev)
    cu = torch.from_numpy(b.cu_seqlens.astype(np.int32)).to(dev)
    cu_h = [int(x) for x in b.cu_seqlens]
    n = b.num_seqs
    cache = torch.zeros((n, b.h_v, b.d, b.d), dtype=torch.float32, device=dev)
    dst = torch.arange(n, dtype=torch.int32, device=dev)
    o = torch.empty((b.total_tokens, b.h_v, b.d), dtype=torch.bfloat16, device=dev)
    n_emit = gdn.gdn_prefill_num_emits(cu_h, E) if E else 0
    cs = torch.empty((max(n_emit, 1), b.h_v, b.d, b.d), dtype=torch.float32, device=dev) if E else None

    def call():
        gdn.gdn_prefill_varlen(q, k, v, g, beta, cu, cu_h, o, state=cache, dst_slot=dst,
                               chunk_states=cs, emit_every_chunks=E)

    ms, clocks = timed_median(torch, call, reps=reps)
    T = b.total_tokens
    fl = prefill_flops_per_token(b.h_k, b.h_v, b.d) * T
    return {"workload": wl["name"], "seqlens": b.seqlens if n <= 16 else f"{n} x {b.seqlens[0]}",
            "tokens": T, "ms": ms, "timing": f"median of {reps} calls after 10 warm-up calls, {FLUSH_NOTE}",
            "tokens_per_s": T / (ms * 1e-3),
            "algorithmic_tflops": fl / (ms * 1e-3) / 1e12, "emit_every_chunks": E,
            "emitted_states": n_emit, "clocks": clocks}


def mixed_case(torch, gdn, dev, reps, peaks):
    wl = gi.mixed_step(0)
    dec, pre = wl["decode"], wl["prefill"]
    nd = dec.num_seqs
    cat = lambda n: np.concatenate([getattr(dec, n), getattr(pre, n)])
    q, k, v = bf16(torch, cat("q"), dev), bf16(torch, cat("k"), dev), bf16(torch, cat("v"), dev)
    g, beta = torch.from_numpy(cat("g")).to(dev), torch.from_numpy(cat("beta")).to(dev)
    slots = torch.from_numpy(wl["src_slot"]).to(dev)
    cache = torch.zeros((wl["n_slots"], H, D, D), dtype=torch.float32, device=dev)
    cache[slots[:nd].long()] = torch.from_numpy(np.swapaxes(dec.init_state, -1, -2).copy()).to(dev)
    o = torch.empty((q.shape[0], H, D), dtype=torch.bfloat16, device=dev)
    cu = torch.from_numpy(pre.cu_seqlens.astype(np.int32)).to(dev)
    cu_h = [int(x) for x in pre.cu_seqlens]

    def call():
        gdn.gdn_mixed_step(nd, q, k, v, g, beta, cu, cu_h, cache, slots[:nd], o, pre_dst_slot=slots[nd:])

    aux, fork, join = torch.cuda.Stream(), torch.cuda.Event(), torch.cuda.Event()

    def colaunch():
        # the same step with the decode rows on a second stream beside the prefill
        gdn.gdn_mixed_step_colaunch(nd, q, k, v, g, beta, cu, cu_h, cache, slots[:nd], o, aux, fork, join,
                                    pre_dst_slot=slots[nd:])

    ms, clocks = timed_median(torch, call, reps=reps)
    ms2, _ = timed_median(torch, colaunch, reps=reps)
    # Roofline of the step: the decode rows are bound by HBM, the prefill by
    # the tensor cores, and the two run one after the other, so the floor is
    # the sum of the two parts' roofline times.
    dec_bytes = nd * DECODE_BYTES_PER_ROW_H16
    pre_flops = pre.total_tokens * prefill_flops_per_token(pre.h_k, pre.h_v, pre.d)
    dec_floor_ms = dec_bytes / (peaks["hbm_gbs"] * 1e9) * 1e3
    pre_floor_ms = pre_flops / (peaks["bf16_tflops"] * 1e12) * 1e3
    floor_ms = dec_floor_ms + pre_floor_ms
    # co-launched, the halves overlap: the floor is the longer of the two
    floor_co_ms = max(dec_floor_ms, pre_floor_ms)
    return {"workload": wl["name"], "decode_rows": nd, "prefill_seqlens": pre.seqlens, "ms": ms,
            "timing": f"median of {reps} calls after 10 warm-up calls, {FLUSH_NOTE}",
            "tokens_per_s": (nd + pre.total_tokens) / (ms * 1e-3), "colaunch_two_streams_ms": ms2,
            "roofline": {"bound": "hbm (decode rows) + tensor (prefill)", "decode_bytes": dec_bytes,
                         "prefill_flops": pre_flops, "floor_ms": floor_ms, "frac": floor_ms / ms,
                         "floor_colaunch_ms": floor_co_ms, "frac_colaunch": floor_co_ms / ms2,
                         "peak_hbm_gbs": peaks["hbm_gbs"], "peak_tflops": peaks["bf16_tflops"],
                         "peak_source": peaks["source"]},
            "clocks": clocks}


def multi_decode_case(torch, gdn, dev, peaks, rows=256, T=4, reps=10):
    """Multi-token decode, 256 rows x 4 tokens (H=16, d=128): with a state
    snapshot after every token, and with only the final state written back.
    Algorithmic bytes per row: state read once + written per snapshot, plus
    q, k, v, o (bf16) and g, beta (fp32) per token."""
    b = gi.token_batch([T] * rows, H, H, D, 6, init_state=True)
    n_slots = rows * (T + 1)
    perm = np.random.default_rng(6).permutation(n_slots).astype(np.int32)
    src, dsts = perm[:rows], perm[rows:].reshape(rows, T)
    cache = torch.zeros((n_slots, H, D, D), dtype=torch.float32, device=dev)
    cache[torch.from_numpy(src.astype(np.int64)).to(dev)] = \
        torch.from_numpy(np.swapaxes(b.init_state, -1, -2).copy()).to(dev)
    q, k, v = bf16(torch, b.q, dev), bf16(torch, b.k, dev), bf16(torch, b.v, dev)
    g, beta = torch.from_numpy(b.g).to(dev), torch.from_numpy(b.beta).to(dev)
    src_t, dst_t = torch.from_numpy(src).to(dev), torch.from_numpy(dsts.reshape(-1)).to(dev)
    o = torch.empty((rows * T, H, D), dtype=torch.bfloat16, device=dev)
    state_b = H * D * D * 4
    tok_b = H * D * 2 * 4 + H * 4 * 2
    out = {"workload": f"decode_multi_r{rows}_t{T}_h16_d128", "rows": rows, "tokens_per_row": T,
           "timing": f"median of {reps} calls after 1 warm-up call, {FLUSH_NOTE}"}
    for name, dst, writes in (("snapshots", dst_t, T), ("final_only", None, 1)):
        def call():
            gdn.gdn_decode_multi(T, q, k, v, g, beta, cache, src_t, o, dst_slots=dst)
        call()
        torch.cuda.synchronize()
        ev = []
        for _ in range(reps):
            l2_flush(torch)
            a0, z0 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a0.record()
            call()
            z0.record()
            ev.append((a0, z0))
        torch.cuda.synchronize()
        ms = statistics.median(a0.elapsed_time(z0) for a0, z0 in ev)
        byts = rows * ((1 + writes) * state_b + T * tok_b)
        gbs = byts / (ms * 1e-3) / 1e9
        out[name] = {"ms": ms, "tokens_per_s": rows * T / (ms * 1e-3), "bytes_per_launch": byts,
                     "roofline": {"bound": "hbm", "kernel": "decode_multi_kernel<128>", "achieved": gbs,
                                  "peak": peaks["hbm_gbs"], "unit": "GB/s", "frac": gbs / peaks["hbm_gbs"]}}
    return out


def prep_case(torch, gdn, dev, peaks, T=131072, h_k=16, h_v=32, reps=20):
    """Input preparation over 131072 tokens (H_k=16, H_v=32, d=128): q, k
    read and written in bf16, a, b read and g, beta written in fp32."""
    raw = gi.raw_inputs(T, h_k, h_v, D, 9)
    q_raw, k_raw = bf16(torch, raw.q, dev), bf16(torch, raw.k, dev)
    a, b_ = torch.from_numpy(raw.a).to(dev), torch.from_numpy(raw.b).to(dev)
    A_log, dt_bias = torch.from_numpy(raw.A_log).to(dev), torch.from_numpy(raw.dt_bias).to(dev)
    q, k = torch.empty_like(q_raw), torch.empty_like(k_raw)
    g, beta = torch.empty_like(a), torch.empty_like(a)

    def call():
        gdn.gdn_prep_inputs(q_raw, k_raw, a, b_, A_log, dt_bias, q, k, g, beta)

    ms, clocks = timed_median(torch, call, reps=reps)
    byts = T * (2 * 2 * h_k * D * 2 + 4 * h_v * 4)
    gbs = byts / (ms * 1e-3) / 1e9
    return {"workload": f"prep_inputs_t{T}_hk{h_k}_hv{h_v}_d128", "ms": ms, "tokens_per_s": T / (ms * 1e-3),
            "bytes_per_launch": byts, "timing": f"median of {reps} calls after 10 warm-up calls, {FLUSH_NOTE}", "clocks": clocks,
            "roofline": {"bound": "hbm", "kernel": "prep_kernel<128>", "achieved": gbs, "peak": peaks["hbm_gbs"],
                         "unit": "GB/s", "frac": gbs / peaks["hbm_gbs"]}}


def decode_latency_case(torch, gdn, dev, rows_list=(1, 8, 64, 256), iters=200):
    """Decode step latency per padded batch size: eager C-ABI calls from
    Python (checked on every call, and prepared once with
    prepare_decode_packed) versus replay of a CUDA graph holding one step
    (H=16, d=128)."""
    cases = []
    for rows in rows_list:
        b = gi.token_batch([1] * rows, H, H, D, 5, init_state=True)
        src, n_slots = gi.slots(rows, 5)
        cache = torch.zeros((n_slots, H, D, D), dtype=torch.float32, device=dev)
        cache[torch.from_numpy(src.astype(np.int64)).to(dev)] = \
            torch.from_numpy(np.swapaxes(b.init_state, -1, -2).copy()).to(dev)
        q, k, v = bf16(torch, b.q, dev), bf16(torch, b.k, dev), bf16(torch, b.v, dev)
        g, beta = torch.from_numpy(b.g).to(dev), torch.from_numpy(b.beta).to(dev)
        src_t = torch.from_numpy(src).to(dev)
        o = torch.empty((rows, H, D), dtype=torch.bfloat16, device=dev)

        def call():
            gdn.gdn_decode_packed(q, k, v, g, beta, cache, src_t, o)

        def per_step_us(fn):
            for _ in range(5):
                fn()
            torch.cuda.synchronize()
            a, z = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record()
            for _ in range(iters):
                fn()
            z.record()
            torch.cuda.synchronize()
            return a.elapsed_time(z) * 1e3 / iters

        eager = per_step_us(call)
        prepared = per_step_us(gdn.prepare_decode_packed(q, k, v, g, beta, cache, src_t, o))
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph):
            call()
        replay = per_step_us(graph.replay)
        cases.append({"rows": rows, "eager_us_per_step": eager, "prepared_us_per_step": prepared,
                      "graph_us_per_step": replay,
                      "graph_rows_per_s": rows / (replay * 1e-6)})
    return {"workload": "decode_latency_h16_d128", "cases": cases}


def run_extra(torch, gdn, dev, wanted, peaks, prefix_seqlen=32768):
    extra = []
    if "prefill" in wanted:
        extra.append(prefill_case(torch, gdn, gi.prefill_qwen3next_gva(0), dev, reps=20))
    if "prefix" in wanted:
        extra.append(prefill_case(torch, gdn, gi.prefix_cache_prefill(0, seqlen=prefix_seqlen), dev, reps=20, E=17))
    if "mixed" in wanted:
        extra.append(mixed_case(torch, gdn, dev, reps=20, peaks=peaks))
    if "graph" in wanted:
        extra.append(decode_latency_case(torch, gdn, dev))
    if "multi" in wanted:
        extra.append(multi_decode_case(torch, gdn, dev, peaks))
    if "prep" in wanted:
        extra.append(prep_case(torch, gdn, dev, peaks))
    for x in extra:
        if "algorithmic_tflops" in x:
            x["roofline"] = {"bound": "tensor", "kernel": "prefill_chain_kernel<128>",
                             "achieved": x["algorithmic_tflops"], "peak": peaks["bf16_tflops"],
                             "unit": "TFLOP/s", "frac": x["algorithmic_tflops"] / peaks["bf16_tflops"],
                             "traffic": measured_traffic("prefill_chain_kernel<128>", x["workload"]),
                             "peak_source": peaks["source"] + " (dense bf16 burst; fp16 runs at the same rate)"}
    return extra


def kernel_source_hash(kernel: str) -> str:
    """Hash of the CUDA sources a kernel is built from (to tie ncu counters to it)."""
    import hashlib
    csrc = os.path.join(ROOT, "linear_attention_serving_gdn_gb300", "csrc")
    files = {"decode_kernel<128>": ["decode.cu", "row_update.cuh", "gdn_internal.cuh"],
             "prefill_chain_kernel<128>": ["prefill.cu", "tc_ptx.cuh", "gdn_internal.cuh"]}[kernel]
    h = hashlib.sha256()
    for f in files:
        h.update(open(os.path.join(csrc, f), "rb").read())
    return h.hexdigest()[:16]


def measured_traffic(kernel: str, workload: str = "decode_r256_h16_d128"):
    """DRAM bytes per launch (read + write) from the committed ncu summary,
    or None when the kernel's sources changed since the counters were taken."""
    p = os.path.join(ROOT, "profiles", "ncu_dram_traffic.json")
    if not os.path.exists(p):
        return None
    try:
        rec = json.load(open(p)).get(kernel, {}).get(workload)
    except (ValueError, AttributeError):
        return None
    if not rec or rec.get("source_hash") != kernel_source_hash(kernel):
        return None
    return rec.get("dram_bytes_per_launch")


# ---------------------------------------------------------------------------
# CPU oracle (baseline and reference arm)
# ---------------------------------------------------------------------------

def cpu_model() -> str:
    """The host CPU's model name (lscpu, else /proc/cpuinfo, else the machine type)."""
    import platform
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        for line in out.splitlines():
            if line.lower().startswith("model name"):
                return line.split(":", 1)[1].strip()
    except (OSError, subprocess.SubprocessError):
        pass
    try:
        for line in open("/proc/cpuinfo"):
            if line.lower().startswith(("model name", "hardware")):
                return line.split(":", 1)[1].strip()
    except OSError:
        pass
    return platform.machine()


def oracle_decode_rate(n_rows, n_steps, threads, seed=0):
    """Time the fp64 oracle on n_rows decode rows x n_steps tokens each (H=16,
    d=128) with `threads` OpenMP threads; returns (rows/s, seconds)."""
    import oracle
    b = gi.token_batch([n_steps] * n_rows, H, H, D, seed, init_state=True)
    t0 = time.perf_counter()
    oracle.run_chains(b, n_threads=threads)
    dt = time.perf_counter() - t0
    return n_rows * n_steps / dt, dt


def decode_steps_for(target_s, threads, rows=DECODE_ROWS):
    """Recurrent steps per row so that `rows` rows take about target_s seconds."""
    steps = 1
    while True:
        rate, dt = oracle_decode_rate(rows, steps, threads)
        if dt >= 0.25 * target_s or steps >= 1 << 14:
            return max(1, int(steps * target_s / max(dt, 1e-3)))
        steps *= 4


def oracle_prefill_rate(threads, target_s):
    """fp64 oracle on the whole 8-sequence GVA prefill (H_k=16, H_v=32,
    d=128, every value head), repeated until about target_s seconds have
    passed; returns (prefill tokens/s, seconds, tokens, repeats)."""
    import oracle
    b = gi.prefill_qwen3next_gva(0)["prefill"]
    reps, dt = 0, 0.0
    while dt < target_s:
        t0 = time.perf_counter()
        oracle.run_chains(b, n_threads=threads)
        dt += time.perf_counter() - t0
        reps += 1
    return b.total_tokens * reps / dt, dt, b.total_tokens, reps


def cpu_baseline(target_s=6.0):
    """The fp64 oracle on the host cores: decode rows/s and prefill tokens/s,
    each on all cores and on one thread, on bounded samples of the workloads."""
    import oracle
    cores = oracle.max_threads()
    nproc = os.cpu_count()
    steps = decode_steps_for(target_s, cores)
    rate_all, dt_all = oracle_decode_rate(DECODE_ROWS, steps, cores)
    rows1 = 16
    rate_1, dt_1 = oracle_decode_rate(rows1, max(1, steps // 2), 1)
    p_all, pdt_all, ptok, preps = oracle_prefill_rate(cores, 3.0)
    p_1, pdt_1, _, preps1 = oracle_prefill_rate(1, 1.0)
    return {"value": rate_all, "unit": "decode rows/s", "cores": cores, "kind": "oracle",
            "seconds": dt_all,
            "sample": f"{DECODE_ROWS} rows x {steps} recurrent steps of the 256-row decode workload "
                      f"(H=16, d=128), fp64 token recurrence, OpenMP over (row, head) chains",
            "one_thread": {"value": rate_1, "unit": "decode rows/s", "seconds": dt_1,
                           "sample": f"{rows1} rows x {max(1, steps // 2)} recurrent steps, 1 thread"},
            "prefill": {"value": p_all, "unit": "prefill tokens/s", "cores": cores, "seconds": pdt_all,
                        "sample": f"the whole 8-sequence GVA prefill ({ptok} tokens, H_k=16, H_v=32, d=128) "
                                  f"x {preps}",
                        "one_thread": {"value": p_1, "unit": "prefill tokens/s", "seconds": pdt_1,
                                       "sample": f"the same workload x {preps1}, 1 thread"}},
            "nproc": nproc, "cpu_model": cpu_model()}


DECODE_METRIC = "GDN decode rows/s (packed recurrent decode, fp32 state)"


def decode_config(n_slots, world=1):
    return {"workload": "decode_r256_h16_d128", "rows": DECODE_ROWS, "heads": H, "d_k": D, "d_v": D,
            "cache_slots": n_slots, "state_bytes": DECODE_ROWS * H * D * D * 4,
            "l2_policy": "inputs larger than L2 (256 MiB of states read+written per step)",
            "parallelism": f"replicas x{world}"}


def reference_arm(args):
    # The oracle runs on the host cores of rank 0 only; no process group or
    # GPU is needed, so the other ranks of a torchrun launch exit at once.
    # Each step is one oracle call on the same sample shape as the decode
    # cpu_baseline: all 256 rows x S recurrent steps (S sized so that a call
    # takes about a second), so the two CPU figures measure the same work.
    import oracle
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return
    threads = oracle.max_threads()
    steps = decode_steps_for(1.0, threads)
    # one sample, built once: generating it costs several times the oracle call
    b = gi.token_batch([steps] * DECODE_ROWS, H, H, D, 0, init_state=True)
    for _ in range(args.warmup):
        oracle.run_chains(b, n_threads=threads)
    times = []
    for _ in range(args.steps):
        t0 = time.perf_counter()
        oracle.run_chains(b, n_threads=threads)
        times.append(time.perf_counter() - t0)
    tot = sum(times)
    value = DECODE_ROWS * steps * args.steps / tot
    line = {"impl": "reference", "metric": DECODE_METRIC, "value": value, "unit": "rows/s",
            "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": tot / args.steps * 1e3, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": decode_config(2 * DECODE_ROWS, world),
            "cpu_baseline": {"value": value, "unit": "rows/s", "cores": threads, "kind": "oracle",
                             "sample": f"{DECODE_ROWS} rows x {steps} recurrent steps per step (H=16, d=128)",
                             "nproc": os.cpu_count(), "cpu_model": cpu_model()},
            "e2e": {"value": value, "unit": "rows/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def host_cost():
    """Host time per C-ABI call measured from C (csrc/tools/host_cost.cpp)."""
    from linear_attention_serving_gdn_gb300 import _build
    exe = _build.HOST_COST
    if not os.path.exists(exe):
        return None
    try:
        out = subprocess.run([exe, "2000"], capture_output=True, text=True, timeout=120)
        return json.loads(out.stdout.strip().splitlines()[-1])
    except (OSError, subprocess.SubprocessError, ValueError, IndexError):
        return None


# ---------------------------------------------------------------------------
# main
# ---------------------------------------------------------------------------

def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=100)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="gdn", choices=["gdn", "reference"])
    ap.add_argument("--no-extra", action="store_true", help="skip the prefill/mixed workloads")
    ap.add_argument("--workloads", default="decode,prefill,prefix,mixed,graph,multi,prep",
                    help="comma list of decode (headline), prefill, prefix, mixed, graph (decode latency), "
                         "multi (multi-token decode), prep (input preparation)")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--prefix-seqlen", type=int, default=32768,
                    help="tokens per sequence of the prefix-cache workload (smaller for profiling captures)")
    args = ap.parse_args()
    if args.warmup < 3:
        args.warmup = 3
    if args.impl == "reference":
        reference_arm(args)
        return

    import torch
    world, rank, local = dist_setup(torch)
    if not torch.cuda.is_available():
        raise SystemExit("bench.py needs a CUDA GPU")
    dev = f"cuda:{local}"
    from linear_attention_serving_gdn_gb300 import _build
    if rank == 0 or world == 1:
        _build.build()
    barrier(torch, world)
    import linear_attention_serving_gdn_gb300 as gdn
    peaks = load_peaks()

    wanted = set(args.workloads.split(","))
    if args.no_extra:
        wanted &= {"decode"}
    if "decode" not in wanted:
        extra = run_extra(torch, gdn, dev, wanted, load_peaks(), args.prefix_seqlen)
        if rank == 0:
            print(json.dumps({"metric": "GDN prefill tokens/s", "workloads": extra}), flush=True)
        return
    wl, t = decode_setup(torch, seed=rank, dev=dev)
    with Clocks(torch.cuda.current_device()) as clk:
        total_ms, per_launch = time_decode(torch, gdn, t, args.steps, args.warmup, world)
    clocks = clk.summary()
    total_ms = max_over_ranks(torch, world, total_ms)
    e2e_ms, h2d, d2h = time_decode_e2e(torch, gdn, t, args.steps, args.warmup, world, parts=E2E_PARTS)
    e2e_ms = max_over_ranks(torch, world, e2e_ms)
    e2e_serial_ms, _, _ = time_decode_e2e(torch, gdn, t, args.steps, args.warmup, world, parts=1)
    e2e_serial_ms = max_over_ranks(torch, world, e2e_serial_ms)
    e2e_eager_ms, _, _ = time_decode_e2e_eager(torch, gdn, t, args.steps, args.warmup, world)
    e2e_eager_ms = max_over_ranks(torch, world, e2e_eager_ms)

    rows_total = DECODE_ROWS * args.steps * world
    value = rows_total / (total_ms * 1e-3)
    launch_ms = statistics.mean(per_launch)
    bytes_per_launch = DECODE_BYTES_PER_ROW * DECODE_ROWS
    achieved = bytes_per_launch / (launch_ms * 1e-3) / 1e9
    line = {
        "metric": DECODE_METRIC,
        "value": value, "unit": "rows/s", "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": total_ms / args.steps, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f32 state / bf16 activations", "data": "synthetic",
        "config": decode_config(wl["n_slots"], world),
        "roofline": {"bound": "hbm", "kernel": "decode_kernel<128>", "achieved": achieved,
                     "peak": peaks["hbm_gbs"], "unit": "GB/s", "frac": achieved / peaks["hbm_gbs"],
                     "traffic": measured_traffic("decode_kernel<128>"),
                     "peak_source": peaks["source"] + " (burst copy)",
                     "bytes_per_launch": bytes_per_launch, "launch_ms": launch_ms},
        "e2e": {"value": rows_total / (e2e_ms * 1e-3), "unit": "rows/s", "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h,
                "mode": f"one CUDA-graph replay per step; the 256 rows in {E2E_PARTS} groups, each [H2D of its "
                        "packed inputs on an input stream, gdn_decode_packed, D2H of its o on an output stream], "
                        "so one group's copies overlap another's decode",
                "serial_value": rows_total / (e2e_serial_ms * 1e-3),
                "serial_mode": "one CUDA-graph replay per step of [H2D packed inputs, gdn_decode_packed, D2H o]",
                "eager_value": rows_total / (e2e_eager_ms * 1e-3),
                "eager_mode": "the same step issued from Python: H2D, decode, D2H on one stream"},
        "gpu_launches": args.steps,
        "clocks": clocks,
    }
    if wanted - {"decode"}:
        line["workloads"] = run_extra(torch, gdn, dev, wanted, peaks, args.prefix_seqlen)
    if rank == 0:
        line["host_us_per_call"] = host_cost()
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline()
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
