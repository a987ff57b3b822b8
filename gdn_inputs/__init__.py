"""Seeded synthetic inputs for the Gated DeltaNet hot path.

This module is shared by the oracle (``oracle/``) and by the CUDA path's tests
and benchmark.  It draws random numbers and rounds them to the storage types;
it holds none of the recurrence's arithmetic.

Recipe (the workloads of the vLLM GDN pages, "Enable batch-invariant mixed
decode and prefill for Qwen GDN" section "Online serving validation" for the
116/321/1,059-token prompt classes, and "Enable GDN batch-invariant prefix
caching" section "Test Result" for the 2000-token prefix and 1088-token
blocks):

* q, k ~ N(0, 1) drawn in fp32, L2-normalised over the head dimension in fp32,
  then rounded to bf16 (round to nearest even);
* v ~ N(0, 1), rounded to bf16;
* g = -softplus(N(0, 1)) * 0.1 (fp32), so alpha = exp(g) lies in (0, 1);
* beta = sigmoid(N(0, 1)) (fp32);
* cached recurrent states ~ N(0, 0.1**2) in fp32 (std 0.1), in the
  mathematical orientation S[d_k][d_v];
* cache slots are a seeded random permutation of a cache with twice as many
  slots as rows.

Every array comes from ``numpy.random.Generator(PCG64(seed))`` drawn in a
fixed order, so both sides of a parity test see identical inputs.
bf16 tensors are returned as their uint16 bit patterns.
"""
from __future__ import annotations

from dataclasses import dataclass, field

import numpy as np

CHUNK = 64

# Prompt-length classes of the pages' workloads.
PROMPT_CLASSES = (116, 321, 1059, 2000)


def bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round fp32 values to bf16 (nearest, ties to even); return uint16 bits."""
    x = np.ascontiguousarray(x, dtype=np.float32)
    u = x.view(np.uint32).astype(np.uint64)
    lsb = (u >> 16) & 1
    r = ((u + 0x7FFF + lsb) >> 16).astype(np.uint16)
    nan = np.isnan(x)
    if nan.any():
        r[nan] = 0x7FC0
    return r


def bf16_to_f32(bits: np.ndarray) -> np.ndarray:
    """Exact widening of bf16 bit patterns to fp32."""
    b = np.ascontiguousarray(bits, dtype=np.uint16)
    return (b.astype(np.uint32) << 16).view(np.float32)


def _normal(rng: np.random.Generator, shape) -> np.ndarray:
    return rng.standard_normal(size=shape, dtype=np.float32)


def _unit_rows_bf16(x: np.ndarray) -> np.ndarray:
    n = np.sqrt(np.sum(x * x, axis=-1, keepdims=True, dtype=np.float32))
    return bf16_bits(x / n)


def _gates(rng: np.random.Generator, shape):
    z = _normal(rng, shape)
    g = (-np.logaddexp(np.float32(0.0), z) * np.float32(0.1)).astype(np.float32)
    zb = _normal(rng, shape)
    beta = (np.float32(1.0) / (np.float32(1.0) + np.exp(-zb))).astype(np.float32)
    return g, beta


@dataclass
class TokenBatch:
    """Packed varlen token batch (decode rows are sequences of length 1).

    q, k: uint16 bf16 bits [T][h_k][d]; v: [T][h_v][d];
    g, beta: fp32 [T][h_v]; cu_seqlens: int32 [n_seq + 1];
    init_state: fp32 [n_seq][h_v][d_k][d_v] (math orientation) or None for
    zero initial states.
    """

    h_k: int
    h_v: int
    d: int
    cu_seqlens: np.ndarray
    q: np.ndarray
    k: np.ndarray
    v: np.ndarray
    g: np.ndarray
    beta: np.ndarray
    init_state: np.ndarray | None = None
    meta: dict = field(default_factory=dict)

    @property
    def num_seqs(self) -> int:
        return len(self.cu_seqlens) - 1

    @property
    def total_tokens(self) -> int:
        return int(self.cu_seqlens[-1])

    @property
    def seqlens(self) -> list[int]:
        c = self.cu_seqlens
        return [int(c[i + 1] - c[i]) for i in range(len(c) - 1)]


def token_batch(seqlens, h_k: int, h_v: int, d: int, seed: int,
                init_state: bool = False, state_std: float = 0.1) -> TokenBatch:
    """Draw a packed batch of sequences with the recipe above."""
    seqlens = [int(x) for x in seqlens]
    rng = np.random.Generator(np.random.PCG64(seed))
    T = sum(seqlens)
    cu = np.zeros(len(seqlens) + 1, dtype=np.int32)
    cu[1:] = np.cumsum(seqlens)
    q = _unit_rows_bf16(_normal(rng, (T, h_k, d)))
    k = _unit_rows_bf16(_normal(rng, (T, h_k, d)))
    v = bf16_bits(_normal(rng, (T, h_v, d)))
    g, beta = _gates(rng, (T, h_v))
    s0 = None
    if init_state:
        s0 = (_normal(rng, (len(seqlens), h_v, d, d)) * np.float32(state_std)).astype(np.float32)
    return TokenBatch(h_k, h_v, d, cu, q, k, v, g, beta, s0,
                      meta={"seed": seed, "seqlens": seqlens})


def slots(n_rows: int, seed: int, n_slots: int | None = None) -> tuple[np.ndarray, int]:
    """Seeded random slot assignment in a cache of ``n_slots`` (default 2x rows)."""
    n_slots = 2 * n_rows if n_slots is None else n_slots
    rng = np.random.Generator(np.random.PCG64(seed + 7919))
    perm = rng.permutation(n_slots).astype(np.int32)
    return perm[:n_rows].copy(), n_slots


def draw_prompt_lengths(n: int, seed: int, classes=PROMPT_CLASSES) -> list[int]:
    """Seeded uniform draw of ``n`` prompt lengths from ``classes``."""
    rng = np.random.Generator(np.random.PCG64(seed + 104729))
    idx = rng.integers(0, len(classes), size=n)
    return [int(classes[i]) for i in idx]


# ---------------------------------------------------------------------------
# The five workloads, by what they are.
# ---------------------------------------------------------------------------

def tiny_mixed(seed: int = 0) -> dict:
    """Tiny correctness case: H=4, d=64; prefills of 64 and 100 tokens (zero
    initial state) plus 2 cached decode rows (state std 0.1)."""
    dec = token_batch([1, 1], 4, 4, 64, seed, init_state=True)
    pre = token_batch([64, 100], 4, 4, 64, seed + 1, init_state=False)
    return {"name": "tiny_h4_d64_mixed", "decode": dec, "prefill": pre}


def decode_qwen35_08b(seed: int = 0, rows: int = 256) -> dict:
    """Packed recurrent decode of a Qwen3.5-0.8B-like GDN layer: 256 rows,
    H=16, d=128, fp32 states in a slot-indexed cache of 2x rows."""
    b = token_batch([1] * rows, 16, 16, 128, seed, init_state=True)
    src, n_slots = slots(rows, seed)
    return {"name": "decode_r256_h16_d128", "decode": b, "src_slot": src,
            "n_slots": n_slots}


def prefill_qwen3next_gva(seed: int = 0, n_seq: int = 8) -> dict:
    """Chunked varlen prefill, Qwen3-Next-like GVA layer: H_k=16, H_v=32,
    d=128; 8 sequences with lengths drawn from {116, 321, 1059, 2000}."""
    lens = draw_prompt_lengths(n_seq, seed)
    b = token_batch(lens, 16, 32, 128, seed, init_state=False)
    return {"name": "prefill_gva_hk16_hv32_d128_8seq", "prefill": b}


def mixed_step(seed: int = 0, n_dec: int = 64, prefill_lens=PROMPT_CLASSES) -> dict:
    """Mixed continuous-batching step: 64 cached decode rows at the front plus
    fresh prefills of lengths {116, 321, 1059, 2000}; H=16, d=128."""
    dec = token_batch([1] * n_dec, 16, 16, 128, seed, init_state=True)
    pre = token_batch(list(prefill_lens), 16, 16, 128, seed + 1, init_state=False)
    src, n_slots = slots(n_dec + len(prefill_lens), seed)
    return {"name": "mixed_d64rows_p4_h16_d128", "decode": dec, "prefill": pre,
            "src_slot": src, "n_slots": n_slots}


def prefix_cache_prefill(seed: int = 0, n_seq: int = 4, seqlen: int = 32768) -> dict:
    """Prefix-cache prefill with state emission on the 1088-token block grid:
    4 sequences of 32768 tokens, H_k=16, H_v=32, d=128, E=17 chunks."""
    b = token_batch([seqlen] * n_seq, 16, 32, 128, seed, init_state=False)
    return {"name": f"prefix_cache_{n_seq}x{seqlen}_hk16_hv32_d128_E17", "prefill": b,
            "emit_every_chunks": 17}


@dataclass
class RawInputs:
    """Raw per-token projections ahead of the layer's input preparation:
    q, k un-normalised (bf16 bits), a and b (fp32, [T][h_v]) from which the
    decay and the write strength are formed, and the per-head parameters
    A_log and dt_bias (fp32, [h_v])."""
    h_k: int
    h_v: int
    d: int
    q: np.ndarray
    k: np.ndarray
    v: np.ndarray
    a: np.ndarray
    b: np.ndarray
    A_log: np.ndarray
    dt_bias: np.ndarray


def raw_inputs(n_tokens: int, h_k: int, h_v: int, d: int, seed: int) -> RawInputs:
    """q, k ~ N(0, 1) times a per-row scale drawn log-uniform in [0.25, 4]
    (so normalisation matters), v ~ N(0, 1), all rounded to bf16; a, b ~
    N(0, 1); A_log ~ log U(0.02, 0.2); dt_bias ~ N(0, 0.5**2)."""
    rng = np.random.default_rng(np.random.PCG64(seed + 271828))
    q = _normal(rng, (n_tokens, h_k, d)) * np.exp2(rng.uniform(-2, 2, (n_tokens, h_k, 1))).astype(np.float32)
    k = _normal(rng, (n_tokens, h_k, d)) * np.exp2(rng.uniform(-2, 2, (n_tokens, h_k, 1))).astype(np.float32)
    v = _normal(rng, (n_tokens, h_v, d))
    a = _normal(rng, (n_tokens, h_v))
    b = _normal(rng, (n_tokens, h_v))
    A_log = np.log(rng.uniform(0.02, 0.2, h_v)).astype(np.float32)
    dt_bias = (0.5 * _normal(rng, (h_v,))).astype(np.float32)
    return RawInputs(h_k, h_v, d, bf16_bits(q), bf16_bits(k), bf16_bits(v), a, b, A_log, dt_bias)
