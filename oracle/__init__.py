"""fp64 CPU oracle for the Gated DeltaNet hot path.  TEST INFRASTRUCTURE.

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU arms of
``bench.py`` may import this package.  It shares no code with the CUDA path
and never imports it; inputs come from ``gdn_inputs``.

Contents
--------
* :func:`run_chains` -- the token-by-token gated delta rule in fp64
  (``gdn_oracle.c``), per (sequence, value head) chain.
* :mod:`oracle.chunked` -- an independent fp64 chunked (UT / WY) form of the
  same recurrence, used only to check the token oracle.
* :mod:`oracle.exact_tiny` -- exact rational brute force for tiny cases.
* :mod:`oracle.grid` -- the prefix-cache grid rules (block size rounded up to
  the 64-token chunk grid, cache hits floored onto it).

Pins (tests/test_oracle_pins.py) tie each of these to closed forms,
invariants, library routines and hand-derived worked examples.
"""
from __future__ import annotations

import ctypes
import os

import numpy as np

from . import build as _build

_lib = None


def load() -> ctypes.CDLL:
    global _lib
    if _lib is None:
        path = _build.build()
        lib = ctypes.CDLL(path)
        lib.gdn_oracle_chains.restype = ctypes.c_int
        lib.gdn_oracle_chains.argtypes = [
            ctypes.c_int, ctypes.c_void_p, ctypes.c_void_p,
            ctypes.c_int, ctypes.c_void_p, ctypes.c_int, ctypes.c_int,
            ctypes.c_int, ctypes.c_int, ctypes.c_double,
            ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p,
            ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p,
            ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int64, ctypes.c_void_p,
            ctypes.c_int,
        ]
        lib.gdn_oracle_max_threads.restype = ctypes.c_int
        _lib = lib
    return _lib


def max_threads() -> int:
    return int(load().gdn_oracle_max_threads())


def _ptr(a):
    return None if a is None else a.ctypes.data


def run_chains(batch, pairs=None, scale: float = 1.0, init_state=None,
               emit_every: int = 0, n_threads: int = 0) -> dict:
    """Run the fp64 token recurrence on the requested (seq, v-head) chains.

    ``batch`` is a :class:`gdn_inputs.TokenBatch`.  ``pairs`` is a list of
    (seq, head); default: every chain.  ``init_state`` overrides
    ``batch.init_state`` with a [n_pairs][d_k][d_v] array, widened exactly to
    fp64 (None with no batch state means zero).  ``emit_every`` is in tokens.

    Returns ``{"o": [array [T_seq][d_v] per pair], "s_final": [n_pairs][d_k][d_v],
    "emits": [array [n_emit][d_k][d_v] per pair], "pairs": pairs}``, fp64.
    """
    lib = load()
    n_seq = batch.num_seqs
    if pairs is None:
        pairs = [(s, h) for s in range(n_seq) for h in range(batch.h_v)]
    pairs = [(int(s), int(h)) for s, h in pairs]
    n = len(pairs)
    d_k = d_v = batch.d
    ps = np.array([p[0] for p in pairs], dtype=np.int32)
    ph = np.array([p[1] for p in pairs], dtype=np.int32)
    cu = batch.cu_seqlens.astype(np.int64)
    if init_state is None and batch.init_state is not None:
        init_state = np.stack([batch.init_state[s, h] for s, h in pairs]) if n else None
    s0 = None
    if init_state is not None:
        s0 = np.ascontiguousarray(init_state, dtype=np.float64).reshape(n, d_k, d_v)
    lens = [int(cu[s + 1] - cu[s]) for s, _ in pairs]
    o = np.zeros((sum(lens), d_v), dtype=np.float64)
    s_final = np.zeros((n, d_k, d_v), dtype=np.float64)
    n_emit = [(L // emit_every) if emit_every > 0 else 0 for L in lens]
    emits = np.zeros((max(sum(n_emit), 1), d_k, d_v), dtype=np.float64)
    q = np.ascontiguousarray(batch.q)
    k = np.ascontiguousarray(batch.k)
    v = np.ascontiguousarray(batch.v)
    g = np.ascontiguousarray(batch.g, dtype=np.float32)
    beta = np.ascontiguousarray(batch.beta, dtype=np.float32)
    rc = lib.gdn_oracle_chains(
        n, _ptr(ps), _ptr(ph), n_seq, _ptr(cu), batch.h_k, batch.h_v, d_k, d_v,
        float(scale), _ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(beta), _ptr(s0),
        _ptr(o), _ptr(s_final), int(emit_every), _ptr(emits), int(n_threads))
    if rc != 0:
        raise ValueError("gdn_oracle_chains rejected its arguments")
    o_list, e_list = [], []
    oo = eo = 0
    for L, ne in zip(lens, n_emit):
        o_list.append(o[oo:oo + L])
        e_list.append(emits[eo:eo + ne])
        oo += L
        eo += ne
    return {"o": o_list, "s_final": s_final, "emits": e_list, "pairs": pairs}
