"""Helpers for the GPU tests: move seeded inputs to the device and compare
the CUDA path's results with the oracle's.

Tolerances (fixed for this hot path): bf16 outputs within max |err| <= 2e-2
absolute of the fp64 oracle; fp32 states within 1e-3 relative Frobenius
error over the whole state tensor of a workload.
"""
from __future__ import annotations

import numpy as np
import torch

import gdn_inputs as gi

O_ATOL = 2e-2
STATE_RTOL = 1e-3


def bf16_tensor(bits: np.ndarray, device="cuda") -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16).to(device)


def batch_to_device(b: gi.TokenBatch, device="cuda") -> dict:
    return {
        "q": bf16_tensor(b.q, device), "k": bf16_tensor(b.k, device), "v": bf16_tensor(b.v, device),
        "g": torch.from_numpy(b.g).to(device), "beta": torch.from_numpy(b.beta).to(device),
        "cu": torch.from_numpy(b.cu_seqlens.astype(np.int32)).to(device),
        "cu_host": [int(x) for x in b.cu_seqlens],
    }


def concat_batches(a: gi.TokenBatch, b: gi.TokenBatch) -> dict:
    """Token-major concatenation of two batches (decode rows first)."""
    return {
        "q": np.concatenate([a.q, b.q]), "k": np.concatenate([a.k, b.k]),
        "v": np.concatenate([a.v, b.v]), "g": np.concatenate([a.g, b.g]),
        "beta": np.concatenate([a.beta, b.beta]),
    }


def arrays_to_device(d: dict, device="cuda") -> dict:
    out = {}
    for name in ("q", "k", "v"):
        out[name] = bf16_tensor(d[name], device)
    for name in ("g", "beta"):
        out[name] = torch.from_numpy(np.ascontiguousarray(d[name])).to(device)
    return out


def empty_cache(n_slots: int, h_v: int, d: int, device="cuda") -> torch.Tensor:
    return torch.zeros((n_slots, h_v, d, d), dtype=torch.float32, device=device)


def put_states(cache: torch.Tensor, slots, states_math: np.ndarray) -> None:
    """Write states given as S [n][h][d_k][d_v] into the S^T cache at slots."""
    st = torch.from_numpy(np.ascontiguousarray(np.swapaxes(states_math, -1, -2)))
    cache[torch.as_tensor(np.asarray(slots, np.int64), device=cache.device)] = st.to(cache.device)


def get_states_math(cache: torch.Tensor, slots) -> np.ndarray:
    """Read states at slots back as S [n][h][d_k][d_v] (fp64)."""
    st = cache[torch.as_tensor(np.asarray(slots, np.int64), device=cache.device)].cpu().numpy()
    return np.swapaxes(st, -1, -2).astype(np.float64)


def o_to_numpy(o: torch.Tensor) -> np.ndarray:
    return o.float().cpu().numpy().astype(np.float64)


def o_ref_dense(batch: gi.TokenBatch, res: dict) -> np.ndarray:
    """Scatter the oracle's per-pair outputs into [T][h_v][d_v]."""
    out = np.zeros((batch.total_tokens, batch.h_v, batch.d))
    for (s, h), o in zip(res["pairs"], res["o"]):
        t0 = int(batch.cu_seqlens[s])
        out[t0:t0 + o.shape[0], h] = o
    return out


def state_rel_frob(got: np.ndarray, ref: np.ndarray) -> float:
    n = np.linalg.norm(ref)
    return float(np.linalg.norm(got - ref) / (n if n > 0 else 1.0))


def assert_o_close(got: np.ndarray, ref: np.ndarray, what: str = "o") -> float:
    err = float(np.max(np.abs(got - ref))) if got.size else 0.0
    assert np.isfinite(got).all(), f"{what}: non-finite values"
    assert err <= O_ATOL, f"{what}: max |err| {err:.3e} > {O_ATOL} (max |ref| {np.max(np.abs(ref)):.3f})"
    return err


def assert_state_close(got: np.ndarray, ref: np.ndarray, what: str = "state") -> float:
    assert np.isfinite(got).all(), f"{what}: non-finite values"
    rel = state_rel_frob(got, ref)
    assert rel <= STATE_RTOL, f"{what}: rel Frobenius {rel:.3e} > {STATE_RTOL}"
    return rel
