"""Prefix-cache grid rules.  TEST INFRASTRUCTURE.

The vLLM page "Enable GDN batch-invariant prefix caching" (section
"Purpose") puts prefill chunks and prefix-cache hits on one shared grid,
lcm(64, block size): the hybrid block size is rounded up to a multiple of the
64-token chunk (1056 becomes 1088), a prefix hit is floored onto the grid,
and a hit that covers the full prompt is not floored.  Its "Test Result"
section gives the worked values (1100 -> 1088, 200 -> 0).
"""
from __future__ import annotations

import math

CHUNK = 64


def align_block_size(block_size: int, chunk: int = CHUNK) -> int:
    """Round the cache block size up to a multiple of the chunk size."""
    if block_size <= 0:
        raise ValueError("block size must be positive")
    return -(-block_size // chunk) * chunk


def grid_tokens(block_size: int, chunk: int = CHUNK) -> int:
    """lcm(chunk, aligned block size)."""
    return math.lcm(chunk, align_block_size(block_size, chunk))


def floor_hit(hit_tokens: int, prompt_tokens: int, block_size: int, chunk: int = CHUNK) -> int:
    """Usable prefix-cache hit: floored onto the grid unless it is the full prompt."""
    if hit_tokens < 0 or hit_tokens > prompt_tokens:
        raise ValueError("hit must lie in [0, prompt]")
    if hit_tokens == prompt_tokens:
        return hit_tokens
    gr = grid_tokens(block_size, chunk)
    return (hit_tokens // gr) * gr
