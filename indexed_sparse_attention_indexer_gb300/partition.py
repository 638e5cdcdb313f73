"""Splitting a causal prefill's query rows over several GPUs.

("Day 0 Inference Support for New LLM Architectures: Optimization Practices",
"Load Imbalance in Causal Indexing and the Zigzag Layout"; "Day 0 Inference
Adaptation and Performance Optimization for New Models" §5.)  Under causal
indexing a late query token scores far more history than an early one, so
equal contiguous row ranges give the last rank most of the work.  The zigzag
layout cuts the rows into 2N equal segments and gives rank r segments r and
2N-1-r: an early and a late segment, whose causal work adds up to the same
amount on every rank.

Each rank then runs the fused layer on its two segments (two calls, query
offsets at the segments' starts) over the whole causal history of the
sequence, which every rank holds (replicated here: every rank builds the same
seeded cache).  Outputs stay on their rank; ``rank_rows`` maps them back.
Host logic only: nothing here touches a GPU or another rank.
"""
from __future__ import annotations

from typing import List, Tuple


def zigzag_segments(T: int, world: int) -> List[List[Tuple[int, int]]]:
    """Per rank, its [start, end) row ranges: 2*world near-equal segments,
    rank r taking segments r and 2*world-1-r (an empty segment is dropped)."""
    if world < 1 or T < 0:
        raise ValueError("world >= 1 and T >= 0")
    n = 2 * world
    bounds = [T * i // n for i in range(n + 1)]
    seg = [(bounds[i], bounds[i + 1]) for i in range(n)]
    out = []
    for r in range(world):
        mine = [seg[r], seg[n - 1 - r]]
        out.append([s for s in mine if s[1] > s[0]])
    return out


def rank_rows(T: int, world: int, rank: int) -> List[int]:
    """Query rows of one rank, in the order its outputs are produced."""
    return [t for a, b in zigzag_segments(T, world)[rank] for t in range(a, b)]


def causal_pairs(segments, q_offset: int = 0) -> int:
    """(query, visible position) pairs of the given row ranges: the indexer's
    work, row t seeing q_offset + t + 1 positions."""
    tot = 0
    for a, b in segments:
        # sum over t in [a, b) of (q_offset + t + 1)
        tot += (b - a) * (q_offset + 1) + (a + b - 1) * (b - a) // 2
    return tot


def contiguous_segments(T: int, world: int) -> List[List[Tuple[int, int]]]:
    """Equal contiguous ranges (the unbalanced split, for comparison)."""
    bounds = [T * i // world for i in range(world + 1)]
    return [[(bounds[r], bounds[r + 1])] for r in range(world)]
