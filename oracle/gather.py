"""KV-cache compaction to the accepted path (oracle; test infrastructure only).

Definitions (mlxcel issue #1204, "The rollback constraint, which decides
feasibility": a chain rolls back by trimming the tail, trim = block_size - n
with n = max(accepted) + 1, correct only because a linear accept set is a
prefix; PR #1212's gather_positions commit: select and compact scattered
positions on the sequence axis, Int8 scale sidecars move with their tokens,
a prefix selection equals trim_to and the identity selection short-circuits;
PR #1212's gather_within_tail commit: offsets within the verify block, only
[tail_start, tail_start + kept_len) is rewritten and the allocation survives).

Reading: rows at and beyond the new length keep whatever bytes they held
(the in-place tail rewrite leaves them; the next append overwrites them).
Arrays here are [..., N, ...] with the sequence on ``axis``.
"""
from __future__ import annotations

import numpy as np


def trim_to(buf, length: int, axis: int = 0):
    """The chain rollback: keep the first ``length`` positions."""
    return np.take(np.asarray(buf), np.arange(length), axis=axis)


def gather_positions(buf, kept, axis: int = 0):
    """Absolute form: new sequence = old positions ``kept`` (strictly increasing), in order."""
    kept = [int(k) for k in kept]
    assert all(a < b for a, b in zip(kept, kept[1:])), "kept must be strictly increasing"
    return np.take(np.asarray(buf), kept, axis=axis)


def gather_within_tail(buf, tail_start: int, kept_offsets, axis: int = 0):
    """In-place tail form: rows tail_start + j <- rows tail_start + kept[j]; others unchanged.

    Returns (new buffer, new length = tail_start + len(kept)).
    """
    b = np.array(buf, copy=True)
    src = np.take(np.asarray(buf), [tail_start + int(k) for k in kept_offsets], axis=axis)
    idx = [slice(None)] * b.ndim
    idx[axis] = slice(tail_start, tail_start + len(kept_offsets))
    b[tuple(idx)] = src
    return b, tail_start + len(kept_offsets)


def is_identity(kept_offsets) -> bool:
    """True when every kept offset is already in place (no data moves)."""
    return all(int(k) == j for j, k in enumerate(kept_offsets))
