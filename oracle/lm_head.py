"""LM-head projection with greedy argmax (oracle; test infrastructure only).

Definition (mlxcel issue #1185, "Phase 2: stop paying the full-vocab LM head",
2a: at temperature 0 the logits are only needed for their argmax, so a fused
projection + argmax never writes them; issue #1204 "What this needs" item 2:
the target emits one argmax per position): logits[r, v] = sum_k W[v, k] h[r, k]
in fp64 with W and h exact; argmax with ties to the lowest index (our reading).
The top-1 minus top-2 logit gap is reported so callers can tell where the
argmax is well defined at a given precision.
"""
from __future__ import annotations

import numpy as np

CHUNK_ROWS = 16384


def logits(W, h) -> np.ndarray:
    """fp64 logits [R, V] = h [R, H] @ W[V, H]^T."""
    return np.asarray(h, dtype=np.float64) @ np.asarray(W, dtype=np.float64).T


def argmax_gap(lg):
    """(argmax with ties to the lowest index, top-1 value, top-1 minus top-2) per row."""
    lg = np.atleast_2d(np.asarray(lg, dtype=np.float64))
    idx = np.argmax(lg, axis=1)  # first occurrence of the maximum
    top = lg[np.arange(lg.shape[0]), idx]
    rest = lg.copy()
    rest[np.arange(lg.shape[0]), idx] = -np.inf
    second = rest.max(axis=1) if lg.shape[1] > 1 else np.full(lg.shape[0], -np.inf)
    return idx.astype(np.int64), top, top - second


def argmax_streamed(weight_rows, h, V: int):
    """Argmax over V rows produced chunk by chunk by ``weight_rows(r0, r1) -> fp64 [r1-r0, H]``.

    Same definition as ``argmax_gap(logits(W, h))``, for heads too large to hold in fp64.
    Returns (argmax, top-1 value, gap) per row of h.
    """
    h = np.atleast_2d(np.asarray(h, dtype=np.float64))
    R = h.shape[0]
    best = np.full(R, -np.inf)
    second = np.full(R, -np.inf)
    arg = np.zeros(R, dtype=np.int64)
    for r0 in range(0, V, CHUNK_ROWS):
        r1 = min(V, r0 + CHUNK_ROWS)
        lg = h @ weight_rows(r0, r1).T  # [R, chunk]
        ci, ctop, cgap = argmax_gap(lg)
        csec = ctop - cgap
        for r in range(R):
            if ctop[r] > best[r]:  # strictly greater: an earlier chunk keeps ties
                second[r] = max(best[r], csec[r])
                best[r] = ctop[r]
                arg[r] = r0 + ci[r]
            else:
                second[r] = max(second[r], ctop[r])
    return arg, best, best - second


def logits_streamed(weight_rows, h, V: int) -> np.ndarray:
    """All fp64 logits [R, V], the head produced chunk by chunk by ``weight_rows(r0, r1)``."""
    h = np.atleast_2d(np.asarray(h, dtype=np.float64))
    return np.concatenate([h @ weight_rows(r0, min(V, r0 + CHUNK_ROWS)).T for r0 in range(0, V, CHUNK_ROWS)], axis=1)
