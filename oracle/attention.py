"""Tree-masked GQA attention of the verify block (oracle; test infrastructure only).

Definition (mlxcel issue #1204, "What this needs" item 1 and "Increment 3";
PR #1212, history-mask and verify_forward_with_mask commits; Splash issue #728,
"Earlier shader evidence", 16 nodes x 24 heads x D256 over histories 0-8192):
the T tree nodes were appended to the cache in topological order at positions
[S, S + T).  Query row (node i, head h) attends to every history position
c < S and to the block positions S + j for j an ancestor of i or i itself;
softmax over those keys of (q . k) / sqrt(D), output sum_c p_c v_c.

Readings where the pages are silent: the score scale is 1/sqrt(D) with no
soft-cap and no attention sinks; query head h reads KV head floor(h / G) with
G = HQ / HKV.  The softmax subtracts the row maximum (the value is the same
mathematically; fp64 keeps it exact enough to be the reference).
"""
from __future__ import annotations

import math

import numpy as np

from . import tree as _tree


def attend_row(q, K, V, S: int, visible_nodes) -> np.ndarray:
    """One query row.  q [D]; K, V [S + T, D] fp64 values of the sequence's cache.

    visible_nodes: the tree nodes whose block entries the row may see.
    """
    cols = list(range(S)) + [S + j for j in sorted(visible_nodes)]
    k = K[cols]
    v = V[cols]
    s = (k @ np.asarray(q, dtype=np.float64)) / math.sqrt(K.shape[1])
    s = s - s.max()
    p = np.exp(s)
    return (p / p.sum()) @ v


def attend_dense_mask(q, K, V, mask_row) -> np.ndarray:
    """The same row through an additive mask over all S + T columns (-1e9 blocks)."""
    s = (K @ np.asarray(q, dtype=np.float64)) / math.sqrt(K.shape[1]) + mask_row
    s = s - s.max()
    p = np.exp(s)
    return (p / p.sum()) @ V


def attend_cols(q, K, V, cols) -> np.ndarray:
    """One query row over an explicit list of cache positions."""
    k = K[cols]
    v = V[cols]
    s = (k @ np.asarray(q, dtype=np.float64)) / math.sqrt(K.shape[1])
    s = s - s.max()
    p = np.exp(s)
    return (p / p.sum()) @ v


def tree_verify_attention(q, K, V, parents, S: int, window: int = 0) -> np.ndarray:
    """All rows of one (sequence, layer).  q [T, HQ, D]; K, V [HKV, S + T, D] -> [T, HQ, D].

    window > 0: a sliding-window layer; node i (at position S + i) sees only the keys of its tree mask that lie
    inside its band, positions > S + i - window (PR #1212, caller masks and the sliding-window band).
    """
    T, HQ, D = q.shape
    HKV = K.shape[0]
    G = HQ // HKV
    out = np.zeros((T, HQ, D), dtype=np.float64)
    for i in range(T):
        if window == 0:
            vis = _tree.ancestors(parents, i)
        cols = _tree.visible_keys(parents, i, S, window)
        for h in range(HQ):
            kv = h // G
            if window == 0:
                out[i, h] = attend_row(q[i, h], K[kv], V[kv], S, vis)
            else:
                out[i, h] = attend_cols(q[i, h], K[kv], V[kv], cols)
    return out
