"""Draft-tree topology, ancestor mask and accept walk (oracle; test infrastructure only).

Definitions followed:

* Topology - mlxcel issue #1204, "Increment 1 landed on a branch: topology,
  mask, walk", and PR #1212's first commit: nodes in topological order with
  parents[i] < i.  Node 0 is the root, the token already committed before the
  round (our reading: its entry in the verify block is always kept, its token
  is never compared, and the accepted path starts at it).
* Mask - issue #1204, "What this needs" item 1: each node attends to its
  ancestors only (and itself), never to a sibling.  PR #1212's history-mask
  commit: the mask is [n, offset + n]; query row q sits at logical position
  q + offset, the first ``offset`` columns (the cached history) are attended in
  full by every node, and the last n follow the tree.  PR #1212's verify
  commit: blocked entries hold -1e9, not -inf.
* Sliding-window layers - PR #1212, the commit on caller masks and the
  sliding-window band: such a layer attends the intersection of the caller's
  (tree) mask and its band; the band of query q (at position offset + q) keeps
  the window positions ending at the query, so every row keeps itself.
* Walk - issue #1204, "What this needs" item 2, and PR #1212's first commit:
  descend the branch the target agreed with; the accepted set is a path, never
  a subtree.  Reading for two siblings that both match: the one with the lower
  index is taken (scan in ascending index order).  Splash issue #728, "What it
  does": every committed token is the target's selection at its path node, so
  emitted = [argmax[p] for p in path] and there are accepted + 1 of them.
"""
from __future__ import annotations

import numpy as np

BLOCKED = -1e9

# Validation results (mirrors of the device status codes are in the C header;
# the oracle only needs "valid" and "why not").
OK, BAD_ROOT, BAD_PARENT = 0, 1, 2


def validate(parents) -> int:
    """0 if ``parents`` is a topological tree: parents[0] == -1 and 0 <= parents[i] < i."""
    parents = [int(p) for p in parents]
    if len(parents) == 0:
        return OK
    if parents[0] != -1:
        return BAD_ROOT
    for i in range(1, len(parents)):
        if not (0 <= parents[i] < i):
            return BAD_PARENT
    return OK


def ancestors(parents, i: int) -> set:
    """anc(i) = {i} union anc(parents[i]), by chasing parents up to the root."""
    out = set()
    node = int(i)
    while node >= 0:
        out.add(node)
        node = int(parents[node])
    return out


def depth(parents, i: int) -> int:
    return len(ancestors(parents, i)) - 1


def ancestor_bits(parents) -> list[int]:
    """Per node, an integer whose bit j is set iff j is an ancestor of the node or the node."""
    return [sum(1 << j for j in ancestors(parents, i)) for i in range(len(parents))]


def tree_mask(parents) -> np.ndarray:
    """The [n, n] additive mask: 0 where column j is an ancestor-or-self of row i, else -1e9."""
    n = len(parents)
    m = np.full((n, n), BLOCKED, dtype=np.float64)
    for i in range(n):
        for j in ancestors(parents, i):
            m[i, j] = 0.0
    return m


def history_mask(parents, offset: int) -> np.ndarray:
    """The [n, offset + n] additive mask: history columns all 0, block columns as tree_mask."""
    n = len(parents)
    m = np.zeros((n, offset + n), dtype=np.float64)
    m[:, offset:] = tree_mask(parents)
    return m


def sliding_band(n: int, offset: int, window: int) -> np.ndarray:
    """The [n, offset + n] additive sliding-window band of a block of n queries after ``offset`` cached positions.

    Query row q sits at position offset + q (PR #1212, history-mask commit).  Column c is inside the band iff
    offset + q - window < c <= offset + q: the query and the window - 1 positions before it.  window >= 1.
    """
    m = np.full((n, offset + n), BLOCKED, dtype=np.float64)
    for q in range(n):
        pos = offset + q
        for c in range(max(0, pos - window + 1), pos + 1):
            m[q, c] = 0.0
    return m


def sliding_mask_from_caller(mask, offset: int, window: int) -> np.ndarray:
    """What a sliding-window layer attends with: the caller's mask intersected with the band.

    PR #1212, the commit on caller masks and the sliding-window band: additive masks intersect by their
    element-wise minimum, and only where the two can disagree - a block of n queries after ``offset`` cached
    positions is left untouched while offset + n <= window (the band then blocks nothing the causal order
    allows).  window == 0 means a full-attention layer (no band).
    """
    mask = np.asarray(mask, dtype=np.float64)
    n = mask.shape[0]
    if window == 0 or offset + n <= window:
        return mask.copy()
    return np.minimum(mask, sliding_band(n, offset, window))


def visible_keys(parents, i: int, offset: int, window: int = 0) -> list[int]:
    """Cache positions node i attends to: every history position and its ancestors' block positions, and with
    a window > 0 only those inside the band (position > offset + i - window)."""
    cols = list(range(offset)) + [offset + j for j in sorted(ancestors(parents, i))]
    if window > 0:
        lo = offset + i - window + 1
        cols = [c for c in cols if c >= lo]
    return cols


def children(parents, u: int) -> list[int]:
    """Children of ``u`` in ascending index order."""
    return [c for c in range(len(parents)) if int(parents[c]) == u]


def accept_walk(argmax, tokens, parents):
    """Descend from the root to the lowest-index child whose token equals argmax(current).

    Returns (path, emitted): path is the list of accepted node indices starting
    at the root; emitted[j] = argmax[path[j]].  accepted = len(path) - 1.
    """
    u = 0
    path = [0]
    while True:
        nxt = None
        for c in children(parents, u):
            if int(tokens[c]) == int(argmax[u]):
                nxt = c
                break
        if nxt is None:
            break
        path.append(nxt)
        u = nxt
    emitted = [int(argmax[p]) for p in path]
    return path, emitted


def speculative_walk(drafts, target_argmax):
    """Chain walk (issue #1204, "What this needs" item 2): accept the longest matching prefix.

    ``drafts`` are the n proposed tokens; ``target_argmax`` has n + 1 entries
    (one per verified position, the last one being the bonus).  Returns
    (accepted, emitted) with emitted = target_argmax[:accepted + 1].
    """
    k = 0
    while k < len(drafts) and int(drafts[k]) == int(target_argmax[k]):
        k += 1
    return k, [int(t) for t in target_argmax[: k + 1]]
