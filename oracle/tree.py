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
