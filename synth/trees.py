"""Seeded draft trees, draft tokens, target argmaxes and planted hidden states.

A "round" is everything the verify step consumes besides the caches and the
weights: the parent array and draft token of every node, and the hidden state
of every node fed to the LM head.  The generator first decides the accepted
path it wants (by the workload's accept-length rule), then picks each node's
target argmax so that the path is the one the walk should find, and finally
plants each target in the node's hidden state: ``h = noise + c * dir(target)``
with ``dir`` a unit-variance vector correlated with the target's LM-head row.
With ``c`` as configured the target's logit exceeds every other by far more than
the required gap; the oracle measures the gap, this module does not.

Only host-side integer/scalar logic lives here (no logits, no masks, no walk).
Scalar float arithmetic is limited to + * / so that trees are identical on
every IEEE machine.
"""
from __future__ import annotations

import numpy as np

from . import rng, tensors
from .configs import BF16, Config


class Stream:
    """Sequential scalar draws from one counter-based stream."""

    def __init__(self, k: int):
        self.k, self.i = k, 0

    def next(self) -> int:
        h = rng.draw_int(self.k, self.i)
        self.i += 1
        return h

    def below(self, n: int) -> int:
        return rng.int_below_scalar(self.next(), n)

    def u01(self) -> float:
        return rng.u01_scalar(self.next())


# ----------------------------------------------------------------------------- topologies
def chain(T: int) -> list[int]:
    return [-1] + list(range(T - 1))


def specinfer(branching, n: int) -> list[int]:
    """Full tree with the given branching per level, truncated to ``n`` nodes.

    Nodes are ranked by (sum of sibling ranks along the path, depth, BFS index)
    and the first ``n`` kept; the result is ancestor-closed and relabelled in
    BFS order so that parents precede children.
    """
    nodes = [()]  # node = tuple of sibling ranks from the root, in BFS order
    frontier = [()]
    for width in branching:
        nxt = []
        for p in frontier:
            for r in range(width):
                nxt.append(p + (r,))
        nodes.extend(nxt)
        frontier = nxt
    order = sorted(range(len(nodes)), key=lambda i: (sum(nodes[i]), len(nodes[i]), i))
    keep = sorted(order[:n])  # BFS index order == parents first
    kept = [nodes[i] for i in keep]
    pos = {t: j for j, t in enumerate(kept)}
    parents = [-1] + [pos[t[:-1]] for t in kept[1:]]
    return parents


def best_first(st: Stream, n: int, k_max: int, depth_max: int, V: int):
    """Best-first (EAGLE-2 style) tree: expand the best-scoring candidate child.

    Every node draws up to ``k_max`` candidate children with distinct tokens and
    draft probabilities (random weights normalised to sum 1, sorted descending).
    A candidate's score is the product of draft probabilities along its path;
    the best candidate on the frontier (ties: earlier creation) becomes the next
    node until ``n`` nodes exist or the frontier is empty.
    Returns (parents, tokens) with tokens[0] the committed root token.
    """
    parents, tokens, depth, score = [-1], [st.below(V)], [0], [1.0]
    frontier = []  # (score, creation, parent, token)
    created = 0

    def spawn(u):
        nonlocal created
        if depth[u] >= depth_max:
            return
        k = 1 + st.below(k_max)
        w = [1.0 + st.u01() * 15.0 for _ in range(k)]
        tot = 0.0
        for x in w:
            tot += x
        p = sorted((x / tot for x in w), reverse=True)
        seen = set()
        for r in range(k):
            t = st.below(V)
            while t in seen:
                t = st.below(V)
            seen.add(t)
            frontier.append((score[u] * p[r], created, u, t))
            created += 1

    spawn(0)
    while len(parents) < n and frontier:
        best = 0
        for j in range(1, len(frontier)):
            a, b = frontier[j], frontier[best]
            if a[0] > b[0] or (a[0] == b[0] and a[1] < b[1]):
                best = j
        s, _, u, t = frontier.pop(best)
        parents.append(u)
        tokens.append(t)
        depth.append(depth[u] + 1)
        score.append(s)
        spawn(len(parents) - 1)
    return parents, tokens


def depths(parents) -> list[int]:
    d = [0] * len(parents)
    for i in range(1, len(parents)):
        d[i] = d[parents[i]] + 1
    return d


def children(parents):
    ch = [[] for _ in parents]
    for i in range(1, len(parents)):
        ch[parents[i]].append(i)
    return ch


def root_path(parents, node: int) -> list[int]:
    p = []
    while node >= 0:
        p.append(node)
        node = parents[node]
    return p[::-1]


def is_identity(path) -> bool:
    return all(p == j for j, p in enumerate(path))


# ----------------------------------------------------------------------------- rounds
def _choose_path(cfg: Config, st: Stream, parents, b: int, round_id: int):
    d = depths(parents)
    ch = children(parents)
    T = len(parents)
    rule = cfg.accept
    if rule == "uniform_node":
        end = st.below(T)
    elif rule == "cycle":
        end = min((round_id + b) % T, T - 1)  # chain: accept length cycles 0..T-1
    elif rule == "uniform_1_5":
        a = 1 + st.below(max(d))
        cand = [i for i in range(T) if d[i] == a]
        end = cand[st.below(len(cand))]
    elif rule in ("leaf_uniform", "geometric"):
        leaves = [i for i in range(T) if not ch[i]]
        leaf = leaves[st.below(len(leaves))]
        lp = root_path(parents, leaf)
        if rule == "leaf_uniform":
            a = st.below(len(lp))
        else:
            a = 0
            while a < len(lp) - 1 and st.u01() >= 0.35:
                a += 1
        end = lp[a]
    else:
        raise ValueError(rule)
    return root_path(parents, end)


def _force(cfg: Config, trees, paths):
    """Make sure the round exercises the gather cases the workload asks for."""
    if cfg.accept == "leaf_uniform":  # >= 4 scattered (non-prefix) paths
        for b in range(len(paths)):
            if sum(not is_identity(p) for p in paths) >= 4:
                break
            if is_identity(paths[b]):
                par = trees[b][0]
                d = depths(par)
                scattered = [i for i in range(len(par)) if not is_identity(root_path(par, i))]
                if scattered:
                    end = max(scattered, key=lambda i: (d[i], -i))
                    paths[b] = root_path(par, end)
    if cfg.accept == "geometric" and len(paths) >= 2:  # one zero accept, one identity (prefix) accept
        paths[0] = [0]
        par = trees[1][0]
        k = 0
        while k + 1 < len(par) and par[k + 1] == k:
            k += 1
        paths[1] = list(range(k + 1))
    return paths


def make_round(cfg: Config, round_id: int = 0, plant: bool = True):
    """Build one round: parents/tokens/targets [B,T], planned paths, hidden bits [B*T,H]."""
    B, T, V = cfg.B, cfg.T, cfg.V
    trees = []
    for b in range(B):
        st = Stream(rng.stream_key(cfg.seed, tensors.tensor_id(tensors.KIND_TREE, b)))
        if cfg.topology == "fixed":
            par = list(cfg.parents0)
            tok = None
        elif cfg.topology == "chain":
            par, tok = chain(T), None
        elif cfg.topology == "specinfer":
            par, tok = specinfer(cfg.branching, T), None
        elif cfg.topology == "best_first":
            par, tok = best_first(st, T, cfg.k_max, cfg.depth_max, V)
            assert len(par) == T, "frontier ran out before T nodes"
        else:
            raise ValueError(cfg.topology)
        trees.append((par, tok))

    parents = np.zeros((B, T), dtype=np.int32)
    tokens = np.zeros((B, T), dtype=np.int32)
    targets = np.zeros((B, T), dtype=np.int32)
    paths = []
    for b in range(B):
        st = Stream(rng.stream_key(cfg.seed, tensors.tensor_id(tensors.KIND_TOK, (round_id << 8) | b)))
        par, tok = trees[b]
        if tok is None:  # fixed topologies: distinct tokens among siblings
            ch = children(par)
            tok = [st.below(V)] + [0] * (T - 1)
            for u in range(T):
                seen = set()
                for c in ch[u]:
                    t = st.below(V)
                    while t in seen:
                        t = st.below(V)
                    seen.add(t)
                    tok[c] = t
        parents[b] = par
        tokens[b] = tok
        paths.append(_choose_path(cfg, st, par, b, round_id))
    paths = _force(cfg, trees, paths)

    for b in range(B):
        st = Stream(rng.stream_key(cfg.seed, tensors.tensor_id(tensors.KIND_TOK, 0x8000 | (round_id << 8) | b)))
        par = parents[b].tolist()
        ch = children(par)
        path = paths[b]
        for i in range(T):
            targets[b, i] = st.below(V)
        for j in range(len(path) - 1):
            targets[b, path[j]] = tokens[b, path[j + 1]]
        last = path[-1]
        bad = {int(tokens[b, c]) for c in ch[last]}
        t = int(targets[b, last])
        while t in bad:
            t = st.below(V)
        targets[b, last] = t

    out = dict(parents=parents, tokens=tokens, targets=targets, paths=paths)
    if plant:
        out["hidden"] = plant_hidden(cfg, round_id, targets.reshape(-1))
    return out


def plant_hidden(cfg: Config, round_id: int, targets_flat) -> np.ndarray:
    """bf16 bits of hidden [B*T, H] = noise + c * dir(target) (fp32, then rounded)."""
    rows = np.arange(len(targets_flat))
    n = tensors.hidden_noise(cfg, round_id, rows)
    d = tensors.w_direction(cfg, np.asarray(targets_flat, dtype=np.int64))
    h = n + (np.float32(cfg.plant_c) * d)
    return rng.f32_to_bf16_bits(h)
