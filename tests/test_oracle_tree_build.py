"""Pins of the oracle's draft-tree construction (drafter top-k children, best-first selection).

Checked against an independent best-first expansion with a priority queue, scipy's log_softmax, and the
properties the verified tree must have (ancestor-closed, topological, within the depth cap).
"""
import heapq

import numpy as np
import pytest
from scipy.special import log_softmax

from oracle import tree as ot
from oracle import tree_build as otb


def random_candidates(rng, n, fan=4):
    parents = [-1]
    for i in range(1, n):
        parents.append(int(rng.integers(max(0, i - 3 * fan), i)))
    logp = np.log(rng.uniform(0.01, 1.0, size=n)).astype(np.float32)
    logp[0] = 0.0
    tokens = rng.integers(0, 1000, size=n)
    return parents, tokens, logp


def heap_best_first(parents, logp, T, depth_max):
    """Best-first expansion: pop the frontier candidate of highest path score (earlier candidate on ties)."""
    score, depth = otb.path_scores(parents, logp)
    children = {}
    for i in range(1, len(parents)):
        children.setdefault(parents[i], []).append(i)
    chosen, heap = [0], []
    for c in children.get(0, []):
        heapq.heappush(heap, (-float(score[c]), c))
    while heap and len(chosen) < T:
        _, c = heapq.heappop(heap)
        if depth[c] > depth_max:
            continue
        chosen.append(c)
        for g in children.get(c, []):
            heapq.heappush(heap, (-float(score[g]), g))
    return chosen


@pytest.mark.parametrize("seed", range(8))
def test_selection_equals_heap_best_first(seed):
    rng = np.random.default_rng(seed)
    n = int(rng.integers(20, 300))
    parents, tokens, logp = random_candidates(rng, n)
    for T, dmax in ((1, 8), (7, 3), (16, 6), (33, 64), (64, 8)):
        par, tok, idx = otb.select_best_first(parents, tokens, logp, T, dmax)
        assert idx == heap_best_first(parents, logp, T, dmax)
        assert ot.validate(par) == ot.OK  # topological: parents[i] < i, root first
        assert tok == [int(tokens[c]) for c in idx]
        for j in range(1, len(idx)):
            assert idx[par[j]] == parents[idx[j]]  # ancestor-closed: every node's parent was chosen
        _, depth = otb.path_scores(parents, logp)
        assert all(depth[c] <= dmax for c in idx)


def test_chain_candidates_give_the_chain():
    n = 10
    parents = [-1] + list(range(n - 1))
    logp = np.full(n, -0.1, dtype=np.float32)
    logp[0] = 0
    par, tok, idx = otb.select_best_first(parents, np.arange(n), logp, 4, 8)
    assert idx == [0, 1, 2, 3] and par == [-1, 0, 1, 2]


def test_equal_scores_prefer_earlier_candidates_and_parents():
    parents = [-1, 0, 0, 1, 2]
    logp = np.array([0, -1, -1, 0, 0], dtype=np.float32)  # children with probability 1 tie with their parents
    par, tok, idx = otb.select_best_first(parents, np.arange(5), logp, 4, 8)
    assert idx == [0, 1, 2, 3] and par == [-1, 0, 0, 1]


def test_draft_children_are_top_k_log_probabilities():
    rng = np.random.default_rng(4)
    x = rng.standard_normal(500) * 3
    x[[10, 20]] = x.max() + 1  # a tie: the lower index first
    toks, lp = otb.draft_children(x, 5)
    assert toks.tolist()[:2] == [10, 20]
    assert toks.tolist() == np.lexsort((np.arange(500), -x))[:5].tolist()
    assert np.allclose(lp, log_softmax(x)[toks], rtol=0, atol=1e-12)
