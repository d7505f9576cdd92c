"""Sampled (temperature > 0) verification: the target's draw at every tree node (oracle; test infrastructure only).

Definition followed - Splash issue #728, "What it does": for sampled requests every node draws from the
nucleus-filtered distribution with its own uniform, so the committed tokens keep the chain verify's output
distribution; the walk then follows the child whose draft token equals the node's draw (the same walk as
greedy verification, with the draw in place of the argmax).  The issue's sampled check uses temperature 1,
top-p 0.95 and top-k 20.

Reading of the filter order (the page lists the three knobs, not their order): logits / temperature, keep the
top_k largest (ties to the lower index), softmax over them, keep the shortest prefix (in descending order) whose
probability mass reaches top_p, renormalise, and invert the cumulative distribution at the node's uniform u in
[0, 1): the token is the first one whose cumulative mass exceeds u.
"""
from __future__ import annotations

import numpy as np


def nucleus(logits, temperature: float, top_k: int, top_p: float):
    """The kept tokens (descending) and their renormalised probabilities, in fp64."""
    logits = np.asarray(logits, dtype=np.float64)
    V = logits.shape[0]
    k = min(int(top_k), V)
    order = np.lexsort((np.arange(V), -logits))[:k]  # descending logit, lower index first among ties
    x = logits[order] / float(temperature)
    p = np.exp(x - x.max())
    p /= p.sum()
    c = np.cumsum(p)
    m = min(int(np.searchsorted(c, float(top_p), side="left")) + 1, k)  # shortest prefix with mass >= top_p
    q = p[:m] / c[m - 1]
    return order[:m], q


def draw(logits, temperature: float, top_k: int, top_p: float, u: float) -> int:
    """The token a node draws with its uniform u."""
    tokens, q = nucleus(logits, temperature, top_k, top_p)
    cq = np.cumsum(q)
    j = int(np.searchsorted(cq, float(u), side="right"))
    return int(tokens[min(j, len(tokens) - 1)])
