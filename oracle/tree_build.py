"""Building the draft tree from the drafter's confidence (oracle; test infrastructure only).

Definitions followed:

* mlxcel issue #1204, "What this needs", the fourth decision: EAGLE-2 branches by the drafter's confidence,
  which needs the drafter's logits (today reduced to an argmax); PR #1212, the commit that adds draft_tree: the
  runner-up at an uncertain step is the alternative worth a verify position; Splash issue #728, "What it does":
  the chain plus likely alternatives from the draft's top-k selector.
* Reading (the pages give the principle, not the steps): a drafter step turns a node's draft logits into
  children candidates - its top_k tokens with their log-probabilities log_softmax(logits)[token]; candidates of
  every expanded node form a candidate tree (topological order, root 0); the verified tree is the root plus the
  T - 1 candidates with the highest cumulative log-probability along their path (the rerank of EAGLE-2; best-first
  expansion by path probability selects the same set), within a maximum depth, ties to the earlier candidate.
  Since a child's cumulative log-probability never exceeds its parent's, the selection is ancestor-closed.
  The verified tree lists the selected nodes in selection order (descending score, ties to the earlier
  candidate), which is topological.  Scores are accumulated in fp32 from the root down, the precision in which
  the kernel takes the same decisions.
"""
from __future__ import annotations

import numpy as np


def draft_children(draft_logits, top_k: int):
    """Per row of drafter logits [V]: (tokens [k], log-probabilities [k]) of its top_k tokens (fp64)."""
    x = np.asarray(draft_logits, dtype=np.float64)
    V = x.shape[0]
    k = min(int(top_k), V)
    order = np.lexsort((np.arange(V), -x))[:k]
    m = x.max()
    lse = m + np.log(np.sum(np.exp(x - m)))
    return order.astype(np.int64), x[order] - lse


def path_scores(parents, logp):
    """fp32 cumulative log-probability of every candidate, summed from the root down; depth of every candidate."""
    n = len(parents)
    score = np.zeros(n, dtype=np.float32)
    depth = np.zeros(n, dtype=np.int64)
    lp = np.asarray(logp, dtype=np.float32)
    for i in range(1, n):
        p = int(parents[i])
        score[i] = np.float32(score[p] + lp[i])
        depth[i] = depth[p] + 1
    return score, depth


def select_best_first(parents, tokens, logp, T: int, depth_max: int):
    """Verified tree of at most T nodes: (parents [t], tokens [t], candidate index [t]) in selection order."""
    score, depth = path_scores(parents, logp)
    n = len(parents)
    eligible = [i for i in range(1, n) if depth[i] <= depth_max]
    order = sorted(eligible, key=lambda i: (-float(score[i]), i))[: max(0, T - 1)]
    chosen = [0] + order
    where = {c: j for j, c in enumerate(chosen)}
    out_par = [-1] + [where[int(parents[c])] for c in order]
    out_tok = [int(tokens[c]) for c in chosen]
    return out_par, out_tok, chosen
