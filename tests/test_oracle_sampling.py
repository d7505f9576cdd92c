"""Pins of the oracle's sampled verification (the node's nucleus-filtered draw).

Checks against a hand-worked draw, against scipy's softmax for the unfiltered case, and against the properties
the draw must have: top-k 1 is the greedy argmax, logit shifts change nothing, and tokens cut by the nucleus are
never drawn.
"""
import math

import numpy as np
import pytest
from scipy.special import softmax

from oracle import sampling as osm


def test_hand_worked_draw():
    # softmax([2, 1, 0]) = [0.665, 0.245, 0.090]; cumulative 0.665, 0.910 >= 0.9 keeps two tokens;
    # renormalised [e/(e+1), 1/(e+1)] = [0.73106, 0.26894]
    logits = [2.0, 1.0, 0.0, -1.0]
    tokens, q = osm.nucleus(logits, 1.0, 3, 0.9)
    assert tokens.tolist() == [0, 1]
    assert np.allclose(q, [math.e / (math.e + 1), 1 / (math.e + 1)], rtol=0, atol=1e-15)
    assert osm.draw(logits, 1.0, 3, 0.9, 0.5) == 0
    assert osm.draw(logits, 1.0, 3, 0.9, 0.7310) == 0
    assert osm.draw(logits, 1.0, 3, 0.9, 0.7312) == 1
    assert osm.draw(logits, 1.0, 3, 0.9, 0.999) == 1
    # two equal logits: renormalised masses exactly [0.5, 0.5]; a uniform on the boundary belongs to the next
    # token (the first whose cumulative mass exceeds u), zero to the first
    assert osm.draw([0.0, 0.0], 1.0, 2, 1.0, 0.5) == 1
    assert osm.draw([0.0, 0.0], 1.0, 2, 1.0, 0.0) == 0
    assert osm.draw([0.0, 0.0], 1.0, 2, 1.0, np.nextafter(0.5, 0.0)) == 0


def test_top_k_one_is_greedy_with_lowest_index_ties():
    rng = np.random.default_rng(1)
    for _ in range(20):
        x = rng.standard_normal(50)
        x[[7, 31]] = x.max() + 1.0  # a tie at the top
        for u in (0.0, 0.3, 0.999):
            assert osm.draw(x, 0.7, 1, 0.95, u) == 7


def test_unfiltered_draw_follows_softmax():
    rng = np.random.default_rng(2)
    x = rng.standard_normal(12) * 2
    T = 1.3
    n = 200000
    us = (np.arange(n) + 0.5) / n
    counts = np.bincount([osm.draw(x, T, 12, 1.0, u) for u in us], minlength=12)
    assert np.allclose(counts / n, softmax(x / T), rtol=0, atol=2.0 / n)


def test_shift_invariance_and_nucleus_cut():
    rng = np.random.default_rng(3)
    x = rng.standard_normal(40)
    tokens, q = osm.nucleus(x, 1.0, 20, 0.8)
    kept = set(tokens.tolist())
    for u in np.linspace(0, 0.999, 97):
        t = osm.draw(x, 1.0, 20, 0.8, u)
        assert t in kept
        assert osm.draw(x + 123.0, 1.0, 20, 0.8, u) == t
        assert osm.draw(2.0 * x, 2.0, 20, 0.8, u) == t
    order = np.argsort(-x)
    assert tokens.tolist() == order[:len(tokens)].tolist()
    mass = softmax(x[order[:20]])
    assert mass[:len(tokens)].sum() >= 0.8 and mass[:len(tokens) - 1].sum() < 0.8
