"""Pins of the oracle's topology, mask and walk against what the pages fix.

Sources: mlxcel issue #1204 ("Increment 1": a linear tree masks as a causal
mask for every block width from 0 to 5 and walks as speculative_walk at every
accept length; the accepted set is a path, pinned with two siblings carrying
the same token; "Increment 3": the history mask equals a causal mask with the
same offset, element for element) and mlxcel PR #1212 (the real-checkpoint
round accounting, the -1e9 blocking value).
"""
import itertools
import os

import numpy as np
import pytest

from oracle import tree as ot

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def causal_mask(n, offset=0):
    """create_causal_mask's convention, built directly: row q at position q + offset sees c <= q + offset."""
    q = np.arange(n)[:, None] + offset
    c = np.arange(offset + n)[None, :]
    return np.where(c <= q, 0.0, -1e9)


def all_trees(T):
    """Every topological parent array with T nodes (prod_{i>=1} i of them)."""
    if T == 0:
        yield []
        return
    for rest in itertools.product(*[range(i) for i in range(1, T)]):
        yield [-1] + list(rest)


def reachability(parents):
    """Ancestor-or-self relation by boolean matrix closure (independent of parent chasing)."""
    n = len(parents)
    A = np.eye(n, dtype=bool)
    for i in range(1, n):
        A[i, parents[i]] = True
    for _ in range(n):
        A = (A.astype(int) @ A.astype(int)) > 0
    return A


@pytest.mark.parametrize("n", range(0, 6))
def test_linear_tree_masks_as_causal(n):
    assert np.array_equal(ot.tree_mask(ot_chain(n)), causal_mask(n))


@pytest.mark.parametrize("n,offset", [(1, 0), (3, 1), (5, 7), (4, 128), (2, 4096)])
def test_linear_history_mask_equals_causal_with_offset(n, offset):
    assert np.array_equal(ot.history_mask(ot_chain(n), offset), causal_mask(n, offset))


def ot_chain(n):
    return [-1] + list(range(n - 1)) if n else []


@pytest.mark.parametrize("T", range(1, 8))
def test_ancestors_brute_force(T):
    for par in all_trees(T):
        R = reachability(par)
        bits = ot.ancestor_bits(par)
        m = ot.tree_mask(par)
        for i in range(T):
            assert bits[i] == sum(1 << j for j in range(T) if R[i, j])
            assert bin(bits[i]).count("1") == ot.depth(par, i) + 1
            assert m[i, i] == 0.0  # self is never blocked, so no row is all -1e9
        for a, b in itertools.permutations(range(T), 2):
            if par[a] == par[b] and a > 0 and b > 0:
                assert m[a, b] == -1e9  # siblings never see each other


def test_history_columns_all_attend():
    par = [-1, 0, 0, 1, 1, 2, 2]
    m = ot.history_mask(par, 128)
    assert m.shape == (7, 135)
    assert np.all(m[:, :128] == 0.0)
    assert np.array_equal(m[:, 128:], ot.tree_mask(par))


def test_validate():
    assert ot.validate([]) == ot.OK
    assert ot.validate([-1]) == ot.OK
    assert ot.validate([-1, 0, 0, 1]) == ot.OK
    assert ot.validate([0, 0]) == ot.BAD_ROOT
    assert ot.validate([-1, 1]) == ot.BAD_PARENT      # self-parent
    assert ot.validate([-1, 0, 3, 0]) == ot.BAD_PARENT  # forward reference
    assert ot.validate([-1, -1]) == ot.BAD_PARENT     # second root


@pytest.mark.parametrize("n", range(1, 7))
def test_linear_tree_walks_as_speculative_walk(n):
    """Every accept length k in 0..n-1 of an n-node chain (n-1 proposals)."""
    rng = np.random.default_rng(n)
    par = ot_chain(n)
    for k in range(n):
        tokens = rng.integers(0, 50, size=n)
        argmax = np.empty(n, dtype=np.int64)
        argmax[:-1] = tokens[1:]
        argmax[-1] = rng.integers(0, 50)
        if k < n - 1:
            argmax[k] = (tokens[k + 1] + 1) % 50  # first mismatch at proposal k
        path, emitted = ot.accept_walk(argmax, tokens, par)
        acc, em2 = ot.speculative_walk(tokens[1:], argmax)
        assert len(path) - 1 == k == acc
        assert path == list(range(k + 1))
        assert emitted == em2 == [int(a) for a in argmax[: k + 1]]


def test_duplicate_siblings_yield_a_path_lowest_index():
    #      0
    #    / | \
    #   1  2  3      tokens 1 and 3 both equal argmax[0]
    #   |     |
    #   4     5
    par = [-1, 0, 0, 0, 1, 3]
    tokens = [9, 7, 8, 7, 5, 5]
    argmax = [7, 5, 0, 5, 1, 1]
    path, emitted = ot.accept_walk(argmax, tokens, par)
    assert path == [0, 1, 4]
    assert emitted == [7, 5, 1]
    for a, b in zip(path, path[1:]):
        assert par[b] == a


def all_root_paths(par):
    out = []
    for i in range(len(par)):
        p, u = [], i
        while u >= 0:
            p.append(u)
            u = par[u]
        out.append(p[::-1])
    return out


@pytest.mark.parametrize("T", range(1, 7))
def test_walk_brute_force(T):
    """The walk's path is consistent and maximal; with distinct sibling tokens it is the
    unique longest consistent root path."""
    rng = np.random.default_rng(100 + T)
    for par in all_trees(T):
        for trial in range(3):
            tokens = rng.permutation(40)[:T]  # distinct everywhere
            argmax = rng.integers(0, 40, size=T)
            # steer half the nodes towards one of their children
            for u in range(T):
                ch = [c for c in range(T) if par[c] == u]
                if ch and rng.random() < 0.6:
                    argmax[u] = tokens[ch[rng.integers(len(ch))]]
            path, emitted = ot.accept_walk(argmax, tokens, par)
            consistent = [p for p in all_root_paths(par)
                          if all(tokens[b] == argmax[a] for a, b in zip(p, p[1:]))]
            longest = max(len(p) for p in consistent)
            assert path in consistent
            assert len(path) == longest
            assert sum(len(p) == longest for p in consistent) == 1
            last = path[-1]
            assert not any(par[c] == last and tokens[c] == argmax[last] for c in range(T))
            assert emitted == [int(argmax[p]) for p in path]


def read_golden(name):
    vals = {}
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.strip()
            if line and not line.startswith("#"):
                k, v = line.split()
                vals[k] = float(v)
    return vals


def test_round_accounting_matches_printed_run():
    """39 linear-tree rounds of 4 nodes with the printed zero/partial/full split reproduce the
    printed proposed/accepted/emitted-per-verify figures through the oracle's walk."""
    g = read_golden("round_accounting_gemma4.txt")
    n_nodes = 4
    # 17 zero, 7 partial (3 x 1 and 4 x 2 accepted make the printed 56 total), 15 full.
    accepts = [0] * 17 + [1] * 3 + [2] * 4 + [3] * 15
    rng = np.random.default_rng(7)
    proposed = accepted = emitted = zero = partial = full = 0
    for k in accepts:
        tokens = rng.integers(0, 100, size=n_nodes)
        argmax = np.append(tokens[1:], rng.integers(0, 100))
        if k < n_nodes - 1:
            argmax[k] = (tokens[k + 1] + 1) % 100
        path, em = ot.accept_walk(argmax, tokens, ot_chain(n_nodes))
        a = len(path) - 1
        proposed += n_nodes - 1
        accepted += a
        emitted += len(em)
        zero += a == 0
        full += a == n_nodes - 1
        partial += 0 < a < n_nodes - 1
    assert len(accepts) == g["rounds"]
    assert proposed == g["proposed"]
    assert accepted == g["accepted"]
    assert round(emitted / len(accepts), 4) == g["emitted_per_verify"]
    assert (zero, partial, full) == (g["zero_accept"], g["partial_accept"], g["full_accept"])
