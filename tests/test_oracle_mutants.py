"""The oracle's pins catch plausible mistakes: each case plants one in a copy of an oracle module, on the CPU.

A mutant is one textual edit of an oracle module's source (a dropped term, a wrong sign or index, an off-by-one,
a transposed operand, a tie broken the other way).  The edited source is executed as a fresh namespace and its
functions replace the module's for the duration of the case; then the pin tests (``tests/test_oracle_*.py``) run
in this process, the mutated module's own pins first, and at least one of them must fail.  A mutant that every
pin accepts would be a mistake the oracle could carry unnoticed into every parity claim built on it.

The edited snippet must occur exactly once in the module, so that a rewrite of the oracle that moves it shows up
here as a stale case rather than as a silently vacuous one.
"""
from __future__ import annotations

import importlib
import inspect
import itertools

import pytest

from tests import (test_oracle_append, test_oracle_numeric, test_oracle_sampling, test_oracle_tree,
                   test_oracle_tree_build)

PIN_MODULES = {
    "oracle.attention": test_oracle_numeric,
    "oracle.gather": test_oracle_numeric,
    "oracle.lm_head": test_oracle_numeric,
    "oracle.storage": test_oracle_numeric,
    "oracle.tree": test_oracle_tree,
    "oracle.append": test_oracle_append,
    "oracle.sampling": test_oracle_sampling,
    "oracle.tree_build": test_oracle_tree_build,
}

# (module, what the mistake is, snippet, its replacement)
MUTANTS = [
    # attention
    ("oracle.attention", "score scale 1/D instead of 1/sqrt(D)",
     "k = K[cols]\n    v = V[cols]\n    s = (k @ np.asarray(q, dtype=np.float64)) / math.sqrt(K.shape[1])\n    s = s - s.max()\n"
     "    p = np.exp(s)\n    return (p / p.sum()) @ v\n\n\ndef attend_dense_mask",
     "k = K[cols]\n    v = V[cols]\n    s = (k @ np.asarray(q, dtype=np.float64)) / K.shape[1]\n    s = s - s.max()\n"
     "    p = np.exp(s)\n    return (p / p.sum()) @ v\n\n\ndef attend_dense_mask"),
    ("oracle.attention", "last history position dropped", "list(range(S))", "list(range(S - 1))"),
    ("oracle.attention", "GQA head map h mod HKV", "kv = h // G", "kv = h % HKV"),
    ("oracle.attention", "explicit-column form without the score scale",
     '"""One query row over an explicit list of cache positions."""\n    k = K[cols]\n    v = V[cols]\n'
     "    s = (k @ np.asarray(q, dtype=np.float64)) / math.sqrt(K.shape[1])",
     '"""One query row over an explicit list of cache positions."""\n    k = K[cols]\n    v = V[cols]\n'
     "    s = k @ np.asarray(q, dtype=np.float64)"),
    ("oracle.attention", "additive mask subtracted", "+ mask_row", "- mask_row"),
    ("oracle.attention", "dense form unnormalised", "return (p / p.sum()) @ V", "return p @ V"),
    # tree
    ("oracle.tree", "ancestors exclude the node itself", "out = set()\n    node = int(i)",
     "out = set()\n    node = int(parents[i])"),
    ("oracle.tree", "ancestors stop below the root", "while node >= 0:", "while node > 0:"),
    ("oracle.tree", "history columns blocked", "m = np.zeros((n, offset + n), dtype=np.float64)",
     "m = np.full((n, offset + n), BLOCKED, dtype=np.float64)"),
    ("oracle.tree", "tree mask transposed", "m[i, j] = 0.0", "m[j, i] = 0.0"),
    ("oracle.tree", "band one position too wide", "range(max(0, pos - window + 1), pos + 1)",
     "range(max(0, pos - window), pos + 1)"),
    ("oracle.tree", "visible keys one position too wide", "lo = offset + i - window + 1", "lo = offset + i - window"),
    ("oracle.tree", "caller mask left untouched only strictly below the window", "or offset + n <= window",
     "or offset + n < window"),
    ("oracle.tree", "walk takes the highest-index matching sibling", "for c in children(parents, u):",
     "for c in reversed(children(parents, u)):"),
    ("oracle.tree", "walk compares with the child's own argmax", "if int(tokens[c]) == int(argmax[u]):",
     "if int(tokens[c]) == int(argmax[c]):"),
    ("oracle.tree", "walk emits the draft tokens", "emitted = [int(argmax[p]) for p in path]",
     "emitted = [int(tokens[p]) for p in path]"),
    ("oracle.tree", "validation accepts a self-parent", "if not (0 <= parents[i] < i):",
     "if not (0 <= parents[i] <= i):"),
    ("oracle.tree", "ancestor bits shifted by one", "sum(1 << j for j in", "sum(1 << (j + 1) for j in"),
    ("oracle.tree", "depth counts the node itself", "return len(ancestors(parents, i)) - 1", "return len(ancestors(parents, i))"),
    ("oracle.tree", "root check skipped", "if parents[0] != -1:\n        return BAD_ROOT",
     "if parents[0] < -1:\n        return BAD_ROOT"),
    ("oracle.tree", "tree columns placed at the start of the history mask", "m[:, offset:] = tree_mask(parents)",
     "m[:, :n] = tree_mask(parents)"),
    ("oracle.tree", "chain walk stops one early", "while k < len(drafts) and", "while k + 1 < len(drafts) and"),
    # append
    ("oracle.append", "inverse frequencies with exponent -j/rot_dim", "-2.0 * j / rot_dim", "-1.0 * j / rot_dim"),
    ("oracle.append", "half-layout rotation turns the wrong way",
     "a, b = x[..., :h], x[..., h:rot_dim]\n        out[..., :h] = a * c - b * s\n        out[..., h:rot_dim] = b * c + a * s",
     "a, b = x[..., :h], x[..., h:rot_dim]\n        out[..., :h] = a * c + b * s\n        out[..., h:rot_dim] = b * c - a * s"),
    ("oracle.append", "interleaved pairs split as halves", "a, b = x[..., 0:rot_dim:2], x[..., 1:rot_dim:2]",
     "a, b = x[..., 0:rot_dim // 2], x[..., rot_dim // 2:rot_dim]"),
    ("oracle.append", "node position S + index instead of S + depth", "S + _tree.depth(parents, i)", "S + i"),
    ("oracle.append", "quantisation scale absmax / 128", "amax / np.float32(127.0)", "amax / np.float32(128.0)"),
    ("oracle.append", "quantisation truncates", "np.rint(x32 / s32)", "np.trunc(x32 / s32)"),
    ("oracle.append", "codes clipped to -128", "np.clip(q, -127, 127)", "np.clip(q, -128, 127)"),
    ("oracle.append", "scale from the first feature instead of the absmax", "np.max(np.abs(x32))", "np.abs(x32[0])"),
    ("oracle.append", "new K rows all at the first node's position", "rope(k_new[i], pos[i],", "rope(k_new[i], pos[0],"),
    ("oracle.append", "appended fp16 rows double-rounded through fp32",
     '"""Round to the nearest fp16 value (ties to even), returned as fp64."""\n'
     "    return np.asarray(x, dtype=np.float64).astype(np.float16)",
     '"""Round to the nearest fp16 value (ties to even), returned as fp64."""\n'
     "    return np.asarray(x, dtype=np.float64).astype(np.float32).astype(np.float16)"),
    # storage
    ("oracle.storage", "bf16 bits shifted by 15", "<< np.uint32(16)", "<< np.uint32(15)"),
    ("oracle.storage", "Int8 codes read unsigned", "np.asarray(codes, dtype=np.int8).astype(np.float64)",
     "np.asarray(codes, dtype=np.int8).view(np.uint8).astype(np.float64)"),
    ("oracle.storage", "nibbles in the wrong order", "out[..., 0::2] = p & 0xF\n    out[..., 1::2] = p >> 4",
     "out[..., 0::2] = p >> 4\n    out[..., 1::2] = p & 0xF"),
    ("oracle.storage", "4-bit codes taken as signed offsets", "return s * q + b", "return s * (q - 8) + b"),
    ("oracle.storage", "bf16 rounding keeps 7 bits", "np.rint(np.ldexp(m, 8)), e - 8)", "np.rint(np.ldexp(m, 7)), e - 7)"),
    ("oracle.storage", "bf16 rounding truncates", "np.rint(np.ldexp(m, 8))", "np.floor(np.ldexp(m, 8))"),
    ("oracle.storage", "fp16 storage double-rounded through fp32",
     '"""fp64 values rounded to the nearest fp16 value (numpy\'s correctly rounded conversion)."""\n'
     "    return np.asarray(x, dtype=np.float64).astype(np.float16)",
     '"""fp64 values rounded to the nearest fp16 value (numpy\'s correctly rounded conversion)."""\n'
     "    return np.asarray(x, dtype=np.float64).astype(np.float32).astype(np.float16)"),
    ("oracle.storage", "formats 0 and 1 swapped", "if dtype == 0:\n        return f16(store)",
     "if dtype == 0:\n        return bf16(store)"),
    # gather
    ("oracle.gather", "tail rewrite one row late", "idx[axis] = slice(tail_start, tail_start + len(kept_offsets))",
     "idx[axis] = slice(tail_start + 1, tail_start + 1 + len(kept_offsets))"),
    ("oracle.gather", "new length one short", "return b, tail_start + len(kept_offsets)",
     "return b, tail_start + len(kept_offsets) - 1"),
    ("oracle.gather", "trim keeps one position too few", "np.arange(length)", "np.arange(length - 1)"),
    ("oracle.gather", "absolute form drops the last kept position", "return np.take(np.asarray(buf), kept, axis=axis)",
     "return np.take(np.asarray(buf), kept[:-1], axis=axis)"),
    ("oracle.gather", "identity test accepts any kept list", "return all(int(k) == j for j, k in enumerate(kept_offsets))",
     "return True"),
    ("oracle.gather", "tail sources read from the start of the cache",
     "[tail_start + int(k) for k in kept_offsets]", "[int(k) for k in kept_offsets]"),
    # LM head
    ("oracle.lm_head", "argmax ties to the highest index", "idx = np.argmax(lg, axis=1)",
     "idx = lg.shape[1] - 1 - np.argmax(lg[:, ::-1], axis=1)"),
    ("oracle.lm_head", "runner-up taken with the top still in", "rest[np.arange(lg.shape[0]), idx] = -np.inf",
     "rest[np.arange(lg.shape[0]), 0] = -np.inf"),
    ("oracle.lm_head", "logits scaled by the hidden size", "return np.asarray(h, dtype=np.float64) @ np.asarray(W, dtype=np.float64).T",
     "return np.asarray(h, dtype=np.float64) @ np.asarray(W, dtype=np.float64).T / np.asarray(h).shape[-1]"),
    ("oracle.lm_head", "a later chunk takes ties", "if ctop[r] > best[r]:", "if ctop[r] >= best[r]:"),
    ("oracle.lm_head", "streamed argmax forgets the chunk offset", "arg[r] = r0 + ci[r]", "arg[r] = ci[r]"),
    ("oracle.lm_head", "streamed gap drops the old best", "second[r] = max(best[r], csec[r])", "second[r] = csec[r]"),
    ("oracle.lm_head", "streamed logits chunks one row short",
     "weight_rows(r0, min(V, r0 + CHUNK_ROWS)).T for r0", "weight_rows(r0, min(V, r0 + CHUNK_ROWS - 1)).T for r0"),
    # sampling
    ("oracle.sampling", "temperature ignored", "x = logits[order] / float(temperature)", "x = logits[order]"),
    ("oracle.sampling", "nucleus one token short",
     'm = min(int(np.searchsorted(c, float(top_p), side="left")) + 1, k)',
     'm = max(1, min(int(np.searchsorted(c, float(top_p), side="left")), k))'),
    ("oracle.sampling", "top-k ties to the higher index", "np.lexsort((np.arange(V), -logits))",
     "np.lexsort((-np.arange(V), -logits))"),
    ("oracle.sampling", "nucleus not renormalised", "q = p[:m] / c[m - 1]", "q = p[:m]"),
    ("oracle.sampling", "draw takes the token whose mass reaches u", 'side="right"', 'side="left"'),
    # tree construction
    ("oracle.tree_build", "log-probabilities without the normaliser", "x[order] - lse", "x[order] - m"),
    ("oracle.tree_build", "scores not accumulated along the path", "score[i] = np.float32(score[p] + lp[i])",
     "score[i] = np.float32(lp[i])"),
    ("oracle.tree_build", "depth cap one short", "depth[i] <= depth_max", "depth[i] < depth_max"),
    ("oracle.tree_build", "equal scores take the later candidate", "key=lambda i: (-float(score[i]), i)",
     "key=lambda i: (-float(score[i]), -i)"),
    ("oracle.tree_build", "selected parents indexed by candidate, not by position", "[where[int(parents[c])] for c in order]",
     "[int(parents[c]) for c in order]"),
    ("oracle.tree_build", "one node too many", "[: max(0, T - 1)]", "[: max(0, T)]"),
    ("oracle.tree_build", "top-k children ties to the higher index", "np.lexsort((np.arange(V), -x))",
     "np.lexsort((-np.arange(V), -x))"),
]


def _cases(mod):
    """Every pin of a test module as (name, callable, kwargs), parametrised ones expanded."""
    for name, fn in inspect.getmembers(mod, inspect.isfunction):
        if not name.startswith("test_") or fn.__module__ != mod.__name__:
            continue
        grids = []
        for mark in getattr(fn, "pytestmark", []):
            if mark.name != "parametrize":
                continue
            names, values = mark.args[0], mark.args[1]
            names = [s.strip() for s in names.split(",")] if isinstance(names, str) else list(names)
            rows = []
            for v in values:
                v = v.values if hasattr(v, "values") and not isinstance(v, (tuple, list)) else v
                v = tuple(v) if len(names) > 1 else (v[0] if isinstance(v, tuple) and len(v) == 1 else v,)
                rows.append(dict(zip(names, v)))
            grids.append(rows)
        for combo in itertools.product(*grids) if grids else [()]:
            kw = {}
            for part in combo:
                kw.update(part)
            yield name, fn, kw


def _first_failing_pin(home):
    order = [home] + [m for m in dict.fromkeys(PIN_MODULES.values()) if m is not home]
    for mod in order:
        for name, fn, kw in _cases(mod):
            try:
                fn(**kw)
            except Exception:  # an assertion, or the mistake breaking a shape the pin relies on
                return f"{mod.__name__.rsplit('.', 1)[-1]}::{name}{kw or ''}"
    return None


def test_pins_pass_on_the_unmodified_oracle():
    assert _first_failing_pin(test_oracle_numeric) is None


@pytest.mark.parametrize("module,what,old,new", MUTANTS, ids=[f"{m.split('.')[-1]}: {w}" for m, w, _, _ in MUTANTS])
def test_a_planted_mistake_fails_a_pin(module, what, old, new, monkeypatch):
    mod = importlib.import_module(module)
    src = inspect.getsource(mod)
    assert src.count(old) == 1, f"stale mutant: the snippet occurs {src.count(old)} times in {module}"
    ns = {"__name__": module, "__package__": "oracle", "__file__": mod.__file__}
    exec(compile(src.replace(old, new), mod.__file__, "exec"), ns)
    for name, obj in ns.items():
        if inspect.isfunction(obj) and obj.__module__ == module and hasattr(mod, name):
            monkeypatch.setattr(mod, name, obj)
    caught = _first_failing_pin(PIN_MODULES[module])
    assert caught is not None, f"no pin fails when the oracle has: {what}"
