"""Source-level invariants of the CUDA library that no GPU test would catch reliably.

Every kernel is launched with programmatic stream serialization, so it may start before the kernel ahead of it on
the stream has finished: its first statement must be the dependency wait (griddep_begin), and every launch must go
through launch_pdl (a bare <<<...>>> launch would lose the overlap, a kernel without the wait would race).

No kernel may hang or fault its GPU by design: every open-ended loop polls the global timer and gives up after a
bounded time (setting the kernel's abort flag or a status the host reads), or is listed here with the bound that
ends it; no device code stops with a trap or a failing assert.
"""
import os
import re

CSRC = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))),
                    "tree_speculative_decoding_array_gb300", "csrc")


def _sources(exts=(".cu",)):
    for f in sorted(os.listdir(CSRC)):
        if f.endswith(exts):
            with open(os.path.join(CSRC, f)) as fh:
                yield f, fh.read()


def _body_start(s, i):
    depth = 0
    while True:
        c = s[i]
        if c == "(":
            depth += 1
        elif c == ")":
            depth -= 1
        elif c == "{" and depth == 0:
            return i + 1
        i += 1


def test_every_kernel_waits_for_its_predecessor_first():
    kernels = 0
    for f, s in _sources():
        for m in re.finditer(r"__global__", s):
            body = s[_body_start(s, m.start()):]
            first = body.lstrip().split(";", 1)[0]
            assert first == "griddep_begin()", (f, s[m.start():m.start() + 120])
            kernels += 1
    assert kernels >= 20


def test_every_launch_goes_through_launch_pdl():
    for f, s in _sources():
        assert "<<<" not in s, f
    assert any("launch_pdl(" in s for _, s in _sources())


# Open-ended loops that need no timer, with the bound that ends them.
BOUNDED_BY_CONSTRUCTION = {
    ("tree_walk.cu", "for (;;)"): "each step moves to a child, whose index is larger than its parent's in a validated "
                                  "topological tree, so the walk ends within T - 1 steps",
}


def _loop_body(s, i):
    """The text of the loop statement starting at index i (its braces matched), or its single statement."""
    j, par = s.index("(", i), 0
    while True:  # the loop header's closing parenthesis
        par += {"(": 1, ")": -1}.get(s[j], 0)
        if par == 0:
            break
        j += 1
    depth = 0
    for k in range(j + 1, len(s)):
        c = s[k]
        if c == "{":
            depth += 1
        elif c == "}":
            depth -= 1
            if depth == 0:
                return s[i:k + 1]
        elif c == ";" and depth == 0:
            return s[i:k + 1]
    return s[i:]


def test_every_open_ended_loop_is_bounded():
    pat = re.compile(r"for\s*\([^;]*;\s*;[^)]*\)|while\s*\(\s*(true|1)\s*\)|while\s*\(\s*!\s*[\w:]*mbar_(try_wait|test)")
    seen = 0
    for f, s in _sources((".cu", ".cuh")):
        for m in pat.finditer(s):
            seen += 1
            head = m.group(0).replace(" ", "")
            if any(f == bf and head.startswith(bh.replace(" ", "")) for bf, bh in BOUNDED_BY_CONSTRUCTION):
                continue
            body = _loop_body(s, m.start())
            assert "globaltimer()" in body, (f, s[m.start():m.start() + 160])
    assert seen >= 5


def test_no_device_trap_or_assert():
    for f, s in _sources((".cu", ".cuh")):
        code = re.sub(r"//[^\n]*", "", s)
        assert "__trap" not in code, f
        assert re.search(r"(?<![\w_])assert\s*\(", code) is None, f
