"""Source-level invariants of the CUDA library that no GPU test would catch reliably.

Every kernel is launched with programmatic stream serialization, so it may start before the kernel ahead of it on
the stream has finished: its first statement must be the dependency wait (griddep_begin), and every launch must go
through launch_pdl (a bare <<<...>>> launch would lose the overlap, a kernel without the wait would race).
"""
import os
import re

CSRC = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))),
                    "tree_speculative_decoding_array_gb300", "csrc")


def _sources():
    for f in sorted(os.listdir(CSRC)):
        if f.endswith(".cu"):
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
