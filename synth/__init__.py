"""Seeded synthetic inputs for the tree-verify step (shared by tests, smoke and bench).

Holds none of the verify step's arithmetic: only counter-based random numbers
(``rng``), the element formulas of every input tensor (``tensors``), the five
workloads (``configs``) and the draft trees with their planted targets
(``trees``).  ``device`` fills large tensors directly in GPU memory with the
same formulas.
"""
