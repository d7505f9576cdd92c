"""Plain CPU oracle of the tree speculative-decoding verify step (TEST INFRASTRUCTURE).

This package is the slow, obviously-correct definition that the CUDA path is
checked against.  It is used only by ``tests/``, ``__graft_entry__.smoke()`` and
``bench.py``'s CPU-baseline leg; the product path never imports it.

Every floating-point quantity is computed in fp64 from the exact value of its
storage (fp16/bf16 bits, or int8 code times fp16 scale, or 4-bit code times
bf16 scale plus bf16 bias).  Sources, by page title:

* mlxcel issue #1204, "draft a tree instead of a chain": "What this needs"
  (ancestor-only mask, tree-aware walk, tree-aware rollback) and the increments
  that define the topology (parents[i] < i), the history mask [n, offset + n]
  and the path property of the walk.
* mlxcel PR #1212, "draft and verify a token tree, behind a flag, default off":
  the commit messages for the topology/mask/walk, gather_positions (Int8 scale
  sidecars move with their tokens, prefix == trim_to, identity short-circuit),
  the history mask, the -1e9 blocking value, and gather_within_tail.
* mlxcel issue #1185, "cut the MTP drafter's per-step cost": Phase 2a (fused
  LM-head projection + argmax, logits never written) and Phase 3 (affine
  group-64 4-bit weights).
* Splash issue #728, "qualify shared-prefix tree verification": every committed
  token is the target's selection at its path node.

Modules: ``storage`` (exact decoding of stored values), ``tree`` (topology, mask,
walk), ``attention``, ``lm_head``, ``gather``.  Readings of points the pages
leave open are stated in each function's docstring.
"""
from . import attention, gather, lm_head, storage, tree  # noqa: F401
