"""Appending the verify block to the cache: rotary positions and Int8 quantisation (oracle; test infrastructure only).

Definitions followed:

* Positions - mlxcel issue #1185, the closing comment's follow-up list: the tree path verifies the tree at its
  own positions, not at its nodes' slots in the flattened block.  Reading:
  node i sits at position S + depth(i) (the root, the last committed token, at S); for a chain depth(i) = i, the
  chain verify's positions.
* Rotary embedding - the pages name it only through "positions"; the plainest reading is the standard rotary
  embedding of the first rot_dim features: feature pairs (j, j + rot_dim/2) (or (2j, 2j + 1) when interleaved)
  are rotated by the angle pos * base^(-2j / rot_dim).  Applied to Q and to the new K rows; V is not rotated.
* Int8 caches - mlxcel PR #1212, gather_positions commit: one scale per token, and a per-token scale maps every
  single-valued token to the same code.  Reading: symmetric absmax scaling, scale = absmax / 127 (stored as
  fp16), code = round-half-to-even(x / scale) clamped to [-127, 127]; an all-zero token has scale 0 and codes 0.
  The integer decisions are taken in the kernel's precision: absmax / 127 as one fp32 division rounded to fp16,
  x / scale as one fp32 division.
"""
from __future__ import annotations

import numpy as np

from . import tree as _tree


def inv_freq(rot_dim: int, base: float) -> np.ndarray:
    """theta_j = base^(-2j / rot_dim), j < rot_dim / 2, in fp64."""
    j = np.arange(rot_dim // 2, dtype=np.float64)
    return np.power(float(base), -2.0 * j / rot_dim)


def rope(x, pos: int, base: float, rot_dim: int, interleaved: bool = False) -> np.ndarray:
    """Rotate the first rot_dim features of x [..., D] to position ``pos`` (fp64)."""
    x = np.asarray(x, dtype=np.float64)
    out = x.copy()
    ang = float(pos) * inv_freq(rot_dim, base)
    c, s = np.cos(ang), np.sin(ang)
    h = rot_dim // 2
    if interleaved:
        a, b = x[..., 0:rot_dim:2], x[..., 1:rot_dim:2]
        out[..., 0:rot_dim:2] = a * c - b * s
        out[..., 1:rot_dim:2] = b * c + a * s
    else:
        a, b = x[..., :h], x[..., h:rot_dim]
        out[..., :h] = a * c - b * s
        out[..., h:rot_dim] = b * c + a * s
    return out


def node_positions(parents, S: int) -> list[int]:
    """Position of every node: S + depth(i)."""
    return [S + _tree.depth(parents, i) for i in range(len(parents))]


def f16_round(x) -> np.ndarray:
    """Round to the nearest fp16 value (ties to even), returned as fp64."""
    return np.asarray(x, dtype=np.float64).astype(np.float16).astype(np.float64)


def quantize_token(x):
    """One token's symmetric Int8 quantisation: (codes int8 [D], scale as fp16 bits uint16).

    x must hold fp32-representable values (the kernel's inputs); the decisions are taken in fp32.
    """
    x32 = np.asarray(x, dtype=np.float64).astype(np.float32)
    amax = np.float32(np.max(np.abs(x32))) if x32.size else np.float32(0)
    scale = (amax / np.float32(127.0)).astype(np.float16)
    s32 = np.float32(scale)
    if s32 == 0:
        return np.zeros(x32.shape, dtype=np.int8), scale.view(np.uint16)
    q = np.rint(x32 / s32)  # fp32 division, then round half to even
    return np.clip(q, -127, 127).astype(np.int8), scale.view(np.uint16)


def append_block(q, k_new, v_new, parents, S: int, base: float, rot_dim: int, interleaved: bool = False):
    """One (sequence, layer): rotate Q and the new K rows to the nodes' positions.

    q [T, HQ, D], k_new / v_new [T, HKV, D] (fp64 values of the bf16 inputs).  Returns (q_rot, k_rot, v) in fp64,
    the exact values the cache rows and the rotated Q approximate; storage (16-bit rounding or Int8 codes) is the
    caller's choice (``quantize_token``, ``f16_round``).
    """
    pos = node_positions(parents, S)
    q_rot = np.stack([rope(q[i], pos[i], base, rot_dim, interleaved) for i in range(len(pos))])
    k_rot = np.stack([rope(k_new[i], pos[i], base, rot_dim, interleaved) for i in range(len(pos))])
    return q_rot, k_rot, np.asarray(v_new, dtype=np.float64)
