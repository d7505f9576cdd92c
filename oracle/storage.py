"""Exact fp64 values of stored tensors (oracle; test infrastructure only).

Readings (the pages name the formats but do not spell out their arithmetic):

* Int8 KV (mlxcel PR #1212, gather_positions commit; Splash #728 "Int8 KV"):
  symmetric codes with one fp16 scale per token and KV head; value = code * scale.
* 4-bit LM head (mlxcel issue #1185, Phase 3 "affine group-64 4-bit", and the
  cost-model table listing weight, scales and biases): value = scale * q + bias
  with q in [0, 15], one bf16 scale and one bf16 bias per 64 consecutive input
  features.  Packing (our convention): byte j of a row holds element 2j in the
  low nibble and element 2j+1 in the high nibble.
"""
from __future__ import annotations

import numpy as np


def f16(bits) -> np.ndarray:
    """fp16 bit patterns -> exact fp64 values."""
    return np.asarray(bits, dtype=np.uint16).view(np.float16).astype(np.float64)


def bf16(bits) -> np.ndarray:
    """bf16 bit patterns -> exact fp64 values (bf16 is the top half of an fp32)."""
    u = np.asarray(bits, dtype=np.uint16).astype(np.uint32) << np.uint32(16)
    return u.view(np.float32).astype(np.float64)


def int8_scaled(codes, scale_bits) -> np.ndarray:
    """Int8 codes [..., N, D] with fp16 per-token scales [..., N] -> fp64 values."""
    return np.asarray(codes, dtype=np.int8).astype(np.float64) * f16(scale_bits)[..., None]


def unpack_q4(packed) -> np.ndarray:
    """uint8 [R, H/2] -> int codes [R, H]; element 2j is the low nibble of byte j."""
    p = np.asarray(packed, dtype=np.uint8).astype(np.int64)
    out = np.empty(p.shape[:-1] + (p.shape[-1] * 2,), dtype=np.int64)
    out[..., 0::2] = p & 0xF
    out[..., 1::2] = p >> 4
    return out


def q4_affine(packed, scale_bits, bias_bits, group: int = 64) -> np.ndarray:
    """Affine group-wise 4-bit weights -> fp64 [R, H]: w = scale[g] * q + bias[g]."""
    q = unpack_q4(packed).astype(np.float64)
    s = np.repeat(bf16(scale_bits), group, axis=-1)
    b = np.repeat(bf16(bias_bits), group, axis=-1)
    return s * q + b


def kv_values(dtype: int, store, scale_bits=None) -> np.ndarray:
    """KV storage of format ``dtype`` (0 fp16, 1 bf16, 2 int8+scales) -> fp64."""
    if dtype == 0:
        return f16(store)
    if dtype == 1:
        return bf16(store)
    if dtype == 2:
        return int8_scaled(store, scale_bits)
    raise ValueError(f"not a KV format: {dtype}")


def round_bf16(x) -> np.ndarray:
    """fp64 values rounded to the nearest bf16 value (8 significant bits, ties to even; normal range)."""
    m, e = np.frexp(np.asarray(x, dtype=np.float64))
    return np.ldexp(np.rint(np.ldexp(m, 8)), e - 8)


def round_f16(x) -> np.ndarray:
    """fp64 values rounded to the nearest fp16 value (numpy's correctly rounded conversion)."""
    return np.asarray(x, dtype=np.float64).astype(np.float16).astype(np.float64)
