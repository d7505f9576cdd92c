"""Counter-based random numbers for the synthetic inputs (host side).

Every synthetic tensor element is a pure function of (seed, tensor id, flat
element index), so any slice of any tensor can be regenerated on its own, on
the host or on the device, without generating the rest.  The generator is
SplitMix64 (Steele, Lea and Flood, "Fast splittable pseudorandom number
generators", OOPSLA 2014): the n-th output from state ``s`` is
``mix64(s + n * 0x9E3779B97F4A7C15)`` with the published two-multiply mixer.
Counter-based use reads output ``idx + 1`` of the stream whose state is
``key = mix64(seed * 2**32 + tensor_id)``.

The device side (``synth/csrc/synth_fill.cu``) implements the same published
definition independently; a GPU test compares the two element by element.

The distributions below use integer arithmetic plus at most two IEEE fp32
operations with round-to-nearest-even, so host and device agree bit for bit:

* ``normal_f32``  - Irwin-Hall sum of the four 16-bit lanes of one draw,
  centred (mean 131070) and scaled by the fp32 constant ``NORMAL_SCALE``
  (1 / sqrt(4 * (65536**2 - 1) / 12)); an approximately N(0, 1) value with
  tails cut at about +-3.46.
* ``uniform_f32`` - ``lo + (h >> 40) * 2**-24 * width`` in fp32.
* ``int_below``   - Lemire's multiply-shift ``((h >> 32) * n) >> 32``.

Nothing here computes any step of the verify path.
"""
from __future__ import annotations

import numpy as np

GAMMA = 0x9E3779B97F4A7C15
MIX1 = 0xBF58476D1CE4E5B9
MIX2 = 0x94D049BB133111EB
MASK64 = (1 << 64) - 1

# fp32 bit pattern 0x37ddb3d7 == 1 / 37837.227 (the Irwin-Hall(4) sigma of 16-bit lanes).
NORMAL_SCALE = np.array([0x37DDB3D7], dtype=np.uint32).view(np.float32)[0]
IRWIN_HALL_MEAN = 131070

_U64 = np.uint64


def mix64_int(z: int) -> int:
    """SplitMix64 output mixer on a Python int (mod 2**64)."""
    z &= MASK64
    z = ((z ^ (z >> 30)) * MIX1) & MASK64
    z = ((z ^ (z >> 27)) * MIX2) & MASK64
    return z ^ (z >> 31)


def stream_key(seed: int, tensor_id: int) -> int:
    """State of the stream that belongs to (seed, tensor_id)."""
    return mix64_int(((seed & 0xFFFFFFFF) << 32) + (tensor_id & 0xFFFFFFFF))


def draw(key: int, idx: np.ndarray) -> np.ndarray:
    """64-bit draw number ``idx`` (uint64 array) of the stream ``key``."""
    idx = np.asarray(idx, dtype=_U64)
    with np.errstate(over="ignore"):
        z = _U64(key) + (idx + _U64(1)) * _U64(GAMMA)
        z = (z ^ (z >> _U64(30))) * _U64(MIX1)
        z = (z ^ (z >> _U64(27))) * _U64(MIX2)
    return z ^ (z >> _U64(31))


def draw_int(key: int, idx: int) -> int:
    """Scalar version of :func:`draw` on Python ints."""
    return mix64_int(key + (idx + 1) * GAMMA)


def normal_f32(h: np.ndarray) -> np.ndarray:
    """Approximately N(0,1) fp32 values from 64-bit draws (exact on any IEEE machine)."""
    m = _U64(0xFFFF)
    s = (h & m) + ((h >> _U64(16)) & m) + ((h >> _U64(32)) & m) + (h >> _U64(48))
    c = (s.astype(np.int64) - IRWIN_HALL_MEAN).astype(np.float32)  # |c| < 2**18: exact
    return c * NORMAL_SCALE


def uniform_f32(h: np.ndarray, lo: np.float32, width: np.float32) -> np.ndarray:
    """lo + U[0,1) * width in fp32, the product rounded before the sum."""
    u = (h >> _U64(40)).astype(np.float32) * np.float32(2.0 ** -24)  # exact
    return (u * np.float32(width)) + np.float32(lo)


def int_below(h: np.ndarray, n: int) -> np.ndarray:
    """Integers uniform in [0, n) (n < 2**32) by multiply-shift."""
    return (((h >> _U64(32)) * _U64(n)) >> _U64(32)).astype(np.int64)


def int_below_scalar(h: int, n: int) -> int:
    return ((h >> 32) * n) >> 32


def u01_scalar(h: int) -> float:
    """Uniform [0,1) double with 53 random bits (host-only structure draws)."""
    return (h >> 11) * (2.0 ** -53)


def f32_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round fp32 to bf16 (nearest, ties to even); returns the uint16 bit patterns."""
    u = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32).astype(np.uint64)
    r = (u + _U64(0x7FFF) + ((u >> _U64(16)) & _U64(1))) >> _U64(16)
    return r.astype(np.uint16)


def f32_to_f16_bits(x: np.ndarray) -> np.ndarray:
    """Round fp32 to fp16 (nearest, ties to even); returns the uint16 bit patterns."""
    return np.asarray(x, dtype=np.float32).astype(np.float16).view(np.uint16)
