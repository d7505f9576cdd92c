"""Element formulas of every synthetic tensor, and host generation of any slice.

A tensor is named by (kind, layer) -> a 32-bit tensor id; element ``i`` of its
*logical* flat index gets ``dist(draw(stream_key(seed, id), i))``.  Logical
shapes (row-major, no capacity padding):

====  =======  ==========================  ===========================================
kind  name     logical shape               value
====  =======  ==========================  ===========================================
1     Q        [B, T, HQ, D]               bf16(normal)
2     K        [B, HKV, S+T, D]            fp16/bf16(normal) or int8 code in [-127,127]
3     V        [B, HKV, S+T, D]            as K
4     KS       [B, HKV, S+T]               fp16(U(0.005, 0.05))   (Int8 caches only)
5     VS       [B, HKV, S+T]               as KS
6     W        [V, H]                      fp16/bf16(0.02 * normal)
7     WQ       [V, H] 4-bit codes          int in [0, 16); byte j of a row packs
                                           element 2j (low nibble) and 2j+1 (high)
8     WS       [V, H/64]                   bf16(U(0.005, 0.008))
9     WB       [V, H/64]                   bf16(-(U(7, 8) * float(WS)))
10    HN       [B*T, H]                    normal noise of the hidden states
====  =======  ==========================  ===========================================

The device fill kernels in ``synth/csrc/synth_fill.cu`` write the same values;
storage formats are returned here as raw bit patterns (uint16 for fp16/bf16,
int8 codes, uint8 packed nibbles) so that nothing in this module interprets them.
"""
from __future__ import annotations

import numpy as np

from . import rng
from .configs import BF16, F16, I8, Q4, Config

KIND_Q, KIND_K, KIND_V, KIND_KS, KIND_VS, KIND_W, KIND_WQ, KIND_WS, KIND_WB, KIND_HN = range(1, 11)
KIND_TREE, KIND_TOK = 11, 12
KIND_KNEW, KIND_VNEW = 13, 14  # the block's K and V rows before the append (K not yet rotated)
KIND_U = 15  # per-node uniforms of sampled verification
KIND_DRAFT = 16  # synthetic drafter logits (tree construction)

W_SIGMA = np.float32(0.02)
KV_SCALE_LO, KV_SCALE_W = np.float32(0.005), np.float32(0.045)
WS_LO, WS_W = np.float32(0.005), np.float32(0.003)
WB_LO, WB_W = np.float32(7.0), np.float32(1.0)

CHUNK = 1 << 22


def tensor_id(kind: int, layer: int = 0) -> int:
    return (kind << 16) | (layer & 0xFFFF)


def key(cfg: Config, kind: int, layer: int = 0) -> int:
    return rng.stream_key(cfg.seed, tensor_id(kind, layer))


def _draws(k: int, idx: np.ndarray) -> np.ndarray:
    return rng.draw(k, idx.astype(np.uint64))


def _normal_bits(h: np.ndarray, fmt: int, mul: np.float32 = np.float32(1.0)) -> np.ndarray:
    x = rng.normal_f32(h) * np.float32(mul)
    return rng.f32_to_bf16_bits(x) if fmt == BF16 else rng.f32_to_f16_bits(x)


def bits_for_index(k: int, idx: np.ndarray, fmt: int, mul=np.float32(1.0)) -> np.ndarray:
    """Storage values (uint16 bits or int8 codes) of logical elements ``idx``."""
    h = _draws(k, idx)
    if fmt == I8:
        return (rng.int_below(h, 255) - 127).astype(np.int8)
    return _normal_bits(h, fmt, mul)


# ----------------------------------------------------------------------------- attention inputs
def q_rows(cfg: Config, layer: int, b: int, node: int, heads) -> np.ndarray:
    """bf16 bits of Q[b, node, heads, :] -> uint16[len(heads), D]."""
    heads = np.asarray(heads, dtype=np.int64)
    base = ((b * cfg.T + node) * cfg.HQ + heads) * cfg.D
    idx = base[:, None] + np.arange(cfg.D, dtype=np.int64)[None, :]
    return bits_for_index(key(cfg, KIND_Q, layer), idx, BF16)


def q_full(cfg: Config, layer: int) -> np.ndarray:
    n = cfg.B * cfg.T * cfg.HQ * cfg.D
    out = _gen_flat(key(cfg, KIND_Q, layer), n, BF16)
    return out.reshape(cfg.B, cfg.T, cfg.HQ, cfg.D)


def node_uniforms(cfg: Config, round_id: int) -> np.ndarray:
    """fp32 uniforms in [0, 1), one per node of the round ([B * T]), for sampled verification."""
    idx = np.arange(cfg.B * cfg.T, dtype=np.int64) + np.int64(round_id) * (cfg.B * cfg.T)
    return rng.uniform_f32(_draws(key(cfg, KIND_U), idx), 0.0, 1.0)


def new_kv_rows(cfg: Config, which: str, layer: int, b: int, node: int) -> np.ndarray:
    """bf16 bits of the new K or V rows [b, node, :, :] handed to the block append -> uint16[HKV, D]."""
    kind = KIND_KNEW if which == "k" else KIND_VNEW
    base = ((b * cfg.T + node) * cfg.HKV + np.arange(cfg.HKV, dtype=np.int64)) * cfg.D
    idx = base[:, None] + np.arange(cfg.D, dtype=np.int64)[None, :]
    return bits_for_index(key(cfg, kind, layer), idx, BF16)


def kv_rows(cfg: Config, which: str, layer: int, b: int, kvh: int, c0: int, c1: int) -> np.ndarray:
    """Storage of K or V[b, kvh, c0:c1, :] (uint16 bits or int8 codes)."""
    kind = KIND_K if which == "k" else KIND_V
    base = ((b * cfg.HKV + kvh) * cfg.NKV + np.arange(c0, c1, dtype=np.int64)) * cfg.D
    idx = base[:, None] + np.arange(cfg.D, dtype=np.int64)[None, :]
    return bits_for_index(key(cfg, kind, layer), idx, cfg.kv_dtype)


def kv_scales(cfg: Config, which: str, layer: int, b: int, kvh: int, c0: int, c1: int) -> np.ndarray:
    """fp16 bits of the per-token scales of K or V[b, kvh, c0:c1]."""
    kind = KIND_KS if which == "k" else KIND_VS
    idx = (b * cfg.HKV + kvh) * cfg.NKV + np.arange(c0, c1, dtype=np.int64)
    h = _draws(key(cfg, kind, layer), idx)
    return rng.f32_to_f16_bits(rng.uniform_f32(h, KV_SCALE_LO, KV_SCALE_W))


def kv_full(cfg: Config, which: str, layer: int) -> np.ndarray:
    """Whole logical K or V of one layer, [B, HKV, S+T, D] (small configs)."""
    kind = KIND_K if which == "k" else KIND_V
    n = cfg.B * cfg.HKV * cfg.NKV * cfg.D
    out = _gen_flat(key(cfg, kind, layer), n, cfg.kv_dtype)
    return out.reshape(cfg.B, cfg.HKV, cfg.NKV, cfg.D)


def kv_scales_full(cfg: Config, which: str, layer: int) -> np.ndarray:
    out = np.concatenate([kv_scales(cfg, which, layer, b, h, 0, cfg.NKV)
                          for b in range(cfg.B) for h in range(cfg.HKV)])
    return out.reshape(cfg.B, cfg.HKV, cfg.NKV)


def _gen_flat(k: int, n: int, fmt: int, mul=np.float32(1.0)) -> np.ndarray:
    dt = np.int8 if fmt == I8 else np.uint16
    out = np.empty(n, dtype=dt)
    for s in range(0, n, CHUNK):
        e = min(n, s + CHUNK)
        out[s:e] = bits_for_index(k, np.arange(s, e, dtype=np.int64), fmt, mul)
    return out


# ----------------------------------------------------------------------------- LM head inputs
def w_rows(cfg: Config, rows) -> np.ndarray:
    """fp16/bf16 bits of W[rows, :] (w_dtype F16/BF16)."""
    rows = np.asarray(rows, dtype=np.int64)
    idx = rows[:, None] * cfg.H + np.arange(cfg.H, dtype=np.int64)[None, :]
    return bits_for_index(key(cfg, KIND_W), idx, cfg.w_dtype, W_SIGMA)


def w_direction(cfg: Config, rows) -> np.ndarray:
    """Unit-variance fp32 direction correlated with W[rows] (used only for planting).

    For fp16/bf16 heads it is the normal draw before the 0.02 scaling; for 4-bit
    heads the centred code ``q - 7.5``.
    """
    rows = np.asarray(rows, dtype=np.int64)
    idx = rows[:, None] * cfg.H + np.arange(cfg.H, dtype=np.int64)[None, :]
    if cfg.w_dtype == Q4:
        h = _draws(key(cfg, KIND_WQ), idx)
        return (rng.int_below(h, 16).astype(np.float32) - np.float32(7.5)) * np.float32(0.2169304578186)
    return rng.normal_f32(_draws(key(cfg, KIND_W), idx))


def wq_codes(cfg: Config, rows) -> np.ndarray:
    """4-bit codes of W[rows, :] as int64 [len(rows), H] (unpacked)."""
    rows = np.asarray(rows, dtype=np.int64)
    idx = rows[:, None] * cfg.H + np.arange(cfg.H, dtype=np.int64)[None, :]
    return rng.int_below(_draws(key(cfg, KIND_WQ), idx), 16)


def wq_packed(cfg: Config, rows) -> np.ndarray:
    """Packed nibbles uint8 [len(rows), H/2]: element 2j low nibble, 2j+1 high nibble."""
    c = wq_codes(cfg, rows)
    return (c[:, 0::2] | (c[:, 1::2] << 4)).astype(np.uint8)


def wq_scales_biases(cfg: Config, rows):
    """bf16 bits of the group scales and biases of W[rows], each [len(rows), H/64]."""
    rows = np.asarray(rows, dtype=np.int64)
    ng = cfg.H // 64
    idx = rows[:, None] * ng + np.arange(ng, dtype=np.int64)[None, :]
    s_bits = rng.f32_to_bf16_bits(rng.uniform_f32(_draws(key(cfg, KIND_WS), idx), WS_LO, WS_W))
    s_f32 = (s_bits.astype(np.uint32) << np.uint32(16)).view(np.float32)
    t = rng.uniform_f32(_draws(key(cfg, KIND_WB), idx), WB_LO, WB_W)
    b_bits = rng.f32_to_bf16_bits(-(t * s_f32))
    return s_bits, b_bits


def w_full(cfg: Config):
    """Whole LM head (small configs): bits [V,H], or (packed, scales, biases) for 4-bit."""
    rows = np.arange(cfg.V)
    if cfg.w_dtype == Q4:
        s, b = wq_scales_biases(cfg, rows)
        return wq_packed(cfg, rows), s, b
    return w_rows(cfg, rows)


def hidden_noise(cfg: Config, round_id: int, rows) -> np.ndarray:
    rows = np.asarray(rows, dtype=np.int64)
    idx = rows[:, None] * cfg.H + np.arange(cfg.H, dtype=np.int64)[None, :]
    return rng.normal_f32(_draws(key(cfg, KIND_HN, round_id), idx))
