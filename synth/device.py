"""Writes synthetic tensors straight into GPU memory (same formulas as synth.tensors).

Used for workloads whose caches and heads are too large to generate on the
host (up to ~140 GB).  Any slice can be regenerated on the host with
``synth.tensors`` for checking.
"""
from __future__ import annotations

import ctypes as C
import os

import torch

from . import tensors as st
from .configs import BF16, F16, I8, Q4, Config

LIB_PATH = os.path.join(os.path.dirname(os.path.abspath(__file__)), "libtsv_synth.so")
NORMAL_F16, NORMAL_BF16, INT8_CODE, UNIFORM_F16, UNIFORM_BF16, Q4_PACKED, Q4_BIAS = range(7)

_lib = None


def lib():
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(f"{LIB_PATH} missing: build with __graft_entry__.build()")
        _lib = C.CDLL(LIB_PATH)
        _lib.tsv_synth_fill.restype = C.c_int
        _lib.tsv_synth_fill.argtypes = [C.c_void_p, C.c_int, C.c_uint64, C.c_uint64] + [C.c_int64] * 7 + \
            [C.c_float] * 4 + [C.c_void_p]
        _lib.tsv_synth_copy_table.restype = C.c_int
        _lib.tsv_synth_copy_table.argtypes = [C.c_void_p, C.c_int, C.c_void_p]
    return _lib


def fill(t: torch.Tensor, dist: int, key: int, n, strides, p=(1.0, 0.0, 0.0, 0.0), key2: int = 0):
    n0, n1, n2, n3 = n
    s0, s1, s2 = strides
    err = lib().tsv_synth_fill(C.c_void_p(t.data_ptr()), dist, key, key2, n0, n1, n2, n3, s0, s1, s2,
                               *[float(x) for x in p], C.c_void_p(torch.cuda.current_stream().cuda_stream))
    if err != 0:
        raise RuntimeError(f"tsv_synth_fill failed with CUDA error {err}")


def _kv_dist(cfg: Config):
    return {F16: NORMAL_F16, BF16: NORMAL_BF16, I8: INT8_CODE}[cfg.kv_dtype]


def alloc_cache(cfg: Config, layer: int, s_cap: int, device) -> dict:
    """K, V (and Int8 scales) of one layer, [B, HKV, s_cap, D], logical rows [0, S+T) filled."""
    B, HKV, D, N = cfg.B, cfg.HKV, cfg.D, cfg.NKV
    dt = {F16: torch.float16, BF16: torch.bfloat16, I8: torch.int8}[cfg.kv_dtype]
    out = {}
    for which, kind in (("k", st.KIND_K), ("v", st.KIND_V)):
        t = torch.zeros(B, HKV, s_cap, D, dtype=dt, device=device)
        fill(t, _kv_dist(cfg), st.key(cfg, kind, layer), (B, HKV, N, D), (HKV * s_cap * D, s_cap * D, D))
        out[which] = t
    if cfg.kv_dtype == I8:
        for which, kind in (("ks", st.KIND_KS), ("vs", st.KIND_VS)):
            t = torch.zeros(B, HKV, s_cap, dtype=torch.float16, device=device)
            fill(t, UNIFORM_F16, st.key(cfg, kind, layer), (1, B, HKV, N), (0, HKV * s_cap, s_cap),
                 (float(st.KV_SCALE_LO), float(st.KV_SCALE_W), 0.0, 0.0))
            out[which] = t
    return out


def alloc_q(cfg: Config, layer: int, device, out: torch.Tensor | None = None) -> torch.Tensor:
    """Q of one layer [B, T, HQ, D] bf16, filled into ``out`` when given (a view into a larger buffer)."""
    t = out if out is not None else torch.empty(cfg.B, cfg.T, cfg.HQ, cfg.D, dtype=torch.bfloat16, device=device)
    fill(t, NORMAL_BF16, st.key(cfg, st.KIND_Q, layer), (1, 1, cfg.B * cfg.T * cfg.HQ, cfg.D), (0, 0, cfg.D))
    return t


def alloc_new_kv(cfg: Config, layer: int, device, out: dict | None = None) -> dict:
    """The block's new K and V rows [B, T, HKV, D] bf16 (inputs of the block append), filled into ``out``'s
    tensors when given."""
    res = {}
    for which, kind in (("k_new", st.KIND_KNEW), ("v_new", st.KIND_VNEW)):
        t = out[which] if out is not None else torch.empty(cfg.B, cfg.T, cfg.HKV, cfg.D, dtype=torch.bfloat16,
                                                            device=device)
        fill(t, NORMAL_BF16, st.key(cfg, kind, layer), (1, 1, cfg.B * cfg.T * cfg.HKV, cfg.D), (0, 0, cfg.D))
        res[which] = t
    return res


def alloc_head(cfg: Config, device) -> dict:
    V, H = cfg.V, cfg.H
    if cfg.w_dtype == Q4:
        w = torch.empty(V, H // 2, dtype=torch.uint8, device=device)
        fill(w, Q4_PACKED, st.key(cfg, st.KIND_WQ), (1, 1, V, H // 2), (0, 0, H // 2))
        s = torch.empty(V, H // 64, dtype=torch.bfloat16, device=device)
        fill(s, UNIFORM_BF16, st.key(cfg, st.KIND_WS), (1, 1, V, H // 64), (0, 0, H // 64),
             (float(st.WS_LO), float(st.WS_W), 0.0, 0.0))
        b = torch.empty(V, H // 64, dtype=torch.bfloat16, device=device)
        fill(b, Q4_BIAS, st.key(cfg, st.KIND_WB), (1, 1, V, H // 64), (0, 0, H // 64),
             (float(st.WB_LO), float(st.WB_W), float(st.WS_LO), float(st.WS_W)), key2=st.key(cfg, st.KIND_WS))
        return dict(W=w, scales=s, biases=b)
    dt = torch.bfloat16 if cfg.w_dtype == BF16 else torch.float16
    w = torch.empty(V, H, dtype=dt, device=device)
    fill(w, NORMAL_BF16 if cfg.w_dtype == BF16 else NORMAL_F16, st.key(cfg, st.KIND_W), (1, 1, V, H), (0, 0, H),
         (float(st.W_SIGMA), 0.0, 0.0, 0.0))
    return dict(W=w, scales=None, biases=None)


def copy_table(table: torch.Tensor):
    """Run the copies listed in ``table`` (int64 [n, 3] on the device: src, dst, bytes) in one launch."""
    err = lib().tsv_synth_copy_table(C.c_void_p(table.data_ptr()), table.shape[0],
                                     C.c_void_p(torch.cuda.current_stream().cuda_stream))
    if err != 0:
        raise RuntimeError(f"tsv_synth_copy_table failed with CUDA error {err}")
