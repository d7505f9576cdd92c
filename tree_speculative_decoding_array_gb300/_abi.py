"""ctypes declarations of the tsv C ABI (include/tsv.h).

Loading fails loudly when ``libtsv.so`` has not been built: there is no
fallback implementation of any call.
"""
from __future__ import annotations

import ctypes as C
import os

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libtsv.so")

OK, EINVAL, ETOPOLOGY, EUNSUPPORTED, ECAPACITY, ECUDA = range(6)
F16, BF16, I8_SCALED, Q4_G64 = range(4)
DEV_OK, DEV_BAD_ROOT, DEV_BAD_PARENT, DEV_BAD_PATH, DEV_BAD_KV_LEN, DEV_TIMEOUT = range(6)
ATTN_AUTO, ATTN_SIMT, ATTN_TCGEN05, ATTN_TCGEN05_64, ATTN_TCGEN05_128 = range(5)
MAX_T = 64
MAX_CANDIDATES = 1024
MAX_LAYERS = 64
NOALLOC_MAX_ROWS = 4096

STATUS_NAMES = {OK: "TSV_OK", EINVAL: "TSV_EINVAL", ETOPOLOGY: "TSV_ETOPOLOGY", EUNSUPPORTED: "TSV_EUNSUPPORTED",
                ECAPACITY: "TSV_ECAPACITY", ECUDA: "TSV_ECUDA"}

# Every exported symbol with (restype, argtypes); tests check the .so exports them all.
_vp, _i32, _i64, _sz = C.c_void_p, C.c_int32, C.c_int64, C.c_size_t


class AttnDesc(C.Structure):
    _fields_ = [
        ("n_layers", _i32), ("B", _i32), ("T", _i32), ("HQ", _i32), ("HKV", _i32), ("D", _i32),
        ("s_cap", _i64), ("max_kv_len", _i32), ("kv_dtype", _i32), ("splits", _i32), ("path", _i32),
        ("q", _vp * MAX_LAYERS), ("k", _vp * MAX_LAYERS), ("v", _vp * MAX_LAYERS),
        ("k_scale", _vp * MAX_LAYERS), ("v_scale", _vp * MAX_LAYERS), ("o", _vp * MAX_LAYERS),
        ("kv_len", _vp), ("anc", _vp), ("window", _i32 * MAX_LAYERS),
    ]


class KvDesc(C.Structure):
    _fields_ = [
        ("n_layers", _i32), ("B", _i32), ("HKV", _i32), ("D", _i32), ("s_cap", _i64), ("kv_dtype", _i32),
        ("reserved", _i32),
        ("k", _vp * MAX_LAYERS), ("v", _vp * MAX_LAYERS), ("k_scale", _vp * MAX_LAYERS), ("v_scale", _vp * MAX_LAYERS),
    ]


class AppendDesc(C.Structure):
    _fields_ = [
        ("n_layers", _i32), ("B", _i32), ("T", _i32), ("HQ", _i32), ("HKV", _i32), ("D", _i32), ("s_cap", _i64),
        ("kv_dtype", _i32), ("rot_dim", _i32), ("interleaved", _i32), ("reserved", _i32), ("rope_base", C.c_double),
        ("q_in", _vp * MAX_LAYERS), ("q_out", _vp * MAX_LAYERS), ("k_new", _vp * MAX_LAYERS),
        ("v_new", _vp * MAX_LAYERS), ("k", _vp * MAX_LAYERS), ("v", _vp * MAX_LAYERS),
        ("k_scale", _vp * MAX_LAYERS), ("v_scale", _vp * MAX_LAYERS), ("depth", _vp),
    ]


SIGNATURES = {
    "tsv_last_error": (C.c_char_p, []),
    "tsv_version": (C.c_int, []),
    "tsv_selftest_bounded_wait": (C.c_int, [_vp, _vp]),
    "tsv_tree_mask": (C.c_int, [_vp, _i32, _i32, _vp, _vp, _vp, _i32, _vp, _vp]),
    "tsv_sliding_band_mask": (C.c_int, [_vp, _i32, _i32, _i32, _i32, _vp]),
    "tsv_draft_children_workspace_size": (_sz, [_i32, _i32, _i32]),
    "tsv_draft_children": (C.c_int, [_vp, _i32, _i32, _i32, _vp, _vp, _vp, _sz, _vp]),
    "tsv_tree_select": (C.c_int, [_vp, _vp, _vp, _i32, _i32, _i32, _i32, _vp, _vp, _vp, _vp, _vp, _vp]),
    "tsv_attention_workspace_size": (_sz, [C.POINTER(AttnDesc)]),
    "tsv_tree_verify_attention": (C.c_int, [C.POINTER(AttnDesc), _vp, _sz, _vp, _vp]),
    "tsv_lm_head_workspace_size": (_sz, [_i32, _i32, _i32, _i32]),
    "tsv_lm_head_argmax": (C.c_int, [_vp, _i32, _i32, _i32, _i32, _vp, _vp, _vp, _vp, _vp, _vp, _sz, _vp]),
    "tsv_lm_head_logits": (C.c_int, [_vp, _i32, _i32, _i32, _i32, _vp, _vp, _vp, _vp, _vp, _sz, _vp]),
    "tsv_sample_workspace_size": (_sz, [_i32, _i32, _i32]),
    "tsv_sample_nucleus": (C.c_int, [_vp, _i32, _i32, C.c_float, _i32, C.c_float, _vp, _vp, _vp, _sz, _vp]),
    "tsv_lm_head_argmax_noalloc": (C.c_int, [_vp, _i32, _i32, _i32, _i32, _vp, _vp, _vp, _vp, _vp, _vp]),
    "tsv_tree_accept_walk": (C.c_int, [_vp, _vp, _vp, _i32, _i32, _vp, _vp, _vp, _vp, _vp]),
    "tsv_kv_gather_positions": (C.c_int, [C.POINTER(KvDesc), _vp, _vp, _vp, _i32, _vp, _vp]),
    "tsv_gather_positions": (C.c_int, [C.POINTER(KvDesc), _vp, _vp, _vp, _i32, _vp, _vp]),
    "tsv_tree_append": (C.c_int, [C.POINTER(AppendDesc), _vp, _vp, _vp]),
}

_lib = None


class TsvError(RuntimeError):
    def __init__(self, status: int, where: str, reason: str):
        self.status = status
        super().__init__(f"{where}: {STATUS_NAMES.get(status, status)}: {reason}")


def load(path: str = LIB_PATH) -> C.CDLL:
    """Load libtsv.so (once).  Raises if it is missing: build it with __graft_entry__.build()."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(path):
        raise RuntimeError(f"{path} is missing: the tsv CUDA library must be built "
                           "(python -c 'import __graft_entry__ as g; g.build()'); there is no fallback")
    lib = C.CDLL(path)
    for name, (res, args) in SIGNATURES.items():
        f = getattr(lib, name)
        f.restype = res
        f.argtypes = args
    _lib = lib
    return lib


def check(status: int, where: str) -> None:
    if status != OK:
        raise TsvError(status, where, load().tsv_last_error().decode())
