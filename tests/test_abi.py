"""The C-ABI library without a GPU: it loads, exports every declared symbol, its struct layouts match the
ctypes binding, and host-side argument validation refuses bad calls before touching the device."""
import ctypes as C
import os
import re
import shutil
import subprocess

import pytest

import tree_speculative_decoding_array_gb300 as tsv
from tree_speculative_decoding_array_gb300 import _abi

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "tsv.h")


def declared_functions():
    src = open(HEADER).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(tsv_[a-z_0-9]+)\s*\(", src)))


def test_every_declared_symbol_is_exported():
    lib = tsv.load()
    names = declared_functions()
    assert len(names) >= 9
    for n in names:
        assert hasattr(lib, n), n
    assert set(names) == set(_abi.SIGNATURES), "binding and header disagree"


def test_version_and_error_string():
    lib = tsv.load()
    assert lib.tsv_version() == 102
    assert lib.tsv_last_error() == b""


@pytest.mark.skipif(shutil.which("gcc") is None, reason="gcc not available")
def test_struct_layouts_match_header(tmp_path):
    fields = {"tsv_attn_desc": _abi.AttnDesc, "tsv_kv_desc": _abi.KvDesc, "tsv_append_desc": _abi.AppendDesc}
    lines = ["#include <stdio.h>", "#include <stddef.h>", '#include "tsv.h"', "int main(void){"]
    for cname, py in fields.items():
        lines.append(f'printf("{cname} %zu\\n", sizeof({cname}));')
        for f, _ in py._fields_:
            lines.append(f'printf("{cname}.{f} %zu\\n", offsetof({cname}, {f}));')
    lines.append("return 0;}")
    c = tmp_path / "layout.c"
    c.write_text("\n".join(lines))
    exe = tmp_path / "layout"
    cuda_inc = "/usr/local/cuda/include"
    subprocess.run(["gcc", "-I", os.path.join(ROOT, "include"), "-I", cuda_inc, str(c), "-o", str(exe)], check=True)
    out = subprocess.run([str(exe)], capture_output=True, text=True, check=True).stdout.split("\n")
    got = dict(l.split() for l in out if l.strip())
    for cname, py in fields.items():
        assert int(got[cname]) == C.sizeof(py)
        for f, _ in py._fields_:
            assert int(got[f"{cname}.{f}"]) == getattr(py, f).offset, f


def test_host_validation_refuses_without_launching():
    lib = tsv.load()
    # T above the 64-node maximum
    st = lib.tsv_tree_mask(C.c_void_p(16), 1, 65, C.c_void_p(16), C.c_void_p(16), None, 0, None, None)
    assert st == _abi.ECAPACITY and b"64" in lib.tsv_last_error()
    st = lib.tsv_tree_mask(None, 1, 3, None, None, None, 0, None, None)
    assert st == _abi.EINVAL
    st = lib.tsv_tree_accept_walk(None, None, None, 1, 0, None, None, None, None, None)
    assert st == _abi.ECAPACITY
    d = _abi.AttnDesc()
    st = lib.tsv_tree_verify_attention(C.byref(d), None, 0, None, None)
    assert st == _abi.ECAPACITY  # n_layers = 0
    d.n_layers, d.B, d.T, d.HQ, d.HKV, d.D, d.kv_dtype = 1, 1, 4, 8, 2, 96, 0
    st = lib.tsv_tree_verify_attention(C.byref(d), None, 0, None, None)
    assert st == _abi.EUNSUPPORTED and b"96" in lib.tsv_last_error()
    d.D, d.kv_dtype = 64, 3  # a weight format for a cache
    assert lib.tsv_tree_verify_attention(C.byref(d), None, 0, None, None) == _abi.EUNSUPPORTED
    d.kv_dtype, d.max_kv_len, d.s_cap, d.window[0] = 0, 8, 8, -1  # a negative sliding window
    st = lib.tsv_tree_verify_attention(C.byref(d), None, 0, None, None)
    assert st == _abi.EINVAL and b"window" in lib.tsv_last_error()
    assert lib.tsv_sliding_band_mask(None, 1, 4, 10, 0, None) == _abi.EINVAL  # window must be >= 1
    assert lib.tsv_sliding_band_mask(None, 1, 4, 10, 14, None) == _abi.OK  # below the window: untouched
    assert lib.tsv_sliding_band_mask(None, 1, 4, 10, 13, None) == _abi.EINVAL  # past it: needs the mask
    k = _abi.KvDesc()
    k.n_layers, k.B, k.HKV, k.D, k.s_cap, k.kv_dtype = 1, 1, 1, 64, 10, 3
    st = lib.tsv_kv_gather_positions(C.byref(k), C.c_void_p(16), C.c_void_p(16), C.c_void_p(16), 4, None, None)
    assert st == _abi.EUNSUPPORTED and b"gather" in lib.tsv_last_error()
    st = lib.tsv_gather_positions(C.byref(k), C.c_void_p(16), C.c_void_p(16), C.c_void_p(16), 4, None, None)
    assert st == _abi.EUNSUPPORTED and b"gather" in lib.tsv_last_error()  # absolute form: same refusal
    k.kv_dtype = 0
    assert lib.tsv_gather_positions(C.byref(k), C.c_void_p(16), C.c_void_p(16), C.c_void_p(16), -1, None,
                                    None) == _abi.EINVAL  # negative max_kept
    assert lib.tsv_gather_positions(C.byref(k), C.c_void_p(16), None, C.c_void_p(16), 4, None,
                                    None) == _abi.EINVAL  # no kept list for max_kept > 0
    k.B = 0
    assert lib.tsv_gather_positions(C.byref(k), None, None, None, 4, None, None) == _abi.OK  # empty batch
    st = lib.tsv_lm_head_argmax(C.c_void_p(16), 1, 100, 10, 1, C.c_void_p(16), None, None, C.c_void_p(16), None,
                                C.c_void_p(16), 64, None)
    assert st == _abi.EINVAL  # H not a multiple of 256
    st = lib.tsv_lm_head_argmax(C.c_void_p(16), 1, 256, 10, 1, C.c_void_p(16), None, None, C.c_void_p(16), None,
                                C.c_void_p(16), 0, None)
    assert st == _abi.ECAPACITY  # workspace too small
    a = _abi.AppendDesc()
    a.n_layers, a.B, a.T, a.HQ, a.HKV, a.D, a.s_cap, a.kv_dtype, a.rot_dim, a.rope_base = 1, 1, 4, 8, 2, 64, 16, 0, 63, 1e4
    st = lib.tsv_tree_append(C.byref(a), C.c_void_p(16), None, None)
    assert st == _abi.EINVAL and b"rot_dim" in lib.tsv_last_error()  # odd rotary width
    a.rot_dim, a.rope_base = 64, 0.0
    assert lib.tsv_tree_append(C.byref(a), C.c_void_p(16), None, None) == _abi.EINVAL
    a.rope_base, a.D = 1e4, 96
    assert lib.tsv_tree_append(C.byref(a), C.c_void_p(16), None, None) == _abi.EUNSUPPORTED
    assert lib.tsv_lm_head_workspace_size(3, 256, 1000, 1) >= 24
    assert lib.tsv_lm_head_workspace_size(16, 512, 1000, 3) >= 16 * 8 + 16 * 512 * 2  # fp16 copy of hidden
    # which kernel a row count selects shows in the workspace it asks for: the tensor-core kernels take every
    # 4-bit head whose H is a multiple of 512 (an fp16 copy of hidden beside the bests) and 16-bit heads above 4
    # rows (fp16 heads need the copy, bf16 heads none); below, the CUDA-core GEMV needs only the bests
    ws = lib.tsv_lm_head_workspace_size
    assert ws(1, 512, 1000, 3) == 256 + 1024 and ws(3, 512, 1000, 3) == 256 + 3072
    assert ws(3, 256, 1000, 3) == 256  # H not a multiple of 512: GEMV
    assert ws(4, 256, 1000, 0) == 256 and ws(5, 256, 1000, 0) == 256 + 2560
    assert ws(8, 256, 1000, 1) == 256
