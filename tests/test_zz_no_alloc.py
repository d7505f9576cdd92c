"""The LM-head entry point that allocates nothing (tsv_lm_head_argmax_noalloc), through the C ABI.

Some callers cannot allocate device memory themselves (their host framework owns every device buffer through
its own pool, or their latency budget cannot absorb cudaMalloc's implicit synchronisation).  For them the
library keeps the LM head's scratch in a fixed device array.  This test compares that entry point with the
workspace entry point on five calls in a row, with different row counts so that entries left over from one
call would show up in the next, in every weight format, on both sides of the point where the tensor-core
kernel's fp16 copy of hidden no longer fits the fixed array.
It runs last in the suite and also passes alone in a fresh process.
"""
import ctypes as C

import numpy as np
import pytest
import torch

pytestmark = pytest.mark.gpu


def _p(t):
    return C.c_void_p(t.data_ptr()) if t is not None else None


def test_noalloc_matches_workspace_entry_point(gpu_lib):
    lib = gpu_lib.load()
    stream = C.c_void_p(torch.cuda.current_stream().cuda_stream)
    V, H = 5003, 512
    # 13 bf16 rows and 3 4-bit rows take the tensor-core kernels in both calls (bf16 needs no copy of hidden, and
    # 3 x 512 x 2 bytes fit the 32 KiB array); 2 fp16 rows take the CUDA-core GEMV in both; 40 4-bit and 37 fp16
    # rows overflow the array (40 KB, 37 KB), so the no-alloc call streams the head once per 8 rows through the
    # CUDA-core kernel while the workspace call takes the tensor-core one
    for call, (rows, w_dtype) in enumerate([(13, 1), (3, 3), (40, 3), (2, 0), (37, 0)]):
        rng = np.random.default_rng(100 + call)
        target = rng.integers(0, V, size=rows)
        if w_dtype == 3:
            codes = rng.integers(0, 16, size=(V, H))
            W = torch.from_numpy((codes[:, 0::2] | (codes[:, 1::2] << 4)).astype(np.uint8)).cuda()
            sc = torch.from_numpy(rng.uniform(0.005, 0.008, size=(V, H // 64)).astype(np.float32)).to(torch.bfloat16).cuda()
            bi = torch.from_numpy(rng.uniform(-0.06, -0.05, size=(V, H // 64)).astype(np.float32)).to(torch.bfloat16).cuda()
            direction = (codes[target] - 7.5) / 4.6
        else:
            w = rng.standard_normal((V, H))
            W = torch.from_numpy((w * 0.05).astype(np.float32)).to(torch.bfloat16 if w_dtype == 1 else torch.float16).cuda()
            sc = bi = None
            direction = w[target]
        # each row leans towards its own target row, so the two kernels' roundings cannot swap the argmax
        h = rng.standard_normal((rows, H)) + 2.0 * direction
        hidden = torch.from_numpy(h.astype(np.float32)).to(torch.bfloat16).cuda()
        ref_arg = torch.full((rows,), -7, dtype=torch.int32, device="cuda")
        ref_max = torch.zeros(rows, dtype=torch.float32, device="cuda")
        ws = torch.empty(lib.tsv_lm_head_workspace_size(rows, H, V, w_dtype), dtype=torch.uint8, device="cuda")
        st = lib.tsv_lm_head_argmax(_p(hidden), rows, H, V, w_dtype, _p(W), _p(sc), _p(bi), _p(ref_arg), _p(ref_max),
                                    _p(ws), ws.numel(), stream)
        assert st == 0, lib.tsv_last_error()
        arg = torch.full((rows,), -7, dtype=torch.int32, device="cuda")
        mx = torch.zeros(rows, dtype=torch.float32, device="cuda")
        st = lib.tsv_lm_head_argmax_noalloc(_p(hidden), rows, H, V, w_dtype, _p(W), _p(sc), _p(bi), _p(arg), _p(mx),
                                            stream)
        assert st == 0, lib.tsv_last_error()
        torch.cuda.synchronize()
        assert torch.equal(arg, ref_arg), call
        assert torch.allclose(mx, ref_max, rtol=1e-4, atol=1e-3), call
        assert int(arg.min()) >= 0 and int(arg.max()) < V
        assert arg.cpu().numpy().tolist() == target.tolist(), call

    too_many = gpu_lib._abi.NOALLOC_MAX_ROWS + 1
    st = lib.tsv_lm_head_argmax_noalloc(_p(hidden), too_many, H, V, 1, _p(W), None, None, _p(arg), None, stream)
    assert st == gpu_lib._abi.ECAPACITY
    assert b"scratch" in lib.tsv_last_error()
