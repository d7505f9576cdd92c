"""GPU parity of tsv_tree_append (the verify block appended at the nodes' own positions) against the oracle.

Rotated values differ from the fp64 oracle by the fp32 arithmetic of the kernel (angles reduced in fp64, fp32
sine/cosine and products): |error| <= 1e-6 (|a| + |b|) for a rotated pair (a, b).  A stored 16-bit value or an
Int8 code is therefore compared exactly except where the oracle's value lies within that bound of a rounding
boundary; there the stored value must be one of the roundings of the values within the bound.  Un-rotated V
rows are exact inputs, so their stored form (16-bit copy or Int8 codes and scale) is compared bit for bit.
"""
import numpy as np
import pytest
import torch

from oracle import append as oap

from .parity import bf16_tensor_to_f64

pytestmark = pytest.mark.gpu
DEV = "cuda"
KVT = {0: torch.float16, 1: torch.bfloat16, 2: torch.int8}


def rnd16(x, kv_dtype):
    """Round fp64 values to fp16 (numpy's correctly rounded conversion) or to bf16 (8 significant bits, ties to
    even, exact for the normal range these values lie in)."""
    x = np.asarray(x, dtype=np.float64)
    if kv_dtype == 0:
        return x.astype(np.float16).astype(np.float64)
    m, e = np.frexp(x)
    return np.ldexp(np.rint(np.ldexp(m, 8)), e - 8)


def within_roundings(got, v, delta, rnd):
    lo, hi = rnd(v - delta), rnd(v + delta)
    return np.all((got >= lo) & (got <= hi))


def rot_error_bound(x, rot_dim, interleaved):
    """Per-feature bound on |kernel - exact| for one row x [D] (0 for features that are not rotated)."""
    x = np.abs(np.asarray(x, dtype=np.float64))
    b = np.zeros_like(x)
    h = rot_dim // 2
    ia = np.arange(0, rot_dim, 2) if interleaved else np.arange(h)
    ib = ia + 1 if interleaved else ia + h
    pair = x[ia] + x[ib]
    b[ia] = b[ib] = 1e-6 * pair + 1e-30
    return b


def run_append_case(gpu_lib, rng, *, B, T, HQ, HKV, D, S_list, kv_dtype, rot_dim, base, interleaved=False,
                    layers=1, in_place=False, trees=None, s_cap=None):
    s_cap = s_cap or max(S_list) + T + 5
    trees = trees or [[-1] + [int(rng.integers(0, i)) for i in range(1, T)] for _ in range(B)]
    par = torch.tensor(np.array(trees, dtype=np.int32), device=DEV)
    anc = torch.zeros(B, T, dtype=torch.int64, device=DEV)
    depth = torch.zeros(B, T, dtype=torch.int32, device=DEV)
    gpu_lib.tree_mask(par, anc, depth)
    L = []
    for _ in range(layers):
        q = torch.from_numpy(rng.standard_normal((B, T, HQ, D)).astype(np.float32)).to(torch.bfloat16).to(DEV)
        kn = torch.from_numpy(rng.standard_normal((B, T, HKV, D)).astype(np.float32) * 2).to(torch.bfloat16).to(DEV)
        vn = torch.from_numpy(rng.standard_normal((B, T, HKV, D)).astype(np.float32)).to(torch.bfloat16).to(DEV)
        if kv_dtype == 2:
            k = torch.full((B, HKV, s_cap, D), 77, dtype=torch.int8, device=DEV)
            v = torch.full((B, HKV, s_cap, D), -5, dtype=torch.int8, device=DEV)
            ks = torch.full((B, HKV, s_cap), 0.25, dtype=torch.float16, device=DEV)
            vs = torch.full((B, HKV, s_cap), 0.5, dtype=torch.float16, device=DEV)
        else:
            k = torch.full((B, HKV, s_cap, D), 3.0, dtype=KVT[kv_dtype], device=DEV)
            v = torch.full((B, HKV, s_cap, D), -7.0, dtype=KVT[kv_dtype], device=DEV)
            ks = vs = None
        qo = q if in_place else torch.full_like(q, float("nan"))
        L.append(dict(q=q.clone(), q_in=q, q_out=qo, kn=kn, vn=vn, k=k, v=v, ks=ks, vs=vs, k0=k.clone(), v0=v.clone()))
    desc = gpu_lib.append_desc([x["q_in"] for x in L], [x["q_out"] for x in L], [x["kn"] for x in L],
                               [x["vn"] for x in L], [x["k"] for x in L], [x["v"] for x in L], depth, T=T, HQ=HQ,
                               HKV=HKV, D=D, kv_dtype=kv_dtype, rot_dim=rot_dim, rope_base=base,
                               interleaved=interleaved, k_scale=[x["ks"] for x in L] if kv_dtype == 2 else None,
                               v_scale=[x["vs"] for x in L] if kv_dtype == 2 else None)
    kv_len = torch.tensor(S_list, dtype=torch.int32, device=DEV)
    st = torch.zeros(4, dtype=torch.int32, device=DEV)
    gpu_lib.tree_append(desc, kv_len, dev_status=st)
    torch.cuda.synchronize()
    return L, trees, kv_len, st


def check_append(L, trees, S_list, kv_dtype, rot_dim, base, interleaved, ok_seqs=None):
    for x in L:
        q = bf16_tensor_to_f64(x["q"])
        kn = bf16_tensor_to_f64(x["kn"])
        vn = bf16_tensor_to_f64(x["vn"])
        qo = bf16_tensor_to_f64(x["q_out"])
        B, T = q.shape[0], q.shape[1]
        for b in range(B):
            S = S_list[b]
            if ok_seqs is not None and b not in ok_seqs:
                assert torch.equal(x["k"][b], x["k0"][b]) and torch.equal(x["v"][b], x["v0"][b])
                continue
            q_rot, k_rot, v = oap.append_block(q[b], kn[b], vn[b], trees[b], S, base, rot_dim, interleaved)
            for i in range(T):
                for h in range(q.shape[2]):
                    bd = rot_error_bound(q[b, i, h], rot_dim, interleaved)
                    assert within_roundings(qo[b, i, h], q_rot[i, h], bd, lambda a: rnd16(a, 1)), (b, i, h)
                for kvh in range(kn.shape[2]):
                    slot = S + i
                    bd = rot_error_bound(kn[b, i, kvh], rot_dim, interleaved)
                    if kv_dtype == 2:
                        codes = x["k"][b, kvh, slot].cpu().numpy().astype(np.float64)
                        s_bits = np.uint16(x["ks"][b, kvh, slot].cpu().view(torch.int16).item() & 0xFFFF)
                        s_g = float(s_bits.view(np.float16))
                        amax, dmax = np.max(np.abs(k_rot[i, kvh])), np.max(bd)
                        s_lo = float(np.float16(np.float32(max(amax - dmax, 0.0)) / np.float32(127)))
                        s_hi = float(np.float16(np.float32(amax + dmax) / np.float32(127)))
                        assert s_lo <= s_g <= s_hi, (b, i, kvh, s_g, s_lo, s_hi)
                        if s_g > 0:
                            lo = np.clip(np.rint((k_rot[i, kvh] - bd) / s_g), -127, 127)
                            hi = np.clip(np.rint((k_rot[i, kvh] + bd) / s_g), -127, 127)
                            assert np.all((codes >= lo) & (codes <= hi)), (b, i, kvh)
                        # V: exact inputs, bit-exact stored form
                        vc, vsb = oap.quantize_token(v[i, kvh])
                        assert np.array_equal(x["v"][b, kvh, slot].cpu().numpy(), vc)
                        assert (x["vs"][b, kvh, slot].cpu().view(torch.int16).item() & 0xFFFF) == int(vsb)
                    else:
                        got_k = x["k"][b, kvh, slot].double().cpu().numpy()
                        assert within_roundings(got_k, k_rot[i, kvh], bd, lambda a: rnd16(a, kv_dtype)), (b, i, kvh)
                        got_v = x["v"][b, kvh, slot].double().cpu().numpy()
                        assert np.array_equal(got_v, rnd16(v[i, kvh], kv_dtype))
            # rows outside [S, S + T) keep their bytes
            for name in ("k", "v"):
                assert torch.equal(x[name][b, :, :S], x[name + "0"][b, :, :S])
                assert torch.equal(x[name][b, :, S + T:], x[name + "0"][b, :, S + T:])


@pytest.mark.parametrize("kv_dtype", [0, 1, 2])
@pytest.mark.parametrize("D,rot_dim,interleaved,base", [(256, 256, False, 1e4), (256, 64, False, 1e6),
                                                       (128, 128, True, 1e4), (64, 32, True, 5e5), (64, 2, False, 10.)])
def test_append_matches_oracle(gpu_lib, kv_dtype, D, rot_dim, interleaved, base):
    rng = np.random.default_rng(D + rot_dim + kv_dtype)
    B, T = 2, 9
    S_list = [0, 4099]
    L, trees, kv_len, st = run_append_case(gpu_lib, rng, B=B, T=T, HQ=6, HKV=2, D=D, S_list=S_list,
                                           kv_dtype=kv_dtype, rot_dim=rot_dim, base=base, interleaved=interleaved,
                                           layers=2)
    assert st.tolist()[0] == 0
    assert kv_len.tolist() == [S + T for S in S_list]
    check_append(L, trees, S_list, kv_dtype, rot_dim, base, interleaved)


@pytest.mark.parametrize("kv_dtype", [1, 2])
def test_append_long_positions_chain_and_in_place_q(gpu_lib, kv_dtype):
    """A chain at position ~131k (the longest workload): positions S + i, Q rotated in place."""
    rng = np.random.default_rng(11 + kv_dtype)
    T = 64
    S_list = [131072]
    L, trees, kv_len, st = run_append_case(gpu_lib, rng, B=1, T=T, HQ=4, HKV=1, D=256, S_list=S_list,
                                           kv_dtype=kv_dtype, rot_dim=256, base=1e6, in_place=True,
                                           trees=[[-1] + list(range(T - 1))])
    assert st.tolist()[0] == 0 and kv_len.tolist() == [131072 + T]
    check_append(L, trees, S_list, kv_dtype, 256, 1e6, False)


def test_append_capacity_error_and_constant_tokens(gpu_lib):
    rng = np.random.default_rng(5)
    B, T, D = 2, 4, 64
    S_list = [10, 13]  # sequence 1: 13 + 4 > s_cap 16
    L, trees, kv_len, st = run_append_case(gpu_lib, rng, B=B, T=T, HQ=2, HKV=1, D=D, S_list=S_list, kv_dtype=2,
                                           rot_dim=D, base=1e4, s_cap=16)
    s = st.tolist()
    assert s[0] == gpu_lib.DEV_BAD_KV_LEN and s[1] == 1 and s[2] == 13
    assert kv_len.tolist() == [14, 13]  # the refused sequence keeps its length
    check_append(L, trees, S_list, 2, D, 1e4, False, ok_seqs={0})
    # a single-valued V token gets code 127 everywhere, an all-zero one scale 0 and zero codes
    x = L[0]
    vn = torch.full((B, T, 1, D), 0.75, dtype=torch.bfloat16, device=DEV)
    vn[:, 1] = 0.0
    kv_len2 = torch.tensor([0, 0], dtype=torch.int32, device=DEV)
    depth = torch.zeros(B, T, dtype=torch.int32, device=DEV)
    par = torch.tensor([[-1, 0, 1, 2]] * B, dtype=torch.int32, device=DEV)
    gpu_lib.tree_mask(par, torch.zeros(B, T, dtype=torch.int64, device=DEV), depth)
    d2 = gpu_lib.append_desc([x["q_in"]], [x["q_out"]], [x["kn"]], [vn], [x["k"]], [x["v"]], depth, T=T, HQ=2, HKV=1,
                             D=D, kv_dtype=2, rot_dim=D, rope_base=1e4, k_scale=[x["ks"]], v_scale=[x["vs"]])
    gpu_lib.tree_append(d2, kv_len2)
    torch.cuda.synchronize()
    assert x["v"][0, 0, 0].tolist() == [127] * D and x["v"][1, 0, 2].tolist() == [127] * D
    assert x["v"][0, 0, 1].tolist() == [0] * D and float(x["vs"][0, 0, 1]) == 0.0
