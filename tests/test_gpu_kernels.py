"""GPU parity of each C-ABI call on small seeded inputs (several tiles, ragged tails, edge cases).

Every expected value comes from the fp64 oracle on the same host-side inputs.
"""
import numpy as np
import pytest
import torch

from oracle import attention as oa
from oracle import gather as og
from oracle import lm_head as ol
from oracle import storage as osd
from oracle import tree as ot

from .parity import ATT_MAX_ABS, ATT_REL_L2, attn_stats, bf16_tensor_to_f64, u64

pytestmark = pytest.mark.gpu
DEV = "cuda"


def random_tree(rng, T, style="random"):
    if T == 0:
        return []
    if style == "chain":
        return [-1] + list(range(T - 1))
    if style == "star":
        return [-1] + [0] * (T - 1)
    return [-1] + [int(rng.integers(0, i)) for i in range(1, T)]


def i32(a):
    return torch.tensor(np.asarray(a, dtype=np.int32), device=DEV)


def status():
    return torch.zeros(4, dtype=torch.int32, device=DEV)


# ----------------------------------------------------------------------------- a1 mask
@pytest.mark.parametrize("T", [1, 2, 3, 7, 16, 31, 32, 33, 63, 64])
def test_tree_mask_exact(gpu_lib, T):
    rng = np.random.default_rng(T)
    B = 3
    par = np.array([random_tree(rng, T, s) for s in ("random", "chain", "star")], dtype=np.int32)
    offset = 5
    anc = torch.zeros(B, T, dtype=torch.int64, device=DEV)
    depth = torch.zeros(B, T, dtype=torch.int32, device=DEV)
    dense = torch.zeros(B, T, offset + T, dtype=torch.float32, device=DEV)
    st = status()
    gpu_lib.tree_mask(i32(par), anc, depth, dense_mask=dense, mask_offset=offset, dev_status=st)
    torch.cuda.synchronize()
    assert st.tolist() == [0, 0, 0, 0]
    want = [a for b in range(B) for a in ot.ancestor_bits(par[b].tolist())]
    assert u64(anc) == want
    assert depth.cpu().numpy().reshape(-1).tolist() == [ot.depth(par[b].tolist(), i) for b in range(B) for i in range(T)]
    dm = dense.cpu().numpy().astype(np.float64)
    for b in range(B):
        assert np.array_equal(dm[b], ot.history_mask(par[b].tolist(), offset).astype(np.float32))


def test_tree_mask_device_errors_and_host_errors(gpu_lib):
    par = np.array([[-1, 0, 1, 0], [-1, 0, 2, 0], [0, 0, 1, 2]], dtype=np.int32)  # seq 1 node 2 self-parent
    anc = torch.zeros(3, 4, dtype=torch.int64, device=DEV)
    depth = torch.zeros(3, 4, dtype=torch.int32, device=DEV)
    st = status()
    gpu_lib.tree_mask(i32(par), anc, depth, dev_status=st)
    torch.cuda.synchronize()
    s = st.tolist()
    assert s[0] in (gpu_lib.DEV_BAD_PARENT, gpu_lib.DEV_BAD_ROOT) and s[1] in (1, 2)
    assert depth[1].tolist() == [-1] * 4 and depth[2].tolist() == [-1] * 4
    assert u64(anc[0]) == ot.ancestor_bits([-1, 0, 1, 0])
    big = torch.zeros(1, 65, dtype=torch.int32, device=DEV)
    with pytest.raises(gpu_lib.TsvError, match="TSV_ECAPACITY"):
        gpu_lib.tree_mask(big, torch.zeros(1, 65, dtype=torch.int64, device=DEV),
                          torch.zeros(1, 65, dtype=torch.int32, device=DEV))
    # T == 0 is valid for the mask and does nothing
    gpu_lib.tree_mask(torch.zeros(2, 0, dtype=torch.int32, device=DEV), torch.zeros(2, 0, dtype=torch.int64, device=DEV),
                      torch.zeros(2, 0, dtype=torch.int32, device=DEV))


# ----------------------------------------------------------------------------- a2 attention
KVT = {0: torch.float16, 1: torch.bfloat16, 2: torch.int8}


def make_attn_case(rng, *, B, T, HQ, HKV, D, S_list, kv_dtype, layers=1, cap_extra=3):
    s_cap = max(S_list) + T + cap_extra
    data = []
    for _ in range(layers):
        q = (rng.standard_normal((B, T, HQ, D)) * 1.0).astype(np.float32)
        if kv_dtype == 2:
            k = rng.integers(-127, 128, size=(B, HKV, s_cap, D)).astype(np.int8)
            v = rng.integers(-127, 128, size=(B, HKV, s_cap, D)).astype(np.int8)
            ks = rng.uniform(0.005, 0.05, size=(B, HKV, s_cap)).astype(np.float16)
            vs = rng.uniform(0.005, 0.05, size=(B, HKV, s_cap)).astype(np.float16)
        else:
            k = rng.standard_normal((B, HKV, s_cap, D)).astype(np.float32)
            v = rng.standard_normal((B, HKV, s_cap, D)).astype(np.float32)
            ks = vs = None
        data.append((q, k, v, ks, vs))
    trees = [random_tree(rng, T) for _ in range(B)]
    return s_cap, data, trees


def run_attn_case(gpu_lib, rng, *, B, T, HQ, HKV, D, S_list, kv_dtype, splits, layers=1, path=0, cap_extra=3,
                  window=None):
    s_cap, data, trees = make_attn_case(rng, B=B, T=T, HQ=HQ, HKV=HKV, D=D, S_list=S_list, kv_dtype=kv_dtype,
                                        layers=layers, cap_extra=cap_extra)
    qs, ks_, vs_, kss, vss, os_ = [], [], [], [], [], []
    for (q, k, v, ksc, vsc) in data:
        qs.append(torch.from_numpy(q).to(torch.bfloat16).to(DEV))
        if kv_dtype == 2:
            ks_.append(torch.from_numpy(k).to(DEV))
            vs_.append(torch.from_numpy(v).to(DEV))
            kss.append(torch.from_numpy(ksc).to(DEV))
            vss.append(torch.from_numpy(vsc).to(DEV))
        else:
            ks_.append(torch.from_numpy(k).to(KVT[kv_dtype]).to(DEV))
            vs_.append(torch.from_numpy(v).to(KVT[kv_dtype]).to(DEV))
        os_.append(torch.full((B, T, HQ, D), float("nan"), dtype=torch.bfloat16, device=DEV))
    par = i32(np.array(trees, dtype=np.int32))
    anc = torch.zeros(B, T, dtype=torch.int64, device=DEV)
    depth = torch.zeros(B, T, dtype=torch.int32, device=DEV)
    gpu_lib.tree_mask(par, anc, depth)
    kv_len = i32([S + T for S in S_list])
    desc = gpu_lib.attn_desc(qs, ks_, vs_, os_, kv_len, anc, T=T, HQ=HQ, HKV=HKV, D=D, kv_dtype=kv_dtype,
                             max_kv_len=max(S_list) + T, k_scale=kss or None, v_scale=vss or None, splits=splits,
                             path=path, window=window)
    ws = torch.empty(max(gpu_lib.attention_workspace_size(desc), 16), dtype=torch.uint8, device=DEV)
    st = status()
    gpu_lib.tree_verify_attention(desc, ws, dev_status=st)
    torch.cuda.synchronize()
    assert st.tolist()[0] == 0
    G = HQ // HKV
    worst = (0.0, 0.0)
    for l, (q, k, v, ksc, vsc) in enumerate(data):
        o = bf16_tensor_to_f64(os_[l])
        qd = bf16_tensor_to_f64(qs[l])
        for b in range(B):
            S = S_list[b]
            ref = np.zeros((T, HQ, D))
            for kvh in range(HKV):
                if kv_dtype == 2:
                    K = osd.int8_scaled(k[b, kvh, :S + T], ksc[b, kvh, :S + T].view(np.uint16))
                    V = osd.int8_scaled(v[b, kvh, :S + T], vsc[b, kvh, :S + T].view(np.uint16))
                else:
                    K = ks_[l][b, kvh, :S + T].double().cpu().numpy()
                    V = vs_[l][b, kvh, :S + T].double().cpu().numpy()
                w = 0 if window is None else window[l]
                for i in range(T):
                    vis = ot.ancestors(trees[b], i)
                    cols = ot.visible_keys(trees[b], i, S, w)
                    for g in range(G):
                        h = kvh * G + g
                        if w == 0:
                            ref[i, h] = oa.attend_row(qd[b, i, h], K, V, S, vis)
                        else:
                            ref[i, h] = oa.attend_cols(qd[b, i, h], K, V, cols)
            a, r = attn_stats(o[b].reshape(-1, D), ref.reshape(-1, D))
            worst = (max(worst[0], a), max(worst[1], r))
    assert worst[0] <= ATT_MAX_ABS and worst[1] <= ATT_REL_L2, worst
    return worst


@pytest.mark.parametrize("kv_dtype", [0, 1, 2])
@pytest.mark.parametrize("T,S_list,splits", [(1, [0, 5], 0), (3, [127, 128], 1), (7, [129, 300], 3),
                                             (16, [1000, 33], 0), (33, [64, 257], 2), (64, [200, 0], 0)])
def test_attention_small(gpu_lib, kv_dtype, T, S_list, splits):
    rng = np.random.default_rng(T * 31 + kv_dtype)
    run_attn_case(gpu_lib, rng, B=2, T=T, HQ=6, HKV=2, D=256 if T < 33 else 128, S_list=S_list, kv_dtype=kv_dtype,
                  splits=splits)


@pytest.mark.parametrize("path", [1, 2, 3, 4])
@pytest.mark.parametrize("kv_dtype", [0, 1, 2])
@pytest.mark.parametrize("T,S_list,splits", [(1, [0, 63], 0), (3, [64, 4096], 0), (16, [65, 1000], 3),
                                             (22, [127, 5], 1), (33, [500, 200], 0), (64, [64, 1337], 2)])
def test_attention_both_kernels(gpu_lib, path, kv_dtype, T, S_list, splits):
    """The CUDA-core kernel (path 1) and the tcgen05 kernels (path 2: the library's choice of score-tile width,
    3: 64-key tiles, 4: 128-key tiles) on the same inputs; 1 to 3 tiles of 128 rows, ragged tails."""
    rng = np.random.default_rng(T * 7 + kv_dtype)
    run_attn_case(gpu_lib, rng, B=2, T=T, HQ=24, HKV=4, D=256, S_list=S_list, kv_dtype=kv_dtype, splits=splits,
                  path=path, cap_extra=70)


def test_attention_tcgen05_refuses_what_it_cannot_do(gpu_lib):
    B, T, HQ, HKV, D = 1, 2, 4, 2, 128
    q = [torch.zeros(B, T, HQ, D, dtype=torch.bfloat16, device=DEV)]
    k = [torch.zeros(B, HKV, 8, D, dtype=torch.float16, device=DEV)]
    desc = gpu_lib.attn_desc(q, k, [k[0].clone()], [q[0].clone()], i32([4]), torch.ones(B, T, dtype=torch.int64,
                             device=DEV), T=T, HQ=HQ, HKV=HKV, D=D, kv_dtype=0, max_kv_len=8, path=2)
    with pytest.raises(gpu_lib.TsvError, match="TSV_EUNSUPPORTED"):
        gpu_lib.tree_verify_attention(desc, torch.empty(1 << 20, dtype=torch.uint8, device=DEV))


@pytest.mark.parametrize("D", [64, 128, 256])
def test_attention_head_dims_and_layers(gpu_lib, D):
    rng = np.random.default_rng(D)
    run_attn_case(gpu_lib, rng, B=1, T=5, HQ=8, HKV=2, D=D, S_list=[77], kv_dtype=0, splits=0, layers=3)


@pytest.mark.parametrize("path", [1, 3, 4])
@pytest.mark.parametrize("kv_dtype", [0, 1, 2])
@pytest.mark.parametrize("T,S_list,splits,window", [(7, [300, 129], 0, [64]), (16, [1000, 33], 3, [5]),
                                                    (33, [500, 200], 0, [1, 100, 0]), (64, [1337, 64], 2, [200]),
                                                    (3, [4096, 70], 0, [1024, 0])])
def test_attention_sliding_window(gpu_lib, path, kv_dtype, T, S_list, splits, window):
    """Sliding-window layers: the tree mask intersected with each layer's band, mixed with full layers."""
    rng = np.random.default_rng(T * 13 + kv_dtype + len(window))
    run_attn_case(gpu_lib, rng, B=2, T=T, HQ=24, HKV=4, D=256, S_list=S_list, kv_dtype=kv_dtype, splits=splits,
                  path=path, cap_extra=70, layers=len(window), window=window)


@pytest.mark.parametrize("window", [1, 3, 8, 40, 100])
def test_sliding_band_mask_exact(gpu_lib, window):
    rng = np.random.default_rng(window)
    B, T, offset = 3, 9, 37
    par = np.array([random_tree(rng, T, s) for s in ("random", "chain", "star")], dtype=np.int32)
    anc = torch.zeros(B, T, dtype=torch.int64, device=DEV)
    depth = torch.zeros(B, T, dtype=torch.int32, device=DEV)
    dense = torch.zeros(B, T, offset + T, dtype=torch.float32, device=DEV)
    gpu_lib.tree_mask(i32(par), anc, depth, dense_mask=dense, mask_offset=offset)
    gpu_lib.sliding_band_mask(dense, offset, window)
    torch.cuda.synchronize()
    dm = dense.cpu().numpy()
    for b in range(B):
        want = ot.sliding_mask_from_caller(ot.history_mask(par[b].tolist(), offset), offset, window)
        assert np.array_equal(dm[b], want.astype(np.float32)), b
    with pytest.raises(gpu_lib.TsvError, match="TSV_EINVAL"):
        gpu_lib.sliding_band_mask(dense, offset, 0)


@pytest.mark.parametrize("path", [3, 4])
def test_attention_splits_agree(gpu_lib, path):
    """The result holds across split counts (two split choices and more), for both score-tile widths."""
    for splits in (1, 2, 5, 0):
        rng = np.random.default_rng(42)
        run_attn_case(gpu_lib, rng, B=1, T=16, HQ=24, HKV=4, D=256, S_list=[2048], kv_dtype=2, splits=splits,
                      path=path)


def test_attention_refuses_too_many_splits(gpu_lib):
    """More than 64 key-range splits per unit is refused before any launch (the merge keeps 64 weights a row)."""
    B, T, HQ, HKV, D = 1, 2, 4, 2, 64
    q = [torch.zeros(B, T, HQ, D, dtype=torch.bfloat16, device=DEV)]
    k = [torch.zeros(B, HKV, 8192, D, dtype=torch.float16, device=DEV)]
    desc = gpu_lib.attn_desc(q, k, [k[0].clone()], [q[0].clone()], i32([8000]), torch.ones(B, T, dtype=torch.int64,
                             device=DEV), T=T, HQ=HQ, HKV=HKV, D=D, kv_dtype=0, max_kv_len=8000, splits=65)
    with pytest.raises(gpu_lib.TsvError, match="TSV_ECAPACITY"):
        gpu_lib.tree_verify_attention(desc, torch.empty(64 << 20, dtype=torch.uint8, device=DEV))


def test_attention_bad_kv_len(gpu_lib):
    rng = np.random.default_rng(1)
    B, T, HQ, HKV, D = 2, 4, 4, 2, 64
    q = [torch.zeros(B, T, HQ, D, dtype=torch.bfloat16, device=DEV)]
    k = [torch.zeros(B, HKV, 40, D, dtype=torch.float16, device=DEV)]
    v = [torch.zeros_like(k[0])]
    o = [torch.zeros_like(q[0])]
    anc = torch.ones(B, T, dtype=torch.int64, device=DEV)
    kv_len = i32([2, 10])  # sequence 0: kv_len < T
    desc = gpu_lib.attn_desc(q, k, v, o, kv_len, anc, T=T, HQ=HQ, HKV=HKV, D=D, kv_dtype=0, max_kv_len=40)
    ws = torch.empty(max(gpu_lib.attention_workspace_size(desc), 16), dtype=torch.uint8, device=DEV)
    st = status()
    gpu_lib.tree_verify_attention(desc, ws, dev_status=st)
    torch.cuda.synchronize()
    assert st.tolist()[:2] == [gpu_lib.DEV_BAD_KV_LEN, 0]
    bad = gpu_lib.attn_desc(q, k, v, o, kv_len, anc, T=T, HQ=HQ, HKV=HKV, D=D, kv_dtype=0, max_kv_len=40)
    bad.kv_dtype = gpu_lib.Q4_G64  # a weight format, refused for caches
    with pytest.raises(gpu_lib.TsvError, match="TSV_EUNSUPPORTED"):
        gpu_lib.tree_verify_attention(bad, ws)
    bad.kv_dtype, bad.T = 0, 65
    with pytest.raises(gpu_lib.TsvError, match="TSV_ECAPACITY"):
        gpu_lib.tree_verify_attention(bad, ws)


# ----------------------------------------------------------------------------- a3 LM head
def q4_pack(codes):
    return (codes[:, 0::2] | (codes[:, 1::2] << 4)).astype(np.uint8)


@pytest.mark.parametrize("w_dtype", [0, 1, 3])
@pytest.mark.parametrize("rows,V,H", [(1, 1000, 256), (2, 1536, 5120), (3, 4099, 512), (5, 777, 256), (8, 2048, 1024), (13, 3001, 256),
                                      (16, 1280, 5120), (17, 257, 512), (29, 3001, 1024), (64, 5003, 512),
                                      (200, 2303, 256), (257, 1000, 1024),
                                      (600, 700, 256), (600, 700, 512)])
def test_lm_head_exact(gpu_lib, w_dtype, rows, V, H):
    rng = np.random.default_rng(rows * 1000 + V + w_dtype)
    h = torch.from_numpy(rng.standard_normal((rows, H)).astype(np.float32)).to(torch.bfloat16)
    if w_dtype == 3:
        codes = rng.integers(0, 16, size=(V, H))
        sc = torch.from_numpy(rng.uniform(0.005, 0.008, size=(V, H // 64)).astype(np.float32)).to(torch.bfloat16)
        bi = torch.from_numpy(rng.uniform(-0.06, -0.05, size=(V, H // 64)).astype(np.float32)).to(torch.bfloat16)
        Wd = torch.from_numpy(q4_pack(codes)).to(DEV)
        W64 = osd.q4_affine(q4_pack(codes), sc.view(torch.int16).numpy().view(np.uint16),
                            bi.view(torch.int16).numpy().view(np.uint16))
        sc, bi = sc.to(DEV), bi.to(DEV)
    else:
        dt = torch.bfloat16 if w_dtype == 1 else torch.float16
        Wt = torch.from_numpy((rng.standard_normal((V, H)) * 0.05).astype(np.float32)).to(dt)
        W64 = Wt.double().numpy()
        Wd, sc, bi = Wt.to(DEV), None, None
    arg = torch.zeros(rows, dtype=torch.int32, device=DEV)
    mx = torch.zeros(rows, dtype=torch.float32, device=DEV)
    gpu_lib.lm_head_argmax(h.to(DEV), Wd, arg, w_dtype=w_dtype, V=V, scales=sc, biases=bi, maxlogit=mx)
    torch.cuda.synchronize()
    o_arg, o_top, o_gap = ol.argmax_gap(ol.logits(W64, h.double().numpy()))
    g_arg = arg.cpu().numpy()
    sure = o_gap > 1e-2
    assert sure.sum() >= max(1, rows // 2)
    assert np.array_equal(g_arg[sure], o_arg[sure])
    assert np.allclose(mx.cpu().numpy(), o_top, rtol=1e-4, atol=1e-3)


def test_lm_head_ties_lowest_index(gpu_lib):
    V, H = 5000, 256
    W = torch.zeros(V, H, dtype=torch.bfloat16)
    W[[17, 1234, 4999], 0] = 1.0  # exact three-way tie
    W[3, 0] = 0.5
    h = torch.zeros(2, H, dtype=torch.bfloat16)
    h[:, 0] = 2.0
    h[1, 1] = 1.0
    W[4998, 1] = 2.5  # row 1: 4998 wins (2.5 vs 2.0)
    arg = torch.zeros(2, dtype=torch.int32, device=DEV)
    gpu_lib.lm_head_argmax(h.to(DEV), W.to(DEV), arg, w_dtype=1, V=V)
    torch.cuda.synchronize()
    assert arg.tolist() == [17, 4998]


# ----------------------------------------------------------------------------- a4 walk
@pytest.mark.parametrize("T", [1, 2, 7, 31, 32, 33, 64])
def test_walk_exact(gpu_lib, T):
    rng = np.random.default_rng(T + 5)
    B = 6
    par = np.array([random_tree(rng, T, ("random", "chain", "star")[b % 3]) for b in range(B)], dtype=np.int32)
    tok = rng.integers(0, 6, size=(B, T)).astype(np.int32)  # small vocab: duplicate siblings happen
    arg = rng.integers(0, 6, size=(B, T)).astype(np.int32)
    path = torch.zeros(B, T, dtype=torch.int32, device=DEV)
    plen = torch.zeros(B, dtype=torch.int32, device=DEV)
    em = torch.zeros(B, T, dtype=torch.int32, device=DEV)
    st = status()
    gpu_lib.tree_accept_walk(i32(arg), i32(tok), i32(par), path, plen, em, dev_status=st)
    torch.cuda.synchronize()
    assert st.tolist()[0] == 0
    for b in range(B):
        p, e = ot.accept_walk(arg[b], tok[b], par[b])
        assert plen[b].item() == len(p)
        assert path[b].tolist() == p + [-1] * (T - len(p))
        assert em[b].tolist() == e + [-1] * (T - len(p))


def test_walk_bad_parent(gpu_lib):
    par = np.array([[-1, 0, 0], [-1, 2, 0]], dtype=np.int32)
    z = np.zeros((2, 3), dtype=np.int32)
    path = torch.zeros(2, 3, dtype=torch.int32, device=DEV)
    plen = torch.zeros(2, dtype=torch.int32, device=DEV)
    em = torch.zeros(2, 3, dtype=torch.int32, device=DEV)
    st = status()
    gpu_lib.tree_accept_walk(i32(z), i32(z), i32(par), path, plen, em, dev_status=st)
    torch.cuda.synchronize()
    assert st.tolist()[:3] == [gpu_lib.DEV_BAD_PARENT, 1, 1]
    assert plen[1].item() == 1 and path[1].tolist() == [0, -1, -1]


# ----------------------------------------------------------------------------- a5 gather
@pytest.mark.parametrize("kv_dtype", [0, 1, 2])
def test_gather_cases(gpu_lib, kv_dtype):
    rng = np.random.default_rng(kv_dtype)
    L, B, HKV, D, T = 2, 5, 2, 64, 9
    S = [10, 0, 33, 7, 20]
    s_cap = 50
    paths = [[0, 2, 5, 8], [0], [0, 1, 2], list(range(9)), [0, 3, 4, 7]]  # scattered, zero, prefix, identity, scattered
    dt = KVT[kv_dtype]
    if kv_dtype == 2:
        K = [torch.from_numpy(rng.integers(-127, 128, size=(B, HKV, s_cap, D)).astype(np.int8)) for _ in range(L)]
        Vv = [torch.from_numpy(rng.integers(-127, 128, size=(B, HKV, s_cap, D)).astype(np.int8)) for _ in range(L)]
        # distinct per-token scales so a scale left behind is caught
        KS = [torch.from_numpy((np.arange(B * HKV * s_cap).reshape(B, HKV, s_cap) * 1e-4 + l + 0.01).astype(np.float16))
              for l in range(L)]
        VS = [x + 0.5 for x in KS]
    else:
        K = [torch.from_numpy(rng.standard_normal((B, HKV, s_cap, D)).astype(np.float32)).to(dt) for _ in range(L)]
        Vv = [torch.from_numpy(rng.standard_normal((B, HKV, s_cap, D)).astype(np.float32)).to(dt) for _ in range(L)]
        KS = VS = None
    before = [(k.clone(), v.clone()) for k, v in zip(K, Vv)]
    sb = [(a.clone(), b.clone()) for a, b in zip(KS, VS)] if KS else None
    Kd = [k.to(DEV) for k in K]
    Vd = [v.to(DEV) for v in Vv]
    KSd = [s.to(DEV) for s in KS] if KS else None
    VSd = [s.to(DEV) for s in VS] if VS else None
    desc = gpu_lib.kv_desc(Kd, Vd, HKV=HKV, D=D, kv_dtype=kv_dtype, k_scale=KSd, v_scale=VSd)
    kv_len = i32([s + T for s in S])
    pth = i32([p + [-1] * (T - len(p)) for p in paths])
    plen = i32([len(p) for p in paths])
    st = status()
    gpu_lib.kv_gather_positions(desc, kv_len, pth, plen, T, dev_status=st)
    torch.cuda.synchronize()
    assert st.tolist()[0] == 0
    assert kv_len.tolist() == [s + len(p) for s, p in zip(S, paths)]
    view = (lambda t: t.view(torch.int16).numpy()) if kv_dtype != 2 else (lambda t: t.numpy())
    for l in range(L):
        for (gpu, orig) in ((Kd[l], before[l][0]), (Vd[l], before[l][1])):
            got, o = view(gpu.cpu()), view(orig)
            for b in range(B):
                exp, n = og.gather_within_tail(o[b], S[b], paths[b], axis=1)
                assert np.array_equal(got[b], exp)
        if KS:
            for (gpu, orig) in ((KSd[l], sb[l][0]), (VSd[l], sb[l][1])):
                got, o = gpu.cpu().view(torch.int16).numpy(), orig.view(torch.int16).numpy()
                for b in range(B):
                    exp, n = og.gather_within_tail(o[b], S[b], paths[b], axis=1)
                    assert np.array_equal(got[b], exp)


def test_gather_bad_path(gpu_lib):
    B, HKV, D, T, s_cap = 2, 1, 64, 4, 16
    K = [torch.zeros(B, HKV, s_cap, D, dtype=torch.float16, device=DEV)]
    V = [torch.zeros_like(K[0])]
    desc = gpu_lib.kv_desc(K, V, HKV=HKV, D=D, kv_dtype=0)
    kv_len = i32([8, 8])
    pth = i32([[0, 2, 1, -1], [0, 1, -1, -1]])  # seq 0 not increasing
    plen = i32([3, 2])
    st = status()
    gpu_lib.kv_gather_positions(desc, kv_len, pth, plen, T, dev_status=st)
    torch.cuda.synchronize()
    assert st.tolist()[:2] == [gpu_lib.DEV_BAD_PATH, 0]
    assert kv_len.tolist() == [8, 6]  # bad sequence untouched, good one advanced


# ----------------------------------------------------------------------------- limits and failure paths
def test_attention_maximum_layer_count(gpu_lib):
    """All TSV_MAX_LAYERS layers in one launch, on both kernels."""
    for path, kv_dtype in ((1, 1), (2, 1), (4, 2)):
        rng = np.random.default_rng(64 + path)
        run_attn_case(gpu_lib, rng, B=1, T=3, HQ=6, HKV=2, D=256, S_list=[70], kv_dtype=kv_dtype, splits=0, layers=64,
                      path=path)


def test_empty_batch_is_a_no_op(gpu_lib):
    T, HQ, HKV, D = 3, 4, 2, 64
    e32 = lambda *s: torch.zeros(*s, dtype=torch.int32, device=DEV)
    par, anc, depth = e32(0, T), torch.zeros(0, T, dtype=torch.int64, device=DEV), e32(0, T)
    gpu_lib.tree_mask(par, anc, depth)
    q = [torch.zeros(0, T, HQ, D, dtype=torch.bfloat16, device=DEV)]
    k = [torch.zeros(0, HKV, 8, D, dtype=torch.float16, device=DEV)]
    desc = gpu_lib.attn_desc(q, k, [k[0].clone()], [q[0].clone()], e32(0), anc, T=T, HQ=HQ, HKV=HKV, D=D,
                             kv_dtype=0, max_kv_len=8)
    gpu_lib.tree_verify_attention(desc, torch.empty(256, dtype=torch.uint8, device=DEV))
    gpu_lib.tree_accept_walk(e32(0, T), e32(0, T), par, e32(0, T), e32(0), e32(0, T))
    gpu_lib.kv_gather_positions(gpu_lib.kv_desc(k, [k[0].clone()], HKV=HKV, D=D, kv_dtype=0), e32(0), e32(0, T),
                                e32(0), T)
    kn = [torch.zeros(0, T, HKV, D, dtype=torch.bfloat16, device=DEV)]
    ad = gpu_lib.append_desc(q, q, kn, kn, k, [k[0].clone()], depth, T=T, HQ=HQ, HKV=HKV, D=D, kv_dtype=0,
                             rot_dim=D, rope_base=1e4)
    gpu_lib.tree_append(ad, e32(0))
    torch.cuda.synchronize()
    with pytest.raises(gpu_lib.TsvError, match="TSV_EINVAL"):  # the LM head needs at least one row
        gpu_lib.lm_head_argmax(torch.zeros(0, 256, dtype=torch.bfloat16, device=DEV),
                               torch.zeros(10, 256, dtype=torch.bfloat16, device=DEV), e32(0), w_dtype=1, V=10)


def test_bounded_wait_times_out_and_device_stays_usable(gpu_lib):
    """A wait that nothing completes ends after its limit with TSV_DEV_TIMEOUT; the context keeps working."""
    import ctypes as C
    lib = gpu_lib.load()
    st = status()
    assert lib.tsv_selftest_bounded_wait(C.c_void_p(st.data_ptr()), C.c_void_p(torch.cuda.current_stream().cuda_stream)) == 0
    torch.cuda.synchronize()
    assert st.tolist()[0] == gpu_lib.DEV_TIMEOUT and st.tolist()[1] == 1
    par = i32(np.array([[-1, 0, 1]], dtype=np.int32))
    anc = torch.zeros(1, 3, dtype=torch.int64, device=DEV)
    depth = torch.zeros(1, 3, dtype=torch.int32, device=DEV)
    gpu_lib.tree_mask(par, anc, depth)
    torch.cuda.synchronize()
    assert depth.tolist() == [[0, 1, 2]]
