"""GPU parity of the absolute-position gather (tsv_gather_positions) against the oracle's gather_positions.

mlxcel PR #1212, gather_positions commit: the kept positions, strictly increasing, become the new sequence in
order; Int8 scale sidecars move with their tokens; a prefix selection equals trim_to; the identity selection
moves nothing.  Every cache byte and scale is compared bit for bit: rows below the new length against the
oracle's selection, rows at or above it against their bytes before the call.
"""
import numpy as np
import pytest
import torch

from oracle import gather as og

pytestmark = pytest.mark.gpu
DEV = "cuda"
KVT = {0: torch.float16, 1: torch.bfloat16, 2: torch.int8}


def i32(a):
    return torch.tensor(np.asarray(a, dtype=np.int32), device=DEV)


def make_caches(rng, kv_dtype, L, B, HKV, s_cap, D):
    if kv_dtype == 2:
        K = [torch.from_numpy(rng.integers(-127, 128, size=(B, HKV, s_cap, D)).astype(np.int8)) for _ in range(L)]
        V = [torch.from_numpy(rng.integers(-127, 128, size=(B, HKV, s_cap, D)).astype(np.int8)) for _ in range(L)]
        # distinct per-token scales, so that a scale left behind or moved to the wrong row is caught
        KS = [torch.from_numpy((np.arange(B * HKV * s_cap).reshape(B, HKV, s_cap) % 30000 * 1e-4 + 0.01 + l)
                               .astype(np.float16)) for l in range(L)]
        VS = [x + 0.5 for x in KS]
    else:
        K = [torch.from_numpy(rng.standard_normal((B, HKV, s_cap, D)).astype(np.float32)).to(KVT[kv_dtype])
             for _ in range(L)]
        V = [torch.from_numpy(rng.standard_normal((B, HKV, s_cap, D)).astype(np.float32)).to(KVT[kv_dtype])
             for _ in range(L)]
        KS = VS = None
    return K, V, KS, VS


def bits(t):
    t = t.cpu()
    return t.numpy() if t.dtype == torch.int8 else t.view(torch.int16).numpy()


def run_and_check(gpu_lib, kv_dtype, D, kv_lens, kept_lists, s_cap, L=2, HKV=2, seed=0):
    rng = np.random.default_rng(seed)
    B = len(kv_lens)
    K, V, KS, VS = make_caches(rng, kv_dtype, L, B, HKV, s_cap, D)
    host = [bits(x) for x in K + V + (KS or []) + (VS or [])]
    dev = [x.to(DEV) for x in K + V + (KS or []) + (VS or [])]
    Kd, Vd = dev[:L], dev[L:2 * L]
    KSd, VSd = (dev[2 * L:3 * L], dev[3 * L:]) if KS else (None, None)
    desc = gpu_lib.kv_desc(Kd, Vd, HKV=HKV, D=D, kv_dtype=kv_dtype, k_scale=KSd, v_scale=VSd)
    max_kept = max(1, max(len(k) for k in kept_lists))
    kept = i32([list(k) + [-1] * (max_kept - len(k)) for k in kept_lists])
    kept_len = i32([len(k) for k in kept_lists])
    kv_len = i32(kv_lens)
    st = torch.zeros(4, dtype=torch.int32, device=DEV)
    gpu_lib.gather_positions(desc, kv_len, kept, kept_len, dev_status=st)
    torch.cuda.synchronize()
    assert st.tolist()[0] == 0
    assert kv_len.tolist() == [len(k) for k in kept_lists]
    for before, after in zip(host, dev):
        got = bits(after)
        for b in range(B):
            n = len(kept_lists[b])
            for h in range(HKV):
                want = og.gather_positions(before[b, h, :kv_lens[b]], kept_lists[b], axis=0)
                assert np.array_equal(got[b, h, :n], want), (b, h)
                assert np.array_equal(got[b, h, n:], before[b, h, n:]), (b, h)  # untouched past the new length
    return Kd, Vd


@pytest.mark.parametrize("kv_dtype", [0, 1, 2])
@pytest.mark.parametrize("D", [64, 256])
def test_gather_positions_cases(gpu_lib, kv_dtype, D):
    rng = np.random.default_rng(100 + kv_dtype * 7 + D)
    s_cap = 700
    kv_lens = [650, 300, 120, 0, 90, 500]
    kept = [
        sorted(rng.choice(650, size=400, replace=False).tolist()),              # scattered, many chunks
        list(range(200)),                                                        # prefix: trim_to(200)
        list(range(120)),                                                        # identity: no-op
        [],                                                                      # empty sequence
        [],                                                                      # keep nothing
        list(range(37)) + sorted(rng.choice(np.arange(40, 500), size=300, replace=False).tolist()),
    ]
    run_and_check(gpu_lib, kv_dtype, D, kv_lens, kept, s_cap, seed=kv_dtype + D)


def test_prefix_equals_trim_and_identity_moves_nothing(gpu_lib):
    """A prefix selection is trim_to: no byte of any cache changes, only kv_len."""
    s_cap, kv_lens = 300, [250, 250]
    kept = [list(range(77)), list(range(250))]
    rng = np.random.default_rng(5)
    K, V, _, _ = make_caches(rng, 1, 1, 2, 2, s_cap, 128)
    before = [bits(K[0]), bits(V[0])]
    Kd, Vd = [K[0].to(DEV)], [V[0].to(DEV)]
    desc = gpu_lib.kv_desc(Kd, Vd, HKV=2, D=128, kv_dtype=1)
    kv_len = i32(kv_lens)
    gpu_lib.gather_positions(desc, kv_len, i32([k + [-1] * (250 - len(k)) for k in kept]), i32([77, 250]))
    torch.cuda.synchronize()
    assert kv_len.tolist() == [77, 250]
    assert np.array_equal(bits(Kd[0]), before[0]) and np.array_equal(bits(Vd[0]), before[1])
    assert np.array_equal(bits(Kd[0])[0, :, :77], og.trim_to(before[0][0], 77, axis=1))


def test_tail_form_equals_absolute_form(gpu_lib):
    """tsv_kv_gather_positions(path) == tsv_gather_positions([0, S) + S + path), byte for byte."""
    T, s_cap, D, HKV = 9, 60, 64, 2
    S = [10, 0, 33, 7, 20]
    paths = [[0, 2, 5, 8], [0], [0, 1, 2], list(range(9)), [0, 3, 4, 7]]
    B = len(S)
    rng = np.random.default_rng(9)
    K, V, KS, VS = make_caches(rng, 2, 1, B, HKV, s_cap, D)
    outs = []
    for form in ("tail", "absolute"):
        Kd, Vd, KSd, VSd = [K[0].to(DEV)], [V[0].to(DEV)], [KS[0].to(DEV)], [VS[0].to(DEV)]
        desc = gpu_lib.kv_desc(Kd, Vd, HKV=HKV, D=D, kv_dtype=2, k_scale=KSd, v_scale=VSd)
        kv_len = i32([s + T for s in S])
        if form == "tail":
            gpu_lib.kv_gather_positions(desc, kv_len, i32([p + [-1] * (T - len(p)) for p in paths]),
                                        i32([len(p) for p in paths]), T)
        else:
            kept = [list(range(s)) + [s + j for j in p] for s, p in zip(S, paths)]
            m = max(len(k) for k in kept)
            gpu_lib.gather_positions(desc, kv_len, i32([k + [-1] * (m - len(k)) for k in kept]),
                                     i32([len(k) for k in kept]))
        torch.cuda.synchronize()
        outs.append([kv_len.tolist()] + [bits(x) for x in (Kd[0], Vd[0], KSd[0], VSd[0])])
    assert outs[0][0] == outs[1][0] == [s + len(p) for s, p in zip(S, paths)]
    for a, b in zip(outs[0][1:], outs[1][1:]):
        assert np.array_equal(a, b)


def test_gather_positions_long_history_int8(gpu_lib):
    """A 131,072-position Int8 history keeping every third position after a 1000-position prefix."""
    n_hist, s_cap, D = 131072, 131072 + 64, 256
    kept = list(range(1000)) + list(range(1001, n_hist, 3))
    run_and_check(gpu_lib, 2, D, [n_hist], [kept], s_cap, L=1, HKV=1, seed=77)


def test_gather_positions_bad_lists(gpu_lib):
    """Bad lists are refused on the device: that sequence keeps its bytes and kv_len, the others proceed."""
    s_cap, D = 64, 64
    kv_lens = [40, 40, 20, 40, 70]
    kept = [[0, 5, 5, 9], [0, 40], list(range(21)), [1, 2, 3], [0, 1]]  # repeat, out of range, too long, ok, ok
    rng = np.random.default_rng(3)
    K, V, _, _ = make_caches(rng, 0, 1, 5, 1, s_cap, D)
    before = bits(K[0])
    Kd, Vd = [K[0].to(DEV)], [V[0].to(DEV)]
    desc = gpu_lib.kv_desc(Kd, Vd, HKV=1, D=D, kv_dtype=0)
    kv_len = i32(kv_lens)
    m = max(len(k) for k in kept)
    st = torch.zeros(4, dtype=torch.int32, device=DEV)
    gpu_lib.gather_positions(desc, kv_len, i32([k + [-1] * (m - len(k)) for k in kept]), i32([len(k) for k in kept]),
                             dev_status=st)
    torch.cuda.synchronize()
    code = st.tolist()[0]
    assert code in (gpu_lib.DEV_BAD_PATH, gpu_lib.DEV_BAD_KV_LEN)
    assert kv_len.tolist() == [40, 40, 20, 3, 70]  # sequence 4 has kv_len 70 > s_cap: refused too
    got = bits(Kd[0])
    for b in (0, 1, 2, 4):
        assert np.array_equal(got[b], before[b])
    assert np.array_equal(got[3, 0, :3], before[3, 0, [1, 2, 3]])
