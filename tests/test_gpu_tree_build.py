"""GPU parity of draft-tree construction: the drafter's top-k children and the best-first selection.

Children tokens are compared exactly (packed keys order equal logits by index on both sides) and their
log-probabilities within 1e-5 (fp32 log-sum-exp against fp64).  The selection takes its decisions on fp32
scores summed from the root down on both sides, so its output is compared exactly.
"""
import numpy as np
import pytest
import torch

from oracle import tree as ot
from oracle import tree_build as otb

pytestmark = pytest.mark.gpu
DEV = "cuda"


@pytest.mark.parametrize("V,k", [(1000, 1), (1000, 4), (50000, 16), (248320, 64), (4097, 20)])
def test_draft_children_match_oracle(gpu_lib, V, k):
    rng = np.random.default_rng(V + k)
    rows = 11
    x = (rng.standard_normal((rows, V)) * 2).astype(np.float32)
    x[2, [7, 9]] = x[2].max() + 0.5  # tied top logits: the lower index first
    toks = torch.zeros(rows, k, dtype=torch.int32, device=DEV)
    lp = torch.zeros(rows, k, dtype=torch.float32, device=DEV)
    gpu_lib.draft_children(torch.from_numpy(x).to(DEV), toks, lp, top_k=k)
    torch.cuda.synchronize()
    for r in range(rows):
        t, l = otb.draft_children(x[r].astype(np.float64), k)
        assert toks[r].tolist() == t.tolist(), r
        assert np.allclose(lp[r].cpu().numpy(), l, rtol=0, atol=1e-5), r


def random_candidates(rng, B, N):
    par = np.zeros((B, N), dtype=np.int32)
    for b in range(B):
        par[b, 0] = -1
        for i in range(1, N):
            par[b, i] = rng.integers(max(0, i - 12), i)
    tok = rng.integers(0, 248320, size=(B, N)).astype(np.int32)
    lp = np.log(rng.uniform(0.02, 1.0, size=(B, N))).astype(np.float32)
    lp[:, 5 % N] = 0.0  # a child as likely as its parent: equal scores, the earlier candidate first
    return par, tok, lp


@pytest.mark.parametrize("B,N,T,depth_max", [(3, 40, 16, 6), (2, 1024, 64, 8), (4, 200, 32, 64), (1, 5, 16, 8),
                                             (2, 300, 1, 4)])
def test_tree_select_matches_oracle(gpu_lib, B, N, T, depth_max):
    rng = np.random.default_rng(N + T)
    par, tok, lp = random_candidates(rng, B, N)
    outs = [torch.full((B, T), 99, dtype=torch.int32, device=DEV) for _ in range(3)]
    sizes = torch.zeros(B, dtype=torch.int32, device=DEV)
    st = torch.zeros(4, dtype=torch.int32, device=DEV)
    gpu_lib.tree_select(torch.from_numpy(par).to(DEV), torch.from_numpy(tok).to(DEV), torch.from_numpy(lp).to(DEV),
                        *outs, sizes, depth_max=depth_max, dev_status=st)
    torch.cuda.synchronize()
    assert st.tolist()[0] == 0
    for b in range(B):
        p, t, idx = otb.select_best_first(par[b].tolist(), tok[b], lp[b], T, depth_max)
        n = len(idx)
        assert sizes[b].item() == n
        assert outs[0][b, :n].tolist() == p and outs[1][b, :n].tolist() == t and outs[2][b, :n].tolist() == idx
        assert outs[0][b, n:].tolist() == [-1] * (T - n)
        assert ot.validate(p) == ot.OK


def test_tree_select_device_errors(gpu_lib):
    B, N, T = 2, 6, 4
    par = np.array([[-1, 0, 0, 1, 1, 2], [-1, 0, 3, 1, 1, 2]], dtype=np.int32)  # sequence 1: parent 3 of node 2
    tok = np.arange(B * N, dtype=np.int32).reshape(B, N)
    lp = np.full((B, N), -0.5, dtype=np.float32)
    outs = [torch.zeros(B, T, dtype=torch.int32, device=DEV) for _ in range(3)]
    sizes = torch.zeros(B, dtype=torch.int32, device=DEV)
    st = torch.zeros(4, dtype=torch.int32, device=DEV)
    gpu_lib.tree_select(torch.from_numpy(par).to(DEV), torch.from_numpy(tok).to(DEV), torch.from_numpy(lp).to(DEV),
                        *outs, sizes, depth_max=8, dev_status=st)
    torch.cuda.synchronize()
    assert st.tolist()[:3] == [gpu_lib.DEV_BAD_PARENT, 1, 2]
    assert sizes.tolist() == [4, 0] and outs[0][1].tolist() == [-1] * T
    p, _, _ = otb.select_best_first(par[0].tolist(), tok[0], lp[0], T, 8)
    assert outs[0][0].tolist() == p


def test_children_then_select_then_mask(gpu_lib):
    """Drafter logits -> children -> a two-level candidate tree -> the verified tree -> a valid mask, against the
    oracle's own children and selection from the same drafter logits."""
    rng = np.random.default_rng(3)
    B, V, k, T = 2, 5000, 4, 8
    root_logits = (rng.standard_normal((B, V)) * 3).astype(np.float32)
    toks = torch.zeros(B, k, dtype=torch.int32, device=DEV)
    lps = torch.zeros(B, k, dtype=torch.float32, device=DEV)
    gpu_lib.draft_children(torch.from_numpy(root_logits).to(DEV), toks, lps, top_k=k)
    lvl2 = (rng.standard_normal((B * k, V)) * 3).astype(np.float32)
    t2 = torch.zeros(B * k, k, dtype=torch.int32, device=DEV)
    l2 = torch.zeros(B * k, k, dtype=torch.float32, device=DEV)
    gpu_lib.draft_children(torch.from_numpy(lvl2).to(DEV), t2, l2, top_k=k)
    torch.cuda.synchronize()
    N = 1 + k + k * k  # root, its k children, their k children each
    par = np.zeros((B, N), dtype=np.int32)
    tok = np.zeros((B, N), dtype=np.int32)
    lp = np.zeros((B, N), dtype=np.float32)
    for b in range(B):
        par[b, 0] = -1
        par[b, 1:1 + k] = 0
        tok[b, 1:1 + k] = toks[b].cpu().numpy()
        lp[b, 1:1 + k] = lps[b].cpu().numpy()
        for c in range(k):
            s = 1 + k + c * k
            par[b, s:s + k] = 1 + c
            tok[b, s:s + k] = t2[b * k + c].cpu().numpy()
            lp[b, s:s + k] = l2[b * k + c].cpu().numpy()
    outs = [torch.zeros(B, T, dtype=torch.int32, device=DEV) for _ in range(3)]
    sizes = torch.zeros(B, dtype=torch.int32, device=DEV)
    gpu_lib.tree_select(torch.from_numpy(par).to(DEV), torch.from_numpy(tok).to(DEV), torch.from_numpy(lp).to(DEV),
                        *outs, sizes, depth_max=8)
    anc = torch.zeros(B, T, dtype=torch.int64, device=DEV)
    depth = torch.zeros(B, T, dtype=torch.int32, device=DEV)
    st = torch.zeros(4, dtype=torch.int32, device=DEV)
    gpu_lib.tree_mask(outs[0], anc, depth, dev_status=st)
    torch.cuda.synchronize()
    assert sizes.tolist() == [T] * B and st.tolist()[0] == 0
    # the oracle's own chain from the same drafter logits: its children, its candidate tree, its selection
    for b in range(B):
        otok = np.zeros(N, dtype=np.int64)
        olp = np.zeros(N, dtype=np.float32)
        ct, cl = otb.draft_children(root_logits[b].astype(np.float64), k)
        otok[1:1 + k], olp[1:1 + k] = ct, cl
        for c in range(k):
            s = 1 + k + c * k
            ct, cl = otb.draft_children(lvl2[b * k + c].astype(np.float64), k)
            otok[s:s + k], olp[s:s + k] = ct, cl
        p, t, idx = otb.select_best_first(par[b].tolist(), otok, olp, T, 8)
        assert outs[0][b].tolist() == p and outs[1][b].tolist() == t
