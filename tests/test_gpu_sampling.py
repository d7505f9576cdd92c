"""GPU parity of sampled verification: every logit of the LM head, and each node's nucleus-filtered draw.

The sampler gets the same fp32 logits the oracle reads, so only its fp32 softmax and prefix sums differ from
the oracle's fp64 ones: a draw must equal the oracle's, except when the uniform or top_p lies within 1e-5 of a
cumulative-mass boundary, where any token the oracle draws within that distance is accepted.
"""
import numpy as np
import pytest
import torch

from oracle import lm_head as ol
from oracle import sampling as osm
from oracle import storage as osd

pytestmark = pytest.mark.gpu
DEV = "cuda"


def q4_pack(codes):
    return (codes[:, 0::2] | (codes[:, 1::2] << 4)).astype(np.uint8)


@pytest.mark.parametrize("w_dtype", [0, 1, 3])
@pytest.mark.parametrize("rows,V,H", [(3, 4099, 512), (16, 1280, 5120), (30, 1100, 1024), (130, 1100, 512)])
def test_lm_head_logits_match_oracle(gpu_lib, w_dtype, rows, V, H):
    rng = np.random.default_rng(rows + V + w_dtype)
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
    logits = torch.full((rows, V), float("nan"), dtype=torch.float32, device=DEV)
    gpu_lib.lm_head_logits(h.to(DEV), Wd, logits, w_dtype=w_dtype, V=V, scales=sc, biases=bi)
    arg = torch.zeros(rows, dtype=torch.int32, device=DEV)
    gpu_lib.lm_head_argmax(h.to(DEV), Wd, arg, w_dtype=w_dtype, V=V, scales=sc, biases=bi)
    torch.cuda.synchronize()
    ref = ol.logits(W64, h.double().numpy())
    got = logits.cpu().numpy().astype(np.float64)
    assert np.allclose(got, ref, rtol=1e-4, atol=1e-3)
    # the argmax entry point picks the largest of the same logits (lowest index among equal ones)
    assert np.array_equal(arg.cpu().numpy(), np.argmax(got, axis=1))


def draws_ok(gpu_tok, logits_row, T, k, p, u, eps=1e-5):
    cands = {osm.draw(logits_row, T, k, pp, uu) for pp in (p - eps, p, min(1.0, p + eps))
             for uu in (max(0.0, u - eps), u, min(1.0 - 1e-12, u + eps))}
    return int(gpu_tok) in cands


@pytest.mark.parametrize("V", [10, 1000, 4096, 4097, 50000])
@pytest.mark.parametrize("T,k,p", [(1.0, 20, 0.95), (0.7, 64, 0.5), (1.5, 1, 0.9), (1.0, 33, 1.0), (0.3, 7, 0.99)])
def test_sample_nucleus_matches_oracle(gpu_lib, V, T, k, p):
    rng = np.random.default_rng(V + k)
    rows = 37
    logits = (rng.standard_normal((rows, V)) * rng.uniform(0.5, 4, size=(rows, 1))).astype(np.float32)
    logits[3, 5 % V] = logits[3, 2 % V] = logits[3].max() + 0.25  # a tie at the top: the lower index first
    u = rng.uniform(0, 1, size=rows).astype(np.float32)
    out = torch.full((rows,), -1, dtype=torch.int32, device=DEV)
    gpu_lib.sample_nucleus(torch.from_numpy(logits).to(DEV), torch.from_numpy(u).to(DEV), out, temperature=T,
                           top_k=k, top_p=p)
    torch.cuda.synchronize()
    got = out.cpu().numpy()
    for r in range(rows):
        assert draws_ok(got[r], logits[r].astype(np.float64), T, k, p, float(u[r])), (r, got[r])
    if k == 1:
        assert got[3] == min(5 % V, 2 % V)


def test_sample_nucleus_full_vocabulary_and_refusals(gpu_lib):
    rng = np.random.default_rng(7)
    rows, V = 5, 248320  # three rounds of top-k merging
    logits = rng.standard_normal((rows, V)).astype(np.float32) * 3
    u = np.array([0.0, 0.25, 0.5, 0.75, 0.999], dtype=np.float32)
    out = torch.zeros(rows, dtype=torch.int32, device=DEV)
    lt = torch.from_numpy(logits).to(DEV)
    gpu_lib.sample_nucleus(lt, torch.from_numpy(u).to(DEV), out, temperature=1.0, top_k=20, top_p=0.95)
    torch.cuda.synchronize()
    for r in range(rows):
        assert draws_ok(out[r].item(), logits[r].astype(np.float64), 1.0, 20, 0.95, float(u[r]))
    with pytest.raises(gpu_lib.TsvError, match="TSV_EUNSUPPORTED"):
        gpu_lib.sample_nucleus(lt, torch.from_numpy(u).to(DEV), out, temperature=1.0, top_k=65, top_p=0.9)
    with pytest.raises(gpu_lib.TsvError, match="TSV_EINVAL"):
        gpu_lib.sample_nucleus(lt, torch.from_numpy(u).to(DEV), out, temperature=0.0, top_k=20, top_p=0.9)
