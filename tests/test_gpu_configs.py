"""GPU parity at the five workloads' full sizes, in the launch configuration the bench times.

Every output is checked on the oracle's side from host-regenerated inputs: the mask, walk, path and gathered
bytes bit-exactly; attention on sampled (layer, sequence, kv head, node) rows within 2e-2 max-abs / 1e-2
relative L2; the argmax exactly: every row against the oracle's whole-vocabulary argmax on the first round of
the chain and 16-node workloads, elsewhere every row against its planted target and 8 sampled rows against the
oracle's whole-vocabulary argmax, top-1 logit and top-1/top-2 gap.
"""
import gc

import numpy as np
import pytest
import torch

from synth import configs, device as sd
from synth.workload import Workload

from .parity import check_round

pytestmark = pytest.mark.gpu


def _free():
    gc.collect()
    torch.cuda.empty_cache()


def _run(wl, round_id=0):
    if round_id:
        wl.set_round(round_id)
    out = wl.vr.run()
    torch.cuda.synchronize()
    return out


def test_device_fill_matches_host_generator(gpu_lib):
    from synth import tensors
    for name in ("tiny_tree7", "specinfer16_27b_i8"):
        cfg = configs.scaled(configs.workload(name), n_layers=1, S=300, V=777)
        c = sd.alloc_cache(cfg, 0, cfg.NKV + 5, "cuda")
        for w in ("k", "v"):
            host = tensors.kv_full(cfg, w, 0)
            dev = c[w][:, :, :cfg.NKV].cpu()
            dev = dev.numpy() if cfg.kv_dtype == configs.I8 else dev.view(torch.int16).numpy().view(np.uint16)
            assert np.array_equal(dev, host)
            assert torch.count_nonzero(c[w][:, :, cfg.NKV:]).item() == 0
            if cfg.kv_dtype == configs.I8:
                hs = tensors.kv_scales_full(cfg, w, 0)
                ds = c["ks" if w == "k" else "vs"][:, :, :cfg.NKV].cpu().view(torch.int16).numpy().view(np.uint16)
                assert np.array_equal(ds, hs)
        q = sd.alloc_q(cfg, 0, "cuda").cpu().view(torch.int16).numpy().view(np.uint16)
        assert np.array_equal(q, tensors.q_full(cfg, 0))
        hd = sd.alloc_head(cfg, "cuda")
        if cfg.w_dtype == configs.Q4:
            p, s, b = tensors.w_full(cfg)
            assert np.array_equal(hd["W"].cpu().numpy(), p)
            assert np.array_equal(hd["scales"].cpu().view(torch.int16).numpy().view(np.uint16), s)
            assert np.array_equal(hd["biases"].cpu().view(torch.int16).numpy().view(np.uint16), b)
        else:
            assert np.array_equal(hd["W"].cpu().view(torch.int16).numpy().view(np.uint16), tensors.w_full(cfg))


def test_tiny_every_round(gpu_lib):
    cfg = configs.workload("tiny_tree7")
    wl = Workload(cfg)
    wl.save_tail()
    for rid in range(6):
        wl.restore_tail()
        out = _run(wl, rid)
        rep = check_round(wl, out, layers=[0], attn_rows="all")
        assert rep["ok"], rep


@pytest.mark.parametrize("name", ["tiny_tree7", "specinfer16_27b_i8"])
def test_replayed_rounds_match_the_oracle(gpu_lib, name):
    """One captured graph serves every later round: new inputs copied into the buffers, then replay()."""
    cfg = configs.workload(name)
    if cfg.n_layers > 2:
        cfg = configs.scaled(cfg, n_layers=2)
    wl = Workload(cfg)
    wl.save_tail()
    _run(wl)  # one eager round on this stream before the capture (loads the kernels)
    wl.restore_tail()
    wl.vr.capture()
    torch.cuda.synchronize()
    for rid in range(4):
        wl.restore_tail()
        wl.set_round(rid)
        out = wl.vr.replay()
        torch.cuda.synchronize()
        rep = check_round(wl, out, layers=[0], attn_rows="all" if cfg.T <= 16 else 4)
        assert rep["ok"], (rid, rep)
    del wl
    _free()


def test_tiny_splits_and_ragged_capacity(gpu_lib):
    cfg = configs.workload("tiny_tree7")
    for splits in (1, 2, 3):
        wl = Workload(cfg, s_cap=cfg.NKV + 61, splits=splits)
        out = _run(wl)
        rep = check_round(wl, out, layers=[0], attn_rows="all")
        assert rep["ok"], rep


def test_chain3_bf16_every_accept_length(gpu_lib):
    """Linear chain T=3: mask == causal, walk == chain walk, gather == trim_to (identity), all accept lengths."""
    cfg = configs.workload("chain3_27b_bf16")
    wl = Workload(cfg)
    wl.save_tail()
    seen = set()
    for rid in range(3):
        wl.restore_tail()
        out = _run(wl, rid)
        rep = check_round(wl, out, layers=[0, 7, 15], attn_rows="all", kv_heads=[0, 3],
                          lm="full" if rid == 0 else "planted")
        assert rep["ok"], rep
        seen.add(len(wl.round["paths"][0]) - 1)
    assert seen == {0, 1, 2}
    del wl
    _free()


def test_specinfer16_int8_q4(gpu_lib):
    cfg = configs.workload("specinfer16_27b_i8")
    wl = Workload(cfg)
    wl.save_tail()
    accepts = set()
    for rid in range(4):
        wl.restore_tail()
        out = _run(wl, rid)
        rep = check_round(wl, out, layers=[0, 15], attn_rows=4, kv_heads=[1, 2],
                          lm="full" if rid == 0 else "planted", rng_seed=rid)
        assert rep["ok"], rep
        accepts.add(len(wl.round["paths"][0]) - 1)
    assert len(accepts) >= 2
    del wl
    _free()


def test_eagle32x8_f16(gpu_lib):
    cfg = configs.workload("eagle32x8_27b_f16")
    wl = Workload(cfg)
    out = _run(wl)
    paths = wl.round["paths"]
    assert sum(1 for p in paths if p != list(range(len(p)))) >= 4  # scattered gathers exercised
    scattered = [b for b, p in enumerate(paths) if p != list(range(len(p)))]
    # nodes from both 128-row tiles of a unit (row = node * 6 + head: node 21 straddles them)
    rep = check_round(wl, out, layers=[0, 7, 15], attn_rows=[0, 9, 20, 21, 22, 31], kv_heads=[0, 3],
                      seqs=sorted({0, 5} | set(scattered[:2])), lm="planted", lm_rows=8)
    assert rep["ok"], rep
    assert rep["lm_rows_oracle"] == 8
    del wl, out
    _free()


def test_eagle64x32_int8_q4_long_context(gpu_lib):
    cfg = configs.workload("eagle64x32_27b_i8")
    free, total = torch.cuda.mem_get_info()
    need = cfg.kv_bytes() + cfg.kv_scale_bytes() + cfg.lm_bytes() + (4 << 30)
    if free < need:
        pytest.skip(f"needs {need / 2**30:.0f} GiB free, have {free / 2**30:.0f}")
    wl = Workload(cfg)
    out = _run(wl)
    paths = wl.round["paths"]
    assert paths[0] == [0] and paths[1] == list(range(len(paths[1])))  # zero accept and identity gather
    scattered = [b for b, p in enumerate(paths) if p != list(range(len(p)))]
    assert len(scattered) >= 3
    seqs = sorted({0, 1, 31} | set(scattered[:3]) | {5, 20})
    # 4 layers x all 4 kv heads x 8 sequences; nodes from all three 128-row tiles of a unit (row = node * 6 +
    # head: nodes 21 and 42 straddle tile boundaries, 43..63 lie in the third tile)
    rep = check_round(wl, out, layers=[0, 5, 10, 15], attn_rows=[0, 10, 21, 30, 42, 43, 55, 63],
                      kv_heads=[0, 1, 2, 3], seqs=seqs, lm="planted", lm_rows=8)
    assert rep["ok"], rep
    assert rep["attn_units"] == 128 and rep["lm_rows_oracle"] == 8
    del wl, out
    _free()


@pytest.mark.parametrize("name,window,every", [("eagle32x8_27b_f16", 1024, 6), ("specinfer16_27b_i8", 2048, 4)])
def test_sliding_hybrid_full_size(gpu_lib, name, window, every):
    """Hybrid sliding/full models at full size: sliding layers see the tree mask intersected with their band."""
    cfg = configs.with_sliding_layers(configs.workload(name), window, every)
    assert cfg.layer_window(0) == window and cfg.layer_window(every - 1) == 0
    wl = Workload(cfg)
    out = _run(wl)
    rep = check_round(wl, out, layers=[0, every - 1, every], attn_rows=3, kv_heads=[1], seqs=[0], lm="planted")
    assert rep["ok"], rep
    del wl, out
    _free()


@pytest.mark.parametrize("name,rot_dim", [("chain3_27b_bf16", 256), ("specinfer16_27b_i8", 64)])
def test_round_that_appends_its_block_full_size(gpu_lib, name, rot_dim):
    """A round that first appends its block (rotary positions S + depth, Int8 quantised on append for the
    specinfer workload), then verifies it: every stage against the oracle of the appended cache."""
    cfg = configs.scaled(configs.workload(name), name=name + f"+append{rot_dim}", rot_dim=rot_dim)
    wl = Workload(cfg)
    assert wl.kv_len.tolist() == [cfg.S] * cfg.B
    out = _run(wl)
    rep = check_round(wl, out, layers=[0, 7], attn_rows="all" if cfg.T <= 16 else 4, kv_heads=[0, 3], lm="planted")
    assert rep["ok"], rep
    del wl, out
    _free()


@pytest.mark.parametrize("name", ["chain3_27b_bf16", "specinfer16_27b_i8"])
def test_sampled_round_full_size(gpu_lib, name):
    """Sampled verification at full vocabulary: each node's draw (temperature 1, top-k 20, top-p 0.95, its own
    uniform) against the oracle's draw from its own fp64 logits; the walk on those draws.  The GPU logits differ
    from the oracle's by fp32 accumulation (and the 4-bit head's fp16 dequantisation), so a draw may take any
    value the oracle draws within 2e-3 of the node's uniform or of top_p."""
    from oracle import lm_head as ol
    from oracle import sampling as osm
    from oracle import storage as osd
    from oracle import tree as ot
    from synth import tensors

    from .oracle_side import oracle_logits_full_parallel

    base = configs.workload(name)
    cfg = configs.scaled(base, name=base.name + "+sampled", sample=(1.0, 20, 0.95))
    wl = Workload(cfg)
    out = _run(wl)
    r = wl.round
    T = cfg.T
    lg = oracle_logits_full_parallel(cfg, r["hidden"])
    u = tensors.node_uniforms(cfg, 0).astype(np.float64)
    got = out["argmax"].cpu().numpy()
    g_path = out["path"].cpu().numpy()
    g_len = out["path_len"].cpu().numpy()
    eps = 2e-3
    for b in range(cfg.B):
        exact = []
        for i in range(T):
            row = b * T + i
            cands = {osm.draw(lg[row], 1.0, 20, pp, uu) for pp in (0.95 - eps, 0.95, 0.95 + eps)
                     for uu in (max(0.0, u[row] - eps), u[row], min(1 - 1e-12, u[row] + eps))}
            assert int(got[row]) in cands, (b, i, int(got[row]), cands)
            exact.append(osm.draw(lg[row], 1.0, 20, 0.95, u[row]) if len(cands) == 1 else None)
        if all(e is not None for e in exact):
            path, em = ot.accept_walk(exact, r["tokens"][b], r["parents"][b])
            assert g_len[b] == len(path) and g_path[b, :len(path)].tolist() == path
    del wl, out
    _free()
