"""Comparisons of one GPU verify round against the fp64 oracle (test infrastructure).

Inputs for the oracle are regenerated on the host from the seeded generator
(``synth.tensors``); nothing the oracle sees comes from the GPU.  Tolerances:
attention within 2e-2 max-abs and 1e-2 relative L2 (bf16 output); argmax
exact (every node is planted with a top-1/top-2 gap of at least 1e-2);
mask, walk, path and gathered cache bytes bit-exact.
"""
from __future__ import annotations

import numpy as np
import torch

from oracle import gather as og
from oracle import storage as osd
from oracle import tree as ot
from synth import configs, tensors

from .oracle_side import (appended_rows, attention_units, head_rows_fn, oracle_lm_full,  # noqa: F401
                          oracle_lm_full_parallel)

ATT_MAX_ABS = 2e-2
ATT_REL_L2 = 1e-2


def u64(t: torch.Tensor) -> list[int]:
    return [int(x) & ((1 << 64) - 1) for x in t.cpu().numpy().reshape(-1).tolist()]


def bf16_tensor_to_f64(t: torch.Tensor) -> np.ndarray:
    return osd.bf16(t.detach().cpu().contiguous().view(torch.int16).numpy().view(np.uint16))


# ----------------------------------------------------------------------------- per-step oracles
def oracle_mask(parents: np.ndarray):
    B, T = parents.shape
    anc = [ot.ancestor_bits(parents[b].tolist()) for b in range(B)]
    depth = [[ot.depth(parents[b].tolist(), i) for i in range(T)] for b in range(B)]
    return anc, depth


def _cache_rows(cfg, c, which, b, kvh, r0, r1):
    """fp64 values of GPU cache rows [r0, r1) of one (sequence, kv head)."""
    t = c[which][b, kvh, r0:r1].cpu()
    if cfg.kv_dtype == configs.I8:
        sc = c["ks" if which == "k" else "vs"][b, kvh, r0:r1].cpu().view(torch.int16).numpy().view(np.uint16)
        return osd.int8_scaled(t.numpy(), sc)
    bits = t.view(torch.int16).numpy().view(np.uint16)
    return osd.f16(bits) if cfg.kv_dtype == configs.F16 else osd.bf16(bits)


def _appended_gather_ok(cfg, c, layer, b, kvh, parents_b, path) -> bool:
    S, T = cfg.S, cfg.T
    kb, vb = appended_rows(cfg, layer, b, kvh, parents_b)
    ok = True
    for which, exp_rows, exact in (("k", kb, False), ("v", vb, True)):
        exp, _ = og.gather_within_tail(exp_rows, 0, path)
        got = _cache_rows(cfg, c, which, b, kvh, S, S + T)
        if exact:
            ok &= bool(np.array_equal(got, exp))
        else:
            ok &= bool(np.max(np.abs(got - exp)) <= 1e-2 * max(float(np.max(np.abs(exp))), 1e-30))
    return ok


# ----------------------------------------------------------------------------- comparison of a round
def attn_stats(gpu: np.ndarray, ref: np.ndarray):
    err = np.abs(gpu - ref)
    rel = float(np.linalg.norm(gpu - ref) / max(np.linalg.norm(ref), 1e-30))
    return float(err.max()), rel


def check_round(wl, out, layers=(0,), attn_rows="all", lm="auto", kv_heads=None, seqs=None, rng_seed=0,
                lm_rows=8):
    """Compare every output of one round on ``wl`` (a synth.workload.Workload) with the oracle.

    attn_rows: "all" (every node), an int = number of nodes sampled per (layer, seq, kv head) (the last node
        always among them), or a list of node indices checked in every unit.
    lm: "full" (the oracle's whole-vocabulary argmax for every row), "planted" (every row's argmax == its
        planted target, and for ``lm_rows`` sampled rows the oracle's whole-vocabulary argmax, top-1 logit and
        top-1/top-2 gap), or "auto" (full when V <= 65536).
    """
    cfg = wl.cfg
    r = wl.round
    rng = np.random.default_rng(rng_seed)
    parents = r["parents"]
    B, T = parents.shape
    rep = {"ok": True}

    # a1 mask
    anc, depth = oracle_mask(parents)
    g_anc = u64(out["anc"])
    g_depth = out["depth"].cpu().numpy().reshape(-1).tolist()
    rep["mask_exact"] = g_anc == [a for row in anc for a in row] and g_depth == [d for row in depth for d in row]

    # a2 attention (sampled (layer, seq, kv head) units; all, sampled or listed nodes)
    seqs = list(range(B)) if seqs is None else seqs
    kv_heads = list(range(cfg.HKV)) if kv_heads is None else kv_heads
    units = []
    for layer in layers:
        for b in seqs:
            for kvh in kv_heads:
                if attn_rows == "all":
                    nodes = list(range(T))
                elif isinstance(attn_rows, (list, tuple)):
                    nodes = sorted(set(int(i) for i in attn_rows))
                else:
                    nodes = sorted(set(rng.choice(T, size=min(T, int(attn_rows)), replace=False).tolist()) | {T - 1})
                units.append((layer, b, kvh, nodes, parents[b].tolist()))
    refs = attention_units(cfg, units, parallel=len(units) > 1 and cfg.S >= 4096)
    worst_abs, worst_rel = 0.0, 0.0
    o_cache = {}
    for (layer, b, kvh, _, _) in units:
        if layer not in o_cache:
            o_cache[layer] = bf16_tensor_to_f64(out["o"][layer])
        o = o_cache[layer]
        ref = refs[(layer, b, kvh)]
        g = np.stack([o[b, i, h] for (i, h) in ref])
        e = np.stack(list(ref.values()))
        a, rl = attn_stats(g, e)
        worst_abs, worst_rel = max(worst_abs, a), max(worst_rel, rl)
    rep["attn_units"] = len(units)
    rep["attn_rows"] = sum(len(refs[k]) for k in refs)
    rep["attn_max_abs"], rep["attn_rel_l2"] = worst_abs, worst_rel
    rep["attn_ok"] = worst_abs <= ATT_MAX_ABS and worst_rel <= ATT_REL_L2

    # a3 LM head
    g_arg = out["argmax"].cpu().numpy().astype(np.int64)
    g_max = out["maxlogit"].cpu().numpy().astype(np.float64)
    targets = r["targets"].reshape(-1).astype(np.int64)
    mode = lm if lm != "auto" else ("full" if cfg.V <= 65536 else "planted")
    lm_fn = oracle_lm_full if cfg.V <= 65536 else oracle_lm_full_parallel
    if mode == "full":
        rows = np.arange(B * T)
        rep["lm_exact"] = True
    else:  # every row against its planted target; sampled rows against the oracle's whole-vocabulary argmax
        rows = np.sort(rng.choice(B * T, size=min(B * T, lm_rows), replace=False))
        rep["lm_exact"] = bool(np.array_equal(g_arg, targets))
    o_arg, o_top, o_gap = lm_fn(cfg, r["hidden"][rows])
    rep["lm_rows_oracle"] = int(len(rows))
    rep["lm_gap_min"] = float(o_gap.min())
    rep["lm_exact"] = rep["lm_exact"] and bool(np.array_equal(g_arg[rows], o_arg)) \
        and bool(np.array_equal(o_arg, targets[rows]))
    rep["lm_maxlogit_err"] = float(np.max(np.abs(g_max[rows] - o_top)))
    # exactness is claimed where the oracle's top-1/top-2 gap exceeds the workload's planted minimum
    rep["lm_ok"] = rep["lm_exact"] and rep["lm_gap_min"] >= cfg.min_gap \
        and rep["lm_maxlogit_err"] <= 1e-3 * (1 + float(np.max(np.abs(g_max))))

    # a4 walk (on the oracle's argmax == the planted targets)
    g_path = out["path"].cpu().numpy()
    g_len = out["path_len"].cpu().numpy()
    g_em = out["emitted"].cpu().numpy()
    walk_ok = True
    for b in range(B):
        path, em = ot.accept_walk(r["targets"][b], r["tokens"][b], parents[b])
        walk_ok &= g_len[b] == len(path) and g_path[b, :len(path)].tolist() == path \
            and bool(np.all(g_path[b, len(path):] == -1)) and g_em[b, :len(path)].tolist() == em \
            and path == r["paths"][b]
    rep["walk_exact"] = bool(walk_ok)

    # a5 gather (the caches were compacted in place by the round)
    kvl = wl.kv_len.cpu().numpy()
    gather_ok = True
    S = cfg.S
    for layer in layers:
        c = wl.caches[layer]
        for b in seqs:
            path = r["paths"][b]
            gather_ok &= int(kvl[b]) == S + len(path)
            for kvh in kv_heads:
                if cfg.rot_dim > 0:  # appended rows: V stored exactly, rotated K within one rounding step
                    gather_ok &= _appended_gather_ok(cfg, c, layer, b, kvh, parents[b].tolist(), path)
                    continue
                for w, key in (("k", "k"), ("v", "v")):
                    orig = tensors.kv_rows(cfg, w, layer, b, kvh, S, S + T)
                    exp, _ = og.gather_within_tail(orig, 0, path)
                    got = c[key][b, kvh, S:S + T].cpu()
                    got = got.view(torch.int8).numpy() if cfg.kv_dtype == configs.I8 else \
                        got.view(torch.int16).numpy().view(np.uint16)
                    gather_ok &= np.array_equal(got, exp)
                    if cfg.kv_dtype == configs.I8:
                        so = tensors.kv_scales(cfg, w, layer, b, kvh, S, S + T)
                        se, _ = og.gather_within_tail(so, 0, path)
                        gs = c["ks" if w == "k" else "vs"][b, kvh, S:S + T].cpu().view(torch.int16).numpy().view(np.uint16)
                        gather_ok &= np.array_equal(gs, se)
    rep["gather_exact"] = bool(gather_ok)
    rep["dev_status"] = out["status"].cpu().tolist()
    rep["ok"] = bool(rep["mask_exact"] and rep["attn_ok"] and rep["lm_ok"] and rep["walk_exact"]
                     and rep["gather_exact"] and rep["dev_status"][0] == 0)
    return rep
