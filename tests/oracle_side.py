"""The oracle's side of a full-size round, spread over worker processes (test infrastructure).

Everything here is numpy: inputs regenerated on the host from the seeded generator (``synth.tensors``), then the
fp64 oracle (``oracle``).  Nothing reads the GPU.  At the full workloads one whole-vocabulary argmax (248,320
LM-head rows regenerated at hidden 5120) or one attention unit over 131,072 keys takes about a minute on one
core, so the work is spread over a process pool.  The pool is started with ``spawn``: a child forked from a
process that already holds a CUDA context can hang.  Workers import only this module, ``synth`` and ``oracle``.
"""
from __future__ import annotations

import atexit
import concurrent.futures as cf
import multiprocessing as mp
import os

import numpy as np

from oracle import append as oap
from oracle import attention as oa
from oracle import lm_head as ol
from oracle import storage as osd
from oracle import tree as ot
from synth import configs, tensors

_POOL = None


def pool() -> cf.ProcessPoolExecutor:
    """The shared spawn pool (one worker per host core, at most 16)."""
    global _POOL
    if _POOL is None:
        n = max(1, min(16, os.cpu_count() or 1))
        _POOL = cf.ProcessPoolExecutor(max_workers=n, mp_context=mp.get_context("spawn"))
        atexit.register(_POOL.shutdown, wait=False, cancel_futures=True)
    return _POOL


# ----------------------------------------------------------------------------- stored values
def stored(cfg, x):
    """The value a cache of cfg's format keeps for fp64 row values x [n, D] (oracle's own rounding)."""
    if cfg.kv_dtype == configs.I8:
        out = []
        for row in x:
            codes, sbits = oap.quantize_token(row)
            out.append(codes.astype(np.float64) * float(np.uint16(sbits).view(np.float16)))
        return np.stack(out)
    return osd.round_f16(x) if cfg.kv_dtype == configs.F16 else osd.round_bf16(x)


def appended_rows(cfg, layer, b, kvh, parents_b):
    """K and V block rows [S, S+T) as an appending round stores them (rotated K, then the cache's format)."""
    pos = oap.node_positions(parents_b, cfg.S)
    kn = osd.bf16(np.stack([tensors.new_kv_rows(cfg, "k", layer, b, i)[kvh] for i in range(cfg.T)]))
    vn = osd.bf16(np.stack([tensors.new_kv_rows(cfg, "v", layer, b, i)[kvh] for i in range(cfg.T)]))
    k_rot = np.stack([oap.rope(kn[i], pos[i], cfg.rope_base, cfg.rot_dim) for i in range(cfg.T)])
    return stored(cfg, k_rot), stored(cfg, vn)


def kv_values(cfg, layer, b, kvh, parents_b=None):
    """fp64 K and V of one (layer, sequence, kv head) over the logical S + T rows."""
    out = []
    for w in ("k", "v"):
        store = tensors.kv_rows(cfg, w, layer, b, kvh, 0, cfg.NKV)
        sc = tensors.kv_scales(cfg, w, layer, b, kvh, 0, cfg.NKV) if cfg.kv_dtype == configs.I8 else None
        out.append(osd.kv_values(cfg.kv_dtype, store, sc))
    if cfg.rot_dim > 0:  # the round appended its own block over rows [S, S + T)
        kb, vb = appended_rows(cfg, layer, b, kvh, parents_b)
        out[0][cfg.S:cfg.NKV], out[1][cfg.S:cfg.NKV] = kb, vb
    return out


# ----------------------------------------------------------------------------- attention
def oracle_attention_rows(cfg, layer, b, kvh, nodes, parents_b):
    """O rows for every (node in nodes, head of the kv group) -> dict[(i, h)] = fp64 [D]."""
    K, V = kv_values(cfg, layer, b, kvh, parents_b)
    G = cfg.G
    heads = [kvh * G + g for g in range(G)]
    res = {}
    w = cfg.layer_window(layer)
    pos = oap.node_positions(parents_b, cfg.S)
    for i in nodes:
        q = osd.bf16(tensors.q_rows(cfg, layer, b, i, heads))
        if cfg.rot_dim > 0:  # the attention reads Q rotated to the node's position, stored as bf16
            q = osd.round_bf16(oap.rope(q, pos[i], cfg.rope_base, cfg.rot_dim))
        vis = ot.ancestors(parents_b, i)
        cols = ot.visible_keys(parents_b, i, cfg.S, w)
        for gi, h in enumerate(heads):
            res[(i, h)] = oa.attend_row(q[gi], K, V, cfg.S, vis) if w == 0 else oa.attend_cols(q[gi], K, V, cols)
    return res


def _attention_unit(args):
    cfg, layer, b, kvh, nodes, parents_b = args
    return (layer, b, kvh), oracle_attention_rows(cfg, layer, b, kvh, nodes, parents_b)


def attention_units(cfg, units, parallel: bool):
    """{(layer, b, kvh): {(i, h): row}} for units = [(layer, b, kvh, nodes, parents_b)], in a pool if asked."""
    jobs = [(cfg, l, b, h, list(nodes), list(par)) for (l, b, h, nodes, par) in units]
    if not parallel or len(jobs) <= 1:
        return dict(map(_attention_unit, jobs))
    return dict(pool().map(_attention_unit, jobs))


# ----------------------------------------------------------------------------- LM head
def head_rows_fn(cfg):
    """weight_rows(r0, r1) -> fp64 [r1 - r0, H]: the exact LM-head rows regenerated from the generator."""
    if cfg.w_dtype == configs.Q4:
        def wr(r0, r1):
            rows = np.arange(r0, r1)
            s, b = tensors.wq_scales_biases(cfg, rows)
            return osd.q4_affine(tensors.wq_packed(cfg, rows), s, b)
        return wr
    dec = osd.bf16 if cfg.w_dtype == configs.BF16 else osd.f16
    return lambda r0, r1: dec(tensors.w_rows(cfg, np.arange(r0, r1)))


def oracle_lm_full(cfg, hidden_bits):
    """Whole-vocabulary (argmax, top-1, gap) of every row, single process."""
    h = osd.bf16(hidden_bits)
    return ol.argmax_streamed(head_rows_fn(cfg), h, cfg.V)


def _lm_chunk(args):
    cfg, hidden_bits, r0, r1 = args
    return r0, ol.logits(head_rows_fn(cfg)(r0, r1), osd.bf16(hidden_bits))


def oracle_logits_full_parallel(cfg, hidden_bits):
    """Every fp64 logit [rows, V] (the definition of ``lm_head.logits_streamed``), chunks spread over the pool."""
    jobs = [(cfg, np.asarray(hidden_bits), r0, min(cfg.V, r0 + ol.CHUNK_ROWS)) for r0 in range(0, cfg.V, ol.CHUNK_ROWS)]
    parts = dict(pool().map(_lm_chunk, jobs))
    return np.concatenate([parts[r0] for r0 in sorted(parts)], axis=1)


def oracle_lm_full_parallel(cfg, hidden_bits):
    """The same (argmax, top-1, gap) as ``oracle_lm_full``, the vocabulary's chunks spread over the pool."""
    return ol.argmax_gap(oracle_logits_full_parallel(cfg, hidden_bits))
