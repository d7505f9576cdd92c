"""Benchmark of the tree-verify step: verified nodes/s and achieved HBM bandwidth.

One step = one whole verify round on one batch of synthetic input: tree_mask -> tree_verify_attention over all
16 layers -> lm_head_argmax -> tree_accept_walk -> kv_gather_positions, plus resetting kv_len to S + T (the
round's tree block is considered appended; the gather advanced kv_len).  Default workload: a 3-node chain over a
4096-token bf16 prefix at the 27B-like shape (16 layers, 24 q / 4 kv heads, D=256, hidden 5120, bf16 LM head
248,320 x 5120); its inputs (2.81 GB per round) are larger than L2, so no flush is needed between steps.

python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference] [--config WORKLOAD]
Under torchrun every rank runs its own replica on its own GPU (the path has no exchange step); rank 0 prints
one JSON line.  --impl reference times the fp64 CPU oracle on a bounded sample on the host cores instead.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "tree-verify nodes/s per round and achieved HBM GB/s as fraction of GB300 peak"
DEFAULT_CONFIG = "chain3_27b_bf16"
DEFAULT_ROUND = {"chain3_27b_bf16": 2}  # the round that accepts the whole chain (3 tokens emitted)

# ncu dram bytes (read + write) per launch of the dominant kernel, with the source hash it was measured on
# (a changed kernel source makes the number stale and it is reported as null).
TRAFFIC = {
    ("chain3_27b_bf16", ("lm_head.cu", "common.cuh")): {"hash": "2530ef189b03e4bc", "bytes": 2543127040 + 2785024},
}


def peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            p = json.load(f)
        return float(p["hbm_gbs"]), "measured"
    except Exception:
        return 6800.0, "fallback"


def src_hash(names):
    h = hashlib.sha256()
    for name in names:
        with open(os.path.join(ROOT, "tree_speculative_decoding_array_gb300", "csrc", name), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


# ----------------------------------------------------------------------------- clocks
REASON_BITS = {0x1: "gpu_idle", 0x2: "applications_clocks_setting", 0x4: "sw_power_cap", 0x8: "hw_slowdown",
               0x10: "sync_boost", 0x20: "sw_thermal_slowdown", 0x40: "hw_thermal_slowdown",
               0x80: "hw_power_brake_slowdown", 0x100: "display_clock_setting"}


class ClockSampler:
    def __init__(self, index: int):
        self.index, self.proc, self.lines = index, None, []

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index),
                 "--query-gpu=clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.t = threading.Thread(target=self._read, daemon=True)
            self.t.start()
        except Exception:
            self.proc = None
        return self

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def __exit__(self, *a):
        if self.proc:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()

    def summary(self):
        sm, mx, reasons = [], [], set()
        for ln in self.lines:
            parts = [x.strip() for x in ln.split(",")]
            if len(parts) < 4:
                continue
            try:
                sm.append(float(parts[0]))
                mx.append(float(parts[1]))
                bits = int(parts[3], 16) if parts[3].startswith("0x") else int(parts[3])
                for b, n in REASON_BITS.items():
                    if bits & b:
                        reasons.add(n)
            except ValueError:
                continue
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"]}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx), "reasons": sorted(reasons), "samples": len(sm)}


# ----------------------------------------------------------------------------- multi-rank helpers
def max_over_ranks(ms: float, device="cpu") -> float:
    """Slowest rank's timed-region length (every rank runs its own replica; no data-path exchange)."""
    import torch

    t = torch.tensor([ms], dtype=torch.float64, device=device)
    torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
    return float(t.item())


def aggregate_nodes_per_s(world: int, nodes_per_round: int, steps: int, ms: float) -> float:
    """Whole-job throughput: every rank verified ``steps`` rounds of ``nodes_per_round`` nodes in ``ms``."""
    return world * nodes_per_round * steps / (ms * 1e-3)


# ----------------------------------------------------------------------------- our arm
def run_ours(args, rank, world, local_rank):
    import torch

    import tree_speculative_decoding_array_gb300 as tsv
    from synth import configs
    from synth.workload import Workload

    tsv.load()
    dev = f"cuda:{local_rank}"
    torch.cuda.set_device(dev)
    cfg = configs.workload(args.config)
    if args.layers:
        cfg = configs.scaled(cfg, n_layers=args.layers)
    if args.sliding:
        w, e = (int(x) for x in args.sliding.split(":"))
        cfg = configs.with_sliding_layers(cfg, w, e)
    if args.append:
        cfg = configs.scaled(cfg, name=f"{cfg.name}+append{args.append}", rot_dim=args.append)
    if args.sampled:
        t, k, p = args.sampled.split(":")
        cfg = configs.scaled(cfg, name=f"{cfg.name}+sampled{args.sampled}", sample=(float(t), int(k), float(p)))
    round_id = args.round if args.round is not None else DEFAULT_ROUND.get(args.config, 0)
    wl = Workload(cfg, device=dev, round_id=round_id, attn_path=args.attn_path)
    vr = wl.vr
    wl.save_tail()
    moved = any(p != list(range(len(p))) for p in wl.round["paths"])
    stream = torch.cuda.current_stream()
    names = (["build"] if args.build_tree else []) + ["mask"] + (["append"] if cfg.rot_dim > 0 else []) + \
        ["attn", "lm", "walk", "gather"]
    build = make_build_stage(cfg, args.build_tree, dev) if args.build_tree else None

    def reset():  # one launch: pristine tails of every cache and kv_len (S + T; S when the round appends)
        wl.restore_tail()

    def step(evs=None):
        reset()
        for i, n in enumerate(names):
            if evs is not None:
                evs[i][0].record(stream)
            if n == "build":
                build()
            else:
                vr.run(stages=(n,))
            if evs is not None:
                evs[i][1].record(stream)

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    ev = [[(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in names]
          for _ in range(args.steps)]
    t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    if args.graph:
        # The round captured once as a CUDA graph and replayed: the same launches on the same buffers, without
        # the host issuing each one.  Per-stage times come from the eager rounds timed below it.
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph):
            step()
        for _ in range(args.warmup):
            graph.replay()
        torch.cuda.synchronize()
    with ClockSampler(torch.cuda.current_device()) as clk:
        t0.record(stream)
        for s in range(args.steps):
            if args.graph:
                graph.replay()
            else:
                step(ev[s])
        t1.record(stream)
        torch.cuda.synchronize()
    if world > 1:
        torch.distributed.barrier()
    ms = t0.elapsed_time(t1)
    if args.graph:  # per-stage times: eager rounds with events
        for s in range(args.steps):
            step(ev[s])
        torch.cuda.synchronize()
    per_kernel = {n: statistics.mean(ev[s][i][0].elapsed_time(ev[s][i][1]) for s in range(args.steps))
                  for i, n in enumerate(names)}
    if world > 1:
        ms = max_over_ranks(ms, dev)

    # correctness of the timed state: one more round, check it against the planted walk
    step()
    torch.cuda.synchronize()
    got_len = vr.outs["path_len"].cpu().tolist()
    want_len = [len(p) for p in wl.round["paths"]]
    if cfg.sample:  # the walk follows each node's draw, not the planted argmax path
        assert all(1 <= n <= cfg.T for n in got_len), got_len
    else:
        assert got_len == want_len, (got_len, want_len)

    # e2e through the public API with host buffers: per step H2D of the round inputs, D2H of the results
    e2e = run_e2e(args, wl, stream) if rank == 0 else None

    # launches of our kernels per step
    if cfg.rows > 8:  # tensor-core LM head: key reset + (fp16 copy of hidden) + kernel + unpack (sampled: + sampler)
        lm_launches = 1 + 1 + (cfg.w_dtype != configs.BF16) + 1
    else:  # CUDA-core GEMV: key reset + one launch per group of up to 8 rows + unpack
        lm_groups, left = 0, cfg.rows
        while left > 0:
            left -= 8 if left >= 8 else (4 if left >= 4 else left)
            lm_groups += 1
        lm_launches = 1 + lm_groups + 1
    if cfg.sample:  # no unpack; top-k passes (one per 4096-entry chunk level) and the draw
        n, passes = cfg.V, 0
        while True:
            passes += 1
            ch = (n + 4095) // 4096
            if ch == 1:
                break
            n = ch * min(int(cfg.sample[1]), cfg.V)
        lm_launches += passes + 1 - 1
    launches = 1 + (1 + (tsv.attention_workspace_size(vr.adesc) > 0)) + lm_launches + 1 + 2 + (2 if cfg.rot_dim > 0 else 0)
    if args.build_tree:  # draft children: top-k passes + output; selection: one
        n, passes = cfg.V, 0
        while True:
            passes += 1
            ch = (n + 4095) // 4096
            if ch == 1:
                break
            n = ch * args.build_tree
        launches += passes + 1 + 1
    return dict(cfg=cfg, ms=ms, per_kernel=per_kernel, clocks=clk.summary(), e2e=e2e, launches=launches,
                round_id=round_id)


def make_build_stage(cfg, k, dev):
    """Tree construction on synthetic drafter output: every node of the round's B trees is expanded (drafter
    logits [B*T, V], N(0, 1) bf16 values widened to fp32), its top-k children become candidates, and the best-first
    selection picks T of the 1 + T*k candidates per sequence.  The verify stages keep the planted trees (the round
    stays checkable); this stage is timed beside them."""
    import torch

    import tree_speculative_decoding_array_gb300 as tsv
    from synth import device as sd
    from synth import tensors as st

    B, T, V = cfg.B, cfg.T, cfg.V
    lg16 = torch.empty(B * T, V, dtype=torch.bfloat16, device=dev)
    sd.fill(lg16, sd.NORMAL_BF16, st.key(cfg, st.KIND_DRAFT), (1, 1, B * T, V), (0, 0, V))
    logits = lg16.float()
    del lg16
    toks = torch.empty(B * T, k, dtype=torch.int32, device=dev)
    lps = torch.empty(B * T, k, dtype=torch.float32, device=dev)
    ws = torch.empty(max(int(tsv.load().tsv_draft_children_workspace_size(B * T, V, k)), 256), dtype=torch.uint8,
                     device=dev)
    N = 1 + T * k
    par = torch.empty(B, N, dtype=torch.int32)
    par[:, 0] = -1
    for m in range(T):  # children of the m-th expanded candidate (0 = the root, then candidates 1, 2, ...)
        par[:, 1 + m * k:1 + (m + 1) * k] = m
    par = par.to(dev)
    ctok = torch.zeros(B, N, dtype=torch.int32, device=dev)
    clp = torch.zeros(B, N, dtype=torch.float32, device=dev)
    outs = [torch.empty(B, T, dtype=torch.int32, device=dev) for _ in range(3)]
    sizes = torch.empty(B, dtype=torch.int32, device=dev)

    def build():
        tsv.draft_children(logits, toks, lps, top_k=k, workspace=ws)
        # candidates 1 + m*k + j of sequence b are child j of its node m (a strided view: no extra copy kernel
        # of ours runs; torch's copy is the only non-tsv launch of the stage)
        clp[:, 1:].copy_(lps.view(B, T * k))
        ctok[:, 1:].copy_(toks.view(B, T * k))
        tsv.tree_select(par, ctok, clp, *outs, sizes, depth_max=cfg.depth_max or T)
    return build


def run_e2e(args, wl, stream):
    import torch

    vr, cfg = wl.vr, wl.cfg
    # the round's inputs (parents, tokens, hidden, Q per layer, ...) are one device buffer: one pinned H2D copy;
    # its int32 results (path, path_len, emitted, argmax) one block: one D2H copy
    h_in = wl.inputs.detach().cpu().pin_memory()
    res = vr.outs["result"]
    h_res = torch.empty(res.shape, dtype=res.dtype).pin_memory()
    h2d = h_in.numel() * h_in.element_size()
    d2h = h_res.numel() * h_res.element_size()

    if args.graph:  # the public capture / replay pair: one graph of the round's calls over its buffers
        vr.capture()
        torch.cuda.synchronize()

    def e2e_step():
        wl.restore_tail()
        wl.inputs.copy_(h_in, non_blocking=True)
        if args.graph:
            vr.replay()
        else:
            vr.run()
        h_res.copy_(res, non_blocking=True)

    for _ in range(3):
        e2e_step()
    torch.cuda.synchronize()
    n = max(3, args.steps // 4)
    t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    t0.record(stream)
    for _ in range(n):
        e2e_step()
    t1.record(stream)
    torch.cuda.synchronize()
    ms = t0.elapsed_time(t1) / n
    return {"value": cfg.rows / (ms * 1e-3), "unit": "nodes/s", "ms_per_step": ms, "steps": n,
            "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
            "launch": "VerifyRound.replay (cuda graph)" if args.graph else "VerifyRound.run (eager)"}


# ----------------------------------------------------------------------------- oracle on the host
ORACLE_SAMPLE = r"""
import json, os, sys, time
sys.path.insert(0, {root!r})
import numpy as np
from oracle import attention as oa, lm_head as ol, storage as osd, tree as ot, gather as og
from synth import configs, tensors, trees
cfg = configs.workload({cfg_name!r})
r = trees.make_round(cfg, {round_id})
par = r["parents"][0].tolist()
# inputs for the sample (untimed): one (layer, kv head) unit of attention, a slice of the LM head
K = osd.kv_values(cfg.kv_dtype, tensors.kv_rows(cfg, "k", 0, 0, 0, 0, cfg.NKV),
                  tensors.kv_scales(cfg, "k", 0, 0, 0, 0, cfg.NKV) if cfg.kv_dtype == configs.I8 else None)
V = osd.kv_values(cfg.kv_dtype, tensors.kv_rows(cfg, "v", 0, 0, 0, 0, cfg.NKV),
                  tensors.kv_scales(cfg, "v", 0, 0, 0, 0, cfg.NKV) if cfg.kv_dtype == configs.I8 else None)
G = cfg.G
q = {{i: osd.bf16(tensors.q_rows(cfg, 0, 0, i, list(range(G)))) for i in range(cfg.T)}}
vr = {vocab_rows}
if cfg.w_dtype == configs.Q4:
    s_, b_ = tensors.wq_scales_biases(cfg, np.arange(vr))
    Wst = (tensors.wq_packed(cfg, np.arange(vr)), s_, b_)
else:
    Wst = tensors.w_rows(cfg, np.arange(vr))
h = osd.bf16(r["hidden"][:cfg.T])
def attn_unit():
    for i in range(cfg.T):
        vis = ot.ancestors(par, i)
        for g in range(G):
            oa.attend_row(q[i][g], K, V, cfg.S, vis)
def lm_slice():
    W = osd.q4_affine(*Wst) if cfg.w_dtype == configs.Q4 else (osd.bf16(Wst) if cfg.w_dtype == configs.BF16 else osd.f16(Wst))
    return ol.argmax_gap(ol.logits(W, h))
def timed(f, budget):
    n, t0 = 0, time.perf_counter()
    while True:
        f(); n += 1
        dt = time.perf_counter() - t0
        if dt > budget: return dt / n, n
t_mask = timed(lambda: [ot.ancestor_bits(par)], 0.5)[0]
t_attn, n_attn = timed(attn_unit, {budget})
t_lm, n_lm = timed(lm_slice, {budget})
t_walk = timed(lambda: ot.accept_walk(r["targets"][0], r["tokens"][0], par), 0.5)[0]
blk = tensors.kv_rows(cfg, "k", 0, 0, 0, cfg.S, cfg.NKV)
t_gather = timed(lambda: og.gather_within_tail(blk, 0, r["paths"][0]), 0.5)[0]
units = cfg.n_layers * cfg.B * cfg.HKV
t_round = cfg.B * t_mask + units * t_attn + (cfg.V / vr) * cfg.B * t_lm + cfg.B * t_walk + 2 * units * t_gather
print(json.dumps(dict(t_round=t_round, t_attn_unit=t_attn, t_lm_slice=t_lm, vocab_rows=vr, units=units,
                      n_attn=n_attn, n_lm=n_lm)))
"""


def run_oracle(cfg_name, round_id, budget=6.0, vocab_rows=16384):
    code = ORACLE_SAMPLE.format(root=ROOT, cfg_name=cfg_name, round_id=round_id, vocab_rows=vocab_rows, budget=budget)
    env = dict(os.environ, OMP_NUM_THREADS="1", OPENBLAS_NUM_THREADS="1", MKL_NUM_THREADS="1")
    t0 = time.perf_counter()
    r = subprocess.run([sys.executable, "-c", code], capture_output=True, text=True, env=env, timeout=900)
    wall = time.perf_counter() - t0
    if r.returncode != 0:
        raise RuntimeError(f"oracle sample failed:\n{r.stderr[-2000:]}")
    res = json.loads(r.stdout.strip().splitlines()[-1])
    from synth import configs

    cfg = configs.workload(cfg_name)
    res["nodes_per_s"] = cfg.rows / res["t_round"]
    res["wall_s"] = wall
    res["sample"] = (f"one (layer, seq, kv head) attention unit over {cfg.NKV} keys (x{res['units']} units) and "
                     f"{vocab_rows} of {cfg.V} LM-head rows for one sequence's {cfg.T} nodes (x{cfg.V / vocab_rows:.1f}"
                     f" x{cfg.B} seqs), plus mask/walk/gather, single thread, extrapolated to one round")
    return res


# ----------------------------------------------------------------------------- main
def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=1000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--config", default=DEFAULT_CONFIG, metavar="WORKLOAD",
                    help="tiny_tree7, chain3_27b_bf16 (default), specinfer16_27b_i8, eagle32x8_27b_f16, "
                         "eagle64x32_27b_i8")
    ap.add_argument("--round", type=int, default=None)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--attn-path", type=int, default=0, help="0 auto, 1 CUDA-core kernel, 2 tcgen05 kernel")
    ap.add_argument("--sliding", default=None,
                    help="W:E = a hybrid model where of every E layers the last is full attention and the others "
                         "slide over W positions")
    ap.add_argument("--append", type=int, default=0, metavar="ROT_DIM",
                    help="> 0: every round first appends its block (rotary width ROT_DIM, base 1e6; Int8 caches "
                         "quantised on append), timed as its own stage")
    ap.add_argument("--sampled", default=None, metavar="T:K:P",
                    help="sampled verification: the LM stage writes every logit and draws each node's token at "
                         "temperature T from the top-K, top-P nucleus (e.g. 1:20:0.95)")
    ap.add_argument("--build-tree", type=int, default=0, metavar="K",
                    help="> 0: time a tree-construction stage first: the drafter's top-K children of every node "
                         "(drafter logits [B*T, V]) and the best-first selection of T nodes from 1 + T*K candidates")
    ap.add_argument("--eager", dest="graph", action="store_false",
                    help="issue every call of every timed round from the host instead of replaying the round as a "
                         "captured CUDA graph (the default; per-stage times are always taken on eager rounds)")
    ap.add_argument("--layers", type=int, default=None,
                    help="attention layers (default: the workload's); fewer only for small profiler captures")
    args = ap.parse_args()
    if args.warmup < 3:
        args.warmup = 3

    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))
    from synth import configs

    cfg = configs.workload(args.config)
    if args.layers:
        cfg = configs.scaled(cfg, n_layers=args.layers)
    if args.sliding:
        w, e = (int(x) for x in args.sliding.split(":"))
        cfg = configs.with_sliding_layers(cfg, w, e)
    if args.append:
        cfg = configs.scaled(cfg, name=f"{cfg.name}+append{args.append}", rot_dim=args.append)
    if args.sampled:
        t, k, p = args.sampled.split(":")
        cfg = configs.scaled(cfg, name=f"{cfg.name}+sampled{args.sampled}", sample=(float(t), int(k), float(p)))
    config = {"workload": cfg.name, "B": cfg.B, "T": cfg.T, "layers": cfg.n_layers, "HQ": cfg.HQ, "HKV": cfg.HKV,
              "D": cfg.D, "S": cfg.S, "H": cfg.H, "V": cfg.V, "kv": configs.DTYPE_NAMES[cfg.kv_dtype],
              "lm_head": configs.DTYPE_NAMES[cfg.w_dtype], "topology": cfg.topology,
              "l2": f"inputs larger than L2 ({cfg.algorithmic_bytes() / 1e9:.2f} GB read per round), no flush",
              "parallelism": f"replicas x{args.gpus}", "launch": "cuda graph" if args.graph else "eager"}
    round_id = args.round if args.round is not None else DEFAULT_ROUND.get(args.config, 0)

    if args.impl == "reference":
        if rank != 0:
            return
        res = run_oracle(args.config, round_id)
        v = res["nodes_per_s"] * 1
        line = {"impl": "reference", "metric": METRIC, "value": v, "unit": "nodes/s", "n_gpus": args.gpus,
                "steps": args.steps, "warmup": args.warmup, "ms_per_step": res["t_round"] * 1e3,
                "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
                "data": "synthetic", "config": config,
                "cpu_baseline": {"value": v, "unit": "nodes/s", "cores": 1, "kind": "oracle", "sample": res["sample"]},
                "e2e": {"value": v, "unit": "nodes/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
        print(json.dumps(line))
        return

    import torch

    if world > 1:
        torch.distributed.init_process_group("nccl")
    r = run_ours(args, rank, world, local_rank)
    if world > 1:
        torch.distributed.destroy_process_group()
    if rank != 0:
        return
    cfg = r["cfg"]
    ms_step = r["ms"] / args.steps
    nodes_per_s = aggregate_nodes_per_s(world, cfg.rows, args.steps, r["ms"])
    peak, peak_kind = peaks()
    round_gbs = cfg.algorithmic_bytes() / (ms_step * 1e-3) / 1e9
    # dominant kernel: the LM head when its bytes dominate, else attention
    dom = "lm" if cfg.lm_bytes() >= cfg.kv_bytes() + cfg.kv_scale_bytes() else "attn"
    dom_bytes = cfg.lm_bytes() if dom == "lm" else cfg.kv_bytes() + cfg.kv_scale_bytes()
    dom_ms = r["per_kernel"][dom]
    achieved = dom_bytes / (dom_ms * 1e-3) / 1e9
    src = {"lm": ("lm_head.cu", "common.cuh"), "attn": ("attention.cu", "attention_tc.cu", "common.cuh", "tc.cuh")}[dom]
    tr = TRAFFIC.get((cfg.name, src))
    traffic = tr["bytes"] if tr and tr["hash"] == src_hash(src) else None
    line = {
        "metric": METRIC, "value": nodes_per_s, "unit": "nodes/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms_step, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16", "data": "synthetic (seeded SplitMix64 inputs, planted argmax)",
        "config": config,
        "rounds_per_s": world * args.steps / (r["ms"] * 1e-3),
        "hbm": {"algorithmic_bytes_per_round": cfg.algorithmic_bytes(), "achieved_gbs": round_gbs,
                "frac_of_peak": round_gbs / peak, "peak_gbs": peak, "peak_kind": peak_kind},
        "roofline": {"kernel": {"lm": "lm_head_argmax", "attn": "tree_verify_attention"}[dom], "bound": "hbm",
                     "achieved": achieved, "peak": peak, "unit": "GB/s", "frac": achieved / peak,
                     "traffic": traffic, "algorithmic_bytes_per_launch": dom_bytes, "avg_launch_ms": dom_ms,
                     "peak_kind": peak_kind},
        "kernels_ms": r["per_kernel"],
        "gpu_launches": r["launches"] * args.steps,
        "clocks": r["clocks"],
        "e2e": r["e2e"],
    }
    if args.sliding:
        config["sliding"] = {"window": int(args.sliding.split(":")[0]), "every": int(args.sliding.split(":")[1])}
    if not args.no_cpu_baseline and not args.sliding and not args.append and not args.sampled and not args.build_tree:
        try:
            o = run_oracle(args.config, r["round_id"])
            line["cpu_baseline"] = {"value": o["nodes_per_s"], "unit": "nodes/s", "cores": 1, "kind": "oracle",
                                    "sample": o["sample"]}
        except Exception as e:  # the baseline is reported, never required for our number
            line["cpu_baseline"] = {"value": None, "unit": "nodes/s", "cores": 1, "kind": "oracle",
                                    "sample": f"failed: {e}"[:300]}
    print(json.dumps(line))


if __name__ == "__main__":
    main()
