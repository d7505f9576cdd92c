"""Benchmark of the tree-verify step: verified nodes/s and achieved HBM bandwidth (and tensor throughput).

One step = one whole verify round on one batch of synthetic input: tree_mask -> tree_verify_attention over all
16 layers -> lm_head_argmax -> tree_accept_walk -> kv_gather_positions, plus the one-launch restore of the
tails the gather rewrote (and of kv_len).  Default workload: the long-context stress case, 32 sequences of
64-node trees over a 131,072-token Int8 prefix with fp16 per-token scales, 16 full-attention layers (24 q / 4 kv
heads, D 256), 4-bit group-64 LM head 248,320 x 5120 -- the largest workload that fits one GPU (139 GB read per
round, far larger than L2, so no flush is needed between steps).  Its attention is bound by the tensor cores
(762 flop per KV byte), so its roofline is TFLOP/s against the sustained bf16/fp16 peak; the HBM fraction is
reported beside it.  At N = 1 the same line also carries the 16-node and 32-node workloads' throughput and HBM
fraction (``configs``).

python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference] [--config WORKLOAD]
Under torchrun every rank runs its own replica on its own GPU (the path has no exchange step); rank 0 prints
one JSON line.  --impl reference times the fp64 CPU oracle on the host cores on a bounded sample of the
workload (one process per core) and extrapolates to a round.
"""
from __future__ import annotations

import argparse
import ctypes
import hashlib
import json
import multiprocessing as mp
import os
import platform
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "tree-verify nodes/s per round and achieved HBM GB/s as fraction of GB300 peak"
DEFAULT_CONFIG = "eagle64x32_27b_i8"
EXTRA_CONFIGS = ("specinfer16_27b_i8", "eagle32x8_27b_f16")  # carried on the default line at N = 1
DEFAULT_ROUND = {"chain3_27b_bf16": 2}  # the round that accepts the whole chain (3 tokens emitted)

# ncu dram bytes (read + write) per launch of a workload's dominant kernel, with the sources that kernel is built
# from and their hash when it was measured (a changed source makes the number stale and it is reported as null).
# The 64-node workload's attention was captured on 1 layer x 4 sequences (1.0867 GB read + 2.978 MB written); a
# launch over 16 layers x 32 sequences reads and writes 128 times that (every unit streams its own keys).
TRAFFIC = {
    # the chain's bf16 LM head (the CUDA-core GEMV), one launch at full size
    "chain3_27b_bf16": {"kernel": "lm", "src": ("lm_head.cu", "common.cuh"), "hash": "46f6f865d5feba27",
                        "bytes": 2543127040 + 2785024},
    # the 16-node workload's 4-bit LM head (lm_q4s_kernel, 16 rows), one launch at full size
    "specinfer16_27b_i8": {"kernel": "lm", "src": ("lm_head.cu", "lm_head_tc.cu", "common.cuh", "tc.cuh"),
                           "hash": "07d6b485b4e260fc", "bytes": 715418368 + 3241984},
    # the 32-node workload's attention (attn_tcw_kernel, 16 layers x 8 sequences), one launch at full size
    "eagle32x8_27b_f16": {"kernel": "attn", "src": ("attention.cu", "attention_tc.cu", "common.cuh", "tc.cuh"),
                          "hash": "af0faa37c76ef2ad", "bytes": 17298162176 + 49117952},
    "eagle64x32_27b_i8": {"kernel": "attn", "src": ("attention.cu", "attention_tc.cu", "common.cuh", "tc.cuh"),
                          "hash": "af0faa37c76ef2ad", "bytes": (1086705920 + 2978048) * 128},
}


def traffic_for(cfg_name, kernel):
    """The recorded traffic of this workload's dominant kernel, or None when none is recorded or it is stale."""
    tr = TRAFFIC.get(cfg_name)
    if tr is None or tr["kernel"] != kernel or tr["hash"] != src_hash(tr["src"]):
        return None
    return tr["bytes"]


def peaks():
    """(HBM GB/s, sustained bf16 TFLOP/s, burst bf16 TFLOP/s, kind)."""
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            p = json.load(f)
        return float(p["hbm_gbs"]), float(p["bf16_tflops_sustained"]), float(p["bf16_tflops"]), "measured"
    except Exception:
        return 6800.0, 1700.0, 1900.0, "fallback"


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
    """Samples the SM clock, its maximum, power and the clock-event reasons of one GPU every ``period`` seconds
    while active, through NVML (read-only queries); falls back to ``nvidia-smi`` when NVML cannot be opened."""

    def __init__(self, torch_device: int, period: float = 0.05):
        import torch

        self.period = period
        self.samples = []  # (sm_mhz, max_mhz, power_w, reason_bits)
        self.source = "none"
        props = torch.cuda.get_device_properties(torch_device)
        self.uuid = "GPU-" + str(getattr(props, "uuid", ""))
        self.bus = None
        if hasattr(props, "pci_bus_id"):
            self.bus = "%08X:%02X:%02X.0" % (getattr(props, "pci_domain_id", 0), props.pci_bus_id,
                                              getattr(props, "pci_device_id", 0))
        self._stop = threading.Event()
        self._nvml = self._handle = None
        self._proc = None

    def _open_nvml(self):
        lib = ctypes.CDLL("libnvidia-ml.so.1")
        if lib.nvmlInit_v2() != 0:
            return False
        h = ctypes.c_void_p()
        ok = lib.nvmlDeviceGetHandleByUUID(self.uuid.encode(), ctypes.byref(h)) == 0
        if not ok and self.bus:
            ok = lib.nvmlDeviceGetHandleByPciBusId_v2(self.bus.encode(), ctypes.byref(h)) == 0
        if not ok:
            return False
        self._nvml, self._handle = lib, h
        self._reasons = getattr(lib, "nvmlDeviceGetCurrentClocksEventReasons", None) or \
            lib.nvmlDeviceGetCurrentClocksThrottleReasons
        return True

    def _sample_nvml(self):
        lib, h = self._nvml, self._handle
        c, m, p, r = ctypes.c_uint(), ctypes.c_uint(), ctypes.c_uint(), ctypes.c_ulonglong()
        while not self._stop.is_set():
            if lib.nvmlDeviceGetClockInfo(h, 1, ctypes.byref(c)) == 0 and \
                    lib.nvmlDeviceGetMaxClockInfo(h, 1, ctypes.byref(m)) == 0 and \
                    self._reasons(h, ctypes.byref(r)) == 0:
                pw = p.value / 1000.0 if lib.nvmlDeviceGetPowerUsage(h, ctypes.byref(p)) == 0 else None
                self.samples.append((float(c.value), float(m.value), pw, int(r.value)))
            self._stop.wait(self.period)

    def _sample_smi(self):
        for line in self._proc.stdout:
            parts = [x.strip() for x in line.split(",")]
            try:
                bits = int(parts[3], 16) if parts[3].startswith("0x") else int(parts[3])
                self.samples.append((float(parts[0]), float(parts[1]), None, bits))
            except (ValueError, IndexError):
                continue

    def __enter__(self):
        try:
            if self._open_nvml():
                self.source = "nvml"
                self._t = threading.Thread(target=self._sample_nvml, daemon=True)
                self._t.start()
                return self
        except OSError:
            pass
        try:
            self._proc = subprocess.Popen(
                ["nvidia-smi", "--id=" + self.uuid, "--query-gpu=clocks.sm,clocks.max.sm,power.draw,"
                 "clocks_event_reasons.active", "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True, bufsize=1)
            self.source = "nvidia-smi"
            self._t = threading.Thread(target=self._sample_smi, daemon=True)
            self._t.start()
            time.sleep(0.3)  # its first line comes after start-up
        except Exception:
            self._proc = None
        return self

    def __exit__(self, *a):
        self._stop.set()
        if self._proc:
            self._proc.terminate()
            try:
                self._proc.wait(timeout=5)
            except Exception:
                self._proc.kill()
        if getattr(self, "_t", None):
            self._t.join(timeout=2)

    def summary(self):
        if not self.samples:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"], "samples": 0, "source": self.source}
        reasons = set()
        for s in self.samples:
            for b, n in REASON_BITS.items():
                if s[3] & b:
                    reasons.add(n)
        pw = [s[2] for s in self.samples if s[2] is not None]
        out = {"sm_mhz": statistics.median(s[0] for s in self.samples), "sm_max_mhz": max(s[1] for s in self.samples),
               "sm_min_mhz": min(s[0] for s in self.samples), "reasons": sorted(reasons),
               "samples": len(self.samples), "source": self.source}
        if pw:
            out["power_w_max"] = max(pw)
        return out


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


def pct(xs, q):
    """q-th percentile (0..100) by linear interpolation of the sorted sample."""
    s = sorted(xs)
    if not s:
        return None
    k = (len(s) - 1) * q / 100.0
    lo, hi = int(k), min(int(k) + 1, len(s) - 1)
    return s[lo] + (s[hi] - s[lo]) * (k - lo)


# ----------------------------------------------------------------------------- workload selection
def make_cfg(args, name=None):
    from synth import configs

    cfg = configs.workload(name or args.config)
    if args.layers:
        cfg = configs.scaled(cfg, n_layers=args.layers)
    if args.batch:
        cfg = configs.scaled(cfg, name=f"{cfg.name}+B{args.batch}", B=args.batch)
    if args.prefix:
        cfg = configs.scaled(cfg, name=f"{cfg.name}+S{args.prefix}", S=args.prefix)
    if args.sliding:
        w, e = (int(x) for x in args.sliding.split(":"))
        cfg = configs.with_sliding_layers(cfg, w, e)
    if args.append:
        cfg = configs.scaled(cfg, name=f"{cfg.name}+append{args.append}", rot_dim=args.append)
    if args.sampled:
        t, k, p = args.sampled.split(":")
        cfg = configs.scaled(cfg, name=f"{cfg.name}+sampled{args.sampled}", sample=(float(t), int(k), float(p)))
    return cfg


def config_json(cfg, args):
    from synth import configs

    return {"workload": cfg.name, "B": cfg.B, "T": cfg.T, "layers": cfg.n_layers, "HQ": cfg.HQ, "HKV": cfg.HKV,
            "D": cfg.D, "S": cfg.S, "H": cfg.H, "V": cfg.V, "kv": configs.DTYPE_NAMES[cfg.kv_dtype],
            "lm_head": configs.DTYPE_NAMES[cfg.w_dtype], "topology": cfg.topology,
            "l2": f"inputs larger than L2 ({cfg.algorithmic_bytes() / 1e9:.2f} GB read per round), no flush",
            "parallelism": f"replicas x{args.gpus}", "launch": "cuda graph" if args.graph else "eager"}


def tensor_bound(cfg) -> bool:
    """Attention is bound by the tensor cores when its flop per KV byte exceeds the machine's balance point."""
    hbm, tf_sus, _, _ = peaks()
    kvb = cfg.kv_bytes() + cfg.kv_scale_bytes()
    return kvb > 0 and cfg.attention_flops() / kvb > tf_sus * 1e12 / (hbm * 1e9)


# ----------------------------------------------------------------------------- our arm
def run_ours(args, cfg, rank, world, local_rank, steps, warmup, e2e=True):
    import torch

    import tree_speculative_decoding_array_gb300 as tsv
    from synth import configs
    from synth.workload import Workload

    tsv.load()
    dev = f"cuda:{local_rank}"
    torch.cuda.set_device(dev)
    round_id = args.round if args.round is not None else DEFAULT_ROUND.get(cfg.name, 0)
    t_setup = time.perf_counter()
    wl = Workload(cfg, device=dev, round_id=round_id, attn_path=args.attn_path)
    vr = wl.vr
    wl.save_tail()
    torch.cuda.synchronize()
    t_setup = time.perf_counter() - t_setup
    stream = torch.cuda.current_stream()
    names = (["build"] if args.build_tree else []) + ["mask"] + (["append"] if cfg.rot_dim > 0 else []) + \
        ["attn", "lm", "walk", "gather"]
    build = make_build_stage(cfg, args.build_tree, dev) if args.build_tree else None

    def step(evs=None):
        wl.restore_tail()  # one launch: pristine tails of every cache and kv_len (S + T; S when the round appends)
        for i, n in enumerate(names):
            if evs is not None:
                evs[i][0].record(stream)
            if n == "build":
                build()
            else:
                vr.run(stages=(n,))
            if evs is not None:
                evs[i][1].record(stream)

    for _ in range(warmup):
        step()
    torch.cuda.synchronize()
    if args.graph:
        # The round captured once as a CUDA graph and replayed: the same launches on the same buffers, without
        # the host issuing each one.  Per-stage times come from the eager rounds timed after it.
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph):
            step()
        for _ in range(warmup):
            graph.replay()
        torch.cuda.synchronize()
    mark = [torch.cuda.Event(enable_timing=True) for _ in range(steps + 1)]
    stage_ev = [[(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in names]
                for _ in range(steps)]
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    with ClockSampler(torch.cuda.current_device()) as clk:
        mark[0].record(stream)
        for s in range(steps):
            if args.graph:
                graph.replay()
            else:
                step(stage_ev[s])
            mark[s + 1].record(stream)
        torch.cuda.synchronize()
    if world > 1:
        torch.distributed.barrier()
    ms = mark[0].elapsed_time(mark[steps])
    per_round = [mark[s].elapsed_time(mark[s + 1]) for s in range(steps)]
    n_stage = min(steps, max(3, args.stage_rounds))
    if args.graph:  # per-stage times: eager rounds with events around every call
        for s in range(n_stage):
            step(stage_ev[s])
        torch.cuda.synchronize()
    per_kernel = {n: statistics.mean(stage_ev[s][i][0].elapsed_time(stage_ev[s][i][1]) for s in range(n_stage))
                  for i, n in enumerate(names)}
    if world > 1:
        ms = max_over_ranks(ms, dev)

    # correctness of the timed state: one more round, checked against the planted walk
    step()
    torch.cuda.synchronize()
    got_len = vr.outs["path_len"].cpu().tolist()
    want_len = [len(p) for p in wl.round["paths"]]
    if cfg.sample:  # the walk follows each node's draw, not the planted argmax path
        assert all(1 <= n <= cfg.T for n in got_len), got_len
    else:
        assert got_len == want_len, (got_len, want_len)
    assert vr.outs["status"].cpu().tolist()[0] == 0, vr.outs["status"].cpu().tolist()

    e2e_res = run_e2e(args, wl, stream, steps, pre=build) if (rank == 0 and e2e) else None
    launches = count_launches(cfg, tsv, vr, args)
    return dict(cfg=cfg, ms=ms, per_round=per_round, per_kernel=per_kernel, clocks=clk.summary(), e2e=e2e_res,
                launches=launches, round_id=round_id, setup_s=t_setup, stage_rounds=n_stage)


def free_device():
    """Return a finished workload's device memory before the next one is built."""
    import gc

    import torch

    gc.collect()
    torch.cuda.synchronize()
    torch.cuda.empty_cache()


def count_launches(cfg, tsv, vr, args):
    """Kernels of this library (and the tail restore of the synthetic workload) launched per round."""
    from synth import configs

    if cfg.rows > 8:  # tensor-core LM head: key reset + (fp16 copy of hidden) + kernel + unpack
        lm = 1 + 1 + (cfg.w_dtype != configs.BF16) + 1
    else:  # CUDA-core GEMV: key reset + one launch per group of up to 8 rows + unpack
        groups, left = 0, cfg.rows
        while left > 0:
            left -= 8 if left >= 8 else (4 if left >= 4 else left)
            groups += 1
        lm = 1 + groups + 1
    if cfg.sample:  # no unpack; top-k passes (one per 4096-entry chunk level) and the draw
        n, passes = cfg.V, 0
        while True:
            passes += 1
            ch = (n + 4095) // 4096
            if ch == 1:
                break
            n = ch * min(int(cfg.sample[1]), cfg.V)
        lm += passes
    attn = 1 + (tsv.attention_workspace_size(vr.adesc) > 0)
    n = 1 + 1 + attn + lm + 1 + 2 + (2 if cfg.rot_dim > 0 else 0)  # restore, mask, attention, LM, walk, gather
    if args.build_tree:  # draft children: top-k passes + output; selection: one
        m, passes = cfg.V, 0
        while True:
            passes += 1
            ch = (m + 4095) // 4096
            if ch == 1:
                break
            m = ch * args.build_tree
        n += passes + 1 + 1
    return n


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


def run_e2e(args, wl, stream, steps, pre=None):
    """Rounds through the public API with host buffers: every round copies its inputs from pinned host memory into
    device memory (one H2D copy) and reads its int32 results back (one D2H copy).  With graphs, two VerifyRounds
    over two input buffers alternate, and round k + 1's inputs are copied on a second stream while round k runs
    (the copy into a buffer waits for the round that last read it).  ``pre`` (the tree-construction stage, when the
    timed round has one) runs at the start of every round, as in the device-timed round."""
    import torch

    vr, cfg = wl.vr, wl.cfg
    # the round's inputs (parents, tokens, hidden, Q per layer, ...) are one device buffer: one pinned H2D copy;
    # its int32 results (path, path_len, emitted, argmax) one block: one D2H copy
    h_in = wl.inputs.detach().cpu().pin_memory()
    res = vr.outs["result"]
    h2d = h_in.numel() * h_in.element_size()
    d2h = res.numel() * res.element_size()
    n = max(3, min(steps, max(3, steps // 4)))
    t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)

    if args.graph:  # the public capture / replay pair, one graph per input buffer
        buf2, vr2 = wl.twin()
        bufs, vrs = [wl.inputs, buf2], [vr, vr2]
        h_res = [torch.empty(res.shape, dtype=res.dtype).pin_memory() for _ in range(2)]
        for r in vrs:
            r.capture()
        torch.cuda.synchronize()
        copy_stream = torch.cuda.Stream()
        ev_in = [torch.cuda.Event(), torch.cuda.Event()]
        ev_done = [torch.cuda.Event(), torch.cuda.Event()]
        start = torch.cuda.Event()

        def rounds(count, timed):
            start.record(stream)
            copy_stream.wait_event(start)
            with torch.cuda.stream(copy_stream):
                bufs[0].copy_(h_in, non_blocking=True)
                ev_in[0].record(copy_stream)
            if timed:
                t0.record(stream)
            for k in range(count):
                a, b = k & 1, (k & 1) ^ 1
                if k + 1 < count:  # the next round's inputs, once the round that last read buffer b is done
                    with torch.cuda.stream(copy_stream):
                        if k >= 1:
                            copy_stream.wait_event(ev_done[b])
                        bufs[b].copy_(h_in, non_blocking=True)
                        ev_in[b].record(copy_stream)
                stream.wait_event(ev_in[a])
                wl.restore_tail()
                if pre is not None:
                    pre()
                vrs[a].replay()
                ev_done[a].record(stream)
                h_res[a].copy_(vrs[a].outs["result"], non_blocking=True)
            if timed:
                t1.record(stream)

        rounds(3, False)
        torch.cuda.synchronize()
        rounds(n, True)
        torch.cuda.synchronize()
        # [t0, t1] holds the first round's copy (round 0 waits for it) and every round; the later copies overlap
        ms = t0.elapsed_time(t1) / n
        for r in vrs:
            r._graph = None
        launch = "VerifyRound.replay (cuda graph), two input buffers, inputs of round k + 1 copied while round k runs"
    else:
        h_res = torch.empty(res.shape, dtype=res.dtype).pin_memory()

        def e2e_step():
            wl.restore_tail()
            wl.inputs.copy_(h_in, non_blocking=True)
            if pre is not None:
                pre()
            vr.run()
            h_res.copy_(res, non_blocking=True)

        for _ in range(3):
            e2e_step()
        torch.cuda.synchronize()
        t0.record(stream)
        for _ in range(n):
            e2e_step()
        t1.record(stream)
        torch.cuda.synchronize()
        ms = t0.elapsed_time(t1) / n
        launch = "VerifyRound.run (eager)"
    return {"value": cfg.rows / (ms * 1e-3), "unit": "nodes/s", "ms_per_step": ms, "steps": n,
            "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "launch": launch}


def gpu_line_parts(cfg, r, world, steps):
    """Throughput, HBM and roofline figures of one measured workload."""
    hbm_peak, tf_sus, _, kind = peaks()
    ms_step = r["ms"] / steps
    out = {"value": aggregate_nodes_per_s(world, cfg.rows, steps, r["ms"]), "ms_per_step": ms_step,
           "rounds_per_s": world * steps / (r["ms"] * 1e-3)}
    pr = r["per_round"]
    out["round_ms"] = {"median": statistics.median(pr), "p10": pct(pr, 10), "p90": pct(pr, 90),
                       "min": min(pr), "max": max(pr), "rounds": len(pr)}
    round_gbs = cfg.algorithmic_bytes() / (ms_step * 1e-3) / 1e9
    out["hbm"] = {"algorithmic_bytes_per_round": cfg.algorithmic_bytes(), "achieved_gbs": round_gbs,
                  "frac_of_peak": round_gbs / hbm_peak, "peak_gbs": hbm_peak, "peak_kind": kind}
    kvb = cfg.kv_bytes() + cfg.kv_scale_bytes()
    attn_ms, lm_ms = r["per_kernel"]["attn"], r["per_kernel"]["lm"]
    if tensor_bound(cfg):
        fl = cfg.attention_flops()
        ach = fl / (attn_ms * 1e-3) / 1e12
        out["roofline"] = {"kernel": "tree_verify_attention", "bound": "tensor", "achieved": ach, "peak": tf_sus,
                           "unit": "TFLOP/s", "frac": ach / tf_sus, "traffic": traffic_for(cfg.name, "attn"),
                           "algorithmic_flops_per_launch": fl, "algorithmic_bytes_per_launch": kvb,
                           "avg_launch_ms": attn_ms, "peak_kind": f"{kind} bf16 sustained",
                           "hbm_gbs": kvb / (attn_ms * 1e-3) / 1e9,
                           "hbm_frac": kvb / (attn_ms * 1e-3) / 1e9 / hbm_peak}
    else:
        dom = "lm" if cfg.lm_bytes() >= kvb else "attn"
        dom_bytes = cfg.lm_bytes() if dom == "lm" else kvb
        dom_ms = lm_ms if dom == "lm" else attn_ms
        ach = dom_bytes / (dom_ms * 1e-3) / 1e9
        out["roofline"] = {"kernel": {"lm": "lm_head_argmax", "attn": "tree_verify_attention"}[dom], "bound": "hbm",
                           "achieved": ach, "peak": hbm_peak, "unit": "GB/s", "frac": ach / hbm_peak,
                           "traffic": traffic_for(cfg.name, dom),
                           "algorithmic_bytes_per_launch": dom_bytes, "avg_launch_ms": dom_ms,
                           "peak_kind": kind}
    return out


# ----------------------------------------------------------------------------- oracle on the host cores
def _oracle_worker(conn, root, cfg_name, round_id, unit, nodes, v0, v1):
    """One host core's share of the oracle sample: one (layer, sequence, kv head) attention unit over its
    ``nodes`` and the LM head's vocabulary rows [v0, v1) for every hidden row of the round.  Inputs are generated
    once (untimed, like weights resident in memory); each command runs the oracle's own functions."""
    sys.path.insert(0, root)
    import numpy as np

    from oracle import attention as oa
    from oracle import lm_head as ol
    from oracle import storage as osd
    from oracle import tree as ot
    from synth import configs, tensors, trees

    cfg = configs.workload(cfg_name)
    layer, b, kvh = unit
    r = trees.make_round(cfg, round_id)
    par = r["parents"][b].tolist()
    i8 = cfg.kv_dtype == configs.I8
    K = osd.kv_values(cfg.kv_dtype, tensors.kv_rows(cfg, "k", layer, b, kvh, 0, cfg.NKV),
                      tensors.kv_scales(cfg, "k", layer, b, kvh, 0, cfg.NKV) if i8 else None)
    V = osd.kv_values(cfg.kv_dtype, tensors.kv_rows(cfg, "v", layer, b, kvh, 0, cfg.NKV),
                      tensors.kv_scales(cfg, "v", layer, b, kvh, 0, cfg.NKV) if i8 else None)
    heads = [kvh * cfg.G + g for g in range(cfg.G)]
    q = {i: osd.bf16(tensors.q_rows(cfg, layer, b, i, heads)) for i in nodes}
    rows = np.arange(v0, v1)
    if cfg.w_dtype == configs.Q4:
        s_, b_ = tensors.wq_scales_biases(cfg, rows)
        W = osd.q4_affine(tensors.wq_packed(cfg, rows), s_, b_)
    else:
        W = (osd.bf16 if cfg.w_dtype == configs.BF16 else osd.f16)(tensors.w_rows(cfg, rows))
    h = osd.bf16(r["hidden"])
    conn.send("ready")
    while True:
        cmd = conn.recv()
        t0 = time.perf_counter()
        if cmd == "attn":
            for i in nodes:
                vis = ot.ancestors(par, i)
                for g in range(cfg.G):
                    oa.attend_row(q[i][g], K, V, cfg.S, vis)
        elif cmd == "lm":
            ol.argmax_gap(ol.logits(W, h))
        else:
            break
        conn.send(time.perf_counter() - t0)
    conn.close()


def cpu_model() -> str:
    try:
        with open("/proc/cpuinfo") as f:
            for line in f:
                k = line.split(":")[0].strip().lower()
                if k in ("model name", "cpu model"):
                    return line.split(":", 1)[1].strip()
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        for line in out.splitlines():
            if line.lower().startswith("model name"):
                return line.split(":", 1)[1].strip()
    except Exception:
        pass
    return platform.processor() or platform.machine()


def host_workers(cfg, want: int) -> int:
    """Worker processes for the oracle sample: one per core, at most ``want``, within half the free memory."""
    n = max(1, min(want, os.cpu_count() or 1))
    per = 2 * cfg.NKV * cfg.D * 8 + 1024 * cfg.H * 8 + cfg.rows * cfg.H * 8 * 2 + (300 << 20)
    try:
        with open("/proc/meminfo") as f:
            avail = next(int(l.split()[1]) * 1024 for l in f if l.startswith("MemAvailable"))
        n = max(1, min(n, int(0.5 * avail // per)))
    except Exception:
        pass
    return n


def run_oracle_sample(cfg_name, round_id, steps, warmup, workers, vocab_per_worker=1024):
    """Times the fp64 oracle on the host cores: ``workers`` processes (spawned), each holding one attention unit
    and one vocabulary slice.  A step is one attention pass (every worker: its nodes x the G heads of its unit,
    over all S keys plus its ancestors) followed by one LM pass (every worker: every hidden row of the round
    against its vocabulary slice, then the argmax).  The round time is extrapolated from the two passes' wall
    times by the round's attention rows and LM products; mask, walk and gather are timed in this process."""
    import numpy as np

    from oracle import gather as og
    from oracle import tree as ot
    from synth import configs, tensors, trees

    cfg = configs.workload(cfg_name)
    r = trees.make_round(cfg, round_id, plant=False)
    rng = np.random.default_rng(12345)
    nodes_per = 1 if cfg.S >= 32768 else (2 if cfg.S >= 4096 else cfg.T)
    ctx = mp.get_context("spawn")
    env0 = {k: os.environ.get(k) for k in ("OMP_NUM_THREADS", "OPENBLAS_NUM_THREADS", "MKL_NUM_THREADS")}
    os.environ.update(OMP_NUM_THREADS="1", OPENBLAS_NUM_THREADS="1", MKL_NUM_THREADS="1")
    procs, conns = [], []
    try:
        for w in range(workers):
            unit = (int(rng.integers(cfg.n_layers)), int(rng.integers(cfg.B)), int(rng.integers(cfg.HKV)))
            nodes = sorted(rng.choice(cfg.T, size=min(cfg.T, nodes_per), replace=False).tolist())
            v0 = (w * vocab_per_worker) % cfg.V
            v1 = min(cfg.V, v0 + vocab_per_worker)
            a, bconn = ctx.Pipe()
            p = ctx.Process(target=_oracle_worker, args=(bconn, ROOT, cfg_name, round_id, unit, nodes, v0, v1),
                            daemon=True)
            p.start()
            procs.append((p, nodes_per, v1 - v0))
            conns.append(a)
        t0 = time.perf_counter()
        for c in conns:
            assert c.recv() == "ready"
        t_setup = time.perf_counter() - t0

        def phase(cmd):
            t = time.perf_counter()
            for c in conns:
                c.send(cmd)
            for c in conns:
                c.recv()
            return time.perf_counter() - t

        walls = []
        for s in range(warmup + steps):
            ta, tl = phase("attn"), phase("lm")
            if s >= warmup:
                walls.append((ta, tl))
        for c in conns:
            c.send("quit")
    finally:
        for (p, _, _) in procs:
            p.join(timeout=30)
            if p.is_alive():
                p.terminate()
        for k, v in env0.items():
            if v is None:
                os.environ.pop(k, None)
            else:
                os.environ[k] = v
    t_attn = statistics.median(w[0] for w in walls)
    t_lm = statistics.median(w[1] for w in walls)
    attn_rows_step = sum(n for (_, n, _) in procs) * cfg.G
    lm_products_step = sum(v for (_, _, v) in procs) * cfg.rows
    attn_rows_round = cfg.n_layers * cfg.B * cfg.T * cfg.HQ
    lm_products_round = cfg.rows * cfg.V
    f_attn, f_lm = attn_rows_round / attn_rows_step, lm_products_round / lm_products_step

    def timed(f, budget=0.3):
        n, t0 = 0, time.perf_counter()
        while True:
            f()
            n += 1
            if time.perf_counter() - t0 > budget:
                return (time.perf_counter() - t0) / n
    par = r["parents"][0].tolist()
    blk = tensors.kv_rows(cfg, "k", 0, 0, 0, cfg.S, cfg.NKV)
    t_small = cfg.B * (timed(lambda: ot.ancestor_bits(par)) + timed(lambda: ot.accept_walk(r["targets"][0],
                                                                                           r["tokens"][0], par)))
    t_small += 2 * cfg.n_layers * cfg.B * cfg.HKV * timed(lambda: og.gather_within_tail(blk, 0, r["paths"][0]))
    t_round = t_attn * f_attn + t_lm * f_lm + t_small
    step_s = [a + l for a, l in walls]
    return {"nodes_per_s": cfg.rows / t_round, "t_round_s": t_round, "workers": workers, "setup_s": t_setup,
            "step_s": statistics.mean(step_s), "steps": len(walls), "attn_pass_s": t_attn, "lm_pass_s": t_lm,
            "factor_attn": f_attn, "factor_lm": f_lm, "small_s": t_small,
            "sample": (f"{workers} processes (one per core) each holding one (layer, sequence, kv head) attention "
                       f"unit over {cfg.NKV} keys ({nodes_per} node(s) x {cfg.G} heads per pass) and a "
                       f"{vocab_per_worker}-row slice of the {cfg.V}-row LM head (every one of the round's "
                       f"{cfg.rows} hidden rows per pass); round time = attention pass x {f_attn:.0f} + LM pass x "
                       f"{f_lm:.1f} + mask/walk/gather ({t_small * 1e3:.1f} ms, one core): extrapolated")}


def cpu_baseline_json(o):
    return {"value": o["nodes_per_s"], "unit": "nodes/s", "cores": o["workers"], "kind": "oracle",
            "sample": o["sample"], "extrapolated": True, "round_s": o["t_round_s"], "nproc": os.cpu_count(),
            "cpu_model": cpu_model(), "machine": platform.machine()}


# ----------------------------------------------------------------------------- main
def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--config", default=DEFAULT_CONFIG, metavar="WORKLOAD",
                    help="tiny_tree7, chain3_27b_bf16, specinfer16_27b_i8, eagle32x8_27b_f16, "
                         "eagle64x32_27b_i8 (default)")
    ap.add_argument("--round", type=int, default=None)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-extra", action="store_true",
                    help="skip the 16-node and 32-node workloads carried on the default line")
    ap.add_argument("--extra-steps", type=int, default=100, help="timed rounds of each extra workload")
    ap.add_argument("--cpu-workers", type=int, default=16, help="host processes of the oracle sample")
    ap.add_argument("--stage-rounds", type=int, default=5, help="eager rounds timed per stage")
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
    ap.add_argument("--batch", type=int, default=None,
                    help="sequences (default: the workload's); fewer only for small profiler captures")
    ap.add_argument("--prefix", type=int, default=None,
                    help="cached prefix length S (default: the workload's); shorter only for small profiler captures")
    args = ap.parse_args()
    if args.warmup < 3:
        args.warmup = 3

    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))
    cfg = make_cfg(args)
    config = config_json(cfg, args)
    if args.sliding:
        config["sliding"] = {"window": int(args.sliding.split(":")[0]), "every": int(args.sliding.split(":")[1])}
    round_id = args.round if args.round is not None else DEFAULT_ROUND.get(args.config, 0)

    if args.impl == "reference":
        if rank != 0:
            return
        o = run_oracle_sample(args.config, round_id, args.steps, args.warmup, host_workers(cfg, args.cpu_workers))
        v = o["nodes_per_s"]
        line = {"impl": "reference", "metric": METRIC, "value": v, "unit": "nodes/s", "n_gpus": args.gpus,
                "steps": o["steps"], "warmup": args.warmup, "ms_per_step": o["step_s"] * 1e3,
                "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
                "data": "synthetic (seeded SplitMix64 inputs)", "config": config,
                "step": "one bounded sample of the round on the host cores (an attention pass and an LM pass); "
                        "value is the round extrapolated from it",
                "extrapolation": {"round_s": o["t_round_s"], "attn_factor": o["factor_attn"],
                                  "lm_factor": o["factor_lm"], "attn_pass_s": o["attn_pass_s"],
                                  "lm_pass_s": o["lm_pass_s"], "mask_walk_gather_s": o["small_s"],
                                  "setup_s": o["setup_s"]},
                "cpu_baseline": cpu_baseline_json(o),
                "e2e": {"value": v, "unit": "nodes/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
        print(json.dumps(line))
        return

    import torch

    if world > 1:
        torch.distributed.init_process_group("nccl")
    r = run_ours(args, cfg, rank, world, local_rank, args.steps, args.warmup)
    free_device()
    extra = {}
    default_line = args.config == DEFAULT_CONFIG and not (args.layers or args.batch or args.prefix or args.sliding
                                                          or args.append or args.sampled or args.build_tree)
    if world == 1 and default_line and not args.no_extra:
        for name in EXTRA_CONFIGS:
            ecfg = make_cfg(args, name)
            er = run_ours(args, ecfg, rank, world, local_rank, args.extra_steps, max(args.warmup, 10), e2e=True)
            free_device()
            p = gpu_line_parts(ecfg, er, world, args.extra_steps)
            extra[name] = {"nodes_per_s": p["value"], "ms_per_round": p["ms_per_step"],
                           "rounds_per_s": p["rounds_per_s"], "round_ms": p["round_ms"],
                           "hbm_frac_of_peak": p["hbm"]["frac_of_peak"], "hbm_gbs": p["hbm"]["achieved_gbs"],
                           "roofline": p["roofline"], "kernels_ms": er["per_kernel"], "clocks": er["clocks"],
                           "e2e_nodes_per_s": er["e2e"]["value"] if er["e2e"] else None, "steps": args.extra_steps}
    if world > 1:
        torch.distributed.destroy_process_group()
    if rank != 0:
        return
    parts = gpu_line_parts(cfg, r, world, args.steps)
    line = {
        "metric": METRIC, "value": parts["value"], "unit": "nodes/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": parts["ms_per_step"], "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16", "data": "synthetic (seeded SplitMix64 inputs, planted argmax)",
        "config": config, "rounds_per_s": parts["rounds_per_s"], "round_ms": parts["round_ms"], "hbm": parts["hbm"],
        "roofline": parts["roofline"], "kernels_ms": r["per_kernel"], "stage_rounds": r["stage_rounds"],
        "gpu_launches": r["launches"] * args.steps, "launches_per_round": r["launches"], "clocks": r["clocks"],
        "e2e": r["e2e"], "setup_s": r["setup_s"],
    }
    if extra:
        line["configs"] = extra
    if not args.no_cpu_baseline and world == 1 and not (args.sliding or args.append or args.sampled or
                                                          args.build_tree or args.layers or args.batch or args.prefix):
        try:
            o = run_oracle_sample(args.config, r["round_id"], 2, 1, host_workers(cfg, args.cpu_workers))
            line["cpu_baseline"] = cpu_baseline_json(o)
        except Exception as e:  # the baseline is reported, never required for our number
            line["cpu_baseline"] = {"value": None, "unit": "nodes/s", "cores": 0, "kind": "oracle",
                                    "sample": f"failed: {e}"[:300]}
    print(json.dumps(line))


if __name__ == "__main__":
    main()
