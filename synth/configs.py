"""The five synthetic workloads of the tree-verify step.

Each workload stands in for the pages' Qwen3.8-27B hybrid target (hidden 5120,
vocabulary 248,320, 16 full-attention layers with 24 query and 4 KV heads of
dimension 256) and their draft trees; the model checkpoints and prompt cohorts
are not available, so every tensor is seeded synthetic data with the stated
shape and distribution.
"""
from __future__ import annotations

from dataclasses import dataclass, field

# KV / weight storage formats (the same numbering as the C-ABI's tsv_dtype).
F16, BF16, I8, Q4 = 0, 1, 2, 3
DTYPE_NAMES = {F16: "f16", BF16: "bf16", I8: "i8_scaled", Q4: "q4_g64"}


@dataclass(frozen=True)
class Config:
    name: str
    seed: int
    n_layers: int
    B: int
    T: int
    HQ: int
    HKV: int
    D: int
    S: int                 # prefix length (offset) before the tree block
    H: int                 # hidden size (LM-head input)
    V: int                 # vocabulary
    kv_dtype: int
    w_dtype: int
    topology: str          # "fixed", "chain", "specinfer", "best_first"
    parents0: tuple = ()   # explicit topology for "fixed"
    branching: tuple = ()  # SpecInfer branching factors
    k_max: int = 4         # best-first: candidates per node
    depth_max: int = 0     # best-first: maximum depth
    accept: str = ""       # accept-length rule
    plant_c: float = 0.25  # planting strength of the target direction in hidden
    min_gap: float = 1e-2  # required top-1/top-2 logit gap (fp64)
    window: tuple = ()     # per-layer sliding windows (0 = full attention); empty = every layer full
    rot_dim: int = 0       # > 0: the round appends its block (rotary width rot_dim, base rope_base) before attention
    rope_base: float = 1e6
    sample: tuple = ()     # (temperature, top_k, top_p): sampled verification; empty = greedy
    notes: str = ""

    @property
    def G(self) -> int:
        return self.HQ // self.HKV

    @property
    def NKV(self) -> int:
        """Logical KV length after the tree block was appended: S + T."""
        return self.S + self.T

    @property
    def rows(self) -> int:
        """LM-head rows per round: one per tree node of every sequence."""
        return self.B * self.T

    # ---- algorithmic bytes per round (HBM reads the method cannot avoid) ----
    def kv_elem_bytes(self) -> int:
        return 1 if self.kv_dtype == I8 else 2

    def layer_window(self, layer: int) -> int:
        return int(self.window[layer]) if self.window else 0

    def kv_positions(self) -> int:
        """Cache positions read per (sequence, KV head), summed over layers: all S+T for a full layer; for a
        sliding-window layer only those inside some node's band, the last window + T - 1."""
        tot = 0
        for l in range(self.n_layers):
            w = self.layer_window(l)
            tot += self.NKV if w == 0 else min(self.NKV, w + self.T - 1)
        return tot

    def kv_bytes(self) -> int:
        """K and V of every layer, sequence and KV head over the positions the layer attends."""
        return 2 * self.B * self.HKV * self.kv_positions() * self.D * self.kv_elem_bytes()

    def kv_scale_bytes(self) -> int:
        if self.kv_dtype != I8:
            return 0
        return 2 * self.B * self.HKV * self.kv_positions() * 2

    def lm_bytes(self) -> int:
        if self.w_dtype == Q4:
            return self.V * self.H // 2 + 2 * (self.V * (self.H // 64) * 2)
        return self.V * self.H * 2

    def algorithmic_bytes(self) -> int:
        return self.kv_bytes() + self.kv_scale_bytes() + self.lm_bytes()

    def attention_flops(self) -> float:
        """2 contractions (QK^T and PV) per query row over its visible keys: on a full layer the S history keys and
        on average (T + 1) / 2 block keys (a chain's mean; a branching tree's nodes see fewer), on a sliding-window
        layer no more than its window."""
        keys = 0.0
        for l in range(self.n_layers):
            w = self.layer_window(l)
            full = self.S + (self.T + 1) / 2
            keys += full if w == 0 else min(full, w)
        return 2 * 2 * self.B * self.HQ * self.T * self.D * keys

    def lm_flops(self) -> int:
        return 2 * self.rows * self.V * self.H


CONFIGS = [
    Config(
        name="tiny_tree7", seed=0, n_layers=1, B=1, T=7, HQ=4, HKV=2, D=64, S=128,
        H=256, V=1024, kv_dtype=F16, w_dtype=F16, topology="fixed",
        parents0=(-1, 0, 0, 1, 1, 2, 2), accept="uniform_node", plant_c=1.0, min_gap=0.05,
        notes="1 layer, 4q/2kv heads, D=64, 128-token fp16 prefix, 7-node tree, fp16 LM head 1024x256",
    ),
    Config(
        name="chain3_27b_bf16", seed=1, n_layers=16, B=1, T=3, HQ=24, HKV=4, D=256, S=4096,
        H=5120, V=248320, kv_dtype=BF16, w_dtype=BF16, topology="chain",
        accept="cycle", notes="linear chain T=3 over a 4096-token bf16 prefix, bf16 LM head",
    ),
    Config(
        name="specinfer16_27b_i8", seed=2, n_layers=16, B=1, T=16, HQ=24, HKV=4, D=256, S=8192,
        H=5120, V=248320, kv_dtype=I8, w_dtype=Q4, topology="specinfer",
        branching=(4, 2, 2, 1, 1), accept="uniform_1_5",
        notes="16-node shared-prefix tree, 8192-token Int8 prefix, 4-bit group-64 LM head",
    ),
    Config(
        name="eagle32x8_27b_f16", seed=3, n_layers=16, B=8, T=32, HQ=24, HKV=4, D=256, S=32768,
        H=5120, V=248320, kv_dtype=F16, w_dtype=BF16, topology="best_first", depth_max=6,
        accept="leaf_uniform", notes="8 sequences of 32-node best-first trees, 32768-token fp16 prefix",
    ),
    Config(
        name="eagle64x32_27b_i8", seed=4, n_layers=16, B=32, T=64, HQ=24, HKV=4, D=256, S=131072,
        H=5120, V=248320, kv_dtype=I8, w_dtype=Q4, topology="best_first", depth_max=8,
        accept="geometric", notes="32 sequences of 64-node trees, 131072-token Int8 prefix, 4-bit LM head",
    ),
]


WORKLOADS = {c.name: c for c in CONFIGS}


def workload(name: str) -> Config:
    """The workload of that name (tiny_tree7, chain3_27b_bf16, specinfer16_27b_i8, eagle32x8_27b_f16,
    eagle64x32_27b_i8)."""
    try:
        return WORKLOADS[name]
    except KeyError:
        raise KeyError(f"unknown workload {name!r}; known: {', '.join(WORKLOADS)}") from None


def scaled(cfg: Config, **kw) -> Config:
    """A copy of ``cfg`` with some fields replaced (reduced-size parity cases)."""
    d = dict(cfg.__dict__)
    d.update(kw)
    if d.get("window") and len(d["window"]) != d["n_layers"]:
        d["window"] = tuple(d["window"][l % len(d["window"])] for l in range(d["n_layers"]))
    return Config(**d)


def with_sliding_layers(cfg: Config, window: int, every: int) -> Config:
    """A hybrid model: of every ``every`` layers the last is full attention and the others slide over
    ``window`` positions (the sliding/full interleave of the hybrid targets the pages verify against)."""
    pattern = tuple(0 if (l % every) == every - 1 else window for l in range(cfg.n_layers))
    return scaled(cfg, name=f"{cfg.name}+sliding{window}x{every - 1}", window=pattern)
