"""The seeded input generator: known-answer, determinism, workload structure, planting.

The planting checks call the oracle (the generator itself computes no logits):
every node's planted target must be the fp64 argmax with at least the
required gap, and the oracle's walk must find the planned path.
"""
import os

import numpy as np
import pytest

from oracle import lm_head as ol
from oracle import storage as osd
from oracle import tree as ot
from synth import configs, rng, tensors, trees

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def test_splitmix64_published_vector():
    with open(os.path.join(GOLDEN, "splitmix64_seed0.txt")) as f:
        want = [int(x, 16) for x in f.read().split() if not x.startswith("#") and len(x) == 16]
    got = rng.draw(0, np.arange(3))
    assert [int(x) for x in got] == want
    assert [rng.draw_int(0, i) for i in range(3)] == want


def test_distributions():
    h = rng.draw(rng.stream_key(5, 1), np.arange(1 << 20))
    x = rng.normal_f32(h).astype(np.float64)
    assert abs(x.mean()) < 0.01 and abs(x.std() - 1.0) < 0.01
    c = rng.int_below(h, 255) - 127
    assert c.min() == -127 and c.max() == 127
    u = rng.uniform_f32(h, np.float32(0.005), np.float32(0.045))
    assert u.min() >= 0.005 and u.max() < 0.05
    b = rng.f32_to_bf16_bits(np.array([1.0, 1.00390625, 1.01171875, -3.0], dtype=np.float32))
    assert b.tolist() == [0x3F80, 0x3F80, 0x3F82, 0xC040]  # ties to even


def test_slices_match_full_tensors():
    cfg = configs.workload("tiny_tree7")
    K = tensors.kv_full(cfg, "k", 0)
    assert np.array_equal(tensors.kv_rows(cfg, "k", 0, 0, 1, 3, 9), K[0, 1, 3:9])
    Q = tensors.q_full(cfg, 0)
    assert np.array_equal(tensors.q_rows(cfg, 0, 0, 4, [1, 3]), Q[0, 4, [1, 3]])
    W = tensors.w_full(cfg)
    assert np.array_equal(tensors.w_rows(cfg, [5, 700]), W[[5, 700]])


def test_specinfer_topology():
    par = trees.specinfer((4, 2, 2, 1, 1), 16)
    assert ot.validate(par) == ot.OK and len(par) == 16
    d = trees.depths(par)
    assert max(d) == 5
    assert sum(1 for x in d if x == 1) == 2  # rank-0 and rank-1 children of the root


@pytest.mark.parametrize("name", ["specinfer16_27b_i8", "eagle32x8_27b_f16", "eagle64x32_27b_i8"])
def test_best_first_topologies(name):
    cfg = configs.workload(name)
    r = trees.make_round(cfg, 0, plant=False)
    for b in range(cfg.B):
        par = r["parents"][b].tolist()
        assert ot.validate(par) == ot.OK
        assert max(trees.depths(par)) <= max(cfg.depth_max, 5)
        ch = trees.children(par)
        for u in range(cfg.T):
            toks = [int(r["tokens"][b, c]) for c in ch[u]]
            assert len(toks) == len(set(toks))  # distinct sibling tokens
    if cfg.accept == "leaf_uniform":
        assert sum(not trees.is_identity(p) for p in r["paths"]) >= 4
    if cfg.accept == "geometric":
        assert r["paths"][0] == [0] and trees.is_identity(r["paths"][1]) and len(r["paths"][1]) >= 2


def test_walk_finds_planned_path_from_targets():
    for cfg in configs.CONFIGS:
        r = trees.make_round(cfg, 1, plant=False)
        for b in range(cfg.B):
            path, _ = ot.accept_walk(r["targets"][b], r["tokens"][b], r["parents"][b])
            assert path == r["paths"][b]


def _check_planting(cfg, round_id):
    r = trees.make_round(cfg, round_id)
    h = osd.bf16(r["hidden"])
    if cfg.w_dtype == configs.Q4:
        def wr(r0, r1):
            p = tensors.wq_packed(cfg, np.arange(r0, r1))
            s, b = tensors.wq_scales_biases(cfg, np.arange(r0, r1))
            return osd.q4_affine(p, s, b)
    else:
        dec = osd.bf16 if cfg.w_dtype == configs.BF16 else osd.f16
        wr = lambda r0, r1: dec(tensors.w_rows(cfg, np.arange(r0, r1)))
    arg, top, gap = ol.argmax_streamed(wr, h, cfg.V)
    assert np.array_equal(arg, r["targets"].reshape(-1))
    assert gap.min() >= cfg.min_gap
    for b in range(cfg.B):
        path, _ = ot.accept_walk(arg.reshape(cfg.B, cfg.T)[b], r["tokens"][b], r["parents"][b])
        assert path == r["paths"][b]
    return gap.min()


def test_planting_tiny():
    for rid in range(4):
        _check_planting(configs.workload("tiny_tree7"), rid)


@pytest.mark.parametrize("name", ["chain3_27b_bf16", "specinfer16_27b_i8", "eagle32x8_27b_f16"])
def test_planting_reduced_vocab(name):
    """The 27B-shaped workloads at hidden 5120 with a 6144-row vocabulary (full vocab: GPU tests)."""
    cfg = configs.scaled(configs.workload(name), V=6144, B=min(configs.workload(name).B, 2))
    g = _check_planting(cfg, 0)
    assert g > 1.0


def test_input_arena_layout():
    """Per-round inputs share one buffer: 256-byte aligned, disjoint, typed views that write through."""
    import torch
    from synth.workload import _arena

    specs = [("parents", (2, 3), torch.int32), ("hidden", (6, 40), torch.bfloat16), ("q0", (2, 3, 4, 8), torch.bfloat16),
             ("u", (5,), torch.float32)]
    buf, views = _arena(specs, "cpu")
    spans = []
    for name, shape, dt in specs:
        v = views[name]
        assert v.dtype == dt and tuple(v.shape) == shape and v.is_contiguous()
        off = v.data_ptr() - buf.data_ptr()
        assert off % 256 == 0
        spans.append((off, off + v.numel() * v.element_size()))
    spans.sort()
    assert all(a[1] <= b[0] for a, b in zip(spans, spans[1:]))
    assert spans[-1][1] <= buf.numel()
    views["u"].fill_(1.5)
    views["parents"].fill_(-1)
    assert torch.equal(buf[spans[-1][0]:spans[-1][1]].view(torch.float32), torch.full((5,), 1.5))
    assert int(buf.view(torch.uint8)[:4].view(torch.int32)[0]) == -1
