"""Pins of the oracle's attention, LM head, gather and storage decoding.

Each check ties the oracle to something other than itself: a library routine
computing a special case (torch CPU fp64 scaled_dot_product_attention, matmul,
argmax), a hand-built value, or an equivalence the pages state (mlxcel PR #1212:
prefix selection == trim_to, identity selection is a no-op, the tail form equals
the absolute form, Int8 scale sidecars move with their tokens).
"""
import math

import numpy as np
import pytest
import torch

from oracle import attention as oa
from oracle import gather as og
from oracle import lm_head as ol
from oracle import storage as osd
from oracle import tree as ot


# ----------------------------------------------------------------------------- storage
def test_storage_known_values():
    assert list(osd.bf16([0x3F80, 0xC000, 0x3F81, 0x0000, 0x8000])) == [1.0, -2.0, 1.0078125, 0.0, -0.0]
    assert list(osd.f16([0x3C00, 0xC000, 0x3C01, 0x0001])) == [1.0, -2.0, 1.0009765625, 2.0 ** -24]
    v = osd.int8_scaled(np.array([[3, -127], [1, 0]], dtype=np.int8), np.array([0x3800, 0x4000], dtype=np.uint16))
    assert v.tolist() == [[1.5, -63.5], [2.0, 0.0]]  # scales 0.5 and 2.0


def test_kv_values_dispatches_each_format_to_its_decoder():
    # Format 0 reads fp16 bit patterns, 1 bf16, 2 Int8 codes times their token's fp16 scale; anything else is refused.
    bits = np.array([[0x3C00, 0xC000]], dtype=np.uint16)
    assert osd.kv_values(0, bits).tolist() == [[1.0, -2.0]]
    assert osd.kv_values(1, bits).tolist() == [[2.0 ** -7, -2.0 ** 1]]  # bf16 0x3C00 = 2^-7, 0xC000 = -2
    codes = np.array([[4, -8]], dtype=np.int8)
    assert osd.kv_values(2, codes, np.array([0x3400], dtype=np.uint16)).tolist() == [[1.0, -2.0]]  # scale 0.25
    with pytest.raises(ValueError):
        osd.kv_values(3, bits)


def test_q4_hand_built_group():
    # byte 0x21 -> element 0 = 1 (low nibble), element 1 = 2 (high nibble)
    assert osd.unpack_q4(np.array([[0x21, 0xF0]], dtype=np.uint8)).tolist() == [[1, 2, 0, 15]]
    codes = np.arange(64) % 16
    packed = (codes[0::2] | (codes[1::2] << 4)).astype(np.uint8)[None, :]
    scale = np.array([[0x3F00]], dtype=np.uint16)  # 0.5
    bias = np.array([[0xBF80]], dtype=np.uint16)   # -1.0
    w = osd.q4_affine(packed, scale, bias)
    assert w.shape == (1, 64)
    assert np.array_equal(w[0], 0.5 * codes - 1.0)


# ----------------------------------------------------------------------------- attention
def torch_sdpa(q, k, v, allowed):
    """torch CPU fp64 SDPA with a boolean mask; q [R, D], k/v [N, D], allowed [R, N]."""
    t = lambda a: torch.from_numpy(np.ascontiguousarray(a, dtype=np.float64))[None, None]
    out = torch.nn.functional.scaled_dot_product_attention(t(q), t(k), t(v), attn_mask=t(allowed).bool())
    return out[0, 0].numpy()


@pytest.mark.parametrize("S,T", [(0, 1), (5, 1), (17, 4), (64, 6)])
def test_linear_tree_is_causal_sdpa(S, T):
    rng = np.random.default_rng(S * 10 + T)
    D = 16
    q = rng.standard_normal((T, 1, D))
    K = rng.standard_normal((1, S + T, D))
    V = rng.standard_normal((1, S + T, D))
    par = [-1] + list(range(T - 1))
    out = oa.tree_verify_attention(q, K, V, par, S)
    allowed = np.arange(S + T)[None, :] <= (np.arange(T)[:, None] + S)
    ref = torch_sdpa(q[:, 0], K[0], V[0], allowed)
    assert np.allclose(out[:, 0], ref, rtol=1e-12, atol=1e-12)


def test_tree_node_equals_causal_attention_over_its_root_path():
    rng = np.random.default_rng(3)
    par = [-1, 0, 0, 1, 1, 2, 2, 3, 5, 8]
    T, S, D = len(par), 9, 8
    q = rng.standard_normal((T, 1, D))
    K = rng.standard_normal((1, S + T, D))
    V = rng.standard_normal((1, S + T, D))
    out = oa.tree_verify_attention(q, K, V, par, S)
    for i in range(T):
        path = sorted(ot.ancestors(par, i))
        cols = list(range(S)) + [S + j for j in path]
        # the node is the last element of its own root path: causal SDPA over that sequence
        n = len(cols)
        allowed = np.ones((1, n), dtype=bool)
        ref = torch_sdpa(q[i, :, :], K[0, cols], V[0, cols], allowed)
        assert np.allclose(out[i, 0], ref[0], rtol=1e-12, atol=1e-12)


def test_dense_mask_form_equals_ancestor_form():
    rng = np.random.default_rng(4)
    par = [-1, 0, 0, 1, 1, 2, 2]
    T, S, D = 7, 33, 8
    K = rng.standard_normal((S + T, D))
    V = rng.standard_normal((S + T, D))
    m = ot.history_mask(par, S)
    for i in range(T):
        q = rng.standard_normal(D)
        a = oa.attend_row(q, K, V, S, ot.ancestors(par, i))
        b = oa.attend_dense_mask(q, K, V, m[i])
        assert np.allclose(a, b, rtol=1e-12, atol=1e-12)


def test_gqa_head_mapping_matches_repeat_interleave():
    rng = np.random.default_rng(5)
    T, HQ, HKV, S, D = 3, 6, 2, 10, 8
    par = [-1, 0, 1]
    q = rng.standard_normal((T, HQ, D))
    K = rng.standard_normal((HKV, S + T, D))
    V = rng.standard_normal((HKV, S + T, D))
    out = oa.tree_verify_attention(q, K, V, par, S)
    Kr = np.repeat(K, HQ // HKV, axis=0)  # query head h reads kv head h // G
    Vr = np.repeat(V, HQ // HKV, axis=0)
    allowed = np.arange(S + T)[None, :] <= (np.arange(T)[:, None] + S)
    for h in range(HQ):
        ref = torch_sdpa(q[:, h], Kr[h], Vr[h], allowed)
        assert np.allclose(out[:, h], ref, rtol=1e-12, atol=1e-12)


def test_single_node_is_decode_attention():
    rng = np.random.default_rng(6)
    S, D = 50, 16
    q = rng.standard_normal(D)
    K = rng.standard_normal((S + 1, D))
    V = rng.standard_normal((S + 1, D))
    s = K @ q / math.sqrt(D)
    p = np.exp(s - s.max())
    ref = (p / p.sum()) @ V
    assert np.allclose(oa.attend_row(q, K, V, S, {0}), ref, rtol=1e-13, atol=1e-13)


# ----------------------------------------------------------------------------- LM head
def test_argmax_matches_torch_fp64():
    rng = np.random.default_rng(8)
    W = rng.standard_normal((1000, 64))
    h = rng.standard_normal((5, 64))
    idx, top, gap = ol.argmax_gap(ol.logits(W, h))
    lt = torch.from_numpy(h) @ torch.from_numpy(W).T
    assert idx.tolist() == torch.argmax(lt, dim=1).tolist()
    srt = torch.sort(lt, dim=1, descending=True).values
    assert np.allclose(gap, (srt[:, 0] - srt[:, 1]).numpy(), rtol=0, atol=1e-12)


def test_argmax_ties_go_to_lowest_index_and_streaming_agrees():
    W = np.zeros((40000, 4))
    W[[7, 20000, 39999], 0] = 2.0  # three-way tie
    W[5, 0] = 1.5
    h = np.array([[1.0, 0, 0, 0]])
    idx, top, gap = ol.argmax_gap(ol.logits(W, h))
    assert (idx[0], top[0], gap[0]) == (7, 2.0, 0.0)
    a, t, g = ol.argmax_streamed(lambda r0, r1: W[r0:r1], h, W.shape[0])
    assert (a[0], t[0], g[0]) == (7, 2.0, 0.0)
    W[7, 0] = 1.0
    a, t, g = ol.argmax_streamed(lambda r0, r1: W[r0:r1], h, W.shape[0])
    assert (a[0], t[0], g[0]) == (20000, 2.0, 0.0)
    W[39999, 0] = 0.5  # the runner-up is now an earlier chunk's best (row 5, 1.5), not the winning chunk's second
    a, t, g = ol.argmax_streamed(lambda r0, r1: W[r0:r1], h, W.shape[0])
    assert (a[0], t[0], g[0]) == (20000, 2.0, 0.5)
    assert (a[0], t[0], g[0]) == tuple(v[0] for v in ol.argmax_gap(ol.logits(W, h)))
    rng = np.random.default_rng(9)
    W2 = rng.standard_normal((50000, 8))
    h2 = rng.standard_normal((3, 8))
    a1 = ol.argmax_gap(ol.logits(W2, h2))
    a2 = ol.argmax_streamed(lambda r0, r1: W2[r0:r1], h2, W2.shape[0])
    assert np.array_equal(a1[0], a2[0])
    assert np.allclose(a1[2], a2[2], rtol=0, atol=1e-12)


# ----------------------------------------------------------------------------- gather
def kv_fixture(n=12, D=8, seed=0):
    rng = np.random.default_rng(seed)
    codes = rng.integers(-127, 128, size=(n, D)).astype(np.int8)
    # distinct per-token scales: a misplaced scale is caught, raw codes would not catch it
    scales = (np.arange(n, dtype=np.float32) * 0.001 + 0.005).astype(np.float16).view(np.uint16)
    return codes, scales


def test_prefix_gather_equals_trim_to():
    codes, scales = kv_fixture()
    S = 5
    for k in range(1, 8):
        kept = list(range(k))
        b, n = og.gather_within_tail(codes, S, kept)
        assert n == S + k
        assert np.array_equal(b[:n], og.trim_to(codes, n))
        assert og.is_identity(kept)


def test_identity_gather_is_a_no_op():
    codes, scales = kv_fixture()
    b, n = og.gather_within_tail(codes, 4, [0, 1, 2, 3, 4, 5, 6, 7])
    assert n == 12 and np.array_equal(b, codes)


def test_tail_form_equals_absolute_form_and_scales_move():
    codes, scales = kv_fixture()
    S, path = 4, [0, 2, 5, 7]
    bc, n = og.gather_within_tail(codes, S, path)
    bs, n2 = og.gather_within_tail(scales, S, path)
    absolute = list(range(S)) + [S + p for p in path]
    assert n == n2 == S + len(path)
    assert np.array_equal(bc[:n], og.gather_positions(codes, absolute))
    assert np.array_equal(bs[:n], og.gather_positions(scales, absolute))
    # every kept token decodes against its own scale
    vals = osd.int8_scaled(bc[:n], bs[:n])
    ref = osd.int8_scaled(codes, scales)[absolute]
    assert np.array_equal(vals, ref)
    # rows past the new length keep their bytes (in-place tail rewrite)
    assert np.array_equal(bc[n:], codes[n:])
    assert not og.is_identity(path)


# ----------------------------------------------------------------------------- sliding-window layers
@pytest.mark.parametrize("n,offset,window", [(1, 0, 1), (4, 0, 2), (3, 10, 1), (5, 7, 4), (6, 2, 50)])
def test_sliding_band_is_the_causal_band_of_numpy_triangles(n, offset, window):
    # Row q sits at position offset + q and keeps the `window` positions ending at itself; a window wider than the
    # history reduces to the plain causal mask with offset.
    ones = np.ones((n, offset + n), dtype=bool)
    inside = np.tril(ones, k=offset) & np.triu(ones, k=offset - window + 1)
    band = ot.sliding_band(n, offset, window)
    assert np.array_equal(band == 0.0, inside)
    assert np.all(band[~inside] == ot.BLOCKED)
    if window >= offset + n:
        assert np.array_equal(inside, np.tril(ones, k=offset))


@pytest.mark.parametrize("S,T,window", [(0, 3, 2), (10, 4, 3), (30, 5, 8), (40, 6, 1), (12, 3, 15)])
def test_sliding_linear_tree_is_banded_causal_sdpa(S, T, window):
    # A linear tree on a sliding-window layer is textbook sliding-window causal attention: query at position
    # S + q sees the `window` positions ending at itself (band built here from numpy's triangle routines).
    rng = np.random.default_rng(S + 7 * T + 31 * window)
    D = 16
    q = rng.standard_normal((T, 1, D))
    K = rng.standard_normal((1, S + T, D))
    V = rng.standard_normal((1, S + T, D))
    par = [-1] + list(range(T - 1))
    out = oa.tree_verify_attention(q, K, V, par, S, window=window)
    ones = np.ones((T, S + T), dtype=bool)
    allowed = np.tril(ones, k=S) & np.triu(ones, k=S - window + 1)
    ref = torch_sdpa(q[:, 0], K[0], V[0], allowed)
    assert np.allclose(out[:, 0], ref, rtol=1e-12, atol=1e-12)


def test_sliding_window_of_one_returns_own_value_and_wide_window_changes_nothing():
    rng = np.random.default_rng(8)
    par = [-1, 0, 0, 1, 2, 2, 5]
    T, S, D = len(par), 20, 8
    q = rng.standard_normal((T, 2, D))
    K = rng.standard_normal((1, S + T, D))
    V = rng.standard_normal((1, S + T, D))
    own = oa.tree_verify_attention(q, K, V, par, S, window=1)
    for i in range(T):
        assert np.allclose(own[i], V[0, S + i], rtol=0, atol=1e-15)  # only the node itself survives the band
    full = oa.tree_verify_attention(q, K, V, par, S)
    assert np.allclose(oa.tree_verify_attention(q, K, V, par, S, window=S + T), full, rtol=1e-13, atol=1e-13)


def test_sliding_mask_from_caller_boundary_is_inclusive():
    # PR #1212 leaves a block untouched while offset + n <= window.  At equality an all-attend mask (whose future
    # columns the band would block) comes back whole; one position past it, the band (numpy triangles) applies.
    T = 5
    for S in (0, 4, 11):
        allatt = np.zeros((T, S + T))
        assert np.array_equal(ot.sliding_mask_from_caller(allatt, S, S + T), allatt)
        window = S + T - 1
        ones = np.ones((T, S + T), dtype=bool)
        inside = np.tril(ones, k=S) & np.triu(ones, k=S - window + 1)
        assert np.array_equal(ot.sliding_mask_from_caller(allatt, S, window) == 0.0, inside)


def test_sliding_mask_from_caller_properties():
    # The properties PR #1212 states for the intersection of a caller mask with the band.
    par = [-1, 0, 0, 1, 1, 2, 2, 4]
    T = len(par)
    for S in (0, 3, 9, 40):
        caller = ot.history_mask(par, S)
        for window in (1, 2, 5, 9, 16, 48, 60):
            got = ot.sliding_mask_from_caller(caller, S, window)
            if S + T <= window:  # below the window the caller mask comes back untouched
                assert np.array_equal(got, caller)
            # intersecting again changes nothing (masks that already carry the band)
            assert np.array_equal(ot.sliding_mask_from_caller(got, S, window), got)
            # every row keeps its own position, so no row is all-masked
            for i in range(T):
                assert got[i, S + i] == 0.0
            # an all-attend caller mask (the draft-tree history shape) reduces to the band past the window
            allatt = np.zeros((T, S + T))
            band_only = ot.sliding_mask_from_caller(allatt, S, window)
            if S + T > window:
                ones = np.ones((T, S + T), dtype=bool)
                inband = np.tril(ones, k=S) & np.triu(ones, k=S - window + 1)  # the causal sliding band
                assert np.array_equal(band_only == 0.0, inband)
            # the dense form and the key lists the attention uses agree
            for i in range(T):
                cols = np.flatnonzero(got[i] == 0.0).tolist()
                assert cols == ot.visible_keys(par, i, S, window)


# ----------------------------------------------------------------------------- rounding to 16-bit storage
# Values are decoded from bit patterns with integer arithmetic (sign, biased exponent, fraction), independently
# of the oracle's view-based decoders; each pattern's neighbours fix where round-to-nearest-even must land.
def bf16_value(p: int) -> float:
    s, e, m = p >> 15, (p >> 7) & 0xFF, p & 0x7F
    assert 0 < e < 255, "normal range only"
    return (-1.0) ** s * math.ldexp(128 + m, e - 127 - 7)


def f16_value(p: int) -> float:
    s, e, m = p >> 15, (p >> 10) & 0x1F, p & 0x3FF
    assert e < 31
    mag = math.ldexp(m, -24) if e == 0 else math.ldexp(1024 + m, e - 15 - 10)
    return -mag if s else mag


def _nearest_even_cases(value, patterns):
    """(x, expected) pairs around every positive pattern p: inside half an ulp -> p, beyond -> the neighbour,
    exactly half an ulp -> whichever of the two has an even fraction (ties to even)."""
    cases = []
    for p in patterns:
        v, up = value(p), value(p + 1)
        dn = value(p - 1) if p > 0 else None
        even = (p & 1) == 0
        cases += [(v, v), (v + 0.49 * (up - v), v), (v + 0.51 * (up - v), up),
                  (v + 0.5 * (up - v), v if even else up)]
        if dn is not None:
            cases += [(v - 0.49 * (v - dn), v), (v - 0.51 * (v - dn), dn), (v - 0.5 * (v - dn), v if even else dn)]
    return cases + [(-x, -y) for x, y in cases]


def test_round_bf16_hand_decoded_values():
    r = lambda x: float(osd.round_bf16(np.array([x]))[0])
    assert r(1.0 + 2.0 ** -8) == 1.0                      # tie between 0x3F80 and 0x3F81 -> even 0x3F80
    assert r(1.0 + 3 * 2.0 ** -8) == 1.0 + 2.0 ** -6      # tie between 0x3F81 and 0x3F82 -> even 0x3F82
    assert r(1.0 + 2.0 ** -8 + 2.0 ** -30) == 1.0 + 2.0 ** -7  # just above the tie -> 0x3F81
    assert r(2.0 - 2.0 ** -10) == 2.0                     # just under a power of two rounds up across it
    assert r(2.0 - 3 * 2.0 ** -9) == bf16_value(0x3FFF) == 1.9921875
    assert r(1.0 / 3.0) == bf16_value(0x3EAB) == 0.333984375
    assert r(-(1.0 + 2.0 ** -8 + 2.0 ** -30)) == bf16_value(0xBF81)
    assert r(3.0e38) == bf16_value(0x7F62)                # large normal values keep 8 significant bits


def test_round_bf16_lands_on_the_nearest_even_neighbour():
    rng = np.random.default_rng(11)
    pats = [0x3F80, 0x3F81, 0x3FFF, 0x4000, 0x0081, 0x7F7E, 0x3E80]
    pats += [int(p) for p in rng.integers(0x0081, 0x7F7E, size=300)]
    cases = _nearest_even_cases(bf16_value, pats)
    x = np.array([c[0] for c in cases])
    want = np.array([c[1] for c in cases])
    assert np.array_equal(osd.round_bf16(x), want)


def test_round_bf16_agrees_with_torch_on_float32_inputs():
    # fp32 -> bf16 in torch is round-to-nearest-even with no intermediate rounding
    rng = np.random.default_rng(12)
    bits = rng.integers(0x00800000, 0x7F000000, size=20000, dtype=np.int64).astype(np.uint32)
    bits |= (rng.integers(0, 2, size=bits.size).astype(np.uint32) << np.uint32(31))
    x = bits.view(np.float32)
    ref = torch.from_numpy(x.copy()).to(torch.bfloat16).to(torch.float64).numpy()
    assert np.array_equal(osd.round_bf16(x.astype(np.float64)), ref)


@pytest.mark.parametrize("fn", ["storage.round_f16", "append.f16_round"])
def test_round_f16_hand_decoded_values(fn):
    from oracle import append as oap
    f = osd.round_f16 if fn == "storage.round_f16" else oap.f16_round
    r = lambda x: float(f(np.array([x]))[0])
    assert r(1.0 + 2.0 ** -11) == 1.0                     # tie -> even 0x3C00
    assert r(1.0 + 3 * 2.0 ** -11) == 1.0 + 2.0 ** -9     # tie -> even 0x3C02
    assert r(1.0 + 2.0 ** -11 + 2.0 ** -30) == 1.0 + 2.0 ** -10  # just past the tie: up (one rounding, not via fp32)
    assert r(1.0 + 2.0 ** -11 - 2.0 ** -30) == 1.0                # just short of it: down
    assert r(2049.0) == 2048.0 and r(2051.0) == 2052.0    # ulp 2 above 2048: ties to even
    with np.errstate(over="ignore"):
        assert r(65519.0) == 65504.0 and r(65520.0) == math.inf  # largest finite, then overflow
    assert r(2.0 ** -25) == 0.0                           # half the smallest subnormal -> even zero
    assert r(3 * 2.0 ** -25) == 2.0 ** -23                # tie between subnormals 1 and 2 -> even 2
    assert r(2.0 ** -24 * 1.49) == 2.0 ** -24
    assert r(-(1.0 / 3.0)) == f16_value(0xB555)           # -0.333251953125


@pytest.mark.parametrize("fn", ["storage.round_f16", "append.f16_round"])
def test_round_f16_lands_on_the_nearest_even_neighbour(fn):
    from oracle import append as oap
    f = osd.round_f16 if fn == "storage.round_f16" else oap.f16_round
    rng = np.random.default_rng(13)
    pats = [0x0001, 0x0002, 0x03FF, 0x0400, 0x3C00, 0x3BFF, 0x7BFE]
    pats += [int(p) for p in rng.integers(0x0001, 0x7BFE, size=300)]
    cases = _nearest_even_cases(f16_value, pats)
    x = np.array([c[0] for c in cases])
    want = np.array([c[1] for c in cases])
    assert np.array_equal(f(x), want)


def test_logits_streamed_equals_integer_matmul_across_chunks():
    # integer-valued weights and hidden rows: every logit is an exact integer, computed independently by an
    # int64 matmul; the head spans two full chunks and a ragged third, so a chunk-offset slip changes values
    V, H = 2 * ol.CHUNK_ROWS + 77, 6
    v = np.arange(V)[:, None]
    k = np.arange(H)[None, :]
    Wi = ((v * 7 + k * 3 + (v // ol.CHUNK_ROWS) * 5) % 11 - 5).astype(np.int64)
    hi = np.array([[1, -2, 3, 0, 5, -1], [2, 2, -1, 4, 0, 3]], dtype=np.int64)
    got = ol.logits_streamed(lambda r0, r1: Wi[r0:r1].astype(np.float64), hi.astype(np.float64), V)
    assert got.shape == (2, V)
    assert np.array_equal(got, (hi @ Wi.T).astype(np.float64))
    a, t, g = ol.argmax_streamed(lambda r0, r1: Wi[r0:r1].astype(np.float64), hi.astype(np.float64), V)
    exact = hi @ Wi.T
    assert a.tolist() == np.argmax(exact, axis=1).tolist()
