"""Pins of the oracle's block append: rotary positions and per-token Int8 quantisation.

Each check ties the oracle to something other than itself: the complex-number form of a rotation, the
relative-position property of rotary embeddings, a hand-worked quantisation, and the property PR #1212 states
for per-token scales (every single-valued token gets the same code).
"""
import numpy as np
import pytest

from oracle import append as oap
from oracle import tree as ot


def test_inverse_frequencies_hand_values():
    f = oap.inv_freq(4, 10000.0)
    assert f.tolist() == [1.0, 0.01]  # 10000^0 and 10000^(-2/4)
    assert np.isclose(oap.inv_freq(8, 1e6)[3], 1e6 ** (-6 / 8), rtol=0, atol=1e-18)


@pytest.mark.parametrize("rot_dim,D", [(8, 8), (16, 24), (64, 64)])
def test_rope_is_complex_multiplication(rot_dim, D):
    rng = np.random.default_rng(rot_dim + D)
    x = rng.standard_normal(D)
    for pos in (0, 1, 17, 4099, 131135):
        got = oap.rope(x, pos, 10000.0, rot_dim)
        h = rot_dim // 2
        z = (x[:h] + 1j * x[h:rot_dim]) * np.exp(1j * pos * 10000.0 ** (-np.arange(h) * 2.0 / rot_dim))
        assert np.allclose(got[:h], z.real, rtol=0, atol=1e-12)
        assert np.allclose(got[h:rot_dim], z.imag, rtol=0, atol=1e-12)
        assert np.array_equal(got[rot_dim:], x[rot_dim:])  # features past rot_dim are not rotated
    assert np.array_equal(oap.rope(x, 0, 10000.0, rot_dim), x)


def test_rope_interleaved_is_a_permutation_of_the_half_layout():
    rng = np.random.default_rng(2)
    D = 32
    x = rng.standard_normal(D)
    perm = np.concatenate([np.arange(0, D, 2), np.arange(1, D, 2)])  # interleaved pairs -> halves
    got = oap.rope(x, 77, 500.0, D, interleaved=True)
    via_half = np.empty(D)
    via_half[perm] = oap.rope(x[perm], 77, 500.0, D)
    assert np.allclose(got, via_half, rtol=0, atol=1e-13)


def test_rope_scores_depend_only_on_relative_position():
    rng = np.random.default_rng(3)
    q, k = rng.standard_normal(64), rng.standard_normal(64)
    ref = oap.rope(q, 40, 1e4, 64) @ oap.rope(k, 33, 1e4, 64)
    for shift in (1, 100, 5000):
        assert np.isclose(oap.rope(q, 40 + shift, 1e4, 64) @ oap.rope(k, 33 + shift, 1e4, 64), ref, rtol=1e-10)


def test_node_positions_follow_depth():
    assert oap.node_positions([-1, 0, 1, 2], 10) == [10, 11, 12, 13]  # a chain: the chain verify's positions
    par = [-1, 0, 0, 1, 1, 2, 2, 4]
    assert oap.node_positions(par, 5) == [5 + ot.depth(par, i) for i in range(len(par))] == [5, 6, 6, 7, 7, 7, 7, 8]


def test_quantize_hand_worked_token():
    # absmax 1.27 -> scale fp32(1.27 / 127) = 0.0099999998 -> fp16 0x211F (0.010002136);
    # codes: 0.5 / s = 49.99 -> 50, -1.27 / s = -126.97 -> -127, 0.01 / s = 0.9998 -> 1, 0 -> 0
    codes, scale = oap.quantize_token([0.5, -1.27, 0.01, 0.0])
    assert codes.tolist() == [50, -127, 1, 0]
    assert int(scale) == 0x211F


@pytest.mark.parametrize("v", [3.0, -1e-3, 0.5, 1000.0, 2.0 ** -14])
def test_single_valued_tokens_all_get_the_same_code(v):
    codes, scale = oap.quantize_token(np.full(16, v))
    assert codes.tolist() == [127 * int(np.sign(v))] * 16


def test_zero_token_and_error_bound():
    codes, scale = oap.quantize_token(np.zeros(8))
    assert codes.tolist() == [0] * 8 and int(scale) == 0
    # a scale below half the smallest fp16 subnormal rounds to 0: such a token stores zeros
    codes, scale = oap.quantize_token(np.full(8, 2.0 ** -20))
    assert codes.tolist() == [0] * 8 and int(scale) == 0
    # absmax 177.8 * 2^-24: the scale absmax / 127 = 1.4 * 2^-24 rounds to the smallest fp16 subnormal 2^-24 (bits
    # 0x0001), so the extreme features divide to -177.8 and 177.8 and clip symmetrically to -127 and 127
    a = float(np.float32(177.8 * 2.0 ** -24))
    codes, scale = oap.quantize_token(np.array([-a, float(np.float32(a / 2)), a]))
    assert int(scale) == 0x0001 and codes.tolist() == [-127, 89, 127]
    rng = np.random.default_rng(9)
    for _ in range(50):
        x = (rng.standard_normal(256) * rng.uniform(1e-3, 10)).astype(np.float32).astype(np.float64)
        codes, sbits = oap.quantize_token(x)
        s = float(np.uint16(sbits).view(np.float16))
        assert codes.min() >= -127 and codes.max() <= 127 and np.abs(codes).max() >= 126
        assert np.max(np.abs(codes * s - x)) <= 0.5 * s + np.max(np.abs(x)) * 2.0 ** -10


def test_append_block_rotates_every_head_to_its_node_position():
    # Each node's Q and new K rows turn by the complex rotation of position S + (edges to the root, counted here by
    # walking the parent links); features past rot_dim and the V rows pass through unchanged.
    rng = np.random.default_rng(11)
    par = [-1, 0, 0, 1, 2, 2, 5, 6]
    T, HQ, HKV, D, rd, S, base = len(par), 4, 2, 20, 12, 1000, 1e4
    q = rng.standard_normal((T, HQ, D))
    k = rng.standard_normal((T, HKV, D))
    v = rng.standard_normal((T, HKV, D))
    q_rot, k_rot, v_out = oap.append_block(q, k, v, par, S, base, rd)
    h = rd // 2
    for i in range(T):
        d, j = 0, i
        while par[j] >= 0:
            j, d = par[j], d + 1
        turn = np.exp(1j * (S + d) * base ** (-np.arange(h) * 2.0 / rd))
        for x, y in ((q[i], q_rot[i]), (k[i], k_rot[i])):
            z = (x[:, :h] + 1j * x[:, h:rd]) * turn
            assert np.allclose(y[:, :h], z.real, rtol=0, atol=1e-12)
            assert np.allclose(y[:, h:rd], z.imag, rtol=0, atol=1e-12)
            assert np.array_equal(y[:, rd:], x[:, rd:])
    assert np.array_equal(v_out, v)
