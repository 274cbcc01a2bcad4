"""Pins of the oracle's steps to facts other than the oracle itself.

Each test checks one step against a hand-enumerated case, a closed form,
an exact-rational evaluation of the step's definition, an invariant, or a
brute force on tiny inputs, chosen so that a plausible slip (a dropped
term, a wrong sign or index, a transposed operand, the wrong rounding
rule) fails at least one of them.
"""
import math
from fractions import Fraction

import numpy as np
import pytest

import oracle
import synth
from tests.exact import F, f32_round, round_half_even, to_f32

# ----------------------------------------------------------------------------
# Quantiser ("Batched Prefill", section "The Solution": per-token int8
# activations, quantised once per chunk; per-token symmetric absmax).
# ----------------------------------------------------------------------------


def test_quantize_hand_enumerated_ties_to_even():
    # amax = 127 makes inv = 127/127 = 1 and a_scale = 1 exactly, so every
    # code is round-half-even(y): 2.5 -> 2, 3.5 -> 4, -2.5 -> -2, -126.5 -> -126.
    y = np.array([[127.0, 2.5, 3.5, -2.5, 0.49999997, -126.5, 0.5, 1.5]], np.float32)
    q, s = oracle.quantize_rows(y)
    assert q.tolist() == [[127, 2, 4, -2, 0, -126, 0, 2]]
    assert s.tolist() == [1.0]


def test_quantize_negative_absmax_and_halves():
    # amax comes from a negative entry; y = [-2, 1, 0.5, -1]: inv = 63.5,
    # codes -127, 63.5 -> 64 (tie to even), 31.75 -> 32, -63.5 -> -64.
    y = np.array([[-2.0, 1.0, 0.5, -1.0]], np.float32)
    q, s = oracle.quantize_rows(y)
    assert q.tolist() == [[-127, 64, 32, -64]]
    assert s[0] == np.float32(2.0) / np.float32(127.0)


def test_quantize_zero_row():
    q, s = oracle.quantize_rows(np.zeros((2, 16), np.float32))
    assert not q.any() and s.tolist() == [0.0, 0.0]


def _quantize_exact(row):
    """The quantiser's definition evaluated on exact rationals, one f32 rounding per operation."""
    amax = max(abs(F(v)) for v in row)
    if amax == 0:
        return [0] * len(row), Fraction(0)
    inv = f32_round(Fraction(127) / amax)
    codes = []
    for v in row:
        t = f32_round(F(v) * inv)
        codes.append(max(-127, min(127, round_half_even(t))))
    return codes, f32_round(amax / 127)


def test_quantize_matches_exact_rational_definition():
    y = synth.uniform_f32(11, 1, (6, 96), -3.0, 3.0)
    y[2] *= 1e-3
    y[3, 5] = 40.0  # one outlier row
    q, s = oracle.quantize_rows(y)
    for r in range(y.shape[0]):
        codes, scale = _quantize_exact(y[r])
        assert q[r].tolist() == codes
        assert F(s[r]) == scale


def test_quantize_multiplies_by_inverse_not_divides():
    # Search for an input where rint(y * fl(127/amax)) and rint(y / fl(amax/127))
    # differ; the oracle must follow the multiply-by-inverse reading.
    # Candidates sit a few ulps around (k + 1/2) * amax / 127, where one
    # rounding step of difference decides the code.
    rng = np.random.default_rng(5)
    found = 0
    for _ in range(300):
        amax = np.float32(rng.uniform(0.5, 3.0))
        inv = f32_round(Fraction(127) / F(amax))
        s = f32_round(F(amax) / 127)
        k = int(rng.integers(0, 126))
        c = np.float32((k + 0.5) * float(amax) / 127.0)
        for d in range(-3, 4):
            v = np.float32(c + d * np.spacing(c))
            a = round_half_even(f32_round(F(v) * inv))
            b = round_half_even(f32_round(F(v) / s))
            if a != b:
                q, _ = oracle.quantize_rows(np.array([[amax, v]], np.float32))
                assert q[0, 1] == a
                found += 1
    assert found > 0


def test_quantize_invariants():
    y = synth.normal_f32(3, 9, (32, 257), 0.0, 1.5)
    q, s = oracle.quantize_rows(y)
    assert np.abs(q.astype(np.int32)).max() <= 127
    am = np.abs(y).argmax(axis=1)
    assert np.all(np.abs(q[np.arange(32), am]) == 127)
    assert np.all((np.sign(q) == np.sign(y)) | (q == 0))
    err = np.abs(q.astype(np.float64) * s[:, None].astype(np.float64) - y.astype(np.float64))
    assert np.all(err <= s[:, None] * 0.5 * (1 + 1e-5) + 1e-30)
    # power-of-two scaling leaves codes unchanged and scales a_scale exactly
    q2, s2 = oracle.quantize_rows(y * np.float32(8.0))
    assert np.array_equal(q, q2) and np.array_equal(s2, s * np.float32(8.0))


# ----------------------------------------------------------------------------
# int8 GEMM ("Batched Prefill", sections "The Solution" and "Correctness").
# ----------------------------------------------------------------------------


def test_gemm_hand_enumerated():
    a = np.array([[1, 2, 3, 4], [-1, 0, 127, -127]], np.int8)
    w = np.array([[1, 1, 1, 1], [127, -127, 1, 0], [0, 0, 0, 1]], np.int8)
    acc = oracle.gemm_i8(a, w, 1)
    # row 0: 1+2+3+4 = 10; 127-254+3 = -124; 4
    # row 1: -1+0+127-127 = -1; -127+0+127+0 = 0; -127
    assert acc.tolist() == [[10, -124, 4], [-1, 0, -127]]


@pytest.mark.parametrize("k", [1, 64, 4096, 14336])
def test_gemm_closed_forms(k):
    ones = np.ones((2, k), np.int8)
    assert np.all(oracle.gemm_i8(ones, ones[:1]) == k)
    hi = np.full((1, k), 127, np.int8)
    lo = np.full((1, k), -127, np.int8)
    assert oracle.gemm_i8(hi, hi)[0, 0] == 127 * 127 * k
    assert oracle.gemm_i8(hi, lo)[0, 0] == -127 * 127 * k


def test_gemm_brute_force_tiny():
    a = synth.uniform_i8(1, 2, (5, 37))
    w = synth.uniform_i8(1, 3, (7, 37))
    acc = oracle.gemm_i8(a, w, 3)
    for t in range(5):
        for r in range(7):
            assert acc[t, r] == sum(int(a[t, i]) * int(w[r, i]) for i in range(37))
    assert oracle.dot_i8(a[2], w[4]) == acc[2, 4]


def test_gemm_thread_split_is_invisible():
    a = synth.uniform_i8(2, 2, (9, 300))
    w = synth.uniform_i8(2, 3, (61, 300))
    assert np.array_equal(oracle.gemm_i8(a, w, 1), oracle.gemm_i8(a, w, 7))


# ----------------------------------------------------------------------------
# Dequantising epilogue: (float(acc) * w_scale) * a_scale in f32, in order.
# ----------------------------------------------------------------------------


def _dequant_exact(acc, ws, as_):
    return f32_round(f32_round(f32_round(Fraction(acc)) * F(ws)) * F(as_))


def test_dequant_exact_and_order():
    rng = np.random.default_rng(7)
    differs = 0
    for _ in range(3000):
        acc = int(rng.integers(-(2**28), 2**28))
        ws = np.float32(rng.uniform(1e-4, 1e-2))
        as_ = np.float32(rng.uniform(1e-3, 1.0))
        got = oracle.dequant(acc, ws, as_)
        assert F(got) == _dequant_exact(acc, ws, as_)
        other = f32_round(f32_round(Fraction(acc)) * f32_round(F(ws) * F(as_)))
        differs += F(got) != other
    assert differs > 0  # the fixed order is observable


def test_dequant_special_cases():
    assert oracle.dequant(16777217, 1.0, 1.0) == np.float32(16777216.0)  # float(acc) rounds to even
    assert oracle.dequant(-5, 1.0, 1.0) == -5.0
    assert oracle.dequant(12345, 0.0, 1.0) == 0.0
    assert oracle.dequant(3, 0.25, 0.5) == 0.375


# ----------------------------------------------------------------------------
# RMSNorm.
# ----------------------------------------------------------------------------


def test_rmsnorm_closed_forms():
    # x = (3, 4): mean square 12.5; with eps = 0, y = x / sqrt(12.5)
    y = oracle.rmsnorm_rows(np.array([[3.0, 4.0]], np.float32), np.ones(2, np.float32), 0.0)
    assert y[0, 0] == np.float32(3 / math.sqrt(12.5)) and y[0, 1] == np.float32(4 / math.sqrt(12.5))
    # constant row c: y_k = g_k * c / sqrt(c^2 + eps)
    g = synth.normal_f32(1, 5, (64,), 1.0, 0.1)
    for c in (-2.0, 0.003, 7.5):
        y = oracle.rmsnorm_rows(np.full((1, 64), c, np.float32), g, 1e-5)
        c32 = np.float64(np.float32(c))
        ref = np.float64(g) * (c32 / math.sqrt(c32 ** 2 + np.float64(np.float32(1e-5))))
        # correctly rounded to f32 up to the double evaluation's own error
        assert np.all(np.abs(y[0].astype(np.float64) - ref) <= 0.5001 * np.spacing(np.abs(y[0])))


def test_rmsnorm_gain_and_scale_invariance():
    x = synth.normal_f32(2, 1, (3, 128), 0.0, 2.0)
    g = synth.normal_f32(2, 2, (128,), 1.0, 0.3)
    y1 = oracle.rmsnorm_rows(x, np.ones(128, np.float32), 0.0)
    yg = oracle.rmsnorm_rows(x, g, 0.0)
    assert np.allclose(yg, y1 * g, rtol=2e-7, atol=0)
    assert np.allclose(np.sqrt((y1.astype(np.float64) ** 2).mean(axis=1)), 1.0, rtol=1e-6)
    y4 = oracle.rmsnorm_rows(x * np.float32(4.0), g, 0.0)
    assert np.array_equal(y4, yg)


# ----------------------------------------------------------------------------
# RoPE: pairs (j, j + hd/2) rotated by pos * theta^(-2j/hd).
# ----------------------------------------------------------------------------


def test_rope_position_zero_is_identity():
    x = synth.normal_f32(4, 1, (1, 3, 64), 0.0, 1.0)
    assert np.array_equal(oracle.rope_rows(x, 0, 10000.0), x)


def test_rope_closed_forms():
    # hd = 2: one pair with frequency theta^0 = 1, so (1, 0) -> (cos p, sin p)
    for p in (1, 7, 300):
        y = oracle.rope_rows(np.array([[[1.0, 0.0]]], np.float32), p, 10000.0)
        assert y[0, 0, 0] == np.float32(math.cos(p)) and y[0, 0, 1] == np.float32(math.sin(p))
    # hd = 4, theta = 10000: pair (0, 2) turns by p, pair (1, 3) by p / 100
    p = 5
    y = oracle.rope_rows(np.array([[[0.0, 1.0, 0.0, 0.0]]], np.float32), p, 10000.0)[0, 0]
    assert y[1] == np.float32(math.cos(p / 100.0)) and y[3] == np.float32(math.sin(p / 100.0))
    assert y[0] == 0.0 and y[2] == 0.0


def test_rope_norms_and_relative_positions():
    hd = 128
    q = synth.normal_f32(5, 1, (1, 1, hd), 0.0, 1.0)
    k = synth.normal_f32(5, 2, (1, 1, hd), 0.0, 1.0)
    qr = oracle.rope_rows(q, 1000, 500000.0)
    half = hd // 2
    n0 = q[0, 0, :half].astype(np.float64) ** 2 + q[0, 0, half:].astype(np.float64) ** 2
    n1 = qr[0, 0, :half].astype(np.float64) ** 2 + qr[0, 0, half:].astype(np.float64) ** 2
    assert np.allclose(n0, n1, rtol=1e-6)
    d1 = np.dot(oracle.rope_rows(q, 40, 10000.0).ravel().astype(np.float64),
                oracle.rope_rows(k, 33, 10000.0).ravel().astype(np.float64))
    d2 = np.dot(oracle.rope_rows(q, 1040, 10000.0).ravel().astype(np.float64),
                oracle.rope_rows(k, 1033, 10000.0).ravel().astype(np.float64))
    assert abs(d1 - d2) < 1e-4 * max(1.0, abs(d1))


# ----------------------------------------------------------------------------
# SwiGLU.
# ----------------------------------------------------------------------------


def test_silu_closed_forms():
    assert oracle.silu_mul(0.0, 5.0) == 0.0
    assert oracle.silu_mul(1.0, 1.0) == np.float32(1.0 / (1.0 + math.exp(-1.0)))
    assert oracle.silu_mul(2.0, -3.0) == np.float32(-3.0 * 2.0 / (1.0 + math.exp(-2.0)))
    assert oracle.silu_mul(40.0, 1.0) == np.float32(40.0)
    assert abs(float(oracle.silu_mul(-40.0, 1.0))) < 1e-15


# ----------------------------------------------------------------------------
# Causal attention.
# ----------------------------------------------------------------------------


def test_attention_single_key_returns_value():
    q = synth.normal_f32(6, 1, (1, 4, 16), 0.0, 3.0)
    K = synth.normal_f32(6, 2, (1, 2, 16), 0.0, 1.0)
    V = synth.normal_f32(6, 3, (1, 2, 16), 0.0, 1.0)
    o = oracle.attention(q, K, V, 0)
    # query heads 0,1 read KV head 0; heads 2,3 read KV head 1
    assert np.array_equal(o[0, 0], V[0, 0]) and np.array_equal(o[0, 1], V[0, 0])
    assert np.array_equal(o[0, 2], V[0, 1]) and np.array_equal(o[0, 3], V[0, 1])


def test_attention_uniform_scores_average_the_prefix():
    # q = 0 makes every score 0: position i averages v_0 .. v_i (inclusive mask)
    rows, start, H, hd = 5, 3, 2, 8
    q = np.zeros((rows, H, hd), np.float32)
    K = synth.normal_f32(7, 2, (start + rows + 4, 1, hd), 0.0, 1.0)
    V = synth.normal_f32(7, 3, (start + rows + 4, 1, hd), 0.0, 1.0)
    o = oracle.attention(q, K, V, start)
    for i in range(rows):
        ref = V[: start + i + 1, 0].astype(np.float64).mean(axis=0)
        assert np.allclose(o[i, 0], ref, rtol=1e-6, atol=1e-7)


def test_attention_ignores_future_keys():
    rows, start, H, hd = 4, 2, 4, 16
    q = synth.normal_f32(8, 1, (rows, H, hd), 0.0, 1.0)
    K = synth.normal_f32(8, 2, (start + rows + 3, 2, hd), 0.0, 1.0)
    V = synth.normal_f32(8, 3, (start + rows + 3, 2, hd), 0.0, 1.0)
    o1 = oracle.attention(q, K, V, start)
    K2, V2 = K.copy(), V.copy()
    K2[start + rows:] = 100.0
    V2[start + rows:] = -100.0
    assert np.array_equal(o1, oracle.attention(q, K2, V2, start))
    # the key at the query's own position is seen
    K3 = K.copy()
    K3[start + rows - 1] *= 2.0
    o3 = oracle.attention(q, K3, V, start)
    assert np.array_equal(o3[:-1], o1[:-1]) and not np.array_equal(o3[-1], o1[-1])


def test_attention_brute_force_softmax():
    from scipy.special import softmax

    rows, start, H, Hkv, hd = 3, 6, 4, 2, 32
    q = synth.normal_f32(9, 1, (rows, H, hd), 0.0, 1.0)
    K = synth.normal_f32(9, 2, (start + rows, Hkv, hd), 0.0, 1.0)
    V = synth.normal_f32(9, 3, (start + rows, Hkv, hd), 0.0, 1.0)
    o = oracle.attention(q, K, V, start)
    for i in range(rows):
        for h in range(H):
            kv = h // (H // Hkv)
            n = start + i + 1
            s = K[:n, kv].astype(np.float64) @ q[i, h].astype(np.float64) / math.sqrt(hd)
            ref = softmax(s) @ V[:n, kv].astype(np.float64)
            assert np.allclose(o[i, h], ref, rtol=1e-6, atol=1e-7)


def test_attention_dominant_key():
    hd = 16
    K = np.zeros((4, 1, hd), np.float32)
    K[2, 0, 0] = 1.0
    V = synth.normal_f32(10, 3, (4, 1, hd), 0.0, 1.0)
    q = np.zeros((1, 1, hd), np.float32)
    q[0, 0, 0] = 400.0  # score 100 at key 2, 0 elsewhere
    o = oracle.attention(q, K, V, 3)
    assert np.allclose(o[0, 0], V[2, 0], rtol=1e-6, atol=1e-6)
