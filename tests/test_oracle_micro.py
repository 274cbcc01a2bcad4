"""A 2-layer, dim-8 micro-model whose every int8 dot product is written out by
hand, run through the oracle's whole prefill path.

Construction (each step exact, so every expected value below is a chain of
binary32 roundings of hand-enumerated integers):
  - the prompt's embedding rows are c * s with one sign pattern
    s = (+1, +1, -1, +1, -1, -1, +1, +1) and c > 0; every RMSNorm gain is 1 and
    eps = 0. A row of uniform magnitude a normalises to exactly s: in double,
    sum(x^2)/8 = a^2, sqrt(a^2) = a and x * (1/a) = s (1 +- 2^-53), which rounds to
    s in binary32 ("Single-pass prefill": RMSNorm, then the projections);
  - so every quantised activation row is q = 127 s with a_scale = fl(1/127)
    ("Batched Prefill", "The Solution": per-token absmax int8), and every
    projection accumulator is acc[r] = 127 * sum_k s_k W[r][k] with weights in
    {-1, 0, 1, 127}: the sums are listed in the test;
  - W_o = 0, so the attention block adds exactly 0 to the residual and its K/V
    rows are checked directly (K at position 0, where RoPE is the identity);
  - the FFN's one live gate row has g > 37, where 1 + exp(-g) is 1.0 in double,
    so SiLU(g) * u = fl(g * u); a gate row with g = 0 gives h = 0 and one with
    g < -37 gives |h| far below half a code step: the codes of h are hand-known;
  - the down projection's live column has the signs of s, so the residual keeps
    one magnitude per row, and the next RMSNorm (and the final one) is exact
    again.
Dequantisation is out = (float(acc) * w_scale[r]) * a_scale[t] in binary32 and
the residual add one binary32 addition (the method's fixed epilogue order).
"""
from fractions import Fraction

import numpy as np

import oracle
import synth
from tests.exact import F, f32_round

S = np.array([1, 1, -1, 1, -1, -1, 1, 1], np.int8)
CFG = synth.ModelConfig("micro-2", dim=8, n_layers=2, n_heads=2, n_kv_heads=1, head_dim=4, ffn=16, vocab=8,
                        rms_eps=0.0, rope_theta=10000.0, max_seq=8)
A_SCALE = f32_round(Fraction(1, 127))  # amax = 1 (rows of +-1)
P = 127  # the code of +1


def _row(*entries):
    r = np.zeros(8, np.int8)
    for k, v in entries:
        r[k] = v
    return r


def _dot_s(w_row) -> int:
    return int(np.dot(S.astype(np.int64), w_row.astype(np.int64)))


def _deq(acc: int, ws: float, a_scale: Fraction) -> Fraction:
    return f32_round(f32_round(Fraction(acc) * F(ws)) * a_scale)


def _model():
    m = synth.make_model(CFG, seed=11)
    D = CFG.dim
    m.tok_emb[1] = 0.5 * S
    m.tok_emb[2] = 1.0 * S
    for L in range(2):
        m.attn_norm[L][:] = 1.0
        m.ffn_norm[L][:] = 1.0
        for kind in range(7):
            m.w[7 * L + kind][:] = 0
    m.final_norm[:] = 1.0
    # ---- layer 0
    wq, wk, wv, wo, wg, wu, wd = (m.w[k] for k in range(7))
    wq[0] = _row((0, 1), (3, 127))
    wq[5] = _row((1, -1), (6, 1))
    wk[0] = _row((1, 1))                              # sum s*w = 1
    wk[1] = _row((4, 127), (5, 127))                  # -127 - 127 = -254
    wk[2] = -np.ones(D, np.int8)                      # -(5 - 3) = -2
    wv[0] = _row((0, 1))                              # 1
    wv[1] = _row((2, 127))                            # -127
    wv[2] = np.ones(D, np.int8)                       # 5 - 3 = 2
    wv[3] = _row((0, -1), (7, 127))                   # -1 + 127 = 126
    # wo stays 0: the attention block adds nothing
    wg[0] = np.where(S > 0, 127, -1).astype(np.int8)  # 5 * 127 + 3 * 1 = 638
    wu[0] = _row((0, 1))                              # 1
    wg[4] = 0                                         # g = 0 -> h = 0
    wu[4] = _row((3, 1))                              # 1 (u != 0, h still 0)
    wd[:, 0] = S                                      # down column 0 carries s
    # ---- layer 1
    wq, wk, wv, wo, wg, wu, wd = (m.w[7 + k] for k in range(7))
    wq[2] = _row((2, 127))
    wk[3] = _row((6, 1), (7, 1))                      # 2
    wv[0] = _row((1, 127), (2, -1))                   # 127 + 1 = 128
    wv[2] = _row((4, -1), (5, -1))                    # 2
    wg[5] = np.array([127, 127, -1, 127, -1, -1, 127, 0], np.int8)  # 127 * 4 + 3 = 511
    wu[5] = _row((7, -1))                             # -1
    wg[2] = np.where(S > 0, -1, 127).astype(np.int8)  # -5 - 3 * 127 = -386
    wu[2] = _row((0, 1))                              # 1
    wd[:, 5] = -S                                     # code of h5 is -127: (-127)(-s) = 127 s
    # ---- scales: powers of two, so acc * w_scale is exact
    for L in range(2):
        m.w_scale[7 * L + 1][:] = [2.0 ** -7, 2.0 ** -10, 2.0 ** -5, 2.0 ** -4]
        m.w_scale[7 * L + 2][:] = [2.0 ** -7, 2.0 ** -12, 2.0 ** -5, 2.0 ** -11]
        m.w_scale[7 * L + 4][:] = 2.0 ** -3
        m.w_scale[7 * L + 5][:] = 2.0 ** -7
        m.w_scale[7 * L + 6][:] = 2.0 ** -6
    # ---- LM head
    m.w_out[:] = 0
    m.w_out[0] = np.ones(D, np.int8)                  # 2
    m.w_out[1] = _row((2, 127))                       # -127
    m.w_out[2] = np.array([127, 127, 0, 127, 0, 0, 127, 127], np.int8)  # 635
    m.w_out[3] = _row((4, -1), (5, 1))                # 1 - 1 = 0
    m.w_out[4] = _row((0, -1))                        # -1
    m.w_out[5] = np.where(S > 0, 1, -1).astype(np.int8)  # 8
    m.w_out[6] = -m.w_out[5]                          # -8
    m.w_out[7] = np.array([127, -1, 0, 0, 0, 0, 0, 0], np.int8)  # 126
    m.w_out_scale[:] = [2.0 ** -7, 2.0 ** -9, 2.0 ** -10, 1.0, 2.0 ** -2, 2.0 ** -3, 2.0 ** -3, 2.0 ** -8]
    return m


def _ffn_delta(g_acc: int, u_acc: int, wd_sign: int) -> Fraction:
    """|down| of the live FFN path: h = fl(g * u), its code is sign(h) * 127 with
    a_scale fl(|h|/127), and the down accumulator is 127 * (code sign * column sign)."""
    g = _deq(g_acc, 2.0 ** -3, A_SCALE)
    assert g > 37  # 1 + exp(-g) == 1.0 in double
    u = _deq(u_acc, 2.0 ** -7, A_SCALE)
    h = f32_round(g * u)
    a_h = f32_round(abs(h) / 127)
    inv = f32_round(Fraction(127) / abs(h))
    assert f32_round(abs(h) * inv) == 127  # the code of h is +-127
    code = 127 if h > 0 else -127
    acc_d = code * wd_sign  # the column's entry for a row whose residual sign is +1
    assert acc_d == 127
    return _deq(acc_d, 2.0 ** -6, a_h)


def test_hand_enumerated_dots():
    m = _model()
    # the hand sums in _model's comments, by brute force over s
    assert [_dot_s(m.w[1][r]) for r in range(3)] == [1, -254, -2]
    assert [_dot_s(m.w[2][r]) for r in range(4)] == [1, -127, 2, 126]
    assert _dot_s(m.w[4][0]) == 638 and _dot_s(m.w[5][0]) == 1 and _dot_s(m.w[5][4]) == 1
    assert _dot_s(m.w[7 + 1][3]) == 2
    assert [_dot_s(m.w[7 + 2][r]) for r in (0, 2)] == [128, 2]
    assert _dot_s(m.w[7 + 4][5]) == 511 and _dot_s(m.w[7 + 5][5]) == -1 and _dot_s(m.w[7 + 4][2]) == -386
    assert [_dot_s(m.w_out[v]) for v in range(8)] == [2, -127, 635, 0, -1, 8, -8, 126]


def test_two_layer_micro_model_by_hand():
    m = _model()
    toks = np.array([1, 2, 1], np.int32)
    om = oracle.OracleModel(m)
    logits, hidden = om.prefill(toks, 0, 2, want_hidden=True)

    # K/V rows: every position's attention input codes are 127 s, so every V row
    # (and K at position 0, where RoPE is the identity) is the same
    v_acc = {0: [P * 1, P * -127, P * 2, P * 126], 1: [P * 128, 0, P * 2, 0]}
    k0_acc = {0: [P * 1, P * -254, P * -2, 0], 1: [0, 0, 0, P * 2]}
    for L in range(2):
        wsk, wsv = m.w_scale[7 * L + 1], m.w_scale[7 * L + 2]
        V = om.kv(L, 1)[:3, 0, :]
        K = om.kv(L, 0)[0, 0, :]
        for j in range(4):
            exp_v = _deq(v_acc[L][j], wsv[j], A_SCALE)
            assert all(F(V[p, j]) == exp_v for p in range(3)), (L, j)
            assert F(K[j]) == _deq(k0_acc[L][j], wsk[j], A_SCALE), (L, j)

    # residual after layer 0: attention adds 0, the FFN adds s * d0;
    # after layer 1 the FFN adds s * d1 (gate 2's h is far below a code step)
    d0 = _ffn_delta(P * 638, P * 1, 1)
    d1 = _ffn_delta(P * 511, P * -1, -1)
    mag = f32_round(f32_round(Fraction(1, 2) + d0) + d1)  # the last token is token 1 (c = 0.5)
    assert all(F(hidden[k]) == int(S[k]) * mag for k in range(8))

    # final RMSNorm gives s again; the LM head's accumulators are 127 * the listed sums
    sums = [2, -127, 635, 0, -1, 8, -8, 126]
    for v in range(8):
        assert F(logits[v]) == _deq(P * sums[v], m.w_out_scale[v], A_SCALE), v


def test_micro_model_chunk_and_order_invariance():
    # the same hand-built model through chunk = 1 and a continuation call
    m = _model()
    toks = np.array([1, 2, 1], np.int32)
    om = oracle.OracleModel(m)
    ref = om.prefill(toks, 0, 3)
    om.kv_reset()
    a = om.prefill(toks, 0, 1)
    om.kv_reset()
    om.prefill(toks[:2], 0, 2)
    b = om.prefill(toks[2:], 2, 1)
    assert np.array_equal(ref.view(np.uint32), a.view(np.uint32))
    assert np.array_equal(ref.view(np.uint32), b.view(np.uint32))
