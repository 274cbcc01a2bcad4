"""Model-level pins of the oracle: invariants the pages state, a closed-form
micro-model, and the block wiring composed from the (separately pinned) steps."""
from fractions import Fraction

import numpy as np
import pytest

import oracle
import synth
from tests.exact import F, f32_round


def _bits(a):
    return np.ascontiguousarray(a).view(np.uint32)


# ----------------------------------------------------------------------------
# "Batched Prefill", section "Correctness": chunked output is identical to the
# per-token path; "Single-pass prefill": per-position results unchanged.
# ----------------------------------------------------------------------------


def test_chunk_invariance_bitwise(tiny_model):
    toks = synth.prompt(tiny_model.cfg)  # 32 tokens
    om = oracle.OracleModel(tiny_model)
    ref = om.prefill(toks, 0, 1)
    kv_ref = [om.kv(L, w) for L in range(4) for w in (0, 1)]
    for chunk in (3, 8, 32, 64):
        om.kv_reset()
        got = om.prefill(toks, 0, chunk)
        assert np.array_equal(_bits(got), _bits(ref)), chunk
        assert all(np.array_equal(a, om.kv(L, w)) for a, (L, w) in zip(kv_ref, [(L, w) for L in range(4) for w in (0, 1)]))


def test_forward_one_loop_equals_prefill(tiny_model):
    toks = synth.prompt(tiny_model.cfg, 13)
    om = oracle.OracleModel(tiny_model)
    for i, t in enumerate(toks):
        last = om.forward_one(int(t), i)
    om2 = oracle.OracleModel(tiny_model)
    assert np.array_equal(_bits(last), _bits(om2.prefill(toks, 0, 8)))


def test_continuation_equals_one_call(tiny_model):
    toks = synth.prompt(tiny_model.cfg, 29)
    om = oracle.OracleModel(tiny_model)
    whole = om.prefill(toks, 0, 8)
    om.kv_reset()
    om.prefill(toks[:11], 0, 8)
    cont = om.prefill(toks[11:], 11, 8)
    assert np.array_equal(_bits(whole), _bits(cont))


def test_causality_appended_tokens_do_not_change_history(tiny_model):
    a = synth.prompt(tiny_model.cfg, 17)
    b = synth.tokens(99, 9, tiny_model.cfg.vocab)
    om = oracle.OracleModel(tiny_model)
    la = om.prefill(a, 0, 8)
    kv_a = [om.kv(L, 0)[:17].copy() for L in range(4)] + [om.kv(L, 1)[:17].copy() for L in range(4)]
    om.kv_reset()
    om.prefill(np.concatenate([a, b]), 0, 8)
    kv_ab = [om.kv(L, 0)[:17] for L in range(4)] + [om.kv(L, 1)[:17] for L in range(4)]
    assert all(np.array_equal(x, y) for x, y in zip(kv_a, kv_ab))
    # dropping the appended tokens again gives back the same last-position logits
    om.kv_reset()
    assert np.array_equal(_bits(om.prefill(a, 0, 5)), _bits(la))


def test_argument_errors(tiny_model):
    om = oracle.OracleModel(tiny_model)
    assert om.prefill_rc(np.zeros(0, np.int32)) == oracle.ORC_ERR_ARG
    assert om.prefill_rc(np.array([1, 2], np.int32), 0, 0) == oracle.ORC_ERR_ARG
    assert om.prefill_rc(np.array([1, 2], np.int32), -1, 1) == oracle.ORC_ERR_ARG
    assert om.prefill_rc(np.array([1, 1024], np.int32), 0, 1) == oracle.ORC_ERR_ARG
    assert om.prefill_rc(np.array([1, -3], np.int32), 0, 1) == oracle.ORC_ERR_ARG
    assert om.prefill_rc(np.ones(65, np.int32), 0, 8) == oracle.ORC_ERR_CAPACITY
    assert om.prefill_rc(np.ones(2, np.int32), 63, 8) == oracle.ORC_ERR_CAPACITY
    assert om.prefill_rc(np.ones(64, np.int32), 0, 8) == oracle.ORC_OK  # exactly max_seq


# ----------------------------------------------------------------------------
# Micro-models built by hand.
# ----------------------------------------------------------------------------

MICRO = synth.ModelConfig("micro", dim=8, n_layers=1, n_heads=2, n_kv_heads=1, head_dim=4, ffn=16, vocab=16,
                          rms_eps=0.0, rope_theta=10000.0, max_seq=8)


def _micro(seed=3, zero=()):
    m = synth.make_model(MICRO, seed=seed)
    for i, k in enumerate(synth.LAYER_KINDS):
        if k in zero:
            m.w[i][:] = 0
    return m


def test_zero_layers_closed_form_logits():
    # All projection weights zero: every projection adds exactly 0, so the last
    # position leaves the stack as its own embedding row. That row is the
    # constant 0.5 and the final gain is 1 with eps = 0, so the final norm is
    # exactly 1.0 everywhere, every code is 127 and a_scale = fl(1/127).
    m = _micro(zero=synth.LAYER_KINDS)
    toks = np.array([3, 5, 9], np.int32)
    m.tok_emb[9, :] = 0.5
    m.final_norm[:] = 1.0
    n_ones = np.arange(16) % 9
    m.w_out[:] = 0
    for v in range(16):
        m.w_out[v, : n_ones[v]] = 1
    m.w_out_scale[:] = np.float32(1.0) / np.float32(127.0)
    logits, hidden = oracle.OracleModel(m).prefill(toks, 0, 2, want_hidden=True)
    assert np.array_equal(hidden, m.tok_emb[9])
    a_scale = f32_round(Fraction(1, 127))
    for v in range(16):
        acc = 127 * int(n_ones[v])
        exp = f32_round(f32_round(Fraction(acc) * F(m.w_out_scale[v])) * a_scale)
        assert F(logits[v]) == exp, v


def _compose_block(m, toks, attn=True, ffn=True):
    """One decoder block composed from the pinned steps, in the pages' order."""
    c = m.cfg
    W, S = m.w, m.w_scale
    x = m.tok_emb[toks].astype(np.float32)
    n = len(toks)
    if attn:
        y = oracle.rmsnorm_rows(x, m.attn_norm[0], c.rms_eps)
        q8, a = oracle.quantize_rows(y)
        Q = oracle.dequant_block(oracle.gemm_i8(q8, W[0]), S[0], a).reshape(n, c.n_heads, c.head_dim)
        K = oracle.dequant_block(oracle.gemm_i8(q8, W[1]), S[1], a).reshape(n, c.n_kv_heads, c.head_dim)
        V = oracle.dequant_block(oracle.gemm_i8(q8, W[2]), S[2], a).reshape(n, c.n_kv_heads, c.head_dim)
        Q = oracle.rope_rows(Q, 0, c.rope_theta)
        K = oracle.rope_rows(K, 0, c.rope_theta)
        o = oracle.attention(Q, K, V, 0).reshape(n, -1)
        q8, a = oracle.quantize_rows(o)
        x = x + oracle.dequant_block(oracle.gemm_i8(q8, W[3]), S[3], a)
    if ffn:
        y = oracle.rmsnorm_rows(x, m.ffn_norm[0], c.rms_eps)
        q8, a = oracle.quantize_rows(y)
        g = oracle.dequant_block(oracle.gemm_i8(q8, W[4]), S[4], a)
        u = oracle.dequant_block(oracle.gemm_i8(q8, W[5]), S[5], a)
        h = np.vectorize(lambda gg, uu: float(oracle.silu_mul(gg, uu)), otypes=[np.float32])(g, u)
        q8, a = oracle.quantize_rows(h)
        x = x + oracle.dequant_block(oracle.gemm_i8(q8, W[6]), S[6], a)
    return x


def test_attention_block_wiring():
    m = _micro(seed=4, zero=("wg", "wu", "wd"))
    toks = np.array([1, 7, 2, 2, 11], np.int32)
    _, hidden = oracle.OracleModel(m).prefill(toks, 0, 2, want_hidden=True)
    assert np.array_equal(hidden, _compose_block(m, toks, attn=True, ffn=False)[-1])


def test_ffn_block_wiring():
    m = _micro(seed=5, zero=("wq", "wk", "wv", "wo"))
    toks = np.array([4, 4, 15], np.int32)
    _, hidden = oracle.OracleModel(m).prefill(toks, 0, 3, want_hidden=True)
    assert np.array_equal(hidden, _compose_block(m, toks, attn=False, ffn=True)[-1])


def test_full_block_wiring():
    m = _micro(seed=6)
    toks = np.array([0, 3, 8, 12, 5, 6], np.int32)
    _, hidden = oracle.OracleModel(m).prefill(toks, 0, 4, want_hidden=True)
    assert np.array_equal(hidden, _compose_block(m, toks)[-1])


@pytest.mark.parametrize("zero", [("wq",), ("wk",), ("wv",), ("wo",), ("wg",), ("wu",), ("wd",)])
def test_every_matrix_reaches_the_output(zero):
    # Zeroing any single projection must change the last hidden state:
    # guards against a matrix that is loaded but never used.
    toks = np.array([0, 3, 8, 12, 5, 6], np.int32)
    _, h_full = oracle.OracleModel(_micro(seed=6)).prefill(toks, 0, 4, want_hidden=True)
    _, h_zero = oracle.OracleModel(_micro(seed=6, zero=zero)).prefill(toks, 0, 4, want_hidden=True)
    assert not np.array_equal(h_full, h_zero)


def test_layer_by_layer_composes_to_prefill(tiny_model):
    # the single-layer entry point, applied layer after layer from the
    # embedding rows, and the final projection reproduce the whole prefill
    toks = synth.prompt(tiny_model.cfg, 20)
    om = oracle.OracleModel(tiny_model)
    ref, hidden = om.prefill(toks, 0, 20, want_hidden=True)
    om.kv_reset()
    x = tiny_model.tok_emb[toks].astype(np.float32)
    for L in range(tiny_model.cfg.n_layers):
        x = om.layer(L, x, 0)
    assert np.array_equal(x[-1], hidden)
    assert np.array_equal(_bits(om.final_logits(x[-1])), _bits(ref))


def test_forced_layer_with_own_codes_is_the_layer():
    # Forcing the oracle's layer with the codes it decides itself (obtained by
    # composing the pinned steps) reports no disagreement and changes nothing.
    m = _micro(seed=7)
    toks = np.array([2, 9, 4, 4, 13, 1], np.int32)
    c = m.cfg
    n = len(toks)
    x = m.tok_emb[toks].astype(np.float32)
    W, S = m.w, m.w_scale
    kmax = max(c.dim, c.n_heads * c.head_dim, c.ffn)
    codes = np.zeros((4, n, kmax), np.int8)
    scales = np.zeros((4, n), np.float32)
    q8, a = oracle.quantize_rows(oracle.rmsnorm_rows(x, m.attn_norm[0], c.rms_eps))
    codes[0, :, :c.dim], scales[0] = q8, a
    Q = oracle.rope_rows(oracle.dequant_block(oracle.gemm_i8(q8, W[0]), S[0], a).reshape(n, c.n_heads, c.head_dim), 0,
                         c.rope_theta)
    K = oracle.rope_rows(oracle.dequant_block(oracle.gemm_i8(q8, W[1]), S[1], a).reshape(n, c.n_kv_heads, c.head_dim),
                         0, c.rope_theta)
    V = oracle.dequant_block(oracle.gemm_i8(q8, W[2]), S[2], a).reshape(n, c.n_kv_heads, c.head_dim)
    q8, a = oracle.quantize_rows(oracle.attention(Q, K, V, 0).reshape(n, -1))
    codes[1, :, :c.n_heads * c.head_dim], scales[1] = q8, a
    x1 = x + oracle.dequant_block(oracle.gemm_i8(q8, W[3]), S[3], a)
    q8, a = oracle.quantize_rows(oracle.rmsnorm_rows(x1, m.ffn_norm[0], c.rms_eps))
    codes[2, :, :c.dim], scales[2] = q8, a
    g = oracle.dequant_block(oracle.gemm_i8(q8, W[4]), S[4], a)
    u = oracle.dequant_block(oracle.gemm_i8(q8, W[5]), S[5], a)
    h = np.vectorize(lambda gg, uu: float(oracle.silu_mul(gg, uu)), otypes=[np.float32])(g, u)
    q8, a = oracle.quantize_rows(h)
    codes[3, :, :c.ffn], scales[3] = q8, a
    om = oracle.OracleModel(m)
    y, st = om.layer_forced(0, x, codes, scales, 0)
    om.kv_reset()
    assert st["mismatches"] == [0, 0, 0, 0] and st["scale_mismatches"] == [0, 0, 0, 0]
    assert np.array_equal(y, om.layer(0, x, 0))


def test_forced_layer_with_zero_codes_adds_nothing_and_counts_disagreements():
    m = _micro(seed=8)
    toks = np.array([5, 6, 7], np.int32)
    c = m.cfg
    x = m.tok_emb[toks].astype(np.float32)
    kmax = max(c.dim, c.n_heads * c.head_dim, c.ffn)
    y, st = oracle.OracleModel(m).layer_forced(0, x, np.zeros((4, 3, kmax), np.int8), np.zeros((4, 3), np.float32), 0)
    # zero codes make every projection add exactly zero
    assert np.array_equal(y, x)
    own, _ = oracle.quantize_rows(oracle.rmsnorm_rows(x, m.attn_norm[0], c.rms_eps))
    assert st["mismatches"][0] == int(np.count_nonzero(own))
    own2, _ = oracle.quantize_rows(oracle.rmsnorm_rows(x, m.ffn_norm[0], c.rms_eps))
    assert st["mismatches"][2] == int(np.count_nonzero(own2))
    assert st["mismatches"][1] == 0 and st["mismatches"][3] == 0  # zero inputs quantise to zero
