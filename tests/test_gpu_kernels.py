"""Parity of each CUDA step with the oracle, through the C ABI.

Integer work (quantised codes, int32 accumulators) and the fixed-order f32
epilogue are compared bit for bit; steps with transcendental functions
(RMSNorm, RoPE, softmax, SiLU) within f32 rounding of the oracle's double
evaluation.
"""
import numpy as np
import pytest

import oracle
import prompt_prefill_gb300 as pp
import synth
from tests.gpu_util import bits, dev, empty, host, swiglu_close, torch_cuda

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def torch():
    return torch_cuda()


def _quantize_gpu(torch, x):
    rows, k = x.shape
    q8 = empty((rows, k), torch.int8)
    q16 = empty((rows, k), torch.float16)
    s = empty((rows,), torch.float32)
    pp.pp_op_quantize(dev(x), rows, k, q8, q16, s)
    return host(q8), host(q16), host(s)


@pytest.mark.parametrize("rows,k", [(1, 4), (7, 256), (33, 4096), (5, 14336)])
def test_quantize_bit_exact(torch, rows, k):
    x = synth.normal_f32(21, k, (rows, k), 0.0, 1.3)
    if rows > 2:
        x[1] = 0.0  # degenerate zero row
        x[2, k // 2] = 55.0  # outlier
    q8, q16, s = _quantize_gpu(torch, x)
    rq, rs = oracle.quantize_rows(x)
    assert np.array_equal(q8, rq)
    assert np.array_equal(bits(s), bits(rs))
    assert np.array_equal(q16.astype(np.float32), rq.astype(np.float32))


def test_quantize_ties_hand_case(torch):
    y = np.array([[127.0, 2.5, 3.5, -2.5, 0.49999997, -126.5, 0.5, 1.5]], np.float32)
    q8, _, s = _quantize_gpu(torch, y)
    assert q8.tolist() == [[127, 2, 4, -2, 0, -126, 0, 2]] and s.tolist() == [1.0]


@pytest.mark.parametrize("k", [4096, 14336, 20000])  # codes kept in registers (two widths) and streamed
def test_quantize_every_tie_and_neighbour(torch, k):
    # amax = 127 makes inv = 1, so y * inv = y: every half-integer in [-127, 127] is a tie, and its float
    # neighbours on either side round away from it; the rest of the row is random
    ties = np.arange(-127, 127, dtype=np.float64) + 0.5
    vals = np.concatenate([ties, np.nextafter(ties.astype(np.float32), np.float32(np.inf)),
                           np.nextafter(ties.astype(np.float32), np.float32(-np.inf)), [127.0, -127.0, 0.0, -0.0]])
    x = synth.normal_f32(23, k, (3, k), 0.0, 40.0)
    x = np.clip(x, -127.0, 127.0).astype(np.float32)
    for r in range(3):
        x[r, r:r + vals.size] = vals
    q8, q16, s = _quantize_gpu(torch, x)
    rq, rs = oracle.quantize_rows(x)
    assert np.array_equal(q8, rq)
    assert np.array_equal(bits(s), bits(rs)) and s.tolist() == [1.0, 1.0, 1.0]
    assert np.array_equal(bits(q16), bits(rq.astype(np.float16)))  # +0 for every zero code


@pytest.mark.parametrize("k", [4096, 14336, 20000])
def test_quantize_tiny_and_non_finite_rows(torch, k):
    # rows outside the conversion-free form: amax below 127 / FLT_MAX (127 / amax overflows to inf, every
    # nonzero code saturates), an infinity (inv = 0) and a NaN (ignored by amax). The definition leaves the
    # code of a NaN product undefined, so those positions are not compared.
    rng = np.random.default_rng(24)
    x = synth.normal_f32(24, k, (4, k), 0.0, 1.0)
    x[0] = (rng.uniform(1e-38, 3e-37, k) * rng.choice([-1.0, 1.0], k)).astype(np.float32)
    x[0, 5] = 0.0
    x[1, 7] = np.inf
    x[2, k - 3] = np.nan
    x[3, 11] = -np.inf
    q8, q16, s = _quantize_gpu(torch, x)
    rq, rs = oracle.quantize_rows(x)
    defined = np.isfinite(x)
    assert np.array_equal(q8[defined], rq[defined])
    assert np.array_equal(q16[defined].astype(np.float32), rq[defined].astype(np.float32))
    assert np.array_equal(bits(s), bits(rs))
    assert set(np.unique(q8[0])) == {-127, 0, 127} and q8[0, 5] == 0
    assert np.isinf(s[1]) and np.isinf(s[3]) and np.isfinite(s[2])


@pytest.mark.parametrize("rows,k", [(3, 256), (17, 1024), (9, 4096)])
def test_rmsnorm_quantize(torch, rows, k):
    x = synth.normal_f32(22, k, (rows, k), 0.0, 3.0)
    g = synth.normal_f32(22, 1, (k,), 1.0, 0.02)
    y = empty((rows, k), torch.float32)
    q8 = empty((rows, k), torch.int8)
    s = empty((rows,), torch.float32)
    pp.pp_op_rmsnorm_quantize(dev(x), dev(g), rows, k, 1e-5, y, q8, None, s)
    y, q8, s = host(y), host(q8), host(s)
    ref = oracle.rmsnorm_rows(x, g, 1e-5)
    # f32 sum of squares: 16-term per-thread partials + an 8-level tree, ~1.5e-6 relative
    assert np.abs(y.astype(np.float64) - ref).max() <= 4e-6 * np.abs(ref).max()
    # the codes from the GPU's own normalised rows are the oracle's codes for them
    rq, rs = oracle.quantize_rows(y)
    assert np.array_equal(q8, rq) and np.array_equal(bits(s), bits(rs))


GEMM_SHAPES = [(1, 128, 64), (8, 768, 256), (37, 256, 768), (130, 160, 320), (200, 2048, 1024)]


@pytest.mark.parametrize("m,n,k", GEMM_SHAPES)
def test_gemm_acc_bit_exact(torch, m, n, k):
    a = synth.uniform_i8(31, m * 7 + k, (m, k))
    w = synth.uniform_i8(32, n * 3 + k, (n, k))
    acc = empty((m, n), torch.int32)
    pp.pp_op_gemm_acc(pp.PP_GEMM_MMA, dev(a), None, dev(w), m, n, k, acc)
    assert np.array_equal(host(acc), oracle.gemm_i8(a, w))


def test_gemm_acc_adversarial_extremes(torch):
    m, n, k = 64, 128, 14336
    a = np.full((m, k), 127, np.int8)
    a[1::2] = -127
    w = np.full((n, k), -127, np.int8)
    w[::3] = 127
    acc = empty((m, n), torch.int32)
    pp.pp_op_gemm_acc(pp.PP_GEMM_MMA, dev(a), None, dev(w), m, n, k, acc)
    got = host(acc)
    assert got[0, 0] == 127 * 127 * k and got[1, 0] == -127 * 127 * k and got[0, 1] == -127 * 127 * k
    assert np.array_equal(got, oracle.gemm_i8(a, w))


@pytest.mark.parametrize("epi", [pp.PP_EPI_STORE, pp.PP_EPI_RESID])
def test_gemm_epilogue_bit_exact(torch, epi):
    m, n, k = 45, 384, 512
    a = synth.uniform_i8(41, 1, (m, k))
    w = synth.uniform_i8(41, 2, (n, k))
    ws = synth.uniform_f32(41, 3, (n,), 1e-4, 2e-3)
    as_ = synth.uniform_f32(41, 4, (m,), 1e-3, 5e-2)
    x0 = synth.normal_f32(41, 5, (m, n), 0.0, 2.0)
    out = dev(x0) if epi == pp.PP_EPI_RESID else empty((m, n), torch.float32)
    pp.pp_op_gemm(pp.PP_GEMM_MMA, epi, dev(a), None, dev(w), dev(ws), dev(as_), m, n, k, out, n)
    got = host(out)
    ref = oracle.dequant_block(oracle.gemm_i8(a, w), ws, as_)
    if epi == pp.PP_EPI_RESID:
        ref = (x0 + ref).astype(np.float32)  # one IEEE f32 add per element
    assert np.array_equal(bits(got), bits(ref))


def test_gemm_swiglu(torch):
    m, F, k = 21, 96, 256
    a = synth.uniform_i8(42, 1, (m, k))
    wg = synth.uniform_i8(42, 2, (F, k))
    wu = synth.uniform_i8(42, 3, (F, k))
    sg = synth.uniform_f32(42, 4, (F,), 1e-4, 1e-3)
    su = synth.uniform_f32(42, 5, (F,), 1e-4, 1e-3)
    as_ = synth.uniform_f32(42, 6, (m,), 1e-2, 5e-2)
    # interleave rows in blocks of 16: gate 16, up 16, ...
    B = 16
    wgu = np.concatenate([np.concatenate([wg[b * B:(b + 1) * B], wu[b * B:(b + 1) * B]]) for b in range(F // B)])
    sgu = np.concatenate([np.concatenate([sg[b * B:(b + 1) * B], su[b * B:(b + 1) * B]]) for b in range(F // B)])
    out = empty((m, F), torch.float32)
    pp.pp_op_gemm(pp.PP_GEMM_MMA, pp.PP_EPI_SWIGLU, dev(a), None, dev(wgu), dev(sgu), dev(as_), m, 2 * F, k, out, F)
    got = host(out)
    g = oracle.dequant_block(oracle.gemm_i8(a, wg), sg, as_)
    u = oracle.dequant_block(oracle.gemm_i8(a, wu), su, as_)
    ref = np.vectorize(lambda x, y: float(oracle.silu_mul(x, y)), otypes=[np.float32])(g, u)
    # full-accuracy expf (<= 2 ulp) and IEEE add, division and multiply: within a few ulp of each value
    assert swiglu_close(got, ref)


@pytest.mark.parametrize("rows,start,H,Hkv,hd,theta", [(5, 0, 4, 4, 64, 1e4), (33, 17, 16, 8, 64, 1e4),
                                                        (9, 4000, 32, 8, 128, 5e5)])
def test_rope_kv(torch, rows, start, H, Hkv, hd, theta):
    max_pos = start + rows + 3
    table = empty((max_pos, hd // 2, 2), torch.float32)
    pp.pp_op_rope_table(max_pos, hd, theta, table)
    qkv = synth.normal_f32(51, rows, (rows, (H + 2 * Hkv) * hd), 0.0, 1.5)
    q = empty((rows, H, hd), torch.float32)
    kc = dev(np.full((max_pos, Hkv, hd), 7.0, np.float32))
    vc = dev(np.full((max_pos, Hkv, hd), 7.0, np.float32))
    pp.pp_op_rope_kv(dev(qkv), rows, start, H, Hkv, hd, table, q, kc, vc)
    q, kc, vc = host(q), host(kc), host(vc)
    ref_q = oracle.rope_rows(qkv[:, :H * hd].reshape(rows, H, hd), start, theta)
    ref_k = oracle.rope_rows(qkv[:, H * hd:(H + Hkv) * hd].reshape(rows, Hkv, hd), start, theta)
    scale = np.abs(qkv).max()
    assert np.abs(q - ref_q).max() <= 2e-6 * scale
    assert np.abs(kc[start:start + rows] - ref_k).max() <= 2e-6 * scale
    assert np.array_equal(vc[start:start + rows], qkv[:, (H + Hkv) * hd:].reshape(rows, Hkv, hd))
    assert np.all(kc[:start] == 7.0) and np.all(kc[start + rows:] == 7.0) and np.all(vc[:start] == 7.0)


# rows, start, H, Hkv, hd. Keys are reduced in ranges of 512 at fixed positions:
# the later cases cross range boundaries (1024, 2048) and merge 16 ranges.
ATTN_CASES = [(1, 0, 4, 4, 64), (8, 0, 4, 4, 64), (32, 5, 16, 8, 64), (37, 100, 32, 8, 64), (64, 250, 32, 8, 128),
              (3, 700, 32, 8, 128), (130, 0, 8, 8, 128), (40, 1000, 32, 8, 128), (64, 2040, 16, 8, 64),
              (16, 8000, 32, 8, 128)]


@pytest.mark.parametrize("rows,start,H,Hkv,hd", ATTN_CASES)
def test_attention_matches_oracle(torch, rows, start, H, Hkv, hd):
    n = start + rows
    q = synth.normal_f32(61, rows, (rows, H, hd), 0.0, 1.0)
    K = synth.normal_f32(62, n, (n + 5, Hkv, hd), 0.0, 1.0)
    V = synth.normal_f32(63, n, (n + 5, Hkv, hd), 0.0, 1.0)
    o = empty((rows, H, hd), torch.float32)
    pp.pp_op_attention(dev(q), dev(K), dev(V), rows, start, H, Hkv, hd, o)
    ref = oracle.attention(q, K, V, start)
    # f32 online softmax over up to ~800 keys vs the double oracle
    assert np.abs(host(o) - ref).max() <= 1e-5 * np.abs(V).max()


@pytest.mark.parametrize("rows,start", [(50, 37), (64, 480), (100, 1500)])
def test_attention_row_result_independent_of_chunk(torch, rows, start):
    # Each query's reduction order depends only on its absolute position:
    # one launch over the rows equals one launch per row, bit for bit, also
    # where the chunk straddles a key-range boundary (512, 1536) so that some
    # of its rows merge two ranges and the rest see one.
    H, Hkv, hd = 32, 8, 128
    n = start + rows
    q = synth.normal_f32(64, 1, (rows, H, hd), 0.0, 2.0)
    K = dev(synth.normal_f32(64, 2, (n, Hkv, hd), 0.0, 1.0))
    V = dev(synth.normal_f32(64, 3, (n, Hkv, hd), 0.0, 1.0))
    dq = dev(q)
    whole = empty((rows, H, hd), torch.float32)
    pp.pp_op_attention(dq, K, V, rows, start, H, Hkv, hd, whole)
    single = empty((rows, H, hd), torch.float32)
    for i in range(rows):
        pp.pp_op_attention(dq[i:i + 1], K, V, 1, start + i, H, Hkv, hd, single[i:i + 1])
    assert np.array_equal(bits(host(whole)), bits(host(single)))


@pytest.mark.parametrize("vocab,dim", [(1024, 256), (5000, 4096), (128257, 2048)])  # last: a ragged group of rows
def test_lm_head_bit_exact(torch, vocab, dim):
    x = synth.normal_f32(71, 1, (1, dim), 0.0, 1.0)
    q8, s = oracle.quantize_rows(x)
    w = synth.uniform_i8(71, 2, (vocab, dim))
    ws = synth.uniform_f32(71, 3, (vocab,), 1e-4, 1e-3)
    logits = empty((vocab,), torch.float32)
    pp.pp_op_lm_head(dev(q8), dev(s), dev(w), dev(ws), vocab, dim, logits)
    ref = oracle.dequant_block(oracle.gemm_i8(q8, w), ws, s)[0]
    assert np.array_equal(bits(host(logits)), bits(ref))


def test_op_argument_errors(torch):
    t = empty((64,), torch.float32)
    with pytest.raises(pp.PPError) as e:
        pp.pp_op_gemm_acc(pp.PP_GEMM_MMA, t, None, t, 4, 32, 60, t)  # k % 64 != 0
    assert e.value.status == pp.PP_ERR_ARG
    with pytest.raises(pp.PPError):
        pp.pp_op_attention(t, t, t, 1, 0, 3, 2, 64, t)  # H % Hkv != 0
